// The loss's small kernels: label check and valid-row count, gradient scale,
// per-row logsumexp combine, the fixed-order loss reduction, the label sort
// and exact one-hot part of grad_W, the grad_b accumulation, and the
// bounded-wait probe.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>

#include "lce_internal.cuh"
#include "lce_ptx.cuh"

namespace lce {

namespace {

constexpr float LN2_F = 0.6931471805599453f;
constexpr float LOG2E_F = 1.4426950408889634f;

// Labels must lie in [0, V) or equal ignore_index (cross_entropy's contract).
// Counts the valid rows; a bad label raises the status bit and is not counted.
// With `label_counts`, also counts each label's valid rows (integer
// atomics: the result does not depend on their order).
__global__ void prepass_kernel(const int64_t* __restrict__ y, int64_t N, int64_t V,
                               int64_t ignore_index, WsHeader* hdr, int* label_counts) {
    unsigned long long cnt = 0;
    bool bad = false;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < N;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t v = y[i];
        if (v == ignore_index) continue;
        if (v < 0 || v >= V) {
            bad = true;
        } else {
            ++cnt;
            if (label_counts) atomicAdd(label_counts + v, 1);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, o);
    __shared__ unsigned long long part[32];
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) part[w] = cnt;
    if (__any_sync(0xFFFFFFFFu, bad) && l == 0) atomicOr(&hdr->status, STATUS_LABEL);
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned long long s = 0;
        for (int k = 0; k < (blockDim.x + 31) / 32; ++k) s += part[k];
        atomicAdd(&hdr->n_valid, s);
    }
}

// s = grad_scale * grad_output / n_valid (0 without valid rows).
__global__ void scale_kernel(WsHeader* hdr, float grad_scale, const float* d_grad_output,
                             int64_t* n_valid_out, int sum_reduction) {
    const unsigned long long nv = hdr->n_valid;
    const double go = d_grad_output ? static_cast<double>(*d_grad_output) : 1.0;
    if (sum_reduction)
        hdr->scale = static_cast<float>(static_cast<double>(grad_scale) * go);
    else
        hdr->scale = nv ? static_cast<float>(static_cast<double>(grad_scale) * go / static_cast<double>(nv)) : 0.f;
    if (n_valid_out) *n_valid_out = static_cast<int64_t>(nv);
}

// lse_i = (M + log2(S + T)) ln 2, where (M, S) merges the per-half-tile
// partial (max, sum of 2^(t - max) over the non-target columns) pairs of row
// i and T = 2^(z_t log2 e - M) is the target's term (0 for an ignored row).
// The target entry's gradient coefficient is c_i = p - 1 = -S / (S + T),
// which has no cancellation however close p is to 1.  Each row's partial list is cut
// into 32 contiguous parts, each merged in order by one thread (S <- S
// 2^(M - M') + s_t 2^(m_t - M') when a larger max m_t = M' arrives, else
// S <- S + s_t 2^(m_t - M)).  The 32 part results are merged by a fixed
// tree: within a warp, parts 4w .. 4w+3 as (0+1) + (2+3) by shuffles; then
// the block's 8 warp results pairwise, ((0+1) + (2+3)) + ((4+5) + (6+7)),
// through shared memory.  The tree depends only on the partial count, so lse
// does not depend on the chunk size.  A block holds 8 rows: the 8 lanes of a
// part read 8 consecutive rows of a partial, one 32-byte sector.  Row loss =
// lse_i - z[i, y_i] for valid rows, 0 for ignored rows, NaN for a label
// outside [0, V).  Without pm (the recompute path) every partial is a plain
// sum of the row's non-target P (max 0: the merge adds them exactly as
// sums), and only c_i = -S is written.
__device__ __forceinline__ void merge_partial(float& M, float& S, float m, float s) {
    if (m > M) {
        S = S * exp2f(M - m) + s;
        M = m;
    } else if (m > -INFINITY) {
        S += s * exp2f(m - M);
    }
}

__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ pm, const float* __restrict__ ps,
                                                      int64_t n_pt, int64_t ldp, int64_t rows,
                                                      const float* __restrict__ zt, const int64_t* __restrict__ y,
                                                      int64_t ignore_index, int64_t V, float* __restrict__ lse,
                                                      float* __restrict__ row_loss, float* __restrict__ tcoef,
                                                      unsigned* status) {
    __shared__ float wm[8][8], wsum[8][8];  // [warp][row of the block]
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int part = warp * 4 + (lane >> 3);
    const int64_t r = static_cast<int64_t>(blockIdx.x) * 8 + (lane & 7);
    const bool ok = r < rows;
    const int64_t per = (n_pt + 31) / 32;
    const int64_t t0 = part * per < n_pt ? part * per : n_pt, t1 = t0 + per < n_pt ? t0 + per : n_pt;
    float M = -INFINITY, S = 0.f;
    if (ok && LCE_IN(r < ldp && t1 <= n_pt, status)) {
        int64_t t = t0;
        for (; t + 8 <= t1; t += 8) {
            float m8[8], s8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                m8[k] = pm ? pm[(t + k) * ldp + r] : 0.f;
                s8[k] = ps[(t + k) * ldp + r];
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) merge_partial(M, S, m8[k], s8[k]);
        }
        for (; t < t1; ++t) merge_partial(M, S, pm ? pm[t * ldp + r] : 0.f, ps[t * ldp + r]);
    }
#pragma unroll
    for (int o = 8; o <= 16; o <<= 1) {
        const float M2 = __shfl_xor_sync(0xFFFFFFFFu, M, o);
        const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, o);
        const bool lower = (lane & o) == 0;  // both partners merge (lower, upper)
        float Ma = lower ? M : M2, Sa = lower ? S : S2;
        merge_partial(Ma, Sa, lower ? M2 : M, lower ? S2 : S);
        M = Ma;
        S = Sa;
    }
    if (lane < 8) {
        wm[warp][lane] = M;
        wsum[warp][lane] = S;
    }
    __syncthreads();
    if (warp != 0 || lane >= 8 || !ok) return;
    float m[8], sv[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        m[w] = wm[w][lane];
        sv[w] = wsum[w][lane];
    }
#pragma unroll
    for (int step = 1; step < 8; step <<= 1)
#pragma unroll
        for (int w = 0; w < 8; w += 2 * step) merge_partial(m[w], sv[w], m[w + step], sv[w + step]);
    const int64_t yv = y[r];
    const bool valid = yv != ignore_index && yv >= 0 && yv < V;
    if (!pm) {
        if (tcoef) tcoef[r] = valid ? -sv[0] : 0.f;
        return;
    }
    const float T = valid ? exp2f(zt[r] * LOG2E_F - m[0]) : 0.f;
    const float St = sv[0] + T;
    const float l = (m[0] + log2f(St)) * LN2_F;
    lse[r] = l;
    if (row_loss) row_loss[r] = valid ? l - zt[r] : (yv == ignore_index ? 0.f : __int_as_float(0x7FC00000));
    if (tcoef) tcoef[r] = valid ? -sv[0] / St : 0.f;
}

__global__ void __launch_bounds__(256) p_rescale_kernel(uint16_t* __restrict__ P, int64_t ldg, int64_t rows,
                                                        int64_t V, const float* __restrict__ pm, int64_t ldp,
                                                        const float* __restrict__ lse,
                                                        const int* __restrict__ crow,
                                                        const int* __restrict__ n_valid,
                                                        float* __restrict__ gb_part, unsigned* status) {
    __shared__ float colsum[8][256 + 4];
    constexpr float LOG2E = 1.4426950408889634f;
    const int cg = threadIdx.x & 31, rr = threadIdx.x >> 5;
    const int64_t tile = blockIdx.y;
    const int64_t row0 = static_cast<int64_t>(blockIdx.x) * 32;
    const int64_t c = tile * 256 + cg * 8;
    const int64_t cend = (tile * 256 + 256 < ldg) ? tile * 256 + 256 : ldg;
    const bool col_ok = c < cend;
    const int64_t nv = *n_valid;
    const int64_t zero_end = (nv + 63) / 64 * 64;
    float sum[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) sum[k] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int64_t j = row0 + rr + 8 * q;  // compact row
        if (j >= rows || !col_ok) continue;
        uint4* ptr = reinterpret_cast<uint4*>(P + j * ldg + c);
        if (j >= nv) {
            if (j < zero_end) *ptr = make_uint4(0u, 0u, 0u, 0u);
            continue;
        }
        const int64_t r = crow[j];  // chunk row
        if (!LCE_IN(r >= 0 && r < ldp, status)) continue;
        // the forward kept one max per 128-column half tile
        const float f = exp2f(pm[(2 * tile + (cg >> 4)) * ldp + r] - lse[r] * LOG2E);
        const uint4 w = *ptr;
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = *reinterpret_cast<const __half2*>(&u[k]);
            const float2 e = __half22float2(h);
            const float p0 = e.x * f, p1 = e.y * f;
            sum[2 * k] += p0;
            sum[2 * k + 1] += p1;
            __half2 out = __floats2half2_rn(p0, p1);
            o[k] = *reinterpret_cast<uint32_t*>(&out);
        }
        *ptr = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (!gb_part) return;
#pragma unroll
    for (int k = 0; k < 8; ++k) colsum[rr][cg * 8 + k] = sum[k];
    __syncthreads();
    const int64_t v = tile * 256 + threadIdx.x;
    if (v < V) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) t += colsum[k][threadIdx.x];
        gb_part[blockIdx.x * V + v] = t * (1.f / static_cast<float>(1 << P_SCALE_EXP));
    }
}

// Valid-row compaction of every chunk: dmap[row] = the row's position among
// its chunk's valid rows (-1 for an ignored or out-of-range label), crow[chunk
// start + position] = the row (relative to the chunk), n_valid[chunk] = count.
// One block per chunk scans its rows in order, 1024 at a time.
__global__ void __launch_bounds__(1024) compact_rows_kernel(const int64_t* __restrict__ y, int64_t N, int64_t C,
                                                            int64_t V, int64_t ignore_index, int* __restrict__ dmap,
                                                            int* __restrict__ crow, int* __restrict__ n_valid) {
    __shared__ int warp_total[32];
    __shared__ int running;
    const int64_t c = blockIdx.x;
    const int64_t r0 = c * C;
    const int64_t rows = (N - r0) < C ? (N - r0) : C;
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (threadIdx.x == 0) running = 0;
    __syncthreads();
    for (int64_t base = 0; base < rows; base += blockDim.x) {
        const int64_t i = base + threadIdx.x;
        bool valid = false;
        if (i < rows) {
            const int64_t v = y[r0 + i];
            valid = v != ignore_index && v >= 0 && v < V;
        }
        const unsigned ballot = __ballot_sync(0xFFFFFFFFu, valid);
        const int before_in_warp = __popc(ballot & ((1u << lane) - 1u));
        if (lane == 0) warp_total[w] = __popc(ballot);
        __syncthreads();
        int before_warp = 0;
        for (int k = 0; k < w; ++k) before_warp += warp_total[k];
        const int d = running + before_warp + before_in_warp;
        if (i < rows) {
            dmap[r0 + i] = valid ? d : -1;
            if (valid) crow[r0 + d] = static_cast<int>(i);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            int t = 0;
            for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) t += warp_total[k];
            running += t;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) n_valid[c] = running;
}

// grad_X rows of ignored rows are zero (the compacted products never write them).
__global__ void zero_ignored_rows_kernel(const int* __restrict__ dmap, int64_t N, int64_t H,
                                         uint16_t* __restrict__ grad_X) {
    for (int64_t r = blockIdx.x; r < N; r += gridDim.x) {
        if (dmap[r] >= 0) continue;
        uint4* row = reinterpret_cast<uint4*>(grad_X + r * H);
        for (int64_t k = threadIdx.x; k < H / 8; k += blockDim.x) row[k] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// X16[j] = fp16(X[crow[j]] 2^k) for the chunk's valid rows in compacted order
// (k from max |X|), zero rows from n_valid to the next multiple of 64; with
// P_tail, the same tail rows of P are zeroed too.
__global__ void gather_f16_kernel(const uint16_t* __restrict__ X_chunk, int64_t H, const int* __restrict__ crow,
                                  const int* __restrict__ n_valid, int64_t max_rows, const unsigned* amax_bits,
                                  uint16_t* __restrict__ X16, uint16_t* __restrict__ P_tail, int64_t ldg,
                                  unsigned* status) {
    const float f = ldexpf(1.f, operand_scale_exp(*amax_bits));
    const int64_t nv = *n_valid;
    int64_t end = (nv + 63) / 64 * 64;
    if (end > max_rows) end = max_rows;
    const int64_t h8 = H / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < end * h8; e += stride) {
        const int64_t j = e / h8, k = e - j * h8;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (j < nv && LCE_IN(crow[j] >= 0 && crow[j] < max_rows, status)) {
            const uint4 w = reinterpret_cast<const uint4*>(X_chunk + static_cast<int64_t>(crow[j]) * H)[k];
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
            uint32_t r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                __half2 hh = __floats2half2_rn(__uint_as_float(u[q] << 16) * f, __uint_as_float(u[q] & 0xFFFF0000u) * f);
                r[q] = *reinterpret_cast<uint32_t*>(&hh);
            }
            o = make_uint4(r[0], r[1], r[2], r[3]);
        }
        reinterpret_cast<uint4*>(X16 + j * H)[k] = o;
    }
    if (P_tail) {
        const int64_t g8 = ldg / 8;
        for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < (end - nv) * g8;
             e += stride) {
            const int64_t j = nv + e / g8, k = e % g8;
            reinterpret_cast<uint4*>(P_tail + j * ldg)[k] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

// loss = sum of row losses / n_valid.  One block; the summation order
// depends on N only, so the result does not depend on the chunk size.  A
// device error raised earlier in the call (a bad label, a timed-out wait)
// makes the loss NaN, so the error also shows in the output itself.
__global__ void loss_kernel(const float* __restrict__ row_loss, int64_t N, const WsHeader* hdr,
                            float* loss, int64_t* n_valid_out, int sum_reduction) {
    __shared__ double red[1024];
    double acc = 0.0;
    for (int64_t i = threadIdx.x; i < N; i += blockDim.x) acc += static_cast<double>(row_loss[i]);
    red[threadIdx.x] = acc;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if (threadIdx.x < s) red[threadIdx.x] += red[threadIdx.x + s];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        const unsigned long long nv = hdr->n_valid;
        if (hdr->status != 0)
            *loss = __int_as_float(0x7FC00000);
        else if (sum_reduction)
            *loss = static_cast<float>(red[0]);
        else
            *loss = nv ? static_cast<float>(red[0] / static_cast<double>(nv)) : 0.f;
        if (n_valid_out) *n_valid_out = static_cast<int64_t>(nv);
    }
}

// grad_b_acc (+)= s * sum over the chunk's partial column sums of P (fixed
// order; P has no target entries); on the last chunk the target entries'
// part, s * (sum of c_i over the rows with label v, summed by the scatter
// kernels in a fixed order), is added and grad_b = bf16(grad_b_acc).
__global__ void grad_b_kernel(const float* __restrict__ gb_part, int64_t parts, int64_t V,
                              const WsHeader* hdr, const float* __restrict__ label_csum, float* grad_b_acc,
                              uint16_t* grad_b, int first, int last) {
    const int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    if (v >= V) return;
    float t = 0.f;
    for (int64_t p = 0; p < parts; ++p) t += gb_part[p * V + v];
    const float s = hdr->scale;
    float a = first ? s * t : fmaf(s, t, grad_b_acc[v]);
    if (last) a = fmaf(s, label_csum[v], a);
    grad_b_acc[v] = a;
    if (last && grad_b) {
        __nv_bfloat16 h = __float2bfloat16_rn(a);
        grad_b[v] = *reinterpret_cast<uint16_t*>(&h);
    }
}

// Sorts one block of up to LABEL_BLOCK rows of a chunk by (label, row) with
// a bitonic network in shared memory.  Ignored rows and out-of-range labels
// get the largest key and end up last.  Key = label << 32 | row-in-chunk,
// so rows of one label stay in row order.
// It also lists the block's runs of equal labels, as (start | end << 32)
// positions in the sorted order, in no particular order, and their count.
__global__ void __launch_bounds__(1024) label_sort_kernel(const int64_t* __restrict__ y, int64_t N, int64_t C,
                                                          int64_t blocks_per_chunk, int64_t V,
                                                          int64_t ignore_index,
                                                          unsigned long long* __restrict__ keys_out,
                                                          unsigned long long* __restrict__ runs_out,
                                                          int* __restrict__ run_count) {
    __shared__ int nrun;
    extern __shared__ unsigned long long sk[];
    const int64_t b = blockIdx.x;
    const int64_t chunk_start = (b / blocks_per_chunk) * C;
    const int64_t chunk_end = chunk_start + C < N ? chunk_start + C : N;
    const int64_t start = chunk_start + (b % blocks_per_chunk) * LABEL_BLOCK;
    const int64_t left = chunk_end - start;
    const int count = left <= 0 ? 0 : (left < LABEL_BLOCK ? static_cast<int>(left) : LABEL_BLOCK);
    for (int i = threadIdx.x; i < LABEL_BLOCK; i += blockDim.x) {
        unsigned long long key = ~0ull;
        if (i < count) {
            const int64_t v = y[start + i];
            if (v != ignore_index && v >= 0 && v < V)
                key = (static_cast<unsigned long long>(v) << 32) |
                      static_cast<unsigned long long>(start + i - chunk_start);
        }
        sk[i] = key;
    }
    __syncthreads();
    for (int size = 2; size <= LABEL_BLOCK; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < LABEL_BLOCK / 2; i += blockDim.x) {
                const int lo = 2 * i - (i & (stride - 1));
                const int hi = lo + stride;
                const bool ascending = (lo & size) == 0;
                const unsigned long long x0 = sk[lo], x1 = sk[hi];
                if ((x0 > x1) == ascending) {
                    sk[lo] = x1;
                    sk[hi] = x0;
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < LABEL_BLOCK; i += blockDim.x) keys_out[b * LABEL_BLOCK + i] = sk[i];
    if (threadIdx.x == 0) nrun = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < LABEL_BLOCK; i += blockDim.x) {
        const unsigned long long k = sk[i];
        if (k == ~0ull) continue;
        const unsigned long long v = k >> 32;
        if (i > 0 && (sk[i - 1] >> 32) == v) continue;
        int lo = i + 1, hi = LABEL_BLOCK;  // first position past the run (invalid keys never match v)
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if ((sk[mid] >> 32) == v)
                lo = mid + 1;
            else
                hi = mid;
        }
        const int slot = atomicAdd(&nrun, 1);
        runs_out[b * LABEL_BLOCK + slot] =
            static_cast<unsigned long long>(i) | (static_cast<unsigned long long>(lo) << 32);
    }
    __syncthreads();
    if (threadIdx.x == 0) run_count[b] = nrun;
}


// The target entries' part of grad_W for one sorted block of a chunk:
//   grad_W_acc[v, :] += s * sum over the block's rows i with y_i = v of c_i X[i, :]
// (c_i = p_{i,y_i} - 1, the entry the tensor-core products leave out).
// Work items are (run of equal labels, 512-column slab).  Within an item,
// 64 threads own 8 columns each and four row groups take every fourth row
// of the run in row order; the four partial sums are added in a fixed
// order, so the result is the same on every call.  Runs have distinct
// labels, so no two items touch the same grad_W elements.  With write_bf16
// the updated elements' bf16 cast is rewritten too.  With label_csum, the
// first slab's item also adds the run's sum of c_i to label_csum[v] (lanes
// of warp 0 take every 32nd row, then a fixed shuffle tree), for grad_b.
__device__ __forceinline__ void fma_bf16x8(float (&sum)[8], float c, const uint4 w) {
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        sum[2 * k] = fmaf(c, __uint_as_float(q[k] << 16), sum[2 * k]);
        sum[2 * k + 1] = fmaf(c, __uint_as_float(q[k] & 0xFFFF0000u), sum[2 * k + 1]);
    }
}

__global__ void __launch_bounds__(256) onehot_scatter_kernel(const unsigned long long* __restrict__ keys,
                                                             const unsigned long long* __restrict__ runs,
                                                             const int* __restrict__ run_count,
                                                             const uint16_t* __restrict__ X_chunk,
                                                             const float* __restrict__ tcoef, int64_t H, int64_t rows,
                                                             int64_t V, WsHeader* hdr, float* grad_W_acc,
                                                             uint16_t* grad_W, float* label_csum, int write_bf16) {
    __shared__ float part[3][64][9];
    const int ct = threadIdx.x & 63, rg = threadIdx.x >> 6;
    const int slabs = static_cast<int>((H + 511) / 512);
    const int items = *run_count * slabs;
    const float s = hdr->scale;
    for (int item = blockIdx.x; item < items; item += gridDim.x) {
        const unsigned long long run = runs[item / slabs];
        int64_t start = static_cast<int64_t>(run & 0xFFFFFFFFull), end = static_cast<int64_t>(run >> 32);
        if (!LCE_IN(start < end && end <= LABEL_BLOCK && item / slabs < LABEL_BLOCK, &hdr->status)) start = end = 0;
        const unsigned long long v = end > start ? keys[start] >> 32 : 0;
        const int64_t h = static_cast<int64_t>(item % slabs) * 512 + ct * 8;
        const bool active = h < H && end > start && LCE_IN(v < static_cast<unsigned long long>(V), &hdr->status);
        float sum[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = 0.f;
        if (active) {
            int64_t j = start + rg;
            for (; j + 12 < end; j += 16) {  // four rows of this group in flight
                uint4 w[4];
                float c[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    int64_t row = static_cast<int64_t>(keys[j + 4 * u] & 0xFFFFFFFFull);
                    if (!LCE_IN(row < rows, &hdr->status)) row = 0;
                    w[u] = *reinterpret_cast<const uint4*>(X_chunk + row * H + h);
                    c[u] = tcoef[row];
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) fma_bf16x8(sum, c[u], w[u]);
            }
            for (; j < end; j += 4) {
                int64_t row = static_cast<int64_t>(keys[j] & 0xFFFFFFFFull);
                if (!LCE_IN(row < rows, &hdr->status)) row = 0;
                fma_bf16x8(sum, tcoef[row], *reinterpret_cast<const uint4*>(X_chunk + row * H + h));
            }
        }
        if (rg > 0) {
#pragma unroll
            for (int k = 0; k < 8; ++k) part[rg - 1][ct][k] = sum[k];
        }
        __syncthreads();
        if (rg == 0 && active) {
#pragma unroll
            for (int k = 0; k < 8; ++k) sum[k] = ((sum[k] + part[0][ct][k]) + part[1][ct][k]) + part[2][ct][k];
            float* acc = grad_W_acc + static_cast<int64_t>(v) * H + h;
            float4 a0 = *reinterpret_cast<float4*>(acc);
            float4 a1 = *reinterpret_cast<float4*>(acc + 4);
            a0.x = fmaf(s, sum[0], a0.x);
            a0.y = fmaf(s, sum[1], a0.y);
            a0.z = fmaf(s, sum[2], a0.z);
            a0.w = fmaf(s, sum[3], a0.w);
            a1.x = fmaf(s, sum[4], a1.x);
            a1.y = fmaf(s, sum[5], a1.y);
            a1.z = fmaf(s, sum[6], a1.z);
            a1.w = fmaf(s, sum[7], a1.w);
            *reinterpret_cast<float4*>(acc) = a0;
            *reinterpret_cast<float4*>(acc + 4) = a1;
            if (write_bf16) {
                __nv_bfloat162 b0 = __floats2bfloat162_rn(a0.x, a0.y), b1 = __floats2bfloat162_rn(a0.z, a0.w);
                __nv_bfloat162 b2 = __floats2bfloat162_rn(a1.x, a1.y), b3 = __floats2bfloat162_rn(a1.z, a1.w);
                uint4 o;
                o.x = *reinterpret_cast<uint32_t*>(&b0);
                o.y = *reinterpret_cast<uint32_t*>(&b1);
                o.z = *reinterpret_cast<uint32_t*>(&b2);
                o.w = *reinterpret_cast<uint32_t*>(&b3);
                *reinterpret_cast<uint4*>(grad_W + static_cast<int64_t>(v) * H + h) = o;
            }
        }
        if (label_csum && item % slabs == 0 && threadIdx.x < 32) {
            float c = 0.f;
            for (int64_t jj = start + threadIdx.x; jj < end; jj += 32) {
                const int64_t row = static_cast<int64_t>(keys[jj] & 0xFFFFFFFFull);
                if (LCE_IN(row < rows, &hdr->status)) c += tcoef[row];
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
            if (threadIdx.x == 0 && end > start && LCE_IN(v < static_cast<unsigned long long>(V), &hdr->status))
                label_csum[v] += c;
        }
        __syncthreads();
    }
}

// The backward of the saved-gradient design: g = *d_grad_output;
// grad_X <- bf16(g grad_X) in place, grad_W <- bf16(g grad_W_acc),
// grad_b <- bf16(g grad_b_acc) (the fp32 accumulators are left as they are).
__global__ void scale_grads_kernel(int64_t nx8, int64_t nw8, int64_t V, const float* d_grad_output,
                                   uint4* __restrict__ grad_X, const float4* __restrict__ grad_W_acc,
                                   uint4* __restrict__ grad_W, const float* __restrict__ grad_b_acc,
                                   uint16_t* __restrict__ grad_b) {
    const float g = *d_grad_output;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    const int64_t t0 = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
    for (int64_t i = t0; i < nx8; i += stride) {
        const uint4 w = grad_X[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(g * __uint_as_float(u[k] << 16),
                                                     g * __uint_as_float(u[k] & 0xFFFF0000u));
            o[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        grad_X[i] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    if (grad_W)
        for (int64_t i = t0; i < nw8; i += stride) {
            const float4 a = grad_W_acc[2 * i], b = grad_W_acc[2 * i + 1];
            __nv_bfloat162 h0 = __floats2bfloat162_rn(g * a.x, g * a.y), h1 = __floats2bfloat162_rn(g * a.z, g * a.w);
            __nv_bfloat162 h2 = __floats2bfloat162_rn(g * b.x, g * b.y), h3 = __floats2bfloat162_rn(g * b.z, g * b.w);
            grad_W[i] = make_uint4(*reinterpret_cast<uint32_t*>(&h0), *reinterpret_cast<uint32_t*>(&h1),
                                   *reinterpret_cast<uint32_t*>(&h2), *reinterpret_cast<uint32_t*>(&h3));
        }
    if (grad_b)
        for (int64_t v = t0; v < V; v += stride) {
            __nv_bfloat16 h = __float2bfloat16_rn(g * grad_b_acc[v]);
            grad_b[v] = *reinterpret_cast<uint16_t*>(&h);
        }
}

// grad_X[crow[j], h .. h+8] = s (f' sum + c W[y, h]) as bf16 from a compacted
// row's summed K slices (f = s 2^-(15+k_W)): the arithmetic of the unsplit
// epilogue.
__device__ __forceinline__ void gradx_finish8(const float (&sum)[8], int64_t j, int64_t h, int64_t H, float s,
                                              float f, const int* __restrict__ crow, const int64_t* __restrict__ y,
                                              int64_t ignore_index, int64_t V, const uint16_t* __restrict__ W,
                                              const float* __restrict__ tcoef, const WsHeader* hdr,
                                              uint16_t* __restrict__ grad_X_chunk, int64_t max_rows) {
    const int64_t r = crow[j];
    if (!LCE_IN(r >= 0 && r < max_rows, const_cast<unsigned*>(&hdr->status))) return;
    const int64_t yr = y[r];
    float w[8];
    const bool valid = yr != ignore_index && yr >= 0 && yr < V;
    const float sc = valid ? s * tcoef[r] : 0.f;
    if (valid) {
        const uint4 q = *reinterpret_cast<const uint4*>(W + yr * H + h);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            w[2 * k] = __uint_as_float(u[k] << 16);
            w[2 * k + 1] = __uint_as_float(u[k] & 0xFFFF0000u);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = 0.f;
    }
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b2 = __floats2bfloat162_rn(fmaf(f, sum[2 * k], sc * w[2 * k]),
                                                  fmaf(f, sum[2 * k + 1], sc * w[2 * k + 1]));
        o[k] = *reinterpret_cast<uint32_t*>(&b2);
    }
    *reinterpret_cast<uint4*>(grad_X_chunk + r * H + h) = make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ void add8(float (&sum)[8], const float* src) {
    const float4 a = *reinterpret_cast<const float4*>(src);
    const float4 b = *reinterpret_cast<const float4*>(src + 4);
    sum[0] += a.x; sum[1] += a.y; sum[2] += a.z; sum[3] += a.w;
    sum[4] += b.x; sum[5] += b.y; sum[6] += b.z; sum[7] += b.w;
}

// Finishes a split grad_X product: for each compacted row j < n_valid and
// column h, sum the K slices' partial sums in slice order, then finish as
// the unsplit epilogue does.
__global__ void gradx_split_reduce_kernel(const float* __restrict__ split_out, int64_t splits, int64_t split_stride,
                                          int64_t H, const int* __restrict__ crow, const int* __restrict__ n_valid,
                                          const int64_t* __restrict__ y, int64_t ignore_index, int64_t V,
                                          const uint16_t* __restrict__ W, const float* __restrict__ tcoef,
                                          const WsHeader* hdr, uint16_t* __restrict__ grad_X_chunk,
                                          int64_t max_rows) {
    const float s = hdr->scale;
    const float f = ldexpf(s, -(P_SCALE_EXP + operand_scale_exp(hdr->amax_w_bits)));
    const int64_t nv = *n_valid, h8 = H / 8;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < nv * h8; e += stride) {
        const int64_t j = e / h8, h = (e - j * h8) * 8;
        float sum[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = 0.f;
        for (int64_t ks = 0; ks < splits; ++ks) add8(sum, split_out + ks * split_stride + j * H + h);
        gradx_finish8(sum, j, h, H, s, f, crow, y, ignore_index, V, W, tcoef, hdr, grad_X_chunk, max_rows);
    }
}

// Finishes the split tail tiles of a grad_X launch of the pair form: the
// plan is recomputed from the chunk's valid rows as the GEMM computed it;
// for each tail tile's valid row and column, the slices' partial tiles are
// summed in slice order, then finished as the unsplit epilogue does.  One
// thread per 8 columns of a row, consecutive threads along the row.  nw: the
// tiles' width in 256-column pieces (1 or 2).
__global__ void gradx_tail_reduce_kernel(const float* __restrict__ tail_out, int slots, int n_tiles, int k_blocks,
                                         int nw, int64_t H, const int* __restrict__ crow,
                                         const int* __restrict__ n_valid, const int64_t* __restrict__ y,
                                         int64_t ignore_index, int64_t V, const uint16_t* __restrict__ W,
                                         const float* __restrict__ tcoef, const WsHeader* hdr,
                                         uint16_t* __restrict__ grad_X_chunk, int64_t max_rows) {
    const int64_t nv = *n_valid;
    const int max_units = TAIL_UNITS_MAX / nw;
    const TailPlan tp =
        gradx_tail_plan(static_cast<int>((nv + 2 * BM - 1) / (2 * BM)) * n_tiles, slots, k_blocks, max_units);
    if (tp.tail == 0) return;
    if (!LCE_IN(tp.tail * tp.s <= max_units, const_cast<unsigned*>(&hdr->status))) return;
    const float s = hdr->scale;
    const float f = ldexpf(s, -(P_SCALE_EXP + operand_scale_exp(hdr->amax_w_bits)));
    const int tw = BN * nw;         // tile width
    const int G = tw / 8;           // 8-column groups per tile row
    const int64_t tile_floats = TAIL_TILE_FLOATS * nw;
    const int64_t total = static_cast<int64_t>(tp.tail) * (2 * BM) * G;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t e = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; e < total; e += stride) {
        const int i = static_cast<int>(e / ((2 * BM) * G));
        const int rem = static_cast<int>(e - static_cast<int64_t>(i) * (2 * BM) * G);
        const int tr = rem / G, g = rem - tr * G;
        const int t = tp.full + i;  // tile order n fastest: tile t is (t / n_tiles, t % n_tiles)
        const int64_t j = static_cast<int64_t>(t / n_tiles) * (2 * BM) + tr;
        const int64_t h = static_cast<int64_t>(t % n_tiles) * tw + 8 * g;
        if (j >= nv || h >= H) continue;
        float sum[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = 0.f;
        for (int ks = 0; ks < tp.s; ++ks)
            add8(sum, tail_out + (static_cast<int64_t>(ks) * tp.tail + i) * tile_floats + static_cast<int64_t>(tr) * tw +
                          8 * g);
        gradx_finish8(sum, j, h, H, s, f, crow, y, ignore_index, V, W, tcoef, hdr, grad_X_chunk, max_rows);
    }
}

// max |x| over bf16 values, as float bits (non-negative floats order like
// their bit patterns, so an integer max is exact and order-independent).
__global__ void amax_kernel(const uint16_t* __restrict__ x, int64_t n, unsigned* amax_bits) {
    unsigned m = 0;
    const int64_t n8 = n / 8;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 w = x8[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            m = max(m, (u[k] & 0x7FFFu) << 16);
            m = max(m, (u[k] >> 16 & 0x7FFFu) << 16);
        }
    }
    for (int64_t i = n8 * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        m = max(m, static_cast<unsigned>(x[i] & 0x7FFFu) << 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    if ((threadIdx.x & 31) == 0) atomicMax(amax_bits, m);
}

// out = fp16(x * 2^k), k = operand_scale_exp(max |x|), round to nearest even.
__global__ void to_f16_scaled_kernel(const uint16_t* __restrict__ x, int64_t n, const unsigned* amax_bits,
                                     uint16_t* __restrict__ out) {
    const float f = ldexpf(1.f, operand_scale_exp(*amax_bits));
    const int64_t n8 = n / 8;
    const uint4* x8 = reinterpret_cast<const uint4*>(x);
    uint4* o8 = reinterpret_cast<uint4*>(out);
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint4 w = x8[i];
        const uint32_t u[4] = {w.x, w.y, w.z, w.w};
        uint32_t r[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __half2 h = __floats2half2_rn(__uint_as_float(u[k] << 16) * f, __uint_as_float(u[k] & 0xFFFF0000u) * f);
            r[k] = *reinterpret_cast<uint32_t*>(&h);
        }
        o8[i] = make_uint4(r[0], r[1], r[2], r[3]);
    }
    for (int64_t i = n8 * 8 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        __half h = __float2half_rn(__uint_as_float(static_cast<uint32_t>(x[i]) << 16) * f);
        out[i] = *reinterpret_cast<uint16_t*>(&h);
    }
}

// One thread waits on a barrier nobody signals, with the pipeline's bounded
// wait; it must come back with the timeout bit set.
__global__ void wait_probe_kernel(unsigned* status, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(b, 0)) {
        if (globaltimer_ns() - t0 > limit_ns) {
            atomicOr(status, STATUS_TIMEOUT);
            break;
        }
    }
}

}  // namespace

cudaError_t launch_prepass(const int64_t* y, int64_t N, int64_t V, int64_t ignore_index, WsHeader* hdr,
                           int* label_counts, cudaStream_t s) {
    const int threads = 256;
    const int64_t want = (N + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 1024 ? want : 1024);
    prepass_kernel<<<blocks, threads, 0, s>>>(y, N, V, ignore_index, hdr, label_counts);
    return cudaGetLastError();
}

cudaError_t launch_label_sort(const int64_t* y, int64_t N, int64_t C, int64_t blocks_per_chunk, int64_t n_blocks,
                              int64_t V, int64_t ignore_index, unsigned long long* keys, unsigned long long* runs,
                              int* run_count, cudaStream_t s) {
    static std::atomic<uint64_t> configured{0};  // bit d: shared-memory limit raised on device d
    constexpr int smem = LABEL_BLOCK * 8;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(label_sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    label_sort_kernel<<<static_cast<unsigned>(n_blocks), 1024, smem, s>>>(y, N, C, blocks_per_chunk, V,
                                                                          ignore_index, keys, runs, run_count);
    return cudaGetLastError();
}

cudaError_t launch_onehot_scatter(const unsigned long long* keys, const unsigned long long* runs, const int* run_count,
                                  const uint16_t* X_chunk, const float* tcoef, int64_t H, int64_t rows, int64_t V,
                                  WsHeader* hdr, float* grad_W_acc, uint16_t* grad_W, float* label_csum,
                                  int write_bf16, int grid, cudaStream_t s) {
    onehot_scatter_kernel<<<grid, 256, 0, s>>>(keys, runs, run_count, X_chunk, tcoef, H, rows, V, hdr, grad_W_acc,
                                               grad_W, label_csum, write_bf16);
    return cudaGetLastError();
}

cudaError_t launch_scale(WsHeader* hdr, float grad_scale, const float* d_grad_output, int64_t* n_valid_out,
                         bool sum_reduction, cudaStream_t s) {
    scale_kernel<<<1, 1, 0, s>>>(hdr, grad_scale, d_grad_output, n_valid_out, sum_reduction ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float* part_m, const float* part_s, int64_t n_pt, int64_t ldp, int64_t rows,
                           const float* zt, const int64_t* y, int64_t ignore_index, int64_t V, float* lse,
                           float* row_loss, float* tcoef, unsigned* status, cudaStream_t s) {
    const int threads = 256;  // 8 rows, 32 threads each
    const int64_t blocks = (rows + 7) / 8;
    combine_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(part_m, part_s, n_pt, ldp, rows, zt, y,
                                                                      ignore_index, V, lse, row_loss, tcoef, status);
    return cudaGetLastError();
}

cudaError_t launch_loss(const float* row_loss, int64_t N, const WsHeader* hdr, float* loss, int64_t* n_valid_out,
                        bool sum_reduction, cudaStream_t s) {
    loss_kernel<<<1, 1024, 0, s>>>(row_loss, N, hdr, loss, n_valid_out, sum_reduction ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_grad_b(const float* gb_part, int64_t parts, int64_t V, const WsHeader* hdr,
                          const float* label_csum, float* grad_b_acc, uint16_t* grad_b, int first, int last,
                          cudaStream_t s) {
    const int threads = 256;
    const int64_t blocks = (V + threads - 1) / threads;
    grad_b_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(gb_part, parts, V, hdr, label_csum,
                                                                     grad_b_acc, grad_b, first, last);
    return cudaGetLastError();
}

cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

cudaError_t launch_amax(const uint16_t* x, int64_t n, unsigned* amax_bits, cudaStream_t s) {
    const int threads = 256;
    const int64_t want = (n / 8 + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 2048 ? want : 2048));
    amax_kernel<<<blocks, threads, 0, s>>>(x, n, amax_bits);
    return cudaGetLastError();
}

cudaError_t launch_to_f16_scaled(const uint16_t* x, int64_t n, const unsigned* amax_bits, uint16_t* out,
                                 cudaStream_t s) {
    const int threads = 256;
    const int64_t want = (n / 8 + threads - 1) / threads;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 4096 ? want : 4096));
    to_f16_scaled_kernel<<<blocks, threads, 0, s>>>(x, n, amax_bits, out);
    return cudaGetLastError();
}

cudaError_t launch_p_rescale(uint16_t* P, int64_t ldg, int64_t rows, int64_t V, const float* pm, int64_t ldp,
                             const float* lse, const int* crow, const int* n_valid, float* gb_part,
                             unsigned* status, cudaStream_t s) {
    // every 32-row block of every 128-row tile writes its column sums (zeros
    // past the last row), the layout the grad_b accumulation reads
    const dim3 grid(static_cast<unsigned>((rows + 127) / 128 * 4), static_cast<unsigned>((V + 255) / 256));
    p_rescale_kernel<<<grid, 256, 0, s>>>(P, ldg, rows, V, pm, ldp, lse, crow, n_valid, gb_part, status);
    return cudaGetLastError();
}

cudaError_t launch_compact_rows(const int64_t* y, int64_t N, int64_t C, int64_t n_chunks, int64_t V,
                                int64_t ignore_index, int* dmap, int* crow, int* n_valid_chunk, cudaStream_t s) {
    compact_rows_kernel<<<static_cast<unsigned>(n_chunks), 1024, 0, s>>>(y, N, C, V, ignore_index, dmap, crow,
                                                                         n_valid_chunk);
    return cudaGetLastError();
}

cudaError_t launch_zero_ignored_rows(const int* dmap, int64_t N, int64_t H, uint16_t* grad_X, cudaStream_t s) {
    const int64_t want = N < 8192 ? N : 8192;
    zero_ignored_rows_kernel<<<static_cast<unsigned>(want), 128, 0, s>>>(dmap, N, H, grad_X);
    return cudaGetLastError();
}

cudaError_t launch_gather_f16(const uint16_t* X_chunk, int64_t H, const int* crow, const int* n_valid,
                              int64_t max_rows, const unsigned* amax_bits, uint16_t* X16, uint16_t* P_tail,
                              int64_t ldg, unsigned* status, cudaStream_t s) {
    const int64_t want = (max_rows * (H / 8) + 255) / 256;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 4096 ? want : 4096));
    gather_f16_kernel<<<blocks, 256, 0, s>>>(X_chunk, H, crow, n_valid, max_rows, amax_bits, X16, P_tail, ldg,
                                             status);
    return cudaGetLastError();
}

cudaError_t launch_scale_grads(int64_t N, int64_t H, int64_t V, const float* d_grad_output, uint16_t* grad_X,
                               const float* grad_W_acc, uint16_t* grad_W, const float* grad_b_acc,
                               uint16_t* grad_b, cudaStream_t s) {
    const int64_t nx8 = grad_X ? N * H / 8 : 0, nw8 = grad_W ? V * H / 8 : 0;
    const int64_t most = nx8 > nw8 ? nx8 : nw8;
    const int64_t want = (most + 255) / 256;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 8192 ? want : 8192));
    scale_grads_kernel<<<blocks, 256, 0, s>>>(nx8, nw8, grad_b ? V : 0, d_grad_output,
                                              reinterpret_cast<uint4*>(grad_X),
                                              reinterpret_cast<const float4*>(grad_W_acc),
                                              reinterpret_cast<uint4*>(grad_W), grad_b_acc, grad_b);
    return cudaGetLastError();
}

cudaError_t launch_gradx_tail_reduce(const float* tail_out, int slots, int n_tiles, int k_blocks, int nw, int64_t H,
                                     const int* crow, const int* n_valid, int64_t max_rows, const int64_t* y,
                                     int64_t ignore_index, int64_t V, const uint16_t* W, const float* tcoef,
                                     const WsHeader* hdr, uint16_t* grad_X_chunk, cudaStream_t s) {
    if (nw != 1 && nw != 2) return cudaErrorInvalidValue;
    // at most slots - 1 tail tiles of 256 rows x (32 nw) groups of 8 columns
    const int64_t want = (static_cast<int64_t>(slots) * 2 * BM * (BN * nw / 8) + 255) / 256;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 1216 ? want : 1216));
    gradx_tail_reduce_kernel<<<blocks, 256, 0, s>>>(tail_out, slots, n_tiles, k_blocks, nw, H, crow, n_valid, y,
                                                    ignore_index, V, W, tcoef, hdr, grad_X_chunk, max_rows);
    return cudaGetLastError();
}

cudaError_t launch_gradx_split_reduce(const float* split_out, int64_t splits, int64_t split_stride, int64_t H,
                                      const int* crow, const int* n_valid, int64_t max_rows, const int64_t* y,
                                      int64_t ignore_index, int64_t V, const uint16_t* W, const float* tcoef,
                                      const WsHeader* hdr, uint16_t* grad_X_chunk, cudaStream_t s) {
    const int64_t want = (max_rows * (H / 8) + 255) / 256;
    const int blocks = static_cast<int>(want < 1 ? 1 : (want < 4096 ? want : 4096));
    gradx_split_reduce_kernel<<<blocks, 256, 0, s>>>(split_out, splits, split_stride, H, crow, n_valid, y,
                                                     ignore_index, V, W, tcoef, hdr, grad_X_chunk, max_rows);
    return cudaGetLastError();
}

}  // namespace lce
