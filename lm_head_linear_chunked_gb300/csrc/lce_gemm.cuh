// The library's one tensor-core GEMM: a persistent, warp-specialised
// tcgen05 kernel for sm_103a, with one fused epilogue per role.
//
//   warp 0 (one lane): TMA producer.  Loads 128x64 A and 256x64 B bf16 slices
//          (128-byte swizzled) into a 4-stage shared-memory ring.
//   warp 1 (one lane): MMA issuer.  Four tcgen05.mma (M=128, N=256, K=16)
//          per slice into one of two 256-column fp32 TMEM accumulators;
//          tcgen05.commit frees ring slots and publishes finished tiles.
//   warps 2..9: epilogue.  Each thread owns one accumulator row (its TMEM
//          lane) and half of its 256 columns, reads them 32 at a time with
//          tcgen05.ld and applies the role's epilogue while the MMA warp
//          fills the other buffer.
//
// Every wait is bounded (globaltimer); a wait that runs out raises the
// status bit, flags the CTA to stop, and the CTA drains its in-flight
// copies and MMAs, frees TMEM and returns.  Nothing traps.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>

#include <atomic>

#include "lce_internal.cuh"
#include "lce_ptx.cuh"

namespace lce {

constexpr float LOG2E_F = 1.4426950408889634f;
constexpr float P_SCALE = static_cast<float>(1 << P_SCALE_EXP);

__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

template <int MODE>
struct ModeTraits {
    static constexpr bool A_MN = (MODE == MODE_PLAIN_MM || MODE == MODE_GRADW);
    static constexpr bool B_MN = (MODE == MODE_PLAIN_KM || MODE == MODE_PLAIN_MM || is_gradx(MODE) ||
                                  MODE == MODE_GRADW);
    static constexpr bool F16 = (is_gradx(MODE) || MODE == MODE_GRADW);
    static constexpr int NW = MODE == MODE_GRADX_W ? 2 : 1;  // output tile width in 256-column MMAs
};

struct SharedCtl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint32_t tmem_base;
    volatile int abort_flag;
};
static_assert(sizeof(SharedCtl) <= CTL_BYTES, "control block too large");

// Waits for the phase of parity `parity` of barrier `bar`.  Gives up, raising
// the CTA's abort flag and the timeout status bit, after `limit_ns`; with
// `honor_abort` it also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, SharedCtl* ctl,
                                           unsigned* status, uint64_t limit_ns,
                                           bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && ctl->abort_flag) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            ctl->abort_flag = 1;
            atomicOr(status, STATUS_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ void tile_coords(int t, const GemmArgs& a, int& m, int& n) {
    if (a.raster == 0) {
        m = t % a.m_tiles;
        n = t / a.m_tiles;
    } else if (a.raster == 1) {
        n = t % a.n_tiles;
        m = t / a.n_tiles;
    } else if (a.raster == 2) {  // groups of group_m m-tiles; m fastest within a group
        const int per = a.group_m * a.n_tiles;
        const int g = t / per;
        const int r = t - g * per;
        const int gm0 = g * a.group_m;
        const int gm = min(a.group_m, a.m_tiles - gm0);
        m = gm0 + r % gm;
        n = r / gm;
    } else {  // groups of group_n n-tiles; n fastest within a group
        const int per = a.group_n * a.m_tiles;
        const int g = t / per;
        const int r = t - g * per;
        const int gn0 = g * a.group_n;
        const int gn = min(a.group_n, a.n_tiles - gn0);
        n = gn0 + r % gn;
        m = r / gn;
    }
}

// Tile t of a launch: output tile (m, n) and K slice ks (0 without a split).
__device__ __forceinline__ void tile_and_slice(int t, const GemmArgs& a, int& m, int& n, int& ks) {
    const int per = a.m_tiles * a.n_tiles;
    ks = t / per;
    tile_coords(t - ks * per, a, m, n);
}

// Work unit u of a launch: output tile (m, n), K slice ks and its k-block
// range [kb0, kb1), and tj = the partial-tile index of a split tail unit
// (-1 otherwise).  With a tail plan (tp.tail > 0) the first tp.full units
// are whole tiles and unit tp.full + j is slice j / tp.tail of tile
// tp.full + j % tp.tail, so one round of units takes every tail tile's
// slice before the next slice of any.
__device__ __forceinline__ void unit_coords(int u, const GemmArgs& a, const TailPlan& tp, int k_blocks, int& m,
                                            int& n, int& ks, int& kb0, int& kb1, int& tj) {
    tj = -1;
    if (tp.tail > 0 && u >= tp.full) {
        const int j = u - tp.full;
        ks = j / tp.tail;
        tile_coords(tp.full + (j - ks * tp.tail), a, m, n);
        kb0 = ks * tp.kps;
        kb1 = min(k_blocks, kb0 + tp.kps);
        tj = j;
        return;
    }
    tile_and_slice(u, a, m, n, ks);
    kb0 = a.k_splits > 1 ? ks * a.k_per_split : 0;
    kb1 = a.k_splits > 1 ? min(k_blocks, kb0 + a.k_per_split) : k_blocks;
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&p);
}

// Adds b[0 .. nv) (bf16, 16-byte aligned when nv == 32) to v[0 .. nv).
__device__ __forceinline__ void add_bias32(float (&v)[32], const uint16_t* b, int nv) {
    if (nv == 32) {
        const uint4* p = reinterpret_cast<const uint4*>(b);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const uint4 w = __ldg(p + g);
            const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                v[8 * g + 2 * k] += bf16_bits_to_float(u[k] & 0xFFFFu);
                v[8 * g + 2 * k + 1] += bf16_bits_to_float(u[k] >> 16);
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < nv) v[i] += bf16_bits_to_float(__ldg(b + i));
    }
}

// Stores v[0 .. nv) as bf16 (round to nearest even); nv is a multiple of 8.
__device__ __forceinline__ void store_bf16_32(uint16_t* dst, const float (&v)[32], int nv) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (8 * g < nv) {
            uint4 w;
            w.x = pack_bf16x2(v[8 * g + 0], v[8 * g + 1]);
            w.y = pack_bf16x2(v[8 * g + 2], v[8 * g + 3]);
            w.z = pack_bf16x2(v[8 * g + 4], v[8 * g + 5]);
            w.w = pack_bf16x2(v[8 * g + 6], v[8 * g + 7]);
            *reinterpret_cast<uint4*>(dst + 8 * g) = w;
        }
    }
}

// Stores v[0 .. nv) as fp16 (round to nearest even); nv is a multiple of 8.
__device__ __forceinline__ void store_f16_32(uint16_t* dst, const float (&v)[32], int nv) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        if (8 * g < nv) {
            __half2 h[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(v[8 * g + 2 * k], v[8 * g + 2 * k + 1]);
            uint4 w;
            w.x = *reinterpret_cast<uint32_t*>(&h[0]);
            w.y = *reinterpret_cast<uint32_t*>(&h[1]);
            w.z = *reinterpret_cast<uint32_t*>(&h[2]);
            w.w = *reinterpret_cast<uint32_t*>(&h[3]);
            *reinterpret_cast<uint4*>(dst + 8 * g) = w;
        }
    }
}

// Stores v[0 .. nv) as fp32; nv is a multiple of 4.
__device__ __forceinline__ void store_f32_32(float* dst, const float (&v)[32], int nv) {
#pragma unroll
    for (int g = 0; g < 8; ++g)
        if (4 * g < nv)
            *reinterpret_cast<float4*>(dst + 4 * g) =
                make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}

// Sum over the warp's 32 rows of each of 32 columns: afterwards lane k holds
// the sum of column k.  Five halving exchange steps (16+8+4+2+1 shuffles).
__device__ __forceinline__ float warp_column_sums(float (&g)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int k = 0; k < w; ++k) {
            const float send = upper ? g[k] : g[k + w];
            const float keep = upper ? g[k + w] : g[k];
            g[k] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, w);
        }
    }
    return g[0];
}

__device__ __forceinline__ bool gradw_nothing_to_add(const GemmArgs& a) {
    return a.dyn_rows && *a.dyn_rows == 0 && !a.acc_first && !a.write_bf16;
}

// Whether the grad_W epilogue reads the accumulator's old values into the
// SM (the read-modify-write path): not on the first chunk, and not when the
// tile is added into the accumulator at L2 by a TMA reduce.
__device__ __forceinline__ bool gradw_reads_old(const GemmArgs& a) {
    return !a.acc_first && (a.write_bf16 || !a.acc_tma);
}

// The FP32 grad_W accumulator values a warp's lane reads for the 32x32 block
// at rows row_base .. +31, columns c0 .. c0+31: rows (lane >> 3) + 4i
// (i = 0..7), columns c0 + 4 (lane & 7) .. +3; rows past m_rows read as 0.
__device__ __forceinline__ void gradw_load_old(const GemmArgs& a, int64_t row_base, int64_t m_rows, int64_t c0,
                                               int lane, float4 (&o)[8]) {
    const float* p = a.out_f32 + c0 + 4 * (lane & 7);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r = row_base + (lane >> 3) + 4 * i;
        o[i] = r < m_rows ? *reinterpret_cast<const float4*>(p + r * a.ld_f32) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
}

// The previous chunk's softmax rescale as a side job of the forward's
// epilogue warps (GemmArgs::side_p): P = fp16(E * 2^(half-tile max - lse
// log2 e)) in place, rows past the compact row count zeroed up to the next
// multiple of 64, exactly as p_rescale_kernel computes it.  Unit u covers
// compact rows 8 (u / n_tiles) .. +8 of vocab tile u % n_tiles; the units
// are dealt round-robin to all epilogue warps of the grid, and each warp
// works off `budget` of its units after each tile, the rest at the end.
struct SideJob {
    int64_t next, stride, units, nv, zero_end;
    int budget;
};

__device__ __forceinline__ void side_init(const GemmArgs& a, SideJob& j, int64_t gwarp, int64_t nwarps,
                                          int64_t tiles_here) {
    j.next = gwarp;
    j.stride = nwarps;
    j.units = 0;
    j.budget = 0;
    if (!a.side_p) return;
    j.nv = *a.side_nvalid;
    j.zero_end = min64((j.nv + 63) / 64 * 64, a.side_rows);
    j.units = (j.zero_end + 7) / 8 * a.n_tiles;
    const int64_t mine = (j.units + nwarps - 1) / nwarps;
    j.budget = static_cast<int>(mine / (tiles_here > 0 ? tiles_here : 1)) + 1;
}

__device__ __forceinline__ void side_unit(const GemmArgs& a, const SideJob& j, int64_t u, int lane) {
    const int64_t tile = u % a.n_tiles, rb = u / a.n_tiles;
    const int64_t c = tile * 256 + lane * 8;
    // The unit's 16 factors (8 rows x 2 half tiles, one max per 128-column
    // half tile) are computed once, by lane 8h + i for row i of half h, and
    // handed to the lanes of that half by shuffles.
    float fl = 0.f;
    {
        const int64_t r8 = rb * 8 + (lane & 7);
        if (lane < 16 && r8 < j.nv && LCE_IN(a.side_crow[r8] >= 0 && a.side_crow[r8] < a.side_rows, a.status)) {
            const int64_t r = a.side_crow[r8];  // chunk row
            const float* pm = a.side_pm + (2 * tile + (lane >> 3)) * a.ldp;
            fl = exp2f(pm[r] - a.side_lse[r] * LOG2E_F);
        }
    }
    float f[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = __shfl_sync(0xFFFFFFFFu, fl, (lane >> 4) * 8 + i);
    if (c >= a.ldg) return;
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r8 = rb * 8 + i;
        if (r8 < j.nv) w[i] = *reinterpret_cast<const uint4*>(a.side_p + r8 * a.ldg + c);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t r8 = rb * 8 + i;
        if (r8 >= j.zero_end) break;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (r8 < j.nv) {
            const uint32_t in[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
            uint32_t out[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float2 e = __half22float2(*reinterpret_cast<const __half2*>(&in[k]));
                __half2 h = __floats2half2_rn(e.x * f[i], e.y * f[i]);
                out[k] = *reinterpret_cast<uint32_t*>(&h);
            }
            o = make_uint4(out[0], out[1], out[2], out[3]);
        }
        *reinterpret_cast<uint4*>(a.side_p + r8 * a.ldg + c) = o;
    }
}

__device__ __forceinline__ void side_work(const GemmArgs& a, SideJob& j, int lane, int64_t budget) {
    for (int64_t k = 0; k < budget && j.next < j.units; ++k, j.next += j.stride) side_unit(a, j, j.next, lane);
}

// Hands an accumulator back to the MMA issuer once a warp has read it: a
// local arrive, or in the pair form an arrive on rank 0's barrier (given by
// its cluster address).
template <bool PAIR>
__device__ __forceinline__ void release_acc(uint32_t bar) {
    if constexpr (PAIR)
        mbar_arrive_cluster(bar);
    else
        mbar_arrive(bar);
}

// m_rows: rows of the output that exist (a.M, or the compacted row count);
// zero_acc: the tile had no K work (an empty compacted chunk), so its
// accumulator reads as zero.
template <int MODE, bool PAIR = false>
__device__ __forceinline__ void epilogue_tile(const GemmArgs& a, int m, int n, int q, int half, int lane,
                                              uint32_t taddr, uint32_t empty_bar, int64_t m_rows,
                                              bool zero_acc, int ks, const float4 (&pre)[8], float* stage,
                                              const CUtensorMap* map_c, int tj = -1) {
    constexpr int TW = BN * ModeTraits<MODE>::NW;  // output tile width
    const int64_t row = static_cast<int64_t>(m) * BM + q * 32 + lane;
    const int64_t col0 = static_cast<int64_t>(n) * TW;
    const int j0 = half * (TW / 64);  // this warp's 32-column chunks: half of the tile's columns
    const bool row_ok = row < m_rows;
    // MODE_LSE / MODE_G: where this row's E or P row goes (-1: not stored)
    const int64_t prow = (a.row_map && row_ok) ? static_cast<int64_t>(a.row_map[row]) : (row_ok ? row : -1);

    if constexpr (MODE == MODE_LSE) {
        // Two passes over the tile's TMEM row.  Pass 1: the tile max of
        // t = z log2(e) and the target logit.  Pass 2: s = sum 2^(t - max)
        // over the columns other than the row's target (the combine kernel
        // adds the target's term), and with a.g set, E = fp16(2^(t - max) *
        // 2^P_SCALE_EXP) for the backward (rescaled to P once lse is known),
        // 0 at the target.
        const int64_t yr = row_ok ? a.y[row] : a.ignore_index;
        // The max is taken over z and scaled once: rounding is monotone, so
        // max(z) * log2(e) rounds to the same float as max(z * log2(e)).
        float mz = -INFINITY, zt = 0.f;
        bool got = false;
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            const int nv = static_cast<int>(min64(32, a.N - c0));
            if (a.bias) add_bias32(v, a.bias + c0, nv);
            const int64_t d = yr - c0;
            const int kk = (d >= 0 && d < 32) ? static_cast<int>(d) : -1;
            got |= kk >= 0;
            if (__any_sync(0xFFFFFFFFu, kk >= 0)) {  // a label of the warp's rows lies in these columns
#pragma unroll
                for (int i = 0; i < 32; ++i) zt = (i == kk) ? v[i] : zt;
            }
            if (nv == 32) {
#pragma unroll
                for (int i = 0; i < 32; ++i) mz = fmaxf(mz, v[i]);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < nv) mz = fmaxf(mz, v[i]);
            }
        }
        const float mx = mz * LOG2E_F;
        float sm = 0.f;
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            const int nv = static_cast<int>(min64(32, a.N - c0));
            if (a.bias) add_bias32(v, a.bias + c0, nv);
            const int64_t d = yr - c0;
            const int kk = (d >= 0 && d < 32) ? static_cast<int>(d) : -1;  // the row's target column here
            const bool tgt = __any_sync(0xFFFFFFFFu, kk >= 0);
            if (nv == 32 && !tgt) {  // a whole chunk without a target: no per-column checks
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float e = fast_exp2(v[i] * LOG2E_F - mx);
                    sm += e;
                    v[i] = e * P_SCALE;
                }
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float e = (i < nv && i != kk) ? fast_exp2(v[i] * LOG2E_F - mx) : 0.f;
                    sm += e;
                    v[i] = e * P_SCALE;
                }
            }
            if (a.g && prow >= 0 && LCE_IN(prow < a.cap_rows, a.status))
                store_f16_32(a.g + prow * a.ldg + c0, v, static_cast<int>(min64(32, a.ldg - c0)));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
        if (row_ok && LCE_IN(2 * n + half < a.cap_pt && row < a.ldp && row < a.cap_rows, a.status)) {
            // one partial per 128-column half tile
            a.part_m[(2 * static_cast<int64_t>(n) + half) * a.ldp + row] = mx;
            a.part_s[(2 * static_cast<int64_t>(n) + half) * a.ldp + row] = sm;
            if (got) a.zt[row] = zt;
        }
    } else if constexpr (MODE == MODE_G) {
        // P = exp(z - lse) without the target entry, and the half tile's sum
        // of it (the combine kernel turns the row's sum into c = -sum P)
        const int64_t yr = row_ok ? a.y[row] : a.ignore_index;
        const bool valid = row_ok && yr != a.ignore_index;
        const float lse2 = row_ok ? a.lse[row] * LOG2E_F : 0.f;
        float se = 0.f;
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            const int nv = static_cast<int>(min64(32, a.N - c0));
            if (a.bias) add_bias32(v, a.bias + c0, nv);
            const int64_t d = yr - c0;
            const int kk = (d >= 0 && d < 32) ? static_cast<int>(d) : -1;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float p = fast_exp2(fmaf(v[i], LOG2E_F, -lse2));
                v[i] = (valid && i < nv && i != kk) ? p : 0.f;
                se += v[i];
            }
            if (prow >= 0 && LCE_IN(prow < a.cap_rows, a.status)) {
                float ps[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) ps[i] = v[i] * P_SCALE;
                store_f16_32(a.g + prow * a.ldg + c0, ps, static_cast<int>(min64(32, a.ldg - c0)));
            }
            if (a.gb_part && static_cast<int64_t>(m) * BM < a.M) {  // (a pair's second tile may lie past M)
                const float cs = warp_column_sums(v, lane);
                if (c0 + lane < a.N && LCE_IN(static_cast<int64_t>(m) * 4 + q < a.cap_gb, a.status))
                    a.gb_part[(static_cast<int64_t>(m) * 4 + q) * a.N + c0 + lane] = cs;
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
        if (row_ok && a.part_s && LCE_IN(2 * n + half < a.cap_pt && row < a.ldp, a.status))
            a.part_s[(2 * static_cast<int64_t>(n) + half) * a.ldp + row] = se;
    } else if constexpr (is_gradx(MODE)) {
      if (a.k_splits > 1 || tj >= 0) {
        // one K slice of a split product: the raw fp32 partial sums, finished
        // by a reduction kernel (fixed slice order).  A split tail unit's
        // slice goes to its own 256 x 256 partial tile (the pair tile's row,
        // this column), the k_splits form's to the slice's rows of the chunk.
        const bool tail = tj >= 0;
        const int64_t trow = row - static_cast<int64_t>(m >> 1) * (2 * BM);  // row within the pair tile
        float* dst = tail ? a.tail_out + static_cast<int64_t>(tj) * (TAIL_TILE_FLOATS * ModeTraits<MODE>::NW) +
                                trow * TW
                          : a.split_out + static_cast<int64_t>(ks) * a.split_stride + row * a.N;
        const int64_t cbase = tail ? col0 : 0;  // dst's first column
        // rows past the valid ones are not stored (and not checked)
        const bool store = row_ok && (tail ? LCE_IN(PAIR && tj < a.tail_units_max && trow >= 0 && trow < 2 * BM,
                                                    a.status)
                                           : LCE_IN(ks < a.k_splits && row < a.cap_rows, a.status));
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            if (zero_acc) {
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            if (store) store_f32_32(dst + (c0 - cbase), v, static_cast<int>(min64(32, a.N - c0)));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
      } else {
        // grad_X[i] = s (sum_v P[i,v] W[v] + c_i W[y_i]), P without the target
        // entry, c_i = p_{i,y_i} - 1; P rows of ignored rows are 0
        const float s = *a.scale;
        const float f = ldexpf(s, -(P_SCALE_EXP + operand_scale_exp(*a.b_amax_bits)));
        int64_t orow = (a.row_map && row_ok) ? static_cast<int64_t>(a.row_map[row]) : row;  // chunk row
        const bool orow_ok = !row_ok || LCE_IN(orow >= 0 && orow < a.cap_rows, a.status);
        if (!orow_ok) orow = 0;
        const int64_t yr = row_ok ? a.y[orow] : a.ignore_index;
        const bool valid = row_ok && orow_ok && yr != a.ignore_index && yr >= 0 && yr < a.V;
        const float sc = valid ? s * a.tcoef[orow] : 0.f;
        const uint16_t* wy = a.w_rows + (valid ? yr : 0) * a.ldw;
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            if (row_ok) {
                if (valid) {
                    float w[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) w[i] = 0.f;
                    add_bias32(w, wy + c0, 32);
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = fmaf(f, v[i], sc * w[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] *= f;
                }
                if (orow_ok) store_bf16_32(a.out_bf16 + orow * a.ld_out + c0, v, static_cast<int>(min64(32, a.N - c0)));
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
      }
    } else if constexpr (MODE == MODE_GRADW) {
        // grad_W_acc[v, h] (+)= s * acc.  Each 32x32 block (the warp's 32
        // rows, 32 columns) goes through the warp's shared-memory buffer, so
        // that the accumulator is read and written a whole 128-byte row
        // segment per 8 lanes (4 rows per instruction) instead of 16 bytes
        // of 32 different rows.  The old values are read one block ahead
        // (the first block by the caller, before the tile's MMAs finished).
        const float s = ldexpf(*a.scale, -(P_SCALE_EXP + operand_scale_exp(*a.b_amax_bits)));
        const int64_t row_base = static_cast<int64_t>(m) * BM + q * 32;
        if (a.acc_tma && !a.write_bf16) {
            // s * block -> buffer -> one TMA store (first chunk) or add at L2
            // (later chunks) per 32x32 block; the accumulator never passes
            // through the SM.  The buffer is the TMA box's 128-byte-swizzled
            // layout: row r's 16-byte slot k at slot k ^ (r & 7).
            const uint32_t sbuf = smem_u32(stage);
#pragma unroll 1
            for (int jj = 0; jj < BN / 64; ++jj) {
                const int64_t c0 = col0 + 32 * (j0 + jj);
                if (c0 >= a.N) break;
                float v[32];
                tmem_load_32cols(taddr + 32 * (j0 + jj), v);
                if (lane == 0) bulk_wait_read_all();  // the previous block has left the buffer
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4*>(stage + lane * 32 + ((k ^ (lane & 7)) << 2)) =
                        zero_acc ? make_float4(0.f, 0.f, 0.f, 0.f)
                                 : make_float4(s * v[4 * k], s * v[4 * k + 1], s * v[4 * k + 2], s * v[4 * k + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0 && row_base < m_rows && LCE_IN((c0 & 3) == 0 && c0 < a.N && row_base >= 0, a.status)) {
                    if (a.acc_first)
                        tma_store_2d(map_c, sbuf, static_cast<int32_t>(c0), static_cast<int32_t>(row_base));
                    else
                        tma_reduce_add_2d(map_c, sbuf, static_cast<int32_t>(c0), static_cast<int32_t>(row_base));
                    bulk_commit_group();
                }
            }
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) release_acc<PAIR>(empty_bar);
            return;
        }
        const int g = lane & 7;
        float4 cur[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[i] = pre[i];
#pragma unroll
        for (int jj = 0; jj < BN / 64; ++jj) {
            const int j = j0 + jj;
            const int64_t c0 = col0 + 32 * j;
            if (c0 < a.N) {
                {
                    float v[32];
                    tmem_load_32cols(taddr + 32 * j, v);
                    if (zero_acc) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] = 0.f;
                    }
                    // lane = row: 16-byte slot k of the row at slot k ^ (row & 7)
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        *reinterpret_cast<float4*>(stage + lane * 32 + ((k ^ (lane & 7)) << 2)) =
                            make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
                }
                __syncwarp();
                float4 nxt[8];
                if (!a.acc_first && jj + 1 < BN / 64 && c0 + 32 < a.N)
                    gradw_load_old(a, row_base, m_rows, c0 + 32, lane, nxt);
                else
#pragma unroll
                    for (int i = 0; i < 8; ++i) nxt[i] = cur[i];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int rr = (lane >> 3) + 4 * i;
                    const float4 x = *reinterpret_cast<const float4*>(stage + rr * 32 + ((g ^ (rr & 7)) << 2));
                    const int64_t r = row_base + rr;
                    if (r < m_rows) {
                        float4 o;
                        if (a.acc_first) {
                            o = make_float4(s * x.x, s * x.y, s * x.z, s * x.w);
                        } else {
                            o = make_float4(fmaf(s, x.x, cur[i].x), fmaf(s, x.y, cur[i].y), fmaf(s, x.z, cur[i].z),
                                            fmaf(s, x.w, cur[i].w));
                        }
                        *reinterpret_cast<float4*>(a.out_f32 + r * a.ld_f32 + c0 + 4 * g) = o;
                        if (a.write_bf16)
                            *reinterpret_cast<uint2*>(a.out_bf16 + r * a.ld_out + c0 + 4 * g) =
                                make_uint2(pack_bf16x2(o.x, o.y), pack_bf16x2(o.z, o.w));
                    }
                }
                __syncwarp();  // the buffer is rewritten by the next block
#pragma unroll
                for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
            }
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
    } else {  // PLAIN: D = fp32 product
#pragma unroll 1
        for (int j = j0; j < j0 + TW / 64; ++j) {
            const int64_t c0 = col0 + 32 * j;
            if (c0 >= a.N) break;
            float v[32];
            tmem_load_32cols(taddr + 32 * j, v);
            if (row_ok) store_f32_32(a.out_f32 + row * a.ld_f32 + c0, v, static_cast<int>(min64(32, a.N - c0)));
        }
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) release_acc<PAIR>(empty_bar);
    }
}

template <int MODE>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                const __grid_constant__ CUtensorMap map_c, const GemmArgs args) {
    using T = ModeTraits<MODE>;
    // A chunk without valid rows adds nothing to the grad_W accumulator: unless
    // its tiles overwrite the accumulator (first chunk) or write its bf16 cast
    // (last chunk), every CTA (both of a pair alike) leaves at once.
    if (MODE == MODE_GRADW && gradw_nothing_to_add(args)) return;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle needs 1024-byte alignment
    // ring | grad_W block buffers (MODE_GRADW) | control block
    constexpr int EPI_BYTES = MODE == MODE_GRADW ? EPI_STAGE_BYTES : 0;
    SharedCtl* ctl = reinterpret_cast<SharedCtl*>(smem_raw + (base - raw) + STAGES * STAGE_BYTES + EPI_BYTES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint64_t limit = args.timeout_ns;
    // grad_W epilogue: this warp's block buffer (launched with the extra bytes)
    float* const epi_stage = reinterpret_cast<float*>(smem_raw + (base - raw) + STAGES * STAGE_BYTES) +
                             (warp >= 2 ? (warp - 2) * EPI_STAGE_FLOATS : 0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tmem_full[b]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[b]), EPI_WARPS);
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        ctl->abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
        if (MODE == MODE_GRADW && args.acc_tma) tma_prefetch_map(&map_c);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&ctl->tmem_base), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = ctl->tmem_base;
    const int num_tiles = args.m_tiles * args.n_tiles * (args.k_splits > 1 ? args.k_splits : 1);
    // Compacted row count (written by an earlier kernel): limits the row tiles
    // of MODE_GRADX and the K loop of MODE_GRADW.  Every role reads the same
    // value, so all three skip the same tiles and run the same K loops.
    const int dyn = args.dyn_rows ? *args.dyn_rows : -1;
    const int64_t m_rows = (MODE == MODE_GRADX && dyn >= 0) ? static_cast<int64_t>(dyn) : args.M;
    const int k_blocks = (MODE == MODE_GRADW && dyn >= 0) ? (dyn + BK - 1) / BK : args.k_blocks;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer
            uint32_t stage = 0, phase = 0;
            uint64_t issued = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int m, n, ks;
                tile_and_slice(t, args, m, n, ks);
                if (static_cast<int64_t>(m) * BM >= m_rows) continue;
                const int kb0 = args.k_splits > 1 ? ks * args.k_per_split : 0;
                const int kb1 = args.k_splits > 1 ? min(k_blocks, kb0 + args.k_per_split) : k_blocks;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(smem_u32(&ctl->empty[stage]), phase ^ 1u, ctl, args.status, limit)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = smem_u32(&ctl->full[stage]);
                    mbar_arrive_expect_tx(fb, STAGE_BYTES);
                    const uint32_t sa = base + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    const int32_t k0 = kb * BK;
                    // innermost coordinates: multiples of 8 16-bit elements (16 bytes)
                    (void)LCE_IN((k0 & 7) == 0 && ((m * BM) & 7) == 0 && ((n * BN) & 7) == 0, args.status);
                    if constexpr (!T::A_MN) {
                        tma_load_2d(sa, &map_a, fb, k0, args.a_y0 + m * BM);
                    } else {
#pragma unroll
                        for (int j = 0; j < BM / 64; ++j)
                            tma_load_2d(sa + j * 8192, &map_a, fb, m * BM + 64 * j, args.a_y0 + k0);
                    }
                    if constexpr (!T::B_MN) {
#pragma unroll
                        for (int j = 0; j < BN / B_BOX_ROWS; ++j)
                            tma_load_2d(sb + j * (B_BOX_ROWS * 128), &map_b, fb, k0,
                                        args.b_y0 + n * BN + B_BOX_ROWS * j);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_2d(sb + j * 8192, &map_b, fb, n * BN + 64 * j, args.b_y0 + k0);
                    }
                    ++issued;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // Let the copies still in flight land before the CTA exits.
                const uint64_t last = issued < STAGES ? issued : STAGES;
                for (uint64_t i = 0; i < last; ++i) {
                    const uint64_t j = issued - 1 - i;
                    wait_phase(smem_u32(&ctl->full[j % STAGES]), static_cast<uint32_t>((j / STAGES) & 1u),
                               ctl, args.status, limit, false);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer
            constexpr uint32_t IDESC = instr_desc_f16kind(BM, BN, T::A_MN, T::B_MN, T::F16);
            // descriptor start-address step per K=16 MMA, in 16-byte units:
            // K-major: 32 bytes along the swizzled row; MN-major: two 8-row groups.
            constexpr uint32_t A_STEP = T::A_MN ? (2048u >> 4) : (32u >> 4);
            constexpr uint32_t B_STEP = T::B_MN ? (2048u >> 4) : (32u >> 4);
            uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
            bool ok = true;
            for (int t = blockIdx.x; t < num_tiles && ok; t += gridDim.x) {
                int m, n, ks;
                tile_and_slice(t, args, m, n, ks);
                if (static_cast<int64_t>(m) * BM >= m_rows) continue;
                const int kb0 = args.k_splits > 1 ? ks * args.k_per_split : 0;
                const int kb1 = args.k_splits > 1 ? min(k_blocks, kb0 + args.k_per_split) : k_blocks;
                if (!wait_phase(smem_u32(&ctl->tmem_empty[acc]), acc_phase ^ 1u, ctl, args.status, limit)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + acc * BN;
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(smem_u32(&ctl->full[stage]), phase, ctl, args.status, limit)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sa = base + stage * STAGE_BYTES;
                    const uint32_t sb = sa + A_STAGE_BYTES;
                    const uint64_t adesc = T::A_MN ? smem_desc_sw128(sa, 8192, 1024) : smem_desc_sw128(sa, 16, 1024);
                    const uint64_t bdesc = T::B_MN ? smem_desc_sw128(sb, 8192, 1024) : smem_desc_sw128(sb, 16, 1024);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k)
                        mma_f16kind(d_tmem, adesc + A_STEP * k, bdesc + B_STEP * k, IDESC,
                                     (kb != kb0 || k != 0) ? 1u : 0u);
                    mma_commit(smem_u32(&ctl->empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(smem_u32(&ctl->tmem_full[acc]));
                acc ^= 1u;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok) {
                // Wait for every MMA this thread issued before TMEM is freed.
                mma_commit(smem_u32(&ctl->drain));
                wait_phase(smem_u32(&ctl->drain), 0, ctl, args.status, limit, false);
            }
        }
    } else {
        // ---------------- epilogue (warps 2..9; warp w reads TMEM lanes 32*(w%4) ..,
        // warps 2..5 the tile's first 128 columns, warps 6..9 the last 128)
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        uint32_t acc = 0, acc_phase = 0;
        SideJob side;
        if constexpr (MODE == MODE_LSE)
            side_init(args, side, static_cast<int64_t>(blockIdx.x) * EPI_WARPS + (warp - 2),
                      static_cast<int64_t>(gridDim.x) * EPI_WARPS, (num_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x);
        for (int t = blockIdx.x; t < num_tiles; t += gridDim.x) {
            int m, n, ks;
            tile_and_slice(t, args, m, n, ks);
            if (static_cast<int64_t>(m) * BM >= m_rows) continue;
            const int kb0 = args.k_splits > 1 ? ks * args.k_per_split : 0;
            const int kb1 = args.k_splits > 1 ? min(k_blocks, kb0 + args.k_per_split) : k_blocks;
            float4 pre[8];
            if constexpr (MODE == MODE_GRADW) {
                // first block of the accumulator's old values, read before the tile's MMAs finish
                const int64_t c0 = static_cast<int64_t>(n) * BN + 128 * half;
                if (gradw_reads_old(args) && c0 < args.N)
                    gradw_load_old(args, static_cast<int64_t>(m) * BM + q * 32, m_rows, c0, lane, pre);
            }
            // (a warp vote keeps the lanes together should their waits end differently)
            if (!__all_sync(0xFFFFFFFFu, wait_phase(smem_u32(&ctl->tmem_full[acc]), acc_phase, ctl, args.status, limit)))
                break;
            tc_fence_after_sync();
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            epilogue_tile<MODE>(args, m, n, q, half, lane, taddr, smem_u32(&ctl->tmem_empty[acc]), m_rows,
                                kb1 <= kb0, ks, pre, epi_stage, &map_c);
            acc ^= 1u;
            if (acc == 0) acc_phase ^= 1u;
            if constexpr (MODE == MODE_LSE) side_work(args, side, lane, side.budget);
        }
        if constexpr (MODE == MODE_LSE) side_work(args, side, lane, side.units);
    }

    __syncwarp();  // reconverge the producer and MMA warps (one lane worked)
    // the epilogue's tile stores/adds read this CTA's shared memory until done
    if (MODE == MODE_GRADW && warp >= 2 && lane == 0) bulk_wait_all();
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int MODE>
cudaError_t launch_gemm_single(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                               const GemmArgs& args, int grid, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};  // bit d: shared-memory limit raised on device d
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (1ull << dev) : 0;
    if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
        e = cudaFuncSetAttribute(gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 gemm_smem_bytes(MODE, false));
        if (e != cudaSuccess) return e;
        configured.fetch_or(bit, std::memory_order_release);
    }
    gemm_kernel<MODE><<<grid, GEMM_THREADS, gemm_smem_bytes(MODE, false), stream>>>(map_a, map_b, map_c, args);
    return cudaGetLastError();
}

}  // namespace lce
