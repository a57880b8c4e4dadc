// Host side of the library: argument checks, the chunk planner, workspace
// carving, TMA descriptor encoding, and the launch sequence of each entry
// point of lce.h.
#include <cudaTypedefs.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "lce_internal.cuh"

namespace lce {
namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Rows per chunk when the caller lets the library choose.  Measured on the
// Qwen3-8B and Qwen3-4B head shapes against 4096-32768: 8192 rows ran 1.5-2.5%
// faster than 16384 (and used less energy per step under the power cap)
// with half the kept-exponential workspace.
constexpr int64_t AUTO_CHUNK_ROWS = 8192;
// Smallest chunk whose forward hosts the previous chunk's softmax rescale.
// Measured on the Qwen3-0.6B head at 256-row chunks: the forward grows by
// 0.9 ms per step and the rescale kernels' 1.3 ms go (+1.2% tokens/s).
constexpr int64_t OVERLAP_MIN_ROWS = 256;
// Tile-order groups: 4096 rows of X (32 MB at H = 4096) for the logits
// passes, 2048 rows of P for grad_X (single form); for the grad_W pass, as
// many 256-column tiles of the fp16 X chunk as make about 32 MB (8 at 8192
// rows), or 64 MB in the pair form.
constexpr int64_t LOGITS_GROUP_ROWS = 4096;
constexpr int64_t GRADX_GROUP_ROWS = 2048;
constexpr int64_t GROUP_BYTES = 32ll << 20;

// grad_X of a chunk with few output tiles (e.g. 256-row chunks) is split
// over K (the vocabulary) so that about two waves of tiles fill the GPU;
// the target does not depend on the device, so neither does the workspace.
constexpr int64_t GRADX_TARGET_TILES = 304;

int64_t gradx_splits(int64_t C, int64_t H, int64_t V) {
    const int64_t tiles = cdiv(C, BM) * cdiv(H, BN);
    if (tiles >= GRADX_TARGET_TILES / 2) return 1;
    int64_t s = cdiv(GRADX_TARGET_TILES, tiles);
    const int64_t kb = cdiv(V, BK);
    if (s > kb / 4) s = kb / 4;
    if (s > 64) s = 64;
    if (s <= 1) return 1;
    return cdiv(kb, cdiv(kb, s));  // every slice gets at least one k-block
}

// The pair form reads less DRAM in the grad_W pass with twice the group
// (measured: 0.4% faster on the Qwen3-8B head at the power cap).
int32_t gradw_group_n(int64_t rows, bool pair) {
    const int64_t g = (pair ? 2 * GROUP_BYTES : GROUP_BYTES) / (rows * BN * 2);
    return static_cast<int32_t>(g < 1 ? 1 : (g > 64 ? 64 : g));
}
constexpr size_t HEADER_BYTES = 1024;


struct Plan {
    int64_t N, H, V, C, n_chunks, n_vt, ldg, mt_chunk, label_blocks_per_chunk, gradx_splits;
    bool has_bias;
    // fused call: chunk c's forward rescales chunk c-1's E (two E and two
    // half-tile-max buffers)
    bool overlap;
    size_t off_row_loss, off_zt, off_pm, off_ps, off_g, off_gb, off_keys, off_runs, off_nrun, off_lcsum, off_w16,
        off_x16, off_dmap, off_crow, off_nvc, off_split, off_g2, off_pm2, off_tcoef, off_tail, total;
};

lce_status_t check_sizes(int64_t N, int64_t H, int64_t V, int64_t chunk_rows) {
    if (N <= 0 || H <= 0 || V <= 0 || chunk_rows < 0) return LCE_ERR_INVALID_ARG;
    if (H % 64 != 0 || N > INT32_MAX || V > INT32_MAX || H > INT32_MAX) return LCE_ERR_UNSUPPORTED;
    return LCE_OK;
}

int64_t rows_per_chunk(int64_t N, int64_t chunk_rows) {
    const int64_t c = chunk_rows > 0 ? chunk_rows : AUTO_CHUNK_ROWS;
    return c < N ? c : N;
}

lce_status_t make_plan(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, bool has_bias, int which,
                       Plan* p) {
    lce_status_t st = check_sizes(N, H, V, chunk_rows);
    if (st != LCE_OK) return st;
    if (which < LCE_WS_FORWARD || which > LCE_WS_FUSED_MIN) return LCE_ERR_INVALID_ARG;
    p->N = N;
    p->H = H;
    p->V = V;
    p->C = rows_per_chunk(N, chunk_rows);
    p->n_chunks = cdiv(N, p->C);
    p->n_vt = cdiv(V, BN);
    p->ldg = align_up(static_cast<size_t>(V), 8);
    p->mt_chunk = cdiv(p->C, BM);
    p->label_blocks_per_chunk = cdiv(p->C, LABEL_BLOCK);
    p->gradx_splits = gradx_splits(p->C, H, V);
    p->has_bias = has_bias;
    // Overlap only where a chunk's forward is long enough to hide the
    // previous chunk's rescale; the bias case keeps the rescale kernel, which
    // also sums P's columns for grad_b.
    p->overlap = which == LCE_WS_FUSED && !has_bias && p->n_chunks >= 2 && p->C >= OVERLAP_MIN_ROWS;
    const bool fwd = which != LCE_WS_BACKWARD, bwd = which != LCE_WS_FORWARD;  // FUSED_MIN: both
    size_t off = HEADER_BYTES;
    auto take = [&](bool use, size_t bytes) -> size_t {
        if (!use) return 0;
        const size_t at = off;
        off = align_up(off + bytes, 1024);
        return at;
    };
    p->off_row_loss = take(fwd, static_cast<size_t>(N) * 4);
    p->off_zt = take(fwd, static_cast<size_t>(p->C) * 4);
    p->off_pm = take(fwd, static_cast<size_t>(2 * p->n_vt) * p->C * 4);  // one per 128-column half tile
    // the forward's half-tile sums, or the recompute's half-tile sums of P
    p->off_ps = take(true, static_cast<size_t>(2 * p->n_vt) * p->C * 4);
    p->off_g = take(bwd, static_cast<size_t>(p->C) * p->ldg * 2);
    p->off_gb = take(bwd && has_bias, static_cast<size_t>(p->mt_chunk) * 4 * V * 4);
    p->off_keys = take(bwd, static_cast<size_t>(p->n_chunks) * p->label_blocks_per_chunk * LABEL_BLOCK * 8);
    p->off_runs = take(bwd, static_cast<size_t>(p->n_chunks) * p->label_blocks_per_chunk * LABEL_BLOCK * 8);
    p->off_nrun = take(bwd, static_cast<size_t>(p->n_chunks) * p->label_blocks_per_chunk * 4);
    p->off_lcsum = take(bwd && has_bias, static_cast<size_t>(V) * 4);
    p->off_w16 = take(bwd, static_cast<size_t>(V) * H * 2);
    p->off_x16 = take(bwd, static_cast<size_t>(p->C) * H * 2);
    p->off_dmap = take(bwd, static_cast<size_t>(N) * 4);
    p->off_crow = take(bwd, static_cast<size_t>(N) * 4);
    p->off_nvc = take(bwd, static_cast<size_t>(p->n_chunks) * 4);
    p->off_split = take(bwd && p->gradx_splits > 1, static_cast<size_t>(p->gradx_splits) * p->C * H * 4);
    p->off_g2 = take(p->overlap, static_cast<size_t>(p->C) * p->ldg * 2);
    p->off_pm2 = take(p->overlap, static_cast<size_t>(2 * p->n_vt) * p->C * 4);
    p->off_tcoef = take(bwd, static_cast<size_t>(N) * 4);  // c_i = p_{i,y_i} - 1 of every row
    // grad_X's split tail tiles (pair form, chunks not split over K as a whole)
    p->off_tail = take(bwd && p->gradx_splits <= 1, static_cast<size_t>(TAIL_UNITS_MAX) * TAIL_TILE_FLOATS * 4);
    p->total = off;
    return LCE_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- TMA maps

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Row-major 16-bit matrix [rows, cols] (bf16, or fp16 with `fp16`) with row
// pitch `pitch` elements; boxes of box_cols (innermost, 64 = one 128-byte
// swizzle row) x box_rows.  Out-of-range elements of a box read as zero.
bool map_16bit_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t pitch,
                  uint32_t box_cols, uint32_t box_rows, bool fp16 = false) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                          const_cast<void*>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Row-major FP32 matrix [rows, cols] with row pitch `pitch` elements, boxes
// of 32 x 32 (128-byte rows, 128-byte swizzle): the grad_W accumulator as
// the target of the epilogue's tile stores and adds.
bool map_f32_acc(CUtensorMap* m, void* base, int64_t rows, int64_t cols, int64_t pitch) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch) * 4};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int sm_count() {
    static std::atomic<int> cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    int n = cached[dev].load(std::memory_order_relaxed);
    if (!n) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev].store(n, std::memory_order_relaxed);
    }
    return n;
}

// The GEMM form of this process's calls (lce_set_gemm_form), read once per call.
std::atomic<int> g_gemm_form{LCE_GEMM_PAIR};

struct Form {
    bool pair;
    int64_t rows;  // output rows per tile: 128, or 256 shared by a pair
    int slots;     // tiles in flight at once: SMs, or resident pairs
};

Form gemm_form() {
    Form f;
    f.pair = g_gemm_form.load(std::memory_order_relaxed) == LCE_GEMM_PAIR && gemm_pair_slots() > 0;
    f.rows = f.pair ? PAIR_BM : BM;
    f.slots = f.pair ? gemm_pair_slots() : sm_count();
    return f;
}

// Grid of a persistent GEMM launch over `units` tiles (x K slices).
int grid_of(const Form& f, int64_t units) {
    if (f.slots <= 0) return 0;
    const int64_t n = units < f.slots ? units : f.slots;
    return static_cast<int>(f.pair ? 2 * n : n);
}

GemmArgs base_args(WsHeader* hdr) {
    GemmArgs a;
    memset(&a, 0, sizeof(a));
    a.group_m = 1;
    a.group_n = 1;
    a.k_splits = 1;
    a.status = &hdr->status;
    a.timeout_ns = WAIT_LIMIT_NS;
    return a;
}

#define LCE_TRY_CUDA(expr)                          \
    do {                                            \
        if ((expr) != cudaSuccess) return LCE_ERR_CUDA; \
    } while (0)

// ---------------------------------------------------------------- profiling

enum ProfKind { PK_LSE = 0, PK_P = 1, PK_GRADX = 2, PK_GRADW = 3, PK_OTHER = 4 };

struct Profiler {
    std::mutex mu;
    bool on = false;
    std::vector<cudaEvent_t> events;  // pairs (start, stop)
    std::vector<int> kinds;
    size_t used = 0;
};

Profiler& profiler() {
    static Profiler p;
    return p;
}

// Records the start event of a profiled launch; returns its slot or -1.
long prof_start(cudaStream_t s, int kind) {
    Profiler& p = profiler();
    if (!p.on) return -1;
    if (2 * p.used + 2 > p.events.size()) {
        for (int i = 0; i < 2; ++i) {
            cudaEvent_t e;
            if (cudaEventCreate(&e) != cudaSuccess) return -1;
            p.events.push_back(e);
        }
    }
    const size_t slot = p.used++;
    if (p.kinds.size() < p.used) p.kinds.resize(p.used);
    p.kinds[slot] = kind;
    cudaEventRecord(p.events[2 * slot], s);
    return static_cast<long>(slot);
}

void prof_stop(cudaStream_t s, long slot) {
    if (slot >= 0) cudaEventRecord(profiler().events[2 * slot + 1], s);
}

#define LCE_LAUNCH(kind, expr)                       \
    do {                                             \
        const long slot_ = prof_start(s, (kind));    \
        const cudaError_t e_ = (expr);               \
        prof_stop(s, slot_);                         \
        if (e_ != cudaSuccess) return LCE_ERR_CUDA;  \
    } while (0)

// ---------------------------------------------------------------- the loss

struct Problem {
    int64_t N, H, V;
    const uint16_t *X, *W, *b;
    const int64_t* y;
    int64_t ignore_index;
};

struct Outputs {
    float* loss;
    float* lse;  // written by the forward; read by the backward
    int64_t* n_valid;
    float grad_scale;
    const float* d_grad_output;
    uint16_t *grad_X, *grad_W, *grad_b;
    float *grad_W_acc, *grad_b_acc;
    uint32_t flags;  // LCE_REDUCTION_SUM | LCE_ACCUMULATE
};

lce_status_t run(const Problem& pb, const Outputs& o, bool do_fwd, bool do_bwd, int64_t chunk_rows, void* ws,
                 size_t ws_bytes, cudaStream_t s) {
    Plan p;
    const int which = do_fwd && do_bwd ? LCE_WS_FUSED : (do_fwd ? LCE_WS_FORWARD : LCE_WS_BACKWARD);
    lce_status_t st = make_plan(pb.N, pb.H, pb.V, chunk_rows, pb.b != nullptr, which, &p);
    if (st != LCE_OK) return st;
    // The fused call overlaps each chunk's softmax rescale with the next
    // chunk's forward when the workspace holds the second chunk of E, and
    // runs them one after the other when it holds only the minimum.
    if (which == LCE_WS_FUSED && ws_bytes < p.total) {
        st = make_plan(pb.N, pb.H, pb.V, chunk_rows, pb.b != nullptr, LCE_WS_FUSED_MIN, &p);
        if (st != LCE_OK) return st;
    }
    // pointer checks
    if (!pb.X || !pb.W || !pb.y || !ws || !o.lse) return LCE_ERR_INVALID_ARG;
    if (!aligned16(pb.X) || !aligned16(pb.W) || !aligned16(pb.b) || !aligned16(pb.y) || !aligned16(o.lse) ||
        (reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
        return LCE_ERR_INVALID_ARG;
    if (do_fwd && !o.loss) return LCE_ERR_INVALID_ARG;
    if (do_bwd) {
        if (!o.grad_W_acc || !aligned16(o.grad_W_acc) || !aligned16(o.grad_W) || !aligned16(o.grad_X))
            return LCE_ERR_INVALID_ARG;
        if (pb.b) {
            if (!o.grad_b_acc) return LCE_ERR_INVALID_ARG;
        } else if (o.grad_b || o.grad_b_acc) {
            return LCE_ERR_INVALID_ARG;
        }
    }
    if (o.flags & ~(LCE_REDUCTION_SUM | LCE_ACCUMULATE)) return LCE_ERR_INVALID_ARG;
    if ((o.flags & LCE_ACCUMULATE) && !do_bwd) return LCE_ERR_INVALID_ARG;
    const bool sum_reduction = (o.flags & LCE_REDUCTION_SUM) != 0;
    const bool accumulate = (o.flags & LCE_ACCUMULATE) != 0;
    if (ws_bytes < p.total) return LCE_ERR_WORKSPACE;
    if (!encode_fn() || sm_count() <= 0) return LCE_ERR_CUDA;
    const Form form = gemm_form();

    uint8_t* wsb = static_cast<uint8_t*>(ws);
    WsHeader* hdr = reinterpret_cast<WsHeader*>(wsb);
    float* row_loss = do_fwd ? reinterpret_cast<float*>(wsb + p.off_row_loss) : nullptr;
    float* zt = do_fwd ? reinterpret_cast<float*>(wsb + p.off_zt) : nullptr;
    float* pm = do_fwd ? reinterpret_cast<float*>(wsb + p.off_pm) : nullptr;
    float* ps = reinterpret_cast<float*>(wsb + p.off_ps);
    uint16_t* G = do_bwd ? reinterpret_cast<uint16_t*>(wsb + p.off_g) : nullptr;
    float* gb = (do_bwd && pb.b) ? reinterpret_cast<float*>(wsb + p.off_gb) : nullptr;
    unsigned long long* keys = do_bwd ? reinterpret_cast<unsigned long long*>(wsb + p.off_keys) : nullptr;
    unsigned long long* runs = do_bwd ? reinterpret_cast<unsigned long long*>(wsb + p.off_runs) : nullptr;
    int* nrun = do_bwd ? reinterpret_cast<int*>(wsb + p.off_nrun) : nullptr;
    uint16_t* W16 = do_bwd ? reinterpret_cast<uint16_t*>(wsb + p.off_w16) : nullptr;
    uint16_t* X16 = do_bwd ? reinterpret_cast<uint16_t*>(wsb + p.off_x16) : nullptr;
    int* dmap = do_bwd ? reinterpret_cast<int*>(wsb + p.off_dmap) : nullptr;  // row -> compacted row or -1
    int* crow = do_bwd ? reinterpret_cast<int*>(wsb + p.off_crow) : nullptr;  // compacted row -> chunk row
    int* nvc = do_bwd ? reinterpret_cast<int*>(wsb + p.off_nvc) : nullptr;    // valid rows per chunk
    float* split_out = (do_bwd && p.gradx_splits > 1) ? reinterpret_cast<float*>(wsb + p.off_split) : nullptr;
    float* lcsum = (do_bwd && pb.b) ? reinterpret_cast<float*>(wsb + p.off_lcsum) : nullptr;  // sum of c per label
    float* tcoef = do_bwd ? reinterpret_cast<float*>(wsb + p.off_tcoef) : nullptr;
    uint16_t* G2 = p.overlap ? reinterpret_cast<uint16_t*>(wsb + p.off_g2) : nullptr;
    float* pm2 = p.overlap ? reinterpret_cast<float*>(wsb + p.off_pm2) : nullptr;
    float* tail = (do_bwd && p.gradx_splits <= 1 && form.pair) ? reinterpret_cast<float*>(wsb + p.off_tail) : nullptr;

    // every GEMM launch of the call: the extents the bounds-checking build checks against
    auto call_args = [&]() {
        GemmArgs g = base_args(hdr);
        g.cap_rows = p.C;
        g.cap_pt = static_cast<int32_t>(2 * p.n_vt);
        g.cap_gb = p.mt_chunk * 4;
        return g;
    };

    // operand maps of the whole X and W
    CUtensorMap mX_k, mW_k, mW16_mn;
    if (!map_16bit_2d(&mX_k, pb.X, pb.N, pb.H, pb.H, 64, BM) || !map_16bit_2d(&mW_k, pb.W, pb.V, pb.H, pb.H, 64, B_BOX_ROWS))
        return LCE_ERR_CUDA;
    if (do_bwd && !map_16bit_2d(&mW16_mn, W16, pb.V, pb.H, pb.H, 64, 64, true)) return LCE_ERR_CUDA;
    CUtensorMap mAcc{};
    if (do_bwd && !map_f32_acc(&mAcc, o.grad_W_acc, pb.V, pb.H, pb.H)) return LCE_ERR_CUDA;

    LCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
    if (lcsum) LCE_TRY_CUDA(cudaMemsetAsync(lcsum, 0, static_cast<size_t>(pb.V) * 4, s));
    LCE_LAUNCH(PK_OTHER, launch_prepass(pb.y, pb.N, pb.V, pb.ignore_index, hdr, nullptr, s));
    if (do_bwd) {
        LCE_LAUNCH(PK_OTHER, launch_scale(hdr, o.grad_scale, o.d_grad_output, nullptr, sum_reduction, s));
        LCE_LAUNCH(PK_OTHER, launch_label_sort(pb.y, pb.N, p.C, p.label_blocks_per_chunk,
                                       p.n_chunks * p.label_blocks_per_chunk, pb.V, pb.ignore_index, keys, runs,
                                       nrun, s));
        // fp16 operands of the gradient GEMMs, with exact power-of-two scales
        LCE_LAUNCH(PK_OTHER, launch_amax(pb.X, pb.N * pb.H, &hdr->amax_x_bits, s));
        LCE_LAUNCH(PK_OTHER, launch_amax(pb.W, pb.V * pb.H, &hdr->amax_w_bits, s));
        LCE_LAUNCH(PK_OTHER, launch_to_f16_scaled(pb.W, pb.V * pb.H, &hdr->amax_w_bits, W16, s));
        // the backward products run over each chunk's valid rows only
        LCE_LAUNCH(PK_OTHER, launch_compact_rows(pb.y, pb.N, p.C, p.n_chunks, pb.V, pb.ignore_index, dmap, crow,
                                                 nvc, s));
        if (o.grad_X) LCE_LAUNCH(PK_OTHER, launch_zero_ignored_rows(dmap, pb.N, pb.H, o.grad_X, s));
    }

    // The forward of chunk c (logits, logsumexp, and in the fused call E kept
    // in Gc), with the previous chunk's rescale as its side job when side >= 0.
    auto forward_chunk = [&](int64_t c, uint16_t* Gc, float* pmc, int64_t side) -> lce_status_t {
        const int64_t r0 = c * p.C;
        const int64_t rows = (pb.N - r0) < p.C ? (pb.N - r0) : p.C;
        const int64_t mtf = cdiv(rows, form.rows);  // tiles of the GEMM form
        GemmArgs a = call_args();
        a.m_tiles = static_cast<int32_t>(mtf);
        a.n_tiles = static_cast<int32_t>(p.n_vt);
        a.k_blocks = static_cast<int32_t>(cdiv(pb.H, BK));
        a.raster = 2;
        a.group_m = static_cast<int32_t>(LOGITS_GROUP_ROWS / form.rows);
        a.a_y0 = static_cast<int32_t>(r0);
        a.M = rows;
        a.N = pb.V;
        a.y = pb.y + r0;
        a.ignore_index = pb.ignore_index;
        a.bias = pb.b;
        a.part_m = pmc;
        a.part_s = ps;
        a.zt = zt;
        a.ldp = p.C;
        if (do_bwd) {  // keep E = 2^(t - tile max) of the valid rows for the backward: no recompute
            a.g = Gc;
            a.ldg = p.ldg;
            a.row_map = dmap + r0;
        }
        if (side >= 0) {  // the epilogue warps rescale the previous chunk's E meanwhile
            const int64_t sr0 = side * p.C;
            a.side_p = (side & 1) ? G2 : G;
            a.side_pm = (side & 1) ? pm2 : pm;
            a.side_lse = o.lse + sr0;
            a.side_crow = crow + sr0;
            a.side_nvalid = nvc + side;
            a.side_rows = (pb.N - sr0) < p.C ? (pb.N - sr0) : p.C;
        }
        LCE_LAUNCH(PK_LSE, launch_gemm(MODE_LSE, mX_k, mW_k, mW_k, a, grid_of(form, mtf * p.n_vt), s, form.pair));
        LCE_LAUNCH(PK_OTHER, launch_combine(pmc, ps, 2 * p.n_vt, p.C, rows, zt, pb.y + r0, pb.ignore_index, pb.V,
                                            o.lse + r0, row_loss + r0, tcoef ? tcoef + r0 : nullptr, &hdr->status,
                                            s));
        return LCE_OK;
    };
    // The backward of chunk c; `rescaled`: its E was already turned into P.
    auto backward_chunk = [&](int64_t c, uint16_t* Gc, const float* pmc, bool rescaled) -> lce_status_t {
        const int64_t r0 = c * p.C;
        const int64_t rows = (pb.N - r0) < p.C ? (pb.N - r0) : p.C;
        const int64_t mt = cdiv(rows, BM);        // 128-row tiles (grad_b partial rows)
        const int64_t mtf = cdiv(rows, form.rows);  // tiles of the GEMM form
        // first: the chunk that overwrites the FP32 accumulators (none when accumulating)
        const bool first = c == 0 && !accumulate, last = c == p.n_chunks - 1;
        if (do_fwd) {  // P = E 2^(tile max - lse), in place (unless the next forward did it)
            if (!rescaled)
                LCE_LAUNCH(PK_OTHER, launch_p_rescale(Gc, p.ldg, rows, pb.V, pmc, p.C, o.lse + r0, crow + r0,
                                                      nvc + c, gb, &hdr->status, s));
        } else {   // recompute the logits; P = softmax (fp16)
            GemmArgs a = call_args();
            a.m_tiles = static_cast<int32_t>(mtf);
            a.n_tiles = static_cast<int32_t>(p.n_vt);
            a.k_blocks = static_cast<int32_t>(cdiv(pb.H, BK));
            a.raster = 2;
            a.group_m = static_cast<int32_t>(LOGITS_GROUP_ROWS / form.rows);
            a.a_y0 = static_cast<int32_t>(r0);
            a.M = rows;
            a.N = pb.V;
            a.y = pb.y + r0;
            a.ignore_index = pb.ignore_index;
            a.bias = pb.b;
            a.lse = o.lse + r0;
            a.g = Gc;
            a.ldg = p.ldg;
            a.gb_part = gb;
            a.row_map = dmap + r0;
            a.part_s = ps;
            a.ldp = p.C;
            LCE_LAUNCH(PK_P, launch_gemm(MODE_G, mX_k, mW_k, mW_k, a, grid_of(form, mtf * p.n_vt), s, form.pair));
            // c_i = -(sum of the row's non-target P), in a fixed order
            LCE_LAUNCH(PK_OTHER, launch_combine(nullptr, ps, 2 * p.n_vt, p.C, rows, nullptr, pb.y + r0,
                                                pb.ignore_index, pb.V, nullptr, nullptr, tcoef + r0, &hdr->status, s));
        }
        // P and X_c maps bounded to this chunk's rows: rows past it read as zero
        LCE_LAUNCH(PK_OTHER, launch_gather_f16(pb.X + r0 * pb.H, pb.H, crow + r0, nvc + c, rows, &hdr->amax_x_bits,
                                               X16, do_fwd ? nullptr : Gc, p.ldg, &hdr->status, s));
        CUtensorMap mG_k, mG_mn, mX16_mn;
        if (!map_16bit_2d(&mG_k, Gc, rows, pb.V, p.ldg, 64, BM, true) ||
            !map_16bit_2d(&mG_mn, Gc, rows, pb.V, p.ldg, 64, 64, true) ||
            !map_16bit_2d(&mX16_mn, X16, rows, pb.H, pb.H, 64, 64, true))
            return LCE_ERR_CUDA;
        if (o.grad_X) {   // grad_X_c = s (P W - W[y])
            // pair form and H a multiple of 512: 256 x 512 tiles (with the tail split)
            const int64_t kbl = cdiv(pb.V, BK);
            const bool wide = form.pair && pb.H % (2 * BN) == 0 && p.gradx_splits <= 1;
            const int nw = wide ? 2 : 1;
            // A small chunk's split product in the pair form: K slices for one round
            // of the pairs, fewer than the workspace holds (measured against two
            // rounds, or 512-column tiles: half the FP32 partial sums to write and
            // add, grad_X 10-14% faster at 256-row chunks)
            int64_t splits = p.gradx_splits;
            if (form.pair && splits > 1) {
                const int64_t sp = cdiv(static_cast<int64_t>(form.slots), mtf * cdiv(pb.H, BN));
                if (sp < splits) splits = sp > 1 ? cdiv(kbl, cdiv(kbl, sp)) : 1;
            }
            GemmArgs a = call_args();
            a.m_tiles = static_cast<int32_t>(mtf);
            a.n_tiles = static_cast<int32_t>(cdiv(pb.H, BN * nw));
            a.k_blocks = static_cast<int32_t>(kbl);
            // pair form: H tiles fastest, so that each wave covers whole rows of
            // grad_X and every tile sharing a P row block runs at once (measured:
            // grad_X 7% faster and ~20% fewer DRAM reads than 2048-row groups)
            a.raster = form.pair ? 1 : 2;
            a.group_m = static_cast<int32_t>(GRADX_GROUP_ROWS / form.rows);
            a.M = rows;
            a.N = pb.H;
            a.scale = &hdr->scale;
            a.out_bf16 = o.grad_X + r0 * pb.H;
            a.ld_out = pb.H;
            a.y = pb.y + r0;
            a.ignore_index = pb.ignore_index;
            a.w_rows = pb.W;
            a.ldw = pb.H;
            a.V = pb.V;
            a.b_amax_bits = &hdr->amax_w_bits;
            a.row_map = crow + r0;
            a.tcoef = tcoef + r0;
            a.dyn_rows = nvc + c;
            a.k_splits = static_cast<int32_t>(splits);
            a.k_per_split = static_cast<int32_t>(cdiv(a.k_blocks, splits));
            a.split_out = split_out;
            a.split_stride = p.C * pb.H;
            a.tail_out = tail;
            a.tail_units_max = TAIL_UNITS_MAX / nw;
            // with the tail split, a chunk of fewer tiles than pairs still gets every
            // pair: its slices spread over them
            const int grid = grid_of(form, static_cast<int64_t>(a.m_tiles) * a.n_tiles *
                                               (tail ? TAIL_SPLIT_MAX : splits));
            LCE_LAUNCH(PK_GRADX, launch_gemm(wide ? MODE_GRADX_W : MODE_GRADX, mG_k, mW16_mn, mW16_mn, a, grid, s,
                                             form.pair));
            if (tail)  // the same plan as the GEMM's: its pairs, tile columns and K extent
                LCE_LAUNCH(PK_GRADX, launch_gradx_tail_reduce(tail, grid / 2, a.n_tiles, a.k_blocks, nw, pb.H, crow + r0,
                                                              nvc + c, rows, pb.y + r0, pb.ignore_index, pb.V, pb.W,
                                                              tcoef + r0, hdr, o.grad_X + r0 * pb.H, s));
            if (split_out && splits > 1)
                LCE_LAUNCH(PK_GRADX, launch_gradx_split_reduce(split_out, splits, p.C * pb.H, pb.H, crow + r0,
                                                               nvc + c, rows, pb.y + r0, pb.ignore_index, pb.V,
                                                               pb.W, tcoef + r0, hdr, o.grad_X + r0 * pb.H, s));
        }
        {   // grad_W_acc (+)= s P^T X_c
            GemmArgs a = call_args();
            a.m_tiles = static_cast<int32_t>(cdiv(pb.V, form.rows));
            a.n_tiles = static_cast<int32_t>(cdiv(pb.H, BN));
            a.k_blocks = static_cast<int32_t>(cdiv(rows, BK));
            a.raster = 3;
            a.group_n = gradw_group_n(rows, form.pair);
            a.M = pb.V;
            a.N = pb.H;
            a.scale = &hdr->scale;
            a.out_f32 = o.grad_W_acc;
            a.ld_f32 = pb.H;
            a.out_bf16 = o.grad_W;
            a.ld_out = pb.H;
            a.acc_first = first;
            a.write_bf16 = last && o.grad_W != nullptr;
            // pair form with whole 256-column tiles: later chunks read the old
            // accumulator blocks by TMA and store them back (plain streams)
            a.acc_tma = (form.pair && pb.H % BN == 0) ? 2 : 1;
            // short K loops (chunks of up to 1024 rows): the tiles wait on the
            // accumulator's traffic, so more of its reads in flight, fewer ring stages
            a.gradw_bufs = a.k_blocks <= 16 ? 4 : 2;
            a.b_amax_bits = &hdr->amax_x_bits;
            a.dyn_rows = nvc + c;
            LCE_LAUNCH(PK_GRADW, launch_gemm(MODE_GRADW, mG_mn, mX16_mn, mAcc, a,
                                             grid_of(form, static_cast<int64_t>(a.m_tiles) * a.n_tiles), s,
                                             form.pair));
        }
        // grad_W_acc[y_i] += s c_i X[i] for the chunk's valid rows, exactly, in row order
        for (int64_t k = 0; k < p.label_blocks_per_chunk; ++k) {
            if (rows - k * LABEL_BLOCK <= 0) break;
            const int64_t blk = c * p.label_blocks_per_chunk + k;
            LCE_LAUNCH(PK_OTHER, launch_onehot_scatter(keys + blk * LABEL_BLOCK, runs + blk * LABEL_BLOCK,
                                                       nrun + blk, pb.X + r0 * pb.H, tcoef + r0, pb.H, rows, pb.V,
                                                       hdr, o.grad_W_acc, o.grad_W, lcsum, last && o.grad_W != nullptr,
                                                       4 * sm_count(), s));
        }
        // grad_b (after the scatter: the last chunk adds the target entries' sums per label)
        if (gb)
            LCE_LAUNCH(PK_OTHER, launch_grad_b(gb, mt * 4, pb.V, hdr, lcsum, o.grad_b_acc, o.grad_b, first, last, s));
        return LCE_OK;
    };

    // With p.overlap, chunk c's forward runs before chunk c-1's backward and
    // rescales chunk c-1's E meanwhile; E and the half-tile maxes alternate
    // between two buffers.
    for (int64_t c = 0; c < p.n_chunks; ++c) {
        uint16_t* Gc = (p.overlap && (c & 1)) ? G2 : G;
        float* pmc = (p.overlap && (c & 1)) ? pm2 : pm;
        if (do_fwd) {
            st = forward_chunk(c, Gc, pmc, p.overlap && c >= 1 ? c - 1 : -1);
            if (st != LCE_OK) return st;
        }
        if (do_bwd && !p.overlap) {
            st = backward_chunk(c, Gc, pmc, false);
            if (st != LCE_OK) return st;
        } else if (do_bwd && c >= 1) {
            st = backward_chunk(c - 1, ((c - 1) & 1) ? G2 : G, ((c - 1) & 1) ? pm2 : pm, true);
            if (st != LCE_OK) return st;
        }
    }
    if (do_bwd && p.overlap) {
        const int64_t c = p.n_chunks - 1;
        st = backward_chunk(c, (c & 1) ? G2 : G, (c & 1) ? pm2 : pm, false);
        if (st != LCE_OK) return st;
    }
    if (do_fwd) LCE_LAUNCH(PK_OTHER, launch_loss(row_loss, pb.N, hdr, o.loss, o.n_valid, sum_reduction, s));
    return LCE_OK;
}

}  // namespace

cudaError_t launch_gemm(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                        const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    if (grid <= 0) return cudaErrorInvalidConfiguration;
    switch (mode) {
        case MODE_LSE:
        case MODE_G: return launch_gemm_logits(mode, map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_GRADX:
        case MODE_GRADW: return launch_gemm_grads(mode, map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_GRADX_W: return launch_gemm_gradx_wide(map_a, map_b, map_c, args, grid, stream, pair);
        default: return launch_gemm_plain(mode, map_a, map_b, map_c, args, grid, stream, pair);
    }
}

}  // namespace lce

using namespace lce;

extern "C" {

lce_status_t lce_workspace_size(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int has_bias, int which,
                                size_t* bytes) {
    if (!bytes) return LCE_ERR_INVALID_ARG;
    Plan p;
    const lce_status_t st = make_plan(N, H, V, chunk_rows, has_bias != 0, which, &p);
    if (st == LCE_OK) *bytes = p.total;
    return st;
}

lce_status_t lce_chunk_rows(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int64_t* out) {
    if (!out) return LCE_ERR_INVALID_ARG;
    const lce_status_t st = check_sizes(N, H, V, chunk_rows);
    if (st == LCE_OK) *out = rows_per_chunk(N, chunk_rows);
    return st;
}

lce_status_t lce_forward_ex(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W,
                            const lce_bf16* b, const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                            float* loss, float* lse, int64_t* n_valid, void* ws, size_t ws_bytes,
                            lce_stream_t stream, uint32_t flags) {
    Problem pb{N, H, V, X, W, b, y, ignore_index};
    Outputs o;
    memset(&o, 0, sizeof(o));
    o.loss = loss;
    o.lse = lse;
    o.n_valid = n_valid;
    o.flags = flags;
    return run(pb, o, true, false, chunk_rows, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

lce_status_t lce_forward(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                         const int64_t* y, int64_t ignore_index, int64_t chunk_rows, float* loss, float* lse,
                         int64_t* n_valid, void* ws, size_t ws_bytes, lce_stream_t stream) {
    return lce_forward_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, loss, lse, n_valid, ws, ws_bytes, stream, 0);
}

lce_status_t lce_backward_ex(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W,
                             const lce_bf16* b, const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                             const float* lse, float grad_scale, const float* d_grad_output, lce_bf16* grad_X,
                             lce_bf16* grad_W, lce_bf16* grad_b, float* grad_W_acc, float* grad_b_acc, void* ws,
                             size_t ws_bytes, lce_stream_t stream, uint32_t flags) {
    Problem pb{N, H, V, X, W, b, y, ignore_index};
    Outputs o;
    memset(&o, 0, sizeof(o));
    o.lse = const_cast<float*>(lse);
    o.grad_scale = grad_scale;
    o.d_grad_output = d_grad_output;
    o.grad_X = grad_X;
    o.grad_W = grad_W;
    o.grad_b = grad_b;
    o.grad_W_acc = grad_W_acc;
    o.grad_b_acc = grad_b_acc;
    o.flags = flags;
    return run(pb, o, false, true, chunk_rows, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

lce_status_t lce_backward(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                          const int64_t* y, int64_t ignore_index, int64_t chunk_rows, const float* lse,
                          float grad_scale, const float* d_grad_output, lce_bf16* grad_X, lce_bf16* grad_W,
                          lce_bf16* grad_b, float* grad_W_acc, float* grad_b_acc, void* ws, size_t ws_bytes,
                          lce_stream_t stream) {
    return lce_backward_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, lse, grad_scale, d_grad_output, grad_X,
                           grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream, 0);
}

lce_status_t lce_fused_fwd_bwd_ex(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W,
                                  const lce_bf16* b, const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                                  float grad_scale, const float* d_grad_output, float* loss, float* lse,
                                  int64_t* n_valid, lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                                  float* grad_W_acc, float* grad_b_acc, void* ws, size_t ws_bytes,
                                  lce_stream_t stream, uint32_t flags) {
    Problem pb{N, H, V, X, W, b, y, ignore_index};
    Outputs o;
    memset(&o, 0, sizeof(o));
    o.loss = loss;
    o.lse = lse;
    o.n_valid = n_valid;
    o.grad_scale = grad_scale;
    o.d_grad_output = d_grad_output;
    o.grad_X = grad_X;
    o.grad_W = grad_W;
    o.grad_b = grad_b;
    o.grad_W_acc = grad_W_acc;
    o.grad_b_acc = grad_b_acc;
    o.flags = flags;
    return run(pb, o, true, true, chunk_rows, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

lce_status_t lce_fused_fwd_bwd(int64_t N, int64_t H, int64_t V, const lce_bf16* X, const lce_bf16* W,
                               const lce_bf16* b, const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                               float grad_scale, const float* d_grad_output, float* loss, float* lse,
                               int64_t* n_valid, lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                               float* grad_W_acc, float* grad_b_acc, void* ws, size_t ws_bytes,
                               lce_stream_t stream) {
    return lce_fused_fwd_bwd_ex(N, H, V, X, W, b, y, ignore_index, chunk_rows, grad_scale, d_grad_output, loss, lse,
                                n_valid, grad_X, grad_W, grad_b, grad_W_acc, grad_b_acc, ws, ws_bytes, stream, 0);
}

lce_status_t lce_scale_grads(int64_t N, int64_t H, int64_t V, const float* d_grad_output, lce_bf16* grad_X,
                             const float* grad_W_acc, lce_bf16* grad_W, const float* grad_b_acc, lce_bf16* grad_b,
                             lce_stream_t stream) {
    if (N <= 0 || H <= 0 || V <= 0 || !d_grad_output) return LCE_ERR_INVALID_ARG;
    if ((grad_W != nullptr) != (grad_W_acc != nullptr) || (grad_b != nullptr) != (grad_b_acc != nullptr))
        return LCE_ERR_INVALID_ARG;
    if (!aligned16(grad_X) || !aligned16(grad_W_acc) || !aligned16(grad_W)) return LCE_ERR_INVALID_ARG;
    if (H % 8 != 0) return LCE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    LCE_LAUNCH(PK_OTHER, launch_scale_grads(N, H, V, d_grad_output, grad_X, grad_W_acc, grad_W, grad_b_acc, grad_b, s));
    return LCE_OK;
}

lce_status_t lce_check_status(const void* ws, lce_stream_t stream) {
    if (!ws) return LCE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return LCE_ERR_CUDA;
    unsigned st = 0;
    if (cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return LCE_ERR_CUDA;
    if (st & STATUS_TIMEOUT) return LCE_ERR_TIMEOUT;
    if (st & STATUS_LABEL) return LCE_ERR_LABEL_RANGE;
    if (st & STATUS_BOUNDS) return LCE_ERR_BOUNDS;
    return LCE_OK;
}

const char* lce_status_string(lce_status_t status) {
    switch (status) {
        case LCE_OK: return "ok";
        case LCE_ERR_INVALID_ARG: return "invalid argument";
        case LCE_ERR_UNSUPPORTED: return "unsupported shape";
        case LCE_ERR_WORKSPACE: return "workspace too small";
        case LCE_ERR_LABEL_RANGE: return "label out of range";
        case LCE_ERR_TIMEOUT: return "device wait timed out";
        case LCE_ERR_CUDA: return "CUDA error";
        case LCE_ERR_BOUNDS: return "index outside its buffer (bounds-checking build)";
        default: return "unknown status";
    }
}

lce_status_t lce_profile_begin(void) {
    Profiler& p = profiler();
    std::lock_guard<std::mutex> g(p.mu);
    p.on = true;
    p.used = 0;
    return LCE_OK;
}

lce_status_t lce_profile_end(double* ms, int64_t* launches) {
    if (!ms || !launches) return LCE_ERR_INVALID_ARG;
    Profiler& p = profiler();
    std::lock_guard<std::mutex> g(p.mu);
    p.on = false;
    for (int k = 0; k < LCE_PROFILE_KINDS; ++k) {
        ms[k] = 0.0;
        launches[k] = 0;
    }
    for (size_t i = 0; i < p.used; ++i) {
        if (cudaEventSynchronize(p.events[2 * i + 1]) != cudaSuccess) return LCE_ERR_CUDA;
        float t = 0.f;
        if (cudaEventElapsedTime(&t, p.events[2 * i], p.events[2 * i + 1]) != cudaSuccess) return LCE_ERR_CUDA;
        ms[p.kinds[i]] += t;
        launches[p.kinds[i]] += 1;
    }
    p.used = 0;
    return LCE_OK;
}

lce_status_t lce_debug_gemm(int layout, int64_t M, int64_t N, int64_t K, const lce_bf16* A, const lce_bf16* B,
                            float* D, void* ws, size_t ws_bytes, lce_stream_t stream) {
    if (layout < 0 || layout > 2 || M <= 0 || N <= 0 || K <= 0 || !A || !B || !D || !ws) return LCE_ERR_INVALID_ARG;
    if (M % 8 || N % 8 || K % 8 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return LCE_ERR_UNSUPPORTED;
    if (!aligned16(A) || !aligned16(B) || !aligned16(D) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return LCE_ERR_INVALID_ARG;
    if (ws_bytes < 256) return LCE_ERR_WORKSPACE;
    if (!encode_fn() || sm_count() <= 0) return LCE_ERR_CUDA;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    CUtensorMap ma, mb;
    bool ok;
    if (layout == 0)
        ok = map_16bit_2d(&ma, A, M, K, K, 64, BM) && map_16bit_2d(&mb, B, N, K, K, 64, B_BOX_ROWS);
    else if (layout == 1)
        ok = map_16bit_2d(&ma, A, M, K, K, 64, BM) && map_16bit_2d(&mb, B, K, N, N, 64, 64);
    else
        ok = map_16bit_2d(&ma, A, K, M, M, 64, 64) && map_16bit_2d(&mb, B, K, N, N, 64, 64);
    if (!ok) return LCE_ERR_CUDA;
    const Form form = gemm_form();
    GemmArgs a = base_args(hdr);
    a.m_tiles = static_cast<int32_t>(cdiv(M, form.rows));
    a.n_tiles = static_cast<int32_t>(cdiv(N, BN));
    a.k_blocks = static_cast<int32_t>(cdiv(K, BK));
    a.raster = 0;
    a.M = M;
    a.N = N;
    a.out_f32 = D;
    a.ld_f32 = N;
    LCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
    LCE_TRY_CUDA(launch_gemm(layout, ma, mb, mb, a, grid_of(form, static_cast<int64_t>(a.m_tiles) * a.n_tiles), s,
                             form.pair));
    return LCE_OK;
}

int lce_gemm_pair_slots(void) { return gemm_pair_slots(); }

int lce_set_gemm_form(int form) {
    if (form != LCE_GEMM_SINGLE && form != LCE_GEMM_PAIR) return -1;
    return g_gemm_form.exchange(form);
}

lce_status_t lce_debug_gradx_tail_plan(int64_t tiles, int64_t slots, int64_t k_blocks, int64_t tile_cols,
                                       int64_t out[4]) {
    if (!out || tiles < 0 || slots < 0 || k_blocks < 0 || tiles > INT32_MAX || slots > INT32_MAX ||
        k_blocks > INT32_MAX || (tile_cols != BN && tile_cols != 2 * BN))
        return LCE_ERR_INVALID_ARG;
    const TailPlan tp = gradx_tail_plan(static_cast<int>(tiles), static_cast<int>(slots), static_cast<int>(k_blocks),
                                        static_cast<int>(TAIL_UNITS_MAX / (tile_cols / BN)));
    out[0] = tp.full;
    out[1] = tp.tail;
    out[2] = tp.s;
    out[3] = tp.kps;
    return LCE_OK;
}

lce_status_t lce_debug_wait_timeout(uint32_t limit_us, void* ws, size_t ws_bytes, lce_stream_t stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return LCE_ERR_INVALID_ARG;
    if (ws_bytes < 256) return LCE_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    WsHeader* hdr = static_cast<WsHeader*>(ws);
    LCE_TRY_CUDA(cudaMemsetAsync(hdr, 0, sizeof(WsHeader), s));
    LCE_TRY_CUDA(launch_wait_probe(&hdr->status, static_cast<uint64_t>(limit_us) * 1000ull, s));
    return LCE_OK;
}

}  // extern "C"
