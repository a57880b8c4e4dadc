// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "lce.h"

namespace lce {

// Roles of the one tensor-core GEMM kernel.  The three PLAIN modes write the
// bare fp32 product (diagnostics); the other four are the loss's GEMMs, each
// with its own fused epilogue.
enum GemmMode : int {
    MODE_PLAIN_KK = 0,  // D = A B^T,  A [M,K], B [N,K]        (both K-major)
    MODE_PLAIN_KM = 1,  // D = A B,    A [M,K], B [K,N]        (B MN-major)
    MODE_PLAIN_MM = 2,  // D = A^T B,  A [K,M], B [K,N]        (both MN-major)
    MODE_LSE = 3,       // logits X_c W^T -> per-row partial (max, sum exp over the non-target columns),
                        //   target logit, optionally E = 2^(t - tile max) (0 at the target) for the backward
    MODE_G = 4,         // logits X_c W^T -> P = softmax without the target entry (fp16, scaled by
                        //   2^P_SCALE_EXP), per-row partial sums of P, bias column sums
    MODE_GRADX = 5,     // grad_X_c = s * (P W + c W[y])         (fp16 operands, bf16 out)
    MODE_GRADW = 6,     // grad_W_acc (+)= s * P^T X_c           (fp16 operands, fp32 accumulator, bf16 cast)
    MODE_GRADX_W = 7,   // MODE_GRADX with 256 x 512 output tiles (pair form only, N a multiple of 512): two
                        //   N = 256 MMAs per K step fill all 512 TMEM columns, so each wave of tiles covers
                        //   twice the rows and streams W half as often; one accumulator, not two
};
constexpr bool is_gradx(int mode) { return mode == MODE_GRADX || mode == MODE_GRADX_W; }

// The softmax's target entry is never a tensor-core operand.  In a peaked
// softmax (a trained head puts p ~ 0.9-0.99 on the label) a 16-bit p would
// carry an error of 2^-11 p against the gradient entry p - 1, which is then
// small.  So every P the GEMMs read has a zero at (i, y_i), and the target
// column's gradient s * c_i with c_i = p_{i,y_i} - 1 is applied exactly, in
// fp32, by the grad_X epilogue (+ s c_i W[y_i]), the label-sorted scatter
// (grad_W_acc[y_i] += s c_i x_i) and the grad_b kernel.  The forward gets
// c_i without cancellation as -S'/(S' + T), S' the row's sum of exponentials
// over the other columns and T the target's; the recompute path sums the
// other columns' p instead.

// Tile shape: 128 rows (TMEM lanes) x 256 columns (fp32 TMEM columns),
// 64-element (128-byte) K slices, a 4-deep shared-memory ring.
constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int A_STAGE_BYTES = BM * BK * 2;                 // 16 KB
constexpr int B_STAGE_BYTES = BN * BK * 2;                 // 32 KB
constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES; // 48 KB
constexpr int CTL_BYTES = 512;
constexpr int GEMM_SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + CTL_BYTES;
// K-major B operands are loaded as boxes of 128 rows (two per 256-row tile
// here; one per CTA in the pair form below).
constexpr int B_BOX_ROWS = 128;
constexpr int EPI_WARPS = 8;        // two per TMEM lane quarter, one per 128-column half
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr uint32_t TMEM_COLS = 512; // two 256-column fp32 accumulators

// Pair form: two CTAs on neighbouring SMs (a cluster of 2) share one
// tcgen05 MMA of M = 256, N = 256 (cta_group::2).  Each CTA loads its own
// 128 rows of A and its own 128 rows (or columns) of B per 64-element K
// slice, 32 KB a stage instead of 48 KB, so the ring is 6 deep; each CTA's
// TMEM holds its 128 rows of the two accumulators.
constexpr int PAIR_BM = 2 * BM;                                      // 256 rows per pair tile
constexpr int PAIR_STAGES = 6;
constexpr int PAIR_B_STAGE_BYTES = (BN / 2) * BK * 2;                // 16 KB
constexpr int PAIR_STAGE_BYTES = A_STAGE_BYTES + PAIR_B_STAGE_BYTES; // 32 KB
constexpr int GEMM_PAIR_SMEM_BYTES = 1024 + PAIR_STAGES * PAIR_STAGE_BYTES + CTL_BYTES;

// The grad_W epilogue passes each warp's 32x32 FP32 blocks through a 4 KB
// shared-memory buffer per epilogue warp (after the ring, before the control
// block; 1024-byte aligned, laid out as a 128-byte-swizzled TMA box).
constexpr int EPI_STAGE_FLOATS = 32 * 32;
constexpr int EPI_STAGE_BYTES = EPI_WARPS * EPI_STAGE_FLOATS * 4;  // 32 KB
// In the pair form the grad_W kernel shares 7 x 32 KB between its ring and
// its epilogue buffers (GemmArgs::gradw_bufs per warp, 2 or 4, so that it can
// read the accumulator's old values that many blocks ahead by TMA; acc_tma 2):
// 5 ring stages and 2 buffers per warp for long K loops, 3 and 4 for short
// ones, whose tiles wait on the accumulator's traffic rather than the MMAs.
constexpr int GRADW_PAIR_SLOTS = 7;
constexpr int GRADW_PAIR_BUFS_MAX = 4;
// MODE_GRADX_W: a K slice is A (16 KB) and two 128-column pieces of B per
// CTA (32 KB); the ring is 4 stages deep.
constexpr int GRADX_W_STAGES = 4;
constexpr int pair_stage_bytes(int mode) {
    return mode == MODE_GRADX_W ? A_STAGE_BYTES + 2 * PAIR_B_STAGE_BYTES : PAIR_STAGE_BYTES;
}
constexpr int pair_ring_bytes(int mode) {
    return mode == MODE_GRADW     ? GRADW_PAIR_SLOTS * PAIR_STAGE_BYTES
           : mode == MODE_GRADX_W ? GRADX_W_STAGES * pair_stage_bytes(mode)
                                  : PAIR_STAGES * PAIR_STAGE_BYTES;
}
constexpr int gemm_smem_bytes(int mode, bool pair) {
    return pair ? 1024 + pair_ring_bytes(mode) + CTL_BYTES
                : GEMM_SMEM_BYTES + (mode == MODE_GRADW ? EPI_STAGE_BYTES : 0);
}
static_assert(PAIR_STAGE_BYTES == EPI_STAGE_BYTES, "a ring stage and a set of epilogue buffers take the same bytes");
static_assert(gemm_smem_bytes(MODE_GRADW, false) <= 232448 && gemm_smem_bytes(MODE_GRADW, true) <= 232448 &&
                  gemm_smem_bytes(MODE_LSE, true) <= 232448 && gemm_smem_bytes(MODE_GRADX_W, true) <= 232448,
              "shared memory of one CTA");

// grad_X's last partial wave (pair form).  Each grad_X tile runs the whole
// vocabulary as its K loop (about a millisecond at V = 151936), so when a
// launch's tiles leave the last round of pairs partly filled, the idle pairs
// wait a whole tile.  The plan keeps the whole rounds of tiles as they are
// and splits each of the r tiles after them into s K slices, dealt out to
// the pairs like tiles; each slice's raw FP32 sum goes to a partial tile of
// the workspace, and a reduction kernel finishes those tiles, adding the
// slices in slice order.  s is the one of 2..TAIL_SPLIT_MAX that makes the
// tail's rounds of slices, ceil(r s / slots) / s of a tile, shortest; no split
// unless that saves at least an eighth of a tile.
struct TailPlan {
    int32_t full;   // tiles computed whole: the first `full` tiles of the launch's tile order
    int32_t tail;   // tiles split over K after them (0: no split)
    int32_t s;      // K slices per split tile
    int32_t kps;    // k-blocks per slice (the last slice may be shorter; none is empty)
};
constexpr int TAIL_SPLIT_MAX = 8;
constexpr int TAIL_UNITS_MAX = 320;     // tail x s partial tiles of 256 x 256 FP32 (80 MB of workspace)
constexpr int TAIL_MIN_KBLOCKS = 16;    // shortest slice, in 64-wide k-blocks
constexpr int64_t TAIL_TILE_FLOATS = static_cast<int64_t>(2 * BM) * BN;  // per 256 output columns

// n_act: output tiles with valid rows; slots: pairs of the launch;
// max_units: partial tiles the workspace holds (TAIL_UNITS_MAX, halved for
// 512-column tiles).
__host__ __device__ inline TailPlan gradx_tail_plan(int n_act, int slots, int k_blocks,
                                                    int max_units = TAIL_UNITS_MAX) {
    TailPlan p{n_act > 0 ? n_act : 0, 0, 1, k_blocks};
    if (n_act <= 0 || slots <= 0) return p;
    const int r = n_act % slots;
    if (r == 0) return p;
    int best = 1, best_rounds = 1;  // tail time = best_rounds / best tiles
    for (int s = 2; s <= TAIL_SPLIT_MAX; ++s) {
        if (r * s > max_units || k_blocks < s * TAIL_MIN_KBLOCKS) break;
        const int rounds = (r * s + slots - 1) / slots;
        if (rounds * best < best_rounds * s) {
            best = s;
            best_rounds = rounds;
        }
    }
    if (best == 1 || 8 * best_rounds > 7 * best) return p;
    p.kps = (k_blocks + best - 1) / best;
    p.s = (k_blocks + p.kps - 1) / p.kps;
    p.full = n_act - r;
    p.tail = r;
    return p;
}

// Device status word bits (bit k set = lce_status_t k was raised).
constexpr unsigned STATUS_LABEL = 1u << LCE_ERR_LABEL_RANGE;
constexpr unsigned STATUS_TIMEOUT = 1u << LCE_ERR_TIMEOUT;
constexpr unsigned STATUS_BOUNDS = 1u << LCE_ERR_BOUNDS;

// Bounds-checking build (LCE_DEBUG): LCE_IN(cond, status) is `cond`, and a
// false condition also raises STATUS_BOUNDS in the call's status word; the
// caller skips the access it guards.  In the release build it is `true` and
// `cond` is not evaluated.
#ifdef LCE_DEBUG
__device__ __forceinline__ bool dbg_in(bool ok, unsigned* status) {
    if (!ok) atomicOr(status, STATUS_BOUNDS);
    return ok;
}
#define LCE_IN(cond, status) (::lce::dbg_in((cond), (status)))
#else
#define LCE_IN(cond, status) (true)
#endif

// The gradient GEMMs take fp16 operands (11 significant bits, against bf16's
// 8): P is stored as fp16(p * 2^P_SCALE_EXP), and W and X are converted to
// fp16 with an exact power-of-two scale 2^k chosen from their largest
// magnitude (k = operand_scale_exp()), so the conversion loses nothing of
// the bf16 values that matter.  Epilogues undo the scales exactly.
constexpr int P_SCALE_EXP = 15;

// Rows per block of the label sort that drives the exact one-hot part of
// grad_W (one CTA sorts one block in shared memory).
constexpr int LABEL_BLOCK = 8192;

// Default limit of one pipeline wait.  The longest legitimate wait is one
// tile's main loop (under a millisecond for K = 151936).
constexpr uint64_t WAIT_LIMIT_NS = 1000000000ull;

// First 256 bytes of every workspace.
struct WsHeader {
    unsigned status;
    unsigned pad0;
    unsigned long long n_valid;
    float scale;          // s = grad_scale * grad_output / n_valid (0 if n_valid == 0)
    unsigned amax_x_bits; // float bits of max |X|
    unsigned amax_w_bits; // float bits of max |W|
    unsigned pad1;
};

// Exponent k with amax * 2^k < 2^15 (so every |value| * 2^k fits fp16's
// range with room to spare); 0 for a zero or non-finite amax.
__host__ __device__ inline int operand_scale_exp(unsigned amax_bits) {
    const int e = static_cast<int>((amax_bits >> 23) & 0xFFu);
    if (e == 0 || e == 255) return 0;
    return 141 - e;  // amax < 2^(e - 126)
}

struct GemmArgs {
    int32_t m_tiles, n_tiles, k_blocks;
    // Tile order.  0: m fastest; 1: n fastest; 2: groups of group_m m-tiles
    // (m fastest inside); 3: groups of group_n n-tiles (n fastest inside).
    // Groups keep the operand that all tiles of a wave share within about
    // 32 MB, which L2 holds across waves (64 MB is re-read from DRAM).
    int32_t raster;
    int32_t group_m;
    int32_t group_n;
    int32_t a_y0;     // added to A's outer (row) TMA coordinate
    int32_t b_y0;     // added to B's outer (row) TMA coordinate
    int64_t M, N;     // valid extent of the output (rows, columns)
    // MODE_LSE / MODE_G
    const int64_t* y;  // labels of this chunk's first row
    int64_t ignore_index;
    const uint16_t* bias;  // nullable
    float* part_m;     // [2 n_tiles, ldp] per-row max of each 128-column half tile (base-2 units)
    float* part_s;     // [2 n_tiles, ldp] MODE_LSE: per-row sum of 2^(t - max) over the half tile's columns
                       //   other than the row's target; MODE_G: per-row sum of P over the same columns
    float* zt;         // [chunk rows] target logit
    int64_t ldp;
    const float* lse;  // this chunk's first row
    uint16_t* g;       // P [chunk rows, ldg] bf16
    int64_t ldg;
    float* gb_part;    // [m_tiles * 4, V] column sums of P (nullable)
    // MODE_GRADX: the target column's part, c_i W[y_i], is applied exactly in the
    // epilogue (tcoef: c_i of this chunk's rows, indexed by chunk row)
    const float* tcoef;
    const uint16_t* w_rows;
    int64_t ldw;
    int64_t V;
    // MODE_GRADX / MODE_GRADW: float bits of max |B operand| (its fp16 scale)
    const unsigned* b_amax_bits;
    // MODE_GRADX / MODE_GRADW / PLAIN
    const float* scale;  // device scalar s
    uint16_t* out_bf16;
    int64_t ld_out;
    float* out_f32;
    int64_t ld_f32;
    int32_t acc_first;   // MODE_GRADW: overwrite instead of accumulate
    int32_t write_bf16;  // MODE_GRADW: also write the bf16 cast
    int32_t gradw_bufs;  // MODE_GRADW, pair form: epilogue buffers per warp (2 or 4; the ring gets 7 - this stages)
    int32_t acc_tma;     // MODE_GRADW: without write_bf16, store (first) or add (later) the tile into
                         // out_f32 through the third tensor map (FP32 [M, N], 32x32 boxes, 128-byte swizzle):
                         // 1: later chunks add at L2 (cp.reduce.async.bulk); 2 (pair form, N a multiple of
                         // 256): later chunks load the old block by TMA, add in registers, store it by TMA
    // Valid-row compaction: the backward products skip ignored rows.
    //   MODE_LSE / MODE_G: row_map[chunk row] = row of the compacted P it is
    //     stored at (-1: ignored, not stored).
    //   MODE_GRADX: row_map[compact row] = chunk row; dyn_rows = number of
    //     compact rows (the M extent; row tiles past it are skipped).
    //   MODE_GRADW: dyn_rows = number of compact rows (the K extent).
    // Both nullable (no compaction).
    const int* row_map;
    const int* dyn_rows;
    // MODE_GRADX split over K (for chunks with few output tiles): tile index
    // t -> (m, n) = the raster of t % (m_tiles n_tiles), K slice
    // t / (m_tiles n_tiles) of k_per_split k-blocks; the raw fp32 accumulator
    // goes to split_out[slice][row][col] (row stride N, slice stride
    // split_stride) and a reduction kernel finishes grad_X.  1 = no split.
    int32_t k_splits;
    int32_t k_per_split;
    float* split_out;
    int64_t split_stride;
    // MODE_GRADX, pair form, no k_splits: split the last partial round of
    // tiles over K (gradx_tail_plan of the valid rows' tiles and the
    // launch's pairs).  Split unit j (< tail_units_max) writes its raw FP32
    // sum to tail_out[j] (a 256 x 256 tile, row stride 256); unit j is slice
    // j / tail of tile full + j % tail.  nullptr: no split.
    float* tail_out;
    int32_t tail_units_max;
    // MODE_LSE side job (fused call): between tiles, the epilogue warps turn
    // the previous chunk's kept exponentials E into P in place, the work of
    // p_rescale_kernel, in units of 8 compact rows x one 256-column vocab
    // tile.  side_p == nullptr: no side job.  n_tiles, ldp, ldg and V are the
    // current chunk's, which the previous chunk shares.
    uint16_t* side_p;          // the previous chunk's E [compact rows, ldg]
    const float* side_pm;      // its [2 n_tiles, ldp] half-tile maxes
    const float* side_lse;     // lse of its first row
    const int* side_crow;      // its compact row -> chunk row
    const int* side_nvalid;    // its number of compact rows (device)
    int64_t side_rows;         // its number of chunk rows
    unsigned* status;
    uint64_t timeout_ns;
    // Extents the bounds-checking build checks against: rows of the buffers
    // indexed by chunk row (target logits, partial columns, E/P rows, split
    // partial rows, c_i), partial rows (2 x vocabulary tiles), grad_b partial rows.
    int64_t cap_rows;
    int32_t cap_pt;
    int64_t cap_gb;
};

// Launches the GEMM kernel of `mode`: with `pair`, the pair form (grid =
// 2 x the number of pairs; m_tiles counts 256-row tiles), else one CTA per
// 128-row tile (grid = CTAs).  The instantiations are spread over four
// translation units so that they compile in parallel.
// map_c: the grad_W accumulator's map (MODE_GRADW with acc_tma), else unused.
cudaError_t launch_gemm(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                        const GemmArgs& args, int grid, cudaStream_t stream, bool pair);
cudaError_t launch_gemm_logits(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                               const GemmArgs& args, int grid, cudaStream_t stream, bool pair);
cudaError_t launch_gemm_grads(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                              const GemmArgs& args, int grid, cudaStream_t stream, bool pair);
cudaError_t launch_gemm_plain(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                              const GemmArgs& args, int grid, cudaStream_t stream, bool pair);
cudaError_t launch_gemm_gradx_wide(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                                   const GemmArgs& args, int grid, cudaStream_t stream, bool pair);
// Pairs of the pair form that can be resident at once on this device (0 if
// the form cannot launch).
int gemm_pair_slots();

// Small kernels (lce_aux.cu).
cudaError_t launch_prepass(const int64_t* y, int64_t N, int64_t V, int64_t ignore_index,
                           WsHeader* hdr, int* label_counts, cudaStream_t s);
cudaError_t launch_label_sort(const int64_t* y, int64_t N, int64_t C, int64_t blocks_per_chunk,
                              int64_t n_blocks, int64_t V, int64_t ignore_index,
                              unsigned long long* keys, unsigned long long* runs, int* run_count,
                              cudaStream_t s);
// grad_W_acc[v] += s * sum of c_i X[i] over the block's rows with y_i = v
// (tcoef: c_i of the chunk's rows); with label_csum, also
// label_csum[v] += sum of those c_i (for grad_b).
cudaError_t launch_onehot_scatter(const unsigned long long* keys, const unsigned long long* runs,
                                  const int* run_count, const uint16_t* X_chunk, const float* tcoef, int64_t H,
                                  int64_t rows, int64_t V, WsHeader* hdr, float* grad_W_acc, uint16_t* grad_W,
                                  float* label_csum, int write_bf16, int grid, cudaStream_t s);
// s = grad_scale * grad_output / n_valid (mean), or grad_scale * grad_output (sum_reduction).
cudaError_t launch_scale(WsHeader* hdr, float grad_scale, const float* d_grad_output,
                         int64_t* n_valid_out, bool sum_reduction, cudaStream_t s);
// Per row of a chunk: merges the partials into lse; row loss lse - z_t (NaN
// for a label outside [0, V) that is not ignore_index); tcoef (nullable):
// c = p_target - 1.  With part_m == nullptr the partials are plain sums of
// the non-target P (the recompute path) and only tcoef = -sum is written.
cudaError_t launch_combine(const float* part_m, const float* part_s, int64_t n_vt, int64_t ldp,
                           int64_t rows, const float* zt, const int64_t* y, int64_t ignore_index, int64_t V,
                           float* lse, float* row_loss, float* tcoef, unsigned* status, cudaStream_t s);
// loss = mean (or, with sum_reduction, sum) of the row losses of the valid rows.
cudaError_t launch_loss(const float* row_loss, int64_t N, const WsHeader* hdr, float* loss,
                        int64_t* n_valid_out, bool sum_reduction, cudaStream_t s);
cudaError_t launch_grad_b(const float* gb_part, int64_t parts, int64_t V, const WsHeader* hdr,
                          const float* label_csum, float* grad_b_acc, uint16_t* grad_b, int first,
                          int last, cudaStream_t s);
cudaError_t launch_wait_probe(unsigned* status, uint64_t limit_ns, cudaStream_t s);
cudaError_t launch_p_rescale(uint16_t* P, int64_t ldg, int64_t rows, int64_t V, const float* pm, int64_t ldp,
                             const float* lse, const int* crow, const int* n_valid, float* gb_part,
                             unsigned* status, cudaStream_t s);
cudaError_t launch_scale_grads(int64_t N, int64_t H, int64_t V, const float* d_grad_output, uint16_t* grad_X,
                               const float* grad_W_acc, uint16_t* grad_W, const float* grad_b_acc,
                               uint16_t* grad_b, cudaStream_t s);
cudaError_t launch_compact_rows(const int64_t* y, int64_t N, int64_t C, int64_t n_chunks, int64_t V,
                                int64_t ignore_index, int* dmap, int* crow, int* n_valid_chunk, cudaStream_t s);
cudaError_t launch_zero_ignored_rows(const int* dmap, int64_t N, int64_t H, uint16_t* grad_X, cudaStream_t s);
cudaError_t launch_gather_f16(const uint16_t* X_chunk, int64_t H, const int* crow, const int* n_valid,
                              int64_t max_rows, const unsigned* amax_bits, uint16_t* X16, uint16_t* P_tail,
                              int64_t ldg, unsigned* status, cudaStream_t s);
cudaError_t launch_gradx_split_reduce(const float* split_out, int64_t splits, int64_t split_stride, int64_t H,
                                      const int* crow, const int* n_valid, int64_t max_rows, const int64_t* y,
                                      int64_t ignore_index, int64_t V, const uint16_t* W, const float* tcoef,
                                      const WsHeader* hdr, uint16_t* grad_X_chunk, cudaStream_t s);
// Finishes the split tail tiles of one grad_X launch of the pair form (slots:
// its pairs; n_tiles, k_blocks: its tile columns and K extent; nw: 1 for
// 256-column tiles, 2 for 512).
cudaError_t launch_gradx_tail_reduce(const float* tail_out, int slots, int n_tiles, int k_blocks, int nw, int64_t H,
                                     const int* crow, const int* n_valid, int64_t max_rows, const int64_t* y,
                                     int64_t ignore_index, int64_t V, const uint16_t* W, const float* tcoef,
                                     const WsHeader* hdr, uint16_t* grad_X_chunk, cudaStream_t s);
cudaError_t launch_amax(const uint16_t* x, int64_t n, unsigned* amax_bits, cudaStream_t s);
cudaError_t launch_to_f16_scaled(const uint16_t* x, int64_t n, const unsigned* amax_bits, uint16_t* out,
                                 cudaStream_t s);

}  // namespace lce
