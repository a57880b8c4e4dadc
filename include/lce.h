/*
 * lce.h -- chunked linear cross-entropy on one GB300 GPU (sm_103a): C ABI.
 *
 * What is computed.  Hidden states X[N,H] times the LM-head weight W[V,H]
 * (the nn.Linear weight layout), plus an optional bias b[V], give logits
 * z[i,v] = sum_h X[i,h] W[v,h] + b[v].  Against labels y[N] the loss is
 *
 *     lse[i] = ln sum_v exp(z[i,v])
 *     loss   = (1 / n_valid) * sum over rows with y[i] != ignore_index
 *                                  of (lse[i] - z[i, y[i]])
 *
 * and the gradients, with s = grad_scale * grad_output / n_valid, are
 *
 *     G[i,v]  = s * (exp(z[i,v] - lse[i]) - [v == y[i]])   (0 for ignored rows)
 *     grad_X  = G W,   grad_W = G^T X,   grad_b = sum_i G[i,:]
 *
 * This is torch's cross_entropy(X W^T + b, y, ignore_index) with a mean over
 * valid rows, as the chunk-loss plugin of LlamaFactory PR #10762 uses it
 * (analysis page, section 4 "Chunk Loss 구현": per-chunk cross_entropy with
 * reduction="none" and ignore_index = IGNORE_INDEX = -100; grad_weight and
 * grad_bias accumulated in FP32 and cast back to the weight dtype), and with
 * the valid-token normalisation of the same page's section 3 (BaseTrainer).
 *
 * Rows are processed in chunks of at most `chunk_rows` rows ("maximum
 * flattened token rows per logits/CE chunk", same page, section 1 and 2);
 * the TRL page "1M 토큰 이상 학습", section "청킹", explains why rows split
 * cleanly.  The N x V logits never exist in memory: only per-chunk pieces do.
 *
 * Conventions for every entry point
 *  - Layouts: row-major, contiguous.  X [N,H], W [V,H], grad_X like X,
 *    grad_W and grad_W_acc like W, lse [N], y int64 [N] (torch.long).
 *    bf16 values are passed as their 16-bit patterns (lce_bf16).
 *  - Device pointers: every tensor argument is a device pointer unless
 *    stated otherwise, aligned to 16 bytes; `ws` is aligned to 256 bytes.
 *  - Sizes: N >= 1, V >= 1, H >= 64 with H % 64 == 0, V <= 2^31 - 1,
 *    N <= 2^31 - 1.  Other shapes return LCE_ERR_UNSUPPORTED.
 *  - chunk_rows: rows per chunk; 0 lets the library choose; < 0 is
 *    LCE_ERR_INVALID_ARG (the plugin rejects a non-positive chunk size).
 *  - Ownership: the caller allocates and owns every buffer, including the
 *    workspace `ws` of at least lce_workspace_size() bytes.  The library
 *    never allocates or frees device memory.
 *  - Streams: all work is enqueued on `stream` in order; no call
 *    synchronises except lce_check_status().
 *  - Errors found on the host (bad sizes, null or misaligned pointers, a
 *    short workspace) are returned before anything is enqueued.  Errors
 *    found on the device (a label outside [0,V) that is not ignore_index,
 *    a pipeline wait that timed out) are recorded in a status word inside
 *    `ws` and read back by lce_check_status(); the loss is then NaN and the
 *    other outputs are undefined.  No kernel traps.
 *  - n_valid == 0 gives loss = 0 and all-zero gradients (the trainer's
 *    guard against dividing by zero); lse is still written for every row,
 *    ignored rows included.
 *  - Results of lse and loss do not depend on chunk_rows (bit for bit);
 *    gradients depend on it only through the FP32 accumulation order.
 */
#ifndef LCE_H_
#define LCE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LCE_API __attribute__((visibility("default")))
#else
#define LCE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t lce_bf16;

/* A CUDA stream (cudaStream_t and CUstream convert to it implicitly). */
struct CUstream_st;
typedef struct CUstream_st* lce_stream_t;

typedef enum {
    LCE_OK = 0,
    LCE_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size or chunk_rows */
    LCE_ERR_UNSUPPORTED = 2,   /* shape outside the supported range (see above) */
    LCE_ERR_WORKSPACE = 3,     /* ws_bytes smaller than lce_workspace_size() */
    LCE_ERR_LABEL_RANGE = 4,   /* device: a label outside [0,V) and != ignore_index */
    LCE_ERR_TIMEOUT = 5,       /* device: a pipeline wait exceeded its time limit */
    LCE_ERR_CUDA = 6,          /* a CUDA runtime call or launch failed */
    LCE_ERR_BOUNDS = 7         /* device, bounds-checking build only: an index or TMA coordinate fell
                                  outside its buffer (the access was skipped) */
} lce_status_t;

/* Which entry point a workspace is sized for.  LCE_WS_FUSED is the size for
 * the fused call's fastest schedule: with chunks of at least 256 rows, no
 * bias and two or more chunks, it holds two chunks of the kept fp16
 * exponentials, so that each chunk's forward also turns the previous
 * chunk's into the softmax while its tensor cores work.  LCE_WS_FUSED_MIN
 * is the smallest workspace the fused call accepts; with less than the
 * LCE_WS_FUSED size it runs the two steps one after the other (same
 * results). */
enum { LCE_WS_FORWARD = 0, LCE_WS_BACKWARD = 1, LCE_WS_FUSED = 2, LCE_WS_FUSED_MIN = 3 };

/* Bytes of workspace the entry point `which` needs for this problem.
 * Host only; enqueues nothing.  Writes *bytes on LCE_OK. */
LCE_API lce_status_t lce_workspace_size(int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                                int has_bias, int which, size_t* bytes);

/* Rows per chunk the library uses for (N, H, V, chunk_rows).  Host only. */
LCE_API lce_status_t lce_chunk_rows(int64_t N, int64_t H, int64_t V, int64_t chunk_rows,
                            int64_t* rows_per_chunk);

/* Forward: loss [1] (float), lse [N] (float) and n_valid [1] (int64).
 * b may be NULL (no bias); n_valid may be NULL.
 * Cost: 2*N*H*V tensor-core FLOPs. */
LCE_API lce_status_t lce_forward(int64_t N, int64_t H, int64_t V,
                         const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                         const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                         float* loss, float* lse, int64_t* n_valid,
                         void* ws, size_t ws_bytes, lce_stream_t stream);

/* Backward from a forward's lse [N]: the logits are recomputed per chunk.
 * The gradient scale is grad_scale (host) times *d_grad_output (a device
 * float; NULL means 1), divided by n_valid.
 * grad_W_acc [V,H] float is required: it receives the FP32 accumulation
 * (overwritten, not added to).  grad_W [V,H] bf16 receives its
 * round-to-nearest-even cast and may be NULL.  grad_X [N,H] bf16 may be
 * NULL (then the grad_X product is skipped).  With a bias, grad_b_acc [V]
 * float and grad_b [V] bf16 follow the same rules (grad_b_acc required,
 * grad_b optional); without a bias both must be NULL.
 * Cost: 6*N*H*V tensor-core FLOPs (4 without grad_X). */
LCE_API lce_status_t lce_backward(int64_t N, int64_t H, int64_t V,
                          const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                          const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                          const float* lse, float grad_scale, const float* d_grad_output,
                          lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                          float* grad_W_acc, float* grad_b_acc,
                          void* ws, size_t ws_bytes, lce_stream_t stream);

/* Forward and backward in one call (the saved-gradient design of the
 * chunk-loss plugin): loss, lse, n_valid, and all gradients, with the same
 * rules as lce_forward and lce_backward.  The forward keeps each chunk's
 * exponentials 2^(z log2 e - tile max) (fp16) in the workspace and rescales
 * them to the softmax once lse is known, so the logits are not recomputed:
 * 6*N*H*V tensor-core FLOPs (forward logits, grad_X, grad_W), against the
 * 8*N*H*V of lce_forward followed by lce_backward. */
LCE_API lce_status_t lce_fused_fwd_bwd(int64_t N, int64_t H, int64_t V,
                               const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                               const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                               float grad_scale, const float* d_grad_output,
                               float* loss, float* lse, int64_t* n_valid,
                               lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                               float* grad_W_acc, float* grad_b_acc,
                               void* ws, size_t ws_bytes, lce_stream_t stream);

/* The same three calls with option flags (flags = 0 is the call above):
 *   LCE_REDUCTION_SUM: loss is the sum, not the mean, of the valid rows'
 *     cross-entropies, and the gradient scale is grad_scale * grad_output
 *     without the division by n_valid.  A trainer that normalises by a
 *     token count of its own (LlamaFactory PR #10762 analysis page, section
 *     3: the valid-token count gathered over all ranks and micro-batches)
 *     passes its 1/count as grad_scale.
 *   LCE_ACCUMULATE (backward and fused only): grad_W_acc and grad_b_acc
 *     hold a running FP32 total (gradient accumulation over micro-batches)
 *     and this call adds its gradients to them instead of overwriting
 *     them; grad_W and grad_b receive the cast of the new totals.  grad_X
 *     is written, as always.  The caller zeroes the accumulators before
 *     the first call of a total.
 * Unknown bits, or LCE_ACCUMULATE given to lce_forward_ex, return
 * LCE_ERR_INVALID_ARG before anything is enqueued. */
#define LCE_REDUCTION_SUM 1u
#define LCE_ACCUMULATE 2u
LCE_API lce_status_t lce_forward_ex(int64_t N, int64_t H, int64_t V,
                            const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                            const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                            float* loss, float* lse, int64_t* n_valid,
                            void* ws, size_t ws_bytes, lce_stream_t stream, uint32_t flags);
LCE_API lce_status_t lce_backward_ex(int64_t N, int64_t H, int64_t V,
                             const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                             const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                             const float* lse, float grad_scale, const float* d_grad_output,
                             lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                             float* grad_W_acc, float* grad_b_acc,
                             void* ws, size_t ws_bytes, lce_stream_t stream, uint32_t flags);
LCE_API lce_status_t lce_fused_fwd_bwd_ex(int64_t N, int64_t H, int64_t V,
                                  const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                                  const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                                  float grad_scale, const float* d_grad_output,
                                  float* loss, float* lse, int64_t* n_valid,
                                  lce_bf16* grad_X, lce_bf16* grad_W, lce_bf16* grad_b,
                                  float* grad_W_acc, float* grad_b_acc,
                                  void* ws, size_t ws_bytes, lce_stream_t stream, uint32_t flags);

/* The backward of the chunk-loss plugin's saved-gradient design (LlamaFactory
 * PR #10762 analysis page, section 4: the Function computes the gradients in
 * its forward, and its backward scales them by grad_output).  After an
 * lce_fused_fwd_bwd call with grad_scale 1 and no grad_output, with
 * g = *d_grad_output (a device float):
 *   grad_X <- bf16(g * grad_X) in place (may be NULL),
 *   grad_W <- bf16(g * grad_W_acc), grad_b <- bf16(g * grad_b_acc)
 * (each output and its accumulator both given or both NULL; the fp32
 * accumulators are not changed).  Device pointers, 16-byte aligned,
 * H % 8 == 0.  Enqueued on `stream`. */
LCE_API lce_status_t lce_scale_grads(int64_t N, int64_t H, int64_t V, const float* d_grad_output,
                             lce_bf16* grad_X, const float* grad_W_acc, lce_bf16* grad_W,
                             const float* grad_b_acc, lce_bf16* grad_b, lce_stream_t stream);

/* Synchronises `stream`, then returns the device status of the last call
 * that used workspace `ws` (LCE_OK, LCE_ERR_LABEL_RANGE, LCE_ERR_TIMEOUT,
 * or LCE_ERR_BOUNDS from the bounds-checking build), or LCE_ERR_CUDA if the
 * stream reported an error.  A call that found an error on the device also
 * writes NaN to its loss.
 *
 * Bounds-checking build.  The same sources compiled with LCE_DEBUG give
 * liblce_debug.so, with the same entry points: there every kernel checks
 * the indices it computes (row maps, sorted label keys, chunk rows, partial
 * and workspace offsets) and the coordinates of its TMA stores against the
 * buffers they address, and a check that fails skips the access and
 * raises LCE_ERR_BOUNDS instead of touching memory outside the buffer.  The
 * release library compiles these checks out. */
LCE_API lce_status_t lce_check_status(const void* ws, lce_stream_t stream);

/* Static, human-readable name of a status code. */
LCE_API const char* lce_status_string(lce_status_t status);

/* ---- diagnostics (used by the tests; not part of the loss) -------------
 *
 * lce_debug_gemm: the library's tensor-core GEMM core alone, FP32 output
 * D [M,N] (row-major) from bf16 operands, for the three operand layouts
 * the loss uses:
 *   layout 0: A [M,K], B [N,K]   D = A B^T   (logits:  X_c W^T)
 *   layout 1: A [M,K], B [K,N]   D = A B     (grad_X:  G W)
 *   layout 2: A [K,M], B [K,N]   D = A^T B   (grad_W:  G^T X_c)
 * M, N, K >= 1 and multiples of 8.  ws >= 256 bytes holds the status word.
 *
 * lce_debug_wait_timeout: one block waits on a pipeline barrier that is
 * never signalled, through the same bounded wait as the GEMM pipeline,
 * with a limit of `limit_us` microseconds; the status word in `ws`
 * (>= 256 bytes) then reads LCE_ERR_TIMEOUT.  Shows that a stuck pipeline
 * ends with an error status instead of a hang.
 *
 * lce_debug_gradx_tail_plan: how the pair form splits the last partial
 * round of a grad_X launch over K.  For `tiles` output tiles of 256 rows x
 * `tile_cols` columns (256, or 512 where H is a multiple of 512) with valid
 * rows, `slots` pairs and a K extent of `k_blocks` blocks of 64, writes
 * out[0] = tiles computed whole, out[1] = tiles split after them (0: no
 * split), out[2] = K slices per split tile, out[3] = k-blocks per slice.
 * Host-only; returns LCE_ERR_INVALID_ARG for a null `out`, a negative or
 * out-of-range count, or another tile width. */
LCE_API lce_status_t lce_debug_gemm(int layout, int64_t M, int64_t N, int64_t K,
                            const lce_bf16* A, const lce_bf16* B, float* D,
                            void* ws, size_t ws_bytes, lce_stream_t stream);

LCE_API lce_status_t lce_debug_wait_timeout(uint32_t limit_us, void* ws, size_t ws_bytes,
                                    lce_stream_t stream);

LCE_API lce_status_t lce_debug_gradx_tail_plan(int64_t tiles, int64_t slots, int64_t k_blocks,
                                       int64_t tile_cols, int64_t out[4]);

/* lce_forward without a caller-provided workspace, for callers that cannot
 * allocate device memory: for example a hook running inside a framework
 * whose allocator owns all of the device's memory, or a C client that links
 * only this library and has no allocator of its own.  (The pages have no
 * counterpart: their plugin lets PyTorch allocate.)
 * Arguments and results are those of lce_forward.  The scratch is one
 * fixed array of LCE_STATIC_SCRATCH_BYTES (32 MiB) in the library's device
 * memory, reserved on every GPU that loads the library until the process
 * exits; this call allocates nothing (no cudaMalloc, no cudaFree).
 * Limits: the forward workspace (lce_workspace_size with LCE_WS_FORWARD)
 * must fit the array.  With chunk_rows == 0 the largest chunk that fits
 * is used (at most 8192 rows); a given chunk_rows whose workspace does not
 * fit, or a problem that does not fit even with one-row chunks (e.g. N
 * above about eight million rows), returns LCE_ERR_WORKSPACE before
 * anything is enqueued.
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress), so make that first call before
 * any stream capture.  Every call on a device uses the same array and
 * leaves its contents behind: calls whose work may overlap on the GPU
 * (different streams, or different host threads) race on it, so issue
 * them in one stream order.  Errors found on the device (a label outside
 * [0, V) that is not ignore_index, a timed-out wait) make the loss NaN;
 * lce_static_ws_check_status() reads their status. */
#define LCE_STATIC_SCRATCH_BYTES (32u << 20)
LCE_API lce_status_t lce_forward_static_ws(int64_t N, int64_t H, int64_t V,
                                   const lce_bf16* X, const lce_bf16* W, const lce_bf16* b,
                                   const int64_t* y, int64_t ignore_index, int64_t chunk_rows,
                                   float* loss, float* lse, int64_t* n_valid,
                                   lce_stream_t stream);

/* The device status of the last lce_forward_static_ws call on the current
 * device, like lce_check_status() for a caller's workspace: synchronises
 * `stream` (the stream of that call), then returns LCE_OK,
 * LCE_ERR_LABEL_RANGE or LCE_ERR_TIMEOUT, or LCE_ERR_CUDA if the stream
 * reported an error.  Allocates nothing. */
LCE_API lce_status_t lce_static_ws_check_status(lce_stream_t stream);

/* lce_set_gemm_form: the tensor-core GEMM form of the calls this process
 * makes after it (each call reads the setting once, when it is made).
 * The default is LCE_GEMM_PAIR.
 *   LCE_GEMM_SINGLE: one CTA per SM computes 128x256 output tiles with
 *     tcgen05.mma cta_group::1 and a 4-stage ring of 48 KB slices.
 *   LCE_GEMM_PAIR: a cluster of two CTAs on neighbouring SMs computes
 *     256x256 tiles with one tcgen05.mma of M = 256 (cta_group::2); each
 *     SM loads its own half of B, so a 64-wide K slice brings 32 KB into
 *     each SM instead of 48 KB, and the ring is 6 stages deep.  grad_X
 *     uses 256x512 tiles where H is a multiple of 512, and splits the tiles
 *     of its last, partly filled round over the vocabulary.  On a device
 *     that cannot keep any cluster of two resident, calls use SINGLE.
 * The products are the ones the documentation of each entry point states
 * in either form.  The forms may differ in the last bits of FP32 sums;
 * each form is deterministic on a given device (grad_X's split depends on
 * the device's number of pairs).  The workspace does not depend on the
 * form.
 * Returns the previous form, or -1 for an unknown value (nothing changes).
 * Host-only; safe to call from any thread. */
#define LCE_GEMM_SINGLE 0
#define LCE_GEMM_PAIR 1
LCE_API int lce_set_gemm_form(int form);

/* lce_gemm_pair_slots: how many CTA pairs of the pair form the current
 * device keeps resident at once (one per two SMs when every pair fits);
 * 0 when the pair form cannot run there (calls then use SINGLE) or no
 * device is usable. */
LCE_API int lce_gemm_pair_slots(void);

/* Per-kernel device time, for benchmarks.  Between lce_profile_begin() and
 * lce_profile_end(), every kernel the library enqueues is bracketed by two
 * CUDA events recorded on the call's own stream (events are created on
 * first use and kept; no device memory is allocated).  lce_profile_end()
 * waits for those events and writes, for each kind k < LCE_PROFILE_KINDS,
 * the summed milliseconds ms[k] and the number of launches launches[k]:
 *   0 forward logits + logsumexp     1 recomputed logits -> softmax P
 *   2 grad_X product                 3 grad_W product                (lce_backward)
 *   4 all other (label checks, combine, softmax rescale, conversions,
 *     one-hot part, loss)
 * Process-wide state: not for concurrent use from several threads. */
#define LCE_PROFILE_KINDS 5
LCE_API lce_status_t lce_profile_begin(void);
LCE_API lce_status_t lce_profile_end(double* ms, int64_t* launches);

#ifdef __cplusplus
}
#endif

#endif /* LCE_H_ */
