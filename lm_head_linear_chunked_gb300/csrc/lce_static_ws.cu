// lce_forward_static_ws: the forward pass for callers that cannot allocate
// device memory.  Its scratch space is a fixed array in the library's own
// device memory instead of a caller-provided workspace.
#include <mutex>

#include "lce_internal.cuh"

namespace {

// The scratch of every lce_forward_static_ws call on this device.  Each GPU
// that loads the library holds these bytes until the process exits.
static __device__ __align__(256) unsigned char lce_static_scratch[LCE_STATIC_SCRATCH_BYTES];

std::mutex g_mu;
void* g_scratch[64];  // device address of lce_static_scratch, per device ordinal

// Set-up, once per device and with that device current: the array's name
// is only a host-side stand-in, so ask the runtime for its device address.
lce_status_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return LCE_ERR_CUDA;
    std::lock_guard<std::mutex> g(g_mu);
    if (!g_scratch[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, lce_static_scratch) != cudaSuccess || !p) return LCE_ERR_CUDA;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return LCE_OK;
}

// Rows per chunk: the caller's choice if its workspace fits the array, else
// (for chunk_rows == 0) the largest chunk whose workspace fits.
lce_status_t pick_chunk(int64_t N, int64_t H, int64_t V, int64_t chunk_rows, int has_bias, int64_t* out) {
    size_t need = 0;
    lce_status_t st = lce_workspace_size(N, H, V, chunk_rows, has_bias, LCE_WS_FORWARD, &need);
    if (st != LCE_OK) return st;
    if (need <= LCE_STATIC_SCRATCH_BYTES) {
        *out = chunk_rows;
        return LCE_OK;
    }
    if (chunk_rows != 0) return LCE_ERR_WORKSPACE;
    int64_t lo = 1, hi = N < 8192 ? N : 8192, best = 0;
    while (lo <= hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        st = lce_workspace_size(N, H, V, mid, has_bias, LCE_WS_FORWARD, &need);
        if (st != LCE_OK) return st;
        if (need <= LCE_STATIC_SCRATCH_BYTES) {
            best = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    if (best == 0) return LCE_ERR_WORKSPACE;
    *out = best >= 128 ? best / 128 * 128 : best;
    return LCE_OK;
}

}  // namespace

extern "C" lce_status_t lce_forward_static_ws(int64_t N, int64_t H, int64_t V, const lce_bf16* X,
                                              const lce_bf16* W, const lce_bf16* b, const int64_t* y,
                                              int64_t ignore_index, int64_t chunk_rows, float* loss, float* lse,
                                              int64_t* n_valid, lce_stream_t stream) {
    if (chunk_rows < 0) return LCE_ERR_INVALID_ARG;
    int64_t rows = 0;
    lce_status_t st = pick_chunk(N, H, V, chunk_rows, b != nullptr, &rows);
    if (st != LCE_OK) return st;
    void* scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != LCE_OK) return st;
    // lce_forward clears the status word and the valid-row count at the start
    // of every call.  The other scratch it reads (per-row partials and target
    // logits) is written earlier in the same call unless the call finds an
    // error on the device: a label outside [0, V) gets a NaN row loss without
    // reading a target logit, and any device error makes the loss NaN and
    // shows in lce_static_ws_check_status.
    return lce_forward(N, H, V, X, W, b, y, ignore_index, rows, loss, lse, n_valid, scratch,
                       LCE_STATIC_SCRATCH_BYTES, stream);
}

extern "C" lce_status_t lce_static_ws_check_status(lce_stream_t stream) {
    void* scratch = nullptr;
    const lce_status_t st = scratch_address(&scratch);
    if (st != LCE_OK) return st;
    return lce_check_status(scratch, stream);
}
