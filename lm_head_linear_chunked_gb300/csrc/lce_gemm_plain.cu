// Instantiations of the bare GEMM (fp32 output) for the three operand
// layouts; used by the diagnostic entry point lce_debug_gemm.
#include "lce_gemm_pair.cuh"

namespace lce {

cudaError_t launch_gemm_plain(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                              const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    switch (mode) {
        case MODE_PLAIN_KK: return launch_gemm_mode<MODE_PLAIN_KK>(map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_PLAIN_KM: return launch_gemm_mode<MODE_PLAIN_KM>(map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_PLAIN_MM: return launch_gemm_mode<MODE_PLAIN_MM>(map_a, map_b, map_c, args, grid, stream, pair);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lce

namespace lce {

int gemm_pair_slots() {
    static std::atomic<int> cached[64];  // pairs + 1; 0 = not yet asked
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int c = cached[dev].load(std::memory_order_relaxed);
    if (c) return c - 1;
    int n = 0, sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && sms >= 2 &&
        cudaFuncSetAttribute(gemm_pair_kernel<MODE_PLAIN_KK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             GEMM_PAIR_SMEM_BYTES) == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(sms / 2 * 2), 1, 1);
        cfg.blockDim = dim3(GEMM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = GEMM_PAIR_SMEM_BYTES;
        if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<MODE_PLAIN_KK>, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();  // a refused query leaves no sticky error behind
    cached[dev].store(n + 1, std::memory_order_relaxed);
    return n;
}

}  // namespace lce
