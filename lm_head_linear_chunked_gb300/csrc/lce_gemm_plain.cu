// Instantiations of the bare GEMM (fp32 output) for the three operand
// layouts; used by the diagnostic entry point lce_debug_gemm.
#include "lce_gemm.cuh"

namespace lce {

cudaError_t launch_gemm_plain(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b,
                              const GemmArgs& args, int grid, cudaStream_t stream) {
    switch (mode) {
        case MODE_PLAIN_KK: return launch_gemm_mode<MODE_PLAIN_KK>(map_a, map_b, args, grid, stream);
        case MODE_PLAIN_KM: return launch_gemm_mode<MODE_PLAIN_KM>(map_a, map_b, args, grid, stream);
        case MODE_PLAIN_MM: return launch_gemm_mode<MODE_PLAIN_MM>(map_a, map_b, args, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lce
