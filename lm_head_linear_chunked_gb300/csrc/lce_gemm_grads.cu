// Instantiations of the GEMM for the two gradient products: grad_X = s G' W
// and grad_W += s G'^T X_c.
#include "lce_gemm_pair.cuh"

namespace lce {

cudaError_t launch_gemm_grads(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                              const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    switch (mode) {
        case MODE_GRADX: return launch_gemm_mode<MODE_GRADX>(map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_GRADW: return launch_gemm_mode<MODE_GRADW>(map_a, map_b, map_c, args, grid, stream, pair);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lce
