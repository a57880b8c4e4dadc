// Instantiation of the pair-form GEMM for grad_X with 512-column output
// tiles (MODE_GRADX_W), in a translation unit of its own so that it compiles
// in parallel with the others.
#include "lce_gemm_pair.cuh"

namespace lce {

cudaError_t launch_gemm_gradx_wide(const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                                   const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    return launch_gemm_mode<MODE_GRADX_W>(map_a, map_b, map_c, args, grid, stream, pair);
}

}  // namespace lce
