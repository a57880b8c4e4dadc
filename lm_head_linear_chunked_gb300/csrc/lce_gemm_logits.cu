// Instantiations of the GEMM for the two logits passes (X_c W^T): the
// forward logsumexp epilogue and the backward softmax-minus-onehot epilogue.
#include "lce_gemm_pair.cuh"

namespace lce {

cudaError_t launch_gemm_logits(int mode, const CUtensorMap& map_a, const CUtensorMap& map_b, const CUtensorMap& map_c,
                               const GemmArgs& args, int grid, cudaStream_t stream, bool pair) {
    switch (mode) {
        case MODE_LSE: return launch_gemm_mode<MODE_LSE>(map_a, map_b, map_c, args, grid, stream, pair);
        case MODE_G: return launch_gemm_mode<MODE_G>(map_a, map_b, map_c, args, grid, stream, pair);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace lce
