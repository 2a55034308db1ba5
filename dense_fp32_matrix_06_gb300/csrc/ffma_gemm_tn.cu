// ffma_gemm_tn.cu -- instantiates the fp32 CUDA-core GEMM for
// op(A) = A^T, op(B) = B (kernel template in ffma_kernel.cuh).
#include "ffma_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_tn(const GemmArgs &a, int tile, bool vec, bool edge,
                           cudaStream_t stream) {
    return tile == kSmallTile
               ? ffma::launch_layout<kSmallTile, false, true, false, true>(a, vec, edge, stream)
               : ffma::launch_layout<128, false, true, false, true>(a, vec, edge, stream);
}

}  // namespace sgemm_impl
