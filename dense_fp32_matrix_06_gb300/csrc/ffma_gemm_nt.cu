// ffma_gemm_nt.cu -- instantiates the fp32 CUDA-core GEMM for
// op(A) = A, op(B) = B^T (kernel template in ffma_kernel.cuh).
#include "ffma_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_nt(const GemmArgs &a, int tile, bool vec, bool edge,
                           cudaStream_t stream) {
    return tile == kSmallTile
               ? ffma::launch_layout<kSmallTile, false, false, true, true>(a, vec, edge, stream)
               : ffma::launch_layout<128, false, false, true, true>(a, vec, edge, stream);
}

}  // namespace sgemm_impl
