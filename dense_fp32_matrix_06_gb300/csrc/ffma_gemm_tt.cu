// ffma_gemm_tt.cu -- instantiates the fp32 CUDA-core GEMM for
// op(A) = A^T, op(B) = B^T (kernel template in ffma_kernel.cuh).
#include "ffma_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_tt(const GemmArgs &a, bool vec, bool edge, cudaStream_t stream) {
    return ffma::launch_layout<false, true, true, true>(a, vec, edge, stream);
}

}  // namespace sgemm_impl
