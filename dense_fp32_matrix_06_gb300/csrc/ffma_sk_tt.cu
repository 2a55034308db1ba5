// ffma_sk_tt.cu -- instantiates the stream-K fp32 GEMM (ffma_sk_kernel.cuh)
// for op(A) = A^T, op(B) = B^T (batch/bias/activation code compiled in).
#include "ffma_sk_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_sk_tt(const SkArgs &a, int tile, int bk, int pages, bool vec,
                              cudaStream_t stream) {
    return vec ? sk::launch_sk_tile<true, true, true, true>(a, tile, bk, pages, stream)
               : sk::launch_sk_tile<true, true, false, true>(a, tile, bk, pages, stream);
}

}  // namespace sgemm_impl
