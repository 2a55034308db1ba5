// ffma_sk_tn.cu -- instantiates the stream-K fp32 GEMM (ffma_sk_kernel.cuh)
// for op(A) = A^T, op(B) = B, with and without the batch/bias/activation
// code: the plain product after A has been transposed once, and sgemm_ex's
// transposed-A form.
#include "ffma_sk_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_sk_tn(const SkArgs &a, int tile, int bk, int pages, bool vec, bool ext,
                              cudaStream_t stream) {
    if (ext)
        return vec ? sk::launch_sk_tile<true, false, true, true>(a, tile, bk, pages, stream)
                   : sk::launch_sk_tile<true, false, false, true>(a, tile, bk, pages, stream);
    return vec ? sk::launch_sk_tile<true, false, true, false>(a, tile, bk, pages, stream)
               : sk::launch_sk_tile<true, false, false, false>(a, tile, bk, pages, stream);
}

}  // namespace sgemm_impl
