// ffma_sk_nn.cu -- instantiates the stream-K fp32 GEMM (ffma_sk_kernel.cuh)
// for op(A) = A, op(B) = B, with and without the batch/bias/activation code,
// and dispatches every layout.
#include "ffma_sk_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_sk_nn(const SkArgs &a, int tile, int bk, int pages, bool vec, bool ext,
                              cudaStream_t stream) {
    if (ext)
        return vec ? sk::launch_sk_tile<false, false, true, true>(a, tile, bk, pages, stream)
                   : sk::launch_sk_tile<false, false, false, true>(a, tile, bk, pages, stream);
    return vec ? sk::launch_sk_tile<false, false, true, false>(a, tile, bk, pages, stream)
               : sk::launch_sk_tile<false, false, false, false>(a, tile, bk, pages, stream);
}

cudaError_t launch_ffma_sk(const SkArgs &a, int tile, int bk, int pages, bool vec, bool trans_a,
                           bool trans_b, bool ext, cudaStream_t stream) {
    if (trans_a) return trans_b ? launch_ffma_sk_tt(a, tile, bk, pages, vec, stream)
                                : launch_ffma_sk_tn(a, tile, bk, pages, vec, ext, stream);
    if (trans_b) return launch_ffma_sk_nt(a, tile, bk, pages, vec, stream);
    return launch_ffma_sk_nn(a, tile, bk, pages, vec, ext, stream);
}

}  // namespace sgemm_impl
