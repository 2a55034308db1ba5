// ffma_gemm_tn_packed.cu -- the op(A) = A^T, op(B) = B product (after A has
// been transposed into the workspace) with its FMAs issued packed
// (fma.rn.f32x2: each lane one round-to-nearest fp32 FMA, the same order, so
// the same C bit for bit as the scalar build in ffma_gemm_tn.cu).  Plain
// products only (no batch, bias or activation); one CTA per (tile, K range),
// or the persistent stream-K schedule.  Kept in its own translation unit so
// the builds run in parallel.
#include "ffma_kernel.cuh"

namespace sgemm_impl {

cudaError_t launch_ffma_tn_wide_packed(const GemmArgs &a, bool vec, bool edge,
                                       cudaStream_t stream) {
    const bool split = a.split_k > 1;
    if (!edge)
        return split ? ffma::launch_variant<128, true, true, false, true, true, false, false,
                                            kWideBK>(a, stream)
                     : ffma::launch_variant<128, true, true, false, false, true, false, false,
                                            kWideBK>(a, stream);
    if (vec)
        return split ? ffma::launch_variant<128, true, true, true, true, true, false, false,
                                            kWideBK>(a, stream)
                     : ffma::launch_variant<128, true, true, true, false, true, false, false,
                                            kWideBK>(a, stream);
    return split ? ffma::launch_variant<128, true, false, true, true, true, false, false,
                                        kWideBK>(a, stream)
                 : ffma::launch_variant<128, true, false, true, false, true, false, false,
                                        kWideBK>(a, stream);
}

cudaError_t launch_ffma_tn_wide_sk_packed(const GemmArgs &a, int64_t grid, bool vec, bool edge,
                                          cudaStream_t stream) {
    if (!edge)
        return ffma::launch_variant<128, true, true, false, false, true, false, false, kWideBK, 1>(
            a, stream, grid);
    if (vec)
        return ffma::launch_variant<128, true, true, true, false, true, false, false, kWideBK, 1>(
            a, stream, grid);
    return ffma::launch_variant<128, true, false, true, false, true, false, false, kWideBK, 1>(
        a, stream, grid);
}

}  // namespace sgemm_impl
