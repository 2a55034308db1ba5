// ffma_gemm_tn_packed.cu -- the op(A) = A^T, op(B) = B product (after A has
// been transposed into the workspace) with its FMAs issued packed
// (fma.rn.f32x2: each lane one round-to-nearest fp32 FMA, the same order, so
// the same C bit for bit as the scalar build in ffma_gemm_tn.cu).  One CTA
// per (tile, K range) -- plain, or with batches, bias and GELU (sgemm_ex) --
// or, for plain products, the persistent stream-K schedule; `pdl` as for
// the scalar build (ffma_gemm_tn.cu).  Kept in its own translation unit so
// the builds run in parallel.
#include "ffma_kernel.cuh"

namespace sgemm_impl {
namespace {

template <bool kExt>
cudaError_t tn_wide_packed(const GemmArgs &a, bool vec, bool edge, bool pdl, cudaStream_t stream) {
    const bool split = a.split_k > 1;
    if (!edge)
        return split ? ffma::launch_variant<128, true, true, false, true, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl)
                     : ffma::launch_variant<128, true, true, false, false, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl);
    if (vec)
        return split ? ffma::launch_variant<128, true, true, true, true, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl)
                     : ffma::launch_variant<128, true, true, true, false, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl);
    return split ? ffma::launch_variant<128, true, false, true, true, true, false, kExt,
                                        kWideBK>(a, stream, 0, pdl)
                 : ffma::launch_variant<128, true, false, true, false, true, false, kExt,
                                        kWideBK>(a, stream, 0, pdl);
}

}  // namespace

cudaError_t launch_ffma_tn_wide_packed(const GemmArgs &a, bool vec, bool edge, bool ext,
                                       bool pdl, cudaStream_t stream) {
    return ext ? tn_wide_packed<true>(a, vec, edge, pdl, stream)
               : tn_wide_packed<false>(a, vec, edge, pdl, stream);
}

cudaError_t launch_ffma_tn_wide_sk_packed(const GemmArgs &a, int64_t grid, bool vec, bool edge,
                                          bool pdl, cudaStream_t stream) {
    if (!edge)
        return ffma::launch_variant<128, true, true, false, false, true, false, false, kWideBK, 1>(
            a, stream, grid, pdl);
    if (vec)
        return ffma::launch_variant<128, true, true, true, false, true, false, false, kWideBK, 1>(
            a, stream, grid, pdl);
    return ffma::launch_variant<128, true, false, true, false, true, false, false, kWideBK, 1>(
        a, stream, grid, pdl);
}

}  // namespace sgemm_impl
