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

// The product after A (and, for sgemm_ex, B^T) has been transposed into the
// workspace: no extension code unless asked for, K slices of 32 (both
// operands are row copies, so the slice is not tied to the tile).  With
// `pdl` it is launched as a programmatic dependent of the kernel before it
// (the transpose pass): its CTAs may start while that grid drains, and wait
// for it before reading.  Measured on GB300 that saves about 2 us a call
// (MLP-down 97.9 -> 95.9, 2048^3 316 -> 314 us) where the grid has more CTAs
// than SMs; on smaller grids the early CTAs land two to an SM on the SMs the
// transpose has left, instead of one to every SM (GPT-2 QKV, 144 CTAs: 72 ->
// 124 us), so the planner asks for it only above one CTA per SM.  Measured
// on GB300 against K slices of 16: 8192^3 65.2 against 63.6 TFLOP/s for the
// product alone.
template <bool kExt>
cudaError_t launch_tn_wide(const GemmArgs &a, bool vec, bool edge, bool pdl, cudaStream_t stream) {
    const bool split = a.split_k > 1;
    if (!edge)
        return split ? ffma::launch_variant<128, false, true, false, true, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl)
                     : ffma::launch_variant<128, false, true, false, false, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl);
    if (vec)
        return split ? ffma::launch_variant<128, false, true, true, true, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl)
                     : ffma::launch_variant<128, false, true, true, false, true, false, kExt,
                                            kWideBK>(a, stream, 0, pdl);
    return split ? ffma::launch_variant<128, false, false, true, true, true, false, kExt,
                                        kWideBK>(a, stream, 0, pdl)
                 : ffma::launch_variant<128, false, false, true, false, true, false, kExt,
                                        kWideBK>(a, stream, 0, pdl);
}

cudaError_t launch_ffma_tn_wide(const GemmArgs &a, bool vec, bool edge, bool ext, bool pdl,
                                cudaStream_t stream) {
    return ext ? launch_tn_wide<true>(a, vec, edge, pdl, stream)
               : launch_tn_wide<false>(a, vec, edge, pdl, stream);
}

// The same kernel scheduled as a persistent stream-K launch (kSched = 1).
template <bool kExt>
cudaError_t launch_tn_wide_sk(const GemmArgs &a, int64_t grid, bool vec, bool edge, bool pdl,
                              cudaStream_t stream) {
    if (!edge)
        return ffma::launch_variant<128, false, true, false, false, true, false, kExt, kWideBK, 1>(
            a, stream, grid, pdl);
    if (vec)
        return ffma::launch_variant<128, false, true, true, false, true, false, kExt, kWideBK, 1>(
            a, stream, grid, pdl);
    return ffma::launch_variant<128, false, false, true, false, true, false, kExt, kWideBK, 1>(
        a, stream, grid, pdl);
}

cudaError_t launch_ffma_tn_wide_sk(const GemmArgs &a, int64_t grid, bool vec, bool edge, bool ext,
                                   bool pdl, cudaStream_t stream) {
    return ext ? launch_tn_wide_sk<true>(a, grid, vec, edge, pdl, stream)
               : launch_tn_wide_sk<false>(a, grid, vec, edge, pdl, stream);
}

}  // namespace sgemm_impl
