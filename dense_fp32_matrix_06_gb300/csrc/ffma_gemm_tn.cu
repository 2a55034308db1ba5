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
// operands are row copies, so the slice is not tied to the tile).  Measured
// on GB300 against K slices of 16: 8192^3 65.2 against 63.6 TFLOP/s for the
// product alone.
template <bool kExt>
cudaError_t launch_tn_wide(const GemmArgs &a, bool vec, bool edge, cudaStream_t stream) {
    const bool split = a.split_k > 1;
    if (!edge)
        return split ? ffma::launch_variant<128, false, true, false, true, true, false, kExt,
                                            kWideBK>(a, stream)
                     : ffma::launch_variant<128, false, true, false, false, true, false, kExt,
                                            kWideBK>(a, stream);
    if (vec)
        return split ? ffma::launch_variant<128, false, true, true, true, true, false, kExt,
                                            kWideBK>(a, stream)
                     : ffma::launch_variant<128, false, true, true, false, true, false, kExt,
                                            kWideBK>(a, stream);
    return split ? ffma::launch_variant<128, false, false, true, true, true, false, kExt,
                                        kWideBK>(a, stream)
                 : ffma::launch_variant<128, false, false, true, false, true, false, kExt,
                                        kWideBK>(a, stream);
}

cudaError_t launch_ffma_tn_wide(const GemmArgs &a, bool vec, bool edge, bool ext,
                                cudaStream_t stream) {
    return ext ? launch_tn_wide<true>(a, vec, edge, stream)
               : launch_tn_wide<false>(a, vec, edge, stream);
}

// The same kernel scheduled as a persistent stream-K launch (kSched = 1).
template <bool kExt>
cudaError_t launch_tn_wide_sk(const GemmArgs &a, int64_t grid, bool vec, bool edge,
                              cudaStream_t stream) {
    if (!edge)
        return ffma::launch_variant<128, false, true, false, false, true, false, kExt, kWideBK, 1>(
            a, stream, grid);
    if (vec)
        return ffma::launch_variant<128, false, true, true, false, true, false, kExt, kWideBK, 1>(
            a, stream, grid);
    return ffma::launch_variant<128, false, false, true, false, true, false, kExt, kWideBK, 1>(
        a, stream, grid);
}

cudaError_t launch_ffma_tn_wide_sk(const GemmArgs &a, int64_t grid, bool vec, bool edge, bool ext,
                                   cudaStream_t stream) {
    return ext ? launch_tn_wide_sk<true>(a, grid, vec, edge, stream)
               : launch_tn_wide_sk<false>(a, grid, vec, edge, stream);
}

}  // namespace sgemm_impl
