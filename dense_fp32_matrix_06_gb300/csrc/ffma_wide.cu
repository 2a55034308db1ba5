// ffma_wide.cu -- instantiates the 16 x 8 per-thread fp32 GEMM kernel
// (ffma_wide_kernel.cuh) for the plans that copy both operands directly.
#include "ffma_wide_kernel.cuh"

namespace sgemm_impl {
namespace {

template <bool kEdge, bool kExt>
cudaError_t launch_16x8(const GemmArgs &a, cudaStream_t stream) {
    auto kernel = wide::ffma16x8_kernel<kEdge, kExt>;
    static bool configured[64];
    const cudaError_t e =
        set_smem_once(reinterpret_cast<const void *>(kernel), wide::kSmemBytes, configured, true);
    if (e != cudaSuccess) return e;
    const int64_t tiles = int64_t(a.tiles_m) * a.tiles_n * a.batch;
    kernel<<<unsigned(tiles), wide::kThreads, wide::kSmemBytes, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ffma16x8(const GemmArgs &a, bool edge, bool ext, cudaStream_t stream) {
    if (a.split_k != 1 || a.tail_split != 1) return cudaErrorInvalidValue;
    if (ext) return edge ? launch_16x8<true, true>(a, stream) : launch_16x8<false, true>(a, stream);
    return edge ? launch_16x8<true, false>(a, stream) : launch_16x8<false, false>(a, stream);
}

}  // namespace sgemm_impl
