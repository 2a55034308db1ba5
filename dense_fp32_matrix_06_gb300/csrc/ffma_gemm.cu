// ffma_gemm.cu -- the fp32 CUDA-core GEMM (kernel template in ffma_kernel.cuh):
// the plain layout (op(A) = A, op(B) = B) in both issue forms, the dispatch
// over layouts, and the small helper kernels (C = beta*C, the FMA-rate probe).
#include <cuda_runtime.h>

#include <cstdint>

#include "ffma_kernel.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

// C = beta * C over the logical M x N part (beta == 0 stores zeros without
// reading C).  Used for K == 0 and alpha == 0.
__global__ void scale_kernel(float *C, int64_t M, int64_t N, int64_t ldc, float beta) {
    const int64_t total = M * N;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t i = e / N, j = e - i * N;
        float *c = C + i * ldc + j;
        *c = (beta == 0.0f) ? 0.0f : beta * *c;
    }
}

// At[k * ldt + m] = A[m * lda + k] for the first K columns of the first M
// rows: 32 x 32 tiles through padded shared memory, so both the reads (along
// k) and the writes (along m) are coalesced.  Feeds the product that reads A
// one k-row at a time (see the planner's transpose_a).
__global__ void transpose_kernel(const float *__restrict__ A, int64_t M, int64_t K, int64_t lda,
                                 float *__restrict__ At, int64_t ldt, int64_t stride_a,
                                 int64_t stride_t) {
    __shared__ float tile[32][33];
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");   // as transpose64_kernel
    A += int64_t(blockIdx.z) * stride_a;    // batch z
    At += int64_t(blockIdx.z) * stride_t;
    const int64_t m0 = int64_t(blockIdx.y) * 32, k0 = int64_t(blockIdx.x) * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
    for (int i = ty; i < 32; i += 8) {
        const int64_t m = m0 + i, k = k0 + tx;
        tile[i][tx] = (m < M && k < K) ? A[m * lda + k] : 0.0f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int64_t k = k0 + i, m = m0 + tx;
        if (k < K && m < M) At[k * ldt + m] = tile[tx][i];
    }
}

// The same with 64 x 64 tiles and 128-bit global accesses (A and At 16-byte
// aligned, lda and ldt multiples of 4, ldt covering M rounded up to 4): each
// of 256 threads loads four float4 along k and stores four float4 along m.
// The shared tile is padded by one float per row; the column reads of the
// store phase then see at most two-way bank conflicts.
// kVecLoad: A's rows start on 16 bytes (lda and stride_a multiples of 4, A
// aligned), so each thread reads its 4 columns with one 128-bit load;
// otherwise with 4 scalar loads (coalesced across the warp all the same).
template <bool kVecLoad>
__global__ void __launch_bounds__(256) transpose64_kernel(const float *__restrict__ A, int64_t M,
                                                          int64_t K, int64_t lda,
                                                          float *__restrict__ At, int64_t ldt,
                                                          int64_t stride_a, int64_t stride_t) {
    __shared__ float tile[64][65];
    // the product that reads A^T is launched as a programmatic dependent: its
    // CTAs may be scheduled once every CTA of this grid has started (they wait
    // for this grid's completion before reading)
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    A += int64_t(blockIdx.z) * stride_a;    // batch z
    At += int64_t(blockIdx.z) * stride_t;
    const int64_t m0 = int64_t(blockIdx.y) * 64, k0 = int64_t(blockIdx.x) * 64;
    const int t = threadIdx.x;
    const int c4 = (t & 15) * 4;   // 4 consecutive columns of the tile
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (t >> 4) + 16 * i;   // tile row (m)
        const int64_t m = m0 + r, k = k0 + c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (m < M) {
            if (kVecLoad && k + 3 < K) {
                v = __ldg(reinterpret_cast<const float4 *>(A + m * lda + k));
            } else {
                const float *src = A + m * lda;
                v.x = k + 0 < K ? src[k + 0] : 0.0f;
                v.y = k + 1 < K ? src[k + 1] : 0.0f;
                v.z = k + 2 < K ? src[k + 2] : 0.0f;
                v.w = k + 3 < K ? src[k + 3] : 0.0f;
            }
        }
        tile[r][c4 + 0] = v.x;
        tile[r][c4 + 1] = v.y;
        tile[r][c4 + 2] = v.z;
        tile[r][c4 + 3] = v.w;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (t >> 4) + 16 * i;   // tile column (k) = output row
        const int64_t k = k0 + r, m = m0 + c4;
        if (k < K && m < M) {
            // m .. m+3 lie inside the row of At (ldt >= M rounded up to 4);
            // entries past M are zeros from the tile
            const float4 v = make_float4(tile[c4 + 0][r], tile[c4 + 1][r], tile[c4 + 2][r],
                                         tile[c4 + 3][r]);
            *reinterpret_cast<float4 *>(At + k * ldt + m) = v;
        }
    }
}

// C_b = act(beta * C_b + bias) for the K == 0 / alpha == 0 case of the
// batched, fused-epilogue call (beta == 0 does not read C).
__global__ void epilogue_only_kernel(float *C, int64_t M, int64_t N, int64_t ldc,
                                     int64_t strideC, int64_t batch, float beta,
                                     const float *bias, int act) {
    const int64_t per = M * N, total = per * batch;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t b = e / per, r = e - b * per;
        const int64_t i = r / N, j = r - i * N;
        float *c = C + b * strideC + i * ldc + j;
        float v = (beta == 0.0f) ? 0.0f : beta * *c;
        if (bias) v += bias[j];
        if (act == kActGeluTanh) v = ffma::gelu_tanh(v);
        *c = v;
    }
}

// Attainable fp32 FMA rate: 64 independent FMA chains per thread, issued as
// 32 packed fp32x2 FMAs or as 64 scalar FMAs per round.
template <bool kPacked>
__global__ void __launch_bounds__(256) ffma_probe_kernel(int64_t iters, float *out) {
    float2 x[32];
    const float seed = 1.0f + 1e-7f * float(threadIdx.x);
#pragma unroll
    for (int r = 0; r < 32; ++r) x[r] = make_float2(seed + r, seed - r);
    const float2 m = make_float2(0.999999f, 0.999998f);
    const float2 c = make_float2(1e-6f, 2e-6f);
    for (int64_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            if constexpr (kPacked) {
                x[r] = __ffma2_rn(x[r], m, c);
            } else {
                x[r].x = fmaf(x[r].x, m.x, c.x);
                x[r].y = fmaf(x[r].y, m.y, c.y);
            }
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int r = 0; r < 32; ++r) s += x[r].x + x[r].y;
    out[int64_t(blockIdx.x) * blockDim.x + threadIdx.x] = s;
}

}  // namespace

cudaError_t launch_ffma(const GemmArgs &a, int kernel, int tile, bool vec, bool edge,
                        bool trans_a, bool trans_b, cudaStream_t stream) {
    if (trans_a) return trans_b ? launch_ffma_tt(a, tile, vec, edge, stream)
                                : launch_ffma_tn(a, tile, vec, edge, stream);
    if (trans_b) return launch_ffma_nt(a, tile, vec, edge, stream);
    const bool ext = a.batch > 1 || a.bias != nullptr || a.act != kActNone;
    if (tile == kSmallTile) {
        if (ext)
            return ffma::launch_layout<kSmallTile, false, false, false, true>(a, vec, edge, stream);
        return kernel == kKernelFfma2x128
                   ? ffma::launch_layout<kSmallTile, true, false, false, false>(a, vec, edge, stream)
                   : ffma::launch_layout<kSmallTile, false, false, false, false>(a, vec, edge,
                                                                                 stream);
    }
    // Plain products can run either instantiation (the extended one with
    // batch 1, no bias, no activation computes the same thing).  ptxas
    // allocates the two differently, and measured on GB300 neither wins
    // everywhere: the extended build is faster for full tiles without
    // split-K (8192^3: 60.8 against 60.0 TFLOP/s) and for bounds-checked
    // vector split-K (1024x1024x16384: 47.0 against 45.4); the plain build
    // for full-tile split-K (GPT-2 QKV 41.8 against 39.9, 1024^3 31.5
    // against 29.7).  The tuning knob kKnobFfmaExt (0/1) overrides the
    // choice for sweeps.
    const bool split = a.split_k > 1 || a.tail_split > 1;
    bool pick_ext = (!edge && !split) || (edge && vec && split);
    if (const int force = tuning(kKnobFfmaExt); force >= 0) pick_ext = force != 0;
    if (ext || (kernel != kKernelFfma2x128 && pick_ext))
        return ffma::launch_layout<128, false, false, false, true>(a, vec, edge, stream);
    return kernel == kKernelFfma2x128
               ? ffma::launch_layout<128, true, false, false, false>(a, vec, edge, stream)
               : ffma::launch_layout<128, false, false, false, false>(a, vec, edge, stream);
}

cudaError_t launch_transpose(const float *A, int64_t M, int64_t K, int64_t lda, float *At,
                             int64_t ldt, cudaStream_t stream, int64_t batch, int64_t stride_a,
                             int64_t stride_t) {
    // the 64 x 64 kernel stores 128-bit rows of A^T; it reads A with 128-bit
    // loads when A's rows allow, with scalar loads otherwise
    const bool vec_store = (reinterpret_cast<uintptr_t>(At) & 15u) == 0 && ldt % 4 == 0 &&
                           ldt >= (M + 3) / 4 * 4 && stride_t % 4 == 0;
    const bool vec_load = (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 4 == 0 &&
                          stride_a % 4 == 0;
    if (vec_store) {
        const dim3 grid(unsigned((K + 63) / 64), unsigned((M + 63) / 64), unsigned(batch));
        if (vec_load)
            transpose64_kernel<true><<<grid, 256, 0, stream>>>(A, M, K, lda, At, ldt, stride_a,
                                                               stride_t);
        else
            transpose64_kernel<false><<<grid, 256, 0, stream>>>(A, M, K, lda, At, ldt, stride_a,
                                                                stride_t);
    } else {
        const dim3 grid(unsigned((K + 31) / 32), unsigned((M + 31) / 32), unsigned(batch));
        transpose_kernel<<<grid, dim3(32, 8), 0, stream>>>(A, M, K, lda, At, ldt, stride_a,
                                                          stride_t);
    }
    return cudaGetLastError();
}

cudaError_t launch_scale(float *C, int64_t M, int64_t N, int64_t ldc, float beta,
                         cudaStream_t stream) {
    const int64_t total = M * N;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    scale_kernel<<<unsigned(blocks), 256, 0, stream>>>(C, M, N, ldc, beta);
    return cudaGetLastError();
}

cudaError_t launch_epilogue_only(float *C, int64_t M, int64_t N, int64_t ldc, int64_t strideC,
                                 int64_t batch, float beta, const float *bias, int act,
                                 cudaStream_t stream) {
    const int64_t total = M * N * batch;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    epilogue_only_kernel<<<unsigned(blocks), 256, 0, stream>>>(C, M, N, ldc, strideC, batch, beta,
                                                               bias, act);
    return cudaGetLastError();
}

cudaError_t launch_ffma_probe(int64_t ctas, int64_t iters, bool packed, float *out,
                              cudaStream_t stream) {
    if (packed)
        ffma_probe_kernel<true><<<unsigned(ctas), 256, 0, stream>>>(iters, out);
    else
        ffma_probe_kernel<false><<<unsigned(ctas), 256, 0, stream>>>(iters, out);
    return cudaGetLastError();
}

cudaError_t ffma_kernel_attributes(cudaFuncAttributes *attr) {
    return cudaFuncGetAttributes(attr,
                                 ffma::ffma_gemm_kernel<128, false, true, false, false, false,
                                                        false, false>);
}

}  // namespace sgemm_impl
