// ffma_tiny.cu -- the fp32 GEMM for small problems with short K: one load of
// each CTA's whole A and B panels, K split across the CTA's warps, the
// partial tiles summed in shared memory.
//
// C = alpha * A * B + beta * C (plain layout, any M, N, K <= 256, any leading
// dimensions), the same arithmetic per K range as the other kernels (one
// round-to-nearest fp32 FMA per accumulator per k, k ascending), then the
// eight warps' partial sums added in warp order.
//
// Why a kernel of its own: at 256^3 the tiled kernels spend their time
// waiting -- on each K slice's load (a pipeline of two to four pages), or on
// the global round trips of a split-K reduction -- not computing (34 MFLOP
// take 0.4 us at the FMA peak).  Here every CTA issues all its copies at
// once, waits once, and reduces in shared memory ("Micro_gemm_4x4 - cuBLAS
// micro GEMM skeleton", section 5: stage the tiles in shared memory, then
// compute from there; the split of K across a CTA's threads is this file's).
//
//  * CTA tile 32 x 32, 256 threads = 8 warps; warp w owns K range
//    [w*kw, (w+1)*kw) with kw = ceil(K/8) rounded up to 4.  Lane (rg, cg) =
//    (lane / 4, lane % 4) owns rows rg + 8i (i < 4) and columns cg*8 .. +7:
//    4 x 8 accumulators, updated in column pairs by packed fma.rn.f32x2 (the
//    same roundings in the same order as scalar FMAs; with two warps per
//    scheduler the kernel is issue-bound, and measured on GB300 the packed
//    form moved 512x512x128 and 256x1024x128 from 10.9 to 8.9 us, 256^3
//    unchanged at 8.9 us, C the same bit for bit).
//  * Shared memory: As[32][Kp + 4] (rows as stored, 16-byte copies; the row
//    stride of Kp/4 + 1 chunks, odd, spreads the eight rows a load touches
//    over distinct banks), Bs[Kp][32].  Per 4 k a lane loads 4 A chunks
//    (4 k of each of its rows) and 8 B chunks for 128 FMAs.
//  * After the FMAs the warps' 32 x 32 partials go to shared memory (over the
//    operand tiles) and each thread sums 4 outputs over the 8 warps in order,
//    then applies alpha and beta and stores with one 128-bit store.
#include <cuda_runtime.h>

#include <cstdint>

#include "ffma_kernel.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace {

constexpr int kTinyT = 32;
constexpr int kTinyThreads = 256;

__host__ __device__ constexpr int tiny_kw(int64_t K) { return int((K + 31) / 32) * 4; }

template <bool kVec>
__global__ void __launch_bounds__(kTinyThreads) ffma_tiny_kernel(const GemmArgs p) {
    extern __shared__ __align__(16) float smem[];
    const int kw = tiny_kw(p.K);     // K per warp, a multiple of 4
    const int Kp = 8 * kw;           // staged K extent (zero past K)
    const int lda_s = Kp + 4;        // A row stride in shared memory (floats)
    float *As = smem;                              // [32][Kp + 4]
    float *Bs = smem + kTinyT * lda_s;             // [Kp][32]

    const int tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    const int64_t tiles_n = (p.N + kTinyT - 1) / kTinyT;
    const int64_t row0 = int64_t(blockIdx.x / tiles_n) * kTinyT;
    const int64_t col0 = int64_t(blockIdx.x % tiles_n) * kTinyT;

    // ---- every copy of the CTA at once (out-of-range elements read as 0) ----
    const int a_chunks = kTinyT * (Kp / 4);
    for (int c = tid; c < a_chunks; c += kTinyThreads) {
        const int r = c / (Kp / 4), k = (c % (Kp / 4)) * 4;
        const int64_t row = row0 + r;
        float *dst = As + r * lda_s + k;
        const float *src = p.A + (row < p.M ? row : 0) * p.lda + k;
        const int64_t left = row < p.M ? p.K - k : 0;
        const int n = left <= 0 ? 0 : (left >= 4 ? 4 : int(left));
        if constexpr (kVec) {
            ffma::cp_async16(dst, n ? src : p.A, n * 4);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) ffma::cp_async4(dst + e, e < n ? src + e : p.A, e < n ? 4 : 0);
        }
    }
    for (int c = tid; c < Kp * (kTinyT / 4); c += kTinyThreads) {
        const int k = c / (kTinyT / 4), j = (c % (kTinyT / 4)) * 4;
        const int64_t col = col0 + j;
        float *dst = Bs + k * kTinyT + j;
        const float *src = p.B + (k < p.K ? k : 0) * p.ldb + (col < p.N ? col : 0);
        const int64_t left = k < p.K ? p.N - col : 0;
        const int n = left <= 0 ? 0 : (left >= 4 ? 4 : int(left));
        if constexpr (kVec) {
            ffma::cp_async16(dst, n ? src : p.B, n * 4);
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) ffma::cp_async4(dst + e, e < n ? src + e : p.B, e < n ? 4 : 0);
        }
    }
    ffma::cp_async_commit();
    ffma::cp_async_wait_all();
    __syncthreads();

    // ---- this warp's K range: 4 x 8 accumulators per lane, as column pairs
    // updated with packed fma.rn.f32x2 (each lane one round-to-nearest fp32
    // FMA, k ascending, as scalar issue would do; half the instructions) ----
    const int rg = lane >> 2, cg = lane & 3;
    float2 acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);
    const int kbeg = warp * kw;
    for (int k4 = kbeg; k4 < kbeg + kw; k4 += 4) {
        float4 a[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            a[i] = *reinterpret_cast<const float4 *>(As + (rg + 8 * i) * lda_s + k4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const float4 b0 = *reinterpret_cast<const float4 *>(Bs + (k4 + kk) * kTinyT + cg * 8);
            const float4 b1 = *reinterpret_cast<const float4 *>(Bs + (k4 + kk) * kTinyT + cg * 8 + 4);
            const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w),
                                 make_float2(b1.x, b1.y), make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float ai = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                const float2 aa = make_float2(ai, ai);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(aa, b[j], acc[i][j]);
            }
        }
    }

    // ---- partials to shared memory (over the operand tiles), summed in warp order ----
    __syncthreads();
    float *red = smem;   // [8][32][32]
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float *dst = red + warp * (kTinyT * kTinyT) + (rg + 8 * i) * kTinyT + cg * 8;
        *reinterpret_cast<float4 *>(dst) =
            make_float4(acc[i][0].x, acc[i][0].y, acc[i][1].x, acc[i][1].y);
        *reinterpret_cast<float4 *>(dst + 4) =
            make_float4(acc[i][2].x, acc[i][2].y, acc[i][3].x, acc[i][3].y);
    }
    __syncthreads();
    const int r = tid >> 3, c4 = (tid & 7) * 4;
    float4 s = *reinterpret_cast<const float4 *>(red + r * kTinyT + c4);
#pragma unroll
    for (int w = 1; w < 8; ++w) {
        const float4 v = *reinterpret_cast<const float4 *>(red + w * (kTinyT * kTinyT) +
                                                          r * kTinyT + c4);
        s.x += v.x;
        s.y += v.y;
        s.z += v.z;
        s.w += v.w;
    }
    const int64_t row = row0 + r, col = col0 + c4;
    if (row >= p.M) return;
    float *cp = p.C + row * p.ldc + col;
    float v[4] = {p.alpha * s.x, p.alpha * s.y, p.alpha * s.z, p.alpha * s.w};
    if (kVec && col + 3 < p.N) {
        if (p.beta != 0.0f) {
            const float4 old = *reinterpret_cast<const float4 *>(cp);
            v[0] = fmaf(p.beta, old.x, v[0]);
            v[1] = fmaf(p.beta, old.y, v[1]);
            v[2] = fmaf(p.beta, old.z, v[2]);
            v[3] = fmaf(p.beta, old.w, v[3]);
        }
        *reinterpret_cast<float4 *>(cp) = make_float4(v[0], v[1], v[2], v[3]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (col + e < p.N) {
                float x = v[e];
                if (p.beta != 0.0f) x = fmaf(p.beta, cp[e], x);
                cp[e] = x;
            }
        }
    }
}

}  // namespace

size_t tiny_smem_bytes(int64_t K) {
    const int Kp = 8 * tiny_kw(K);
    const size_t operands = (size_t(kTinyT) * (Kp + 4) + size_t(Kp) * kTinyT) * sizeof(float);
    const size_t partials = size_t(8) * kTinyT * kTinyT * sizeof(float);
    return operands > partials ? operands : partials;
}

cudaError_t launch_ffma_tiny(const GemmArgs &a, bool vec, cudaStream_t stream) {
    if (a.K < 1 || a.K > kTinyMaxK) return cudaErrorInvalidValue;
    const int bytes = int(tiny_smem_bytes(a.K));
    const int64_t tiles = ((a.M + kTinyT - 1) / kTinyT) * ((a.N + kTinyT - 1) / kTinyT);
    if (vec) {
        static bool configured[64];
        const cudaError_t e = set_smem_once(reinterpret_cast<const void *>(ffma_tiny_kernel<true>),
                                            int(tiny_smem_bytes(kTinyMaxK)), configured);
        if (e != cudaSuccess) return e;
        ffma_tiny_kernel<true><<<unsigned(tiles), kTinyThreads, bytes, stream>>>(a);
    } else {
        static bool configured[64];
        const cudaError_t e = set_smem_once(reinterpret_cast<const void *>(ffma_tiny_kernel<false>),
                                            int(tiny_smem_bytes(kTinyMaxK)), configured);
        if (e != cudaSuccess) return e;
        ffma_tiny_kernel<false><<<unsigned(tiles), kTinyThreads, bytes, stream>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace sgemm_impl
