// ffma_wide_kernel.cuh -- the fp32 CUDA-core GEMM with a 16 x 8 block of
// accumulators per thread, for large products whose operands both arrive by
// direct row copies (op(A) = A^T from the transposed copy, op(B) = B).
//
// Same arithmetic as ffma_kernel.cuh (one round-to-nearest fp32 FMA per
// accumulator per k, k ascending; alpha * acc, then fma(beta, C_old, .)),
// but each thread owns 16 rows x 8 columns of C instead of 8 x 8, so per
// k step it does 128 FMAs for 6 shared loads of 128 bits (4 of A, 2 of B)
// where the 8 x 8 tile does 64 for 4: fewer issue slots go to anything but
// FMAs (velog @levelstage "AutoMinepp7", section "세부 조정": a larger
// per-thread block raises the arithmetic per load until registers run out;
// the accumulators here take 128 of the 255 a thread may hold).
//
//  * CTA tile 128 x 128, 128 threads (4 warps of 4 (M) x 8 (N) threads),
//    two CTAs per SM.  Thread (tm, tn) owns rows q*32 + tm*4 + i (q, i <
//    4) and columns h*64 + tn*4 + j (h < 2, j < 4): a warp's 128-bit loads
//    of A hit 4 distinct 16-byte chunks and of B 8, conflict-free.
//  * K slices of 32 through a three-page cp.async ring (two slices in flight
//    while one is computed), one barrier per slice; fragments double-buffered
//    across the 32 k steps.
//  * FMAs in boustrophedon order (odd rows right to left), so every two
//    consecutive FMAs share a source operand.
//  * Edges: zero-filled copies and predicated stores, as the 8 x 8 kernel.
//
// Measured on GB300 it is slower than the 8 x 8 kernel (8192^3: 60.4
// against 65.9 TFLOP/s): FFMA rises to 92 % of issued instructions, but
// with 245 registers a thread only 8 warps fit on an SM, and the issue
// slots go from 90 % to 85 % busy.  It is kept as an option (tuning knob
// kKnobKernel = 2) with its own parity tests.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ffma_kernel.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace wide {

using ffma::cp_async16;
using ffma::cp_async_commit;
using ffma::gelu_tanh;

constexpr int kT = 128;        // CTA tile
constexpr int kBK = 32;        // K slice
constexpr int kThreads = 128;
constexpr int kPages = 3;
constexpr int kPage = kBK * kT;                           // floats per operand page
constexpr int kSmemBytes = 2 * kPages * kPage * 4;        // 96 KiB
constexpr int kChunks = kPage / 4 / kThreads;             // 16-byte copies per operand per slice
// k steps per unrolled pass (even).  Measured at 8192^3 (TFLOP/s): 4: 59.8,
// 8: 60.4, 16: 56.2, 32 (all): 58.9.
constexpr int kUnroll = 8;
static_assert(kUnroll % 2 == 0 && kBK % kUnroll == 0, "fragment double buffering needs pairs");

template <bool kEdge, bool kExt>
__global__ void __launch_bounds__(kThreads, 2) ffma16x8_kernel(const GemmArgs p) {
    extern __shared__ __align__(16) float smem[];
    float *const ringA = smem;                    // [page][k][m]
    float *const ringB = smem + kPages * kPage;   // [page][k][n]

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tm = (warp >> 1) * 4 + (lane >> 3);   // 0..7
    const int tn = (warp & 1) * 8 + (lane & 7);     // 0..15

    int64_t row0, col0, bidx;
    {
        const ffma::WorkItem w = ffma::work_item(p, blockIdx.x, kT);
        row0 = w.row0;
        col0 = w.col0;
        bidx = kExt ? w.batch : 0;
    }
    const float *Ab = kExt ? p.A + bidx * p.strideA : p.A;   // A^T: K x M
    const float *Bb = kExt ? p.B + bidx * p.strideB : p.B;   // B:   K x N
    const int nsl = int((p.K + kBK - 1) / kBK);

    // copy mapping: chunk c = tid + h * kThreads of a page [kBK][kT] is k row
    // c / 32, columns 4 (c % 32) ..; chunk h sits 4 k rows after chunk h - 1
    const int c_k = tid >> 5;
    const int c_x = (tid & 31) * 4;
    const float *a_src = Ab + int64_t(c_k) * p.lda + row0 + c_x;
    const float *b_src = Bb + int64_t(c_k) * p.ldb + col0 + c_x;
    int a_cols = 4, b_cols = 4;
    if constexpr (kEdge) {
        const int64_t la = p.M - (row0 + c_x), lb = p.N - (col0 + c_x);
        a_cols = la <= 0 ? 0 : (la >= 4 ? 4 : int(la));
        b_cols = lb <= 0 ? 0 : (lb >= 4 ? 4 : int(lb));
        if (a_cols == 0) a_src = p.A;
        if (b_cols == 0) b_src = p.B;
    }

    auto issue = [&](int t, int page) {
        const int64_t k_slice = int64_t(t) * kBK;
        float *da = ringA + page * kPage + c_k * kT + c_x;
        float *db = ringB + page * kPage + c_k * kT + c_x;
#pragma unroll
        for (int h = 0; h < kChunks; ++h) {
            const int64_t k = k_slice + c_k + 4 * h;
            const float *sa = a_src + (k_slice + 4 * h) * p.lda;
            const float *sb = b_src + (k_slice + 4 * h) * p.ldb;
            if constexpr (!kEdge) {
                cp_async16(da + 4 * h * kT, sa, 16);
                cp_async16(db + 4 * h * kT, sb, 16);
            } else {
                const bool k_ok = k < p.K;
                const int na = k_ok ? a_cols : 0, nb = k_ok ? b_cols : 0;
                cp_async16(da + 4 * h * kT, na ? sa : p.A, na * 4);
                cp_async16(db + 4 * h * kT, nb ? sb : p.B, nb * 4);
            }
        }
    };

    float2 acc[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

#pragma unroll
    for (int q = 0; q < kPages - 1; ++q) {
        if (q < nsl) issue(q, q);
        cp_async_commit();   // one group per slice, empty ones included
    }

    for (int t = 0; t < nsl; ++t) {
        const int page = t % kPages;
        asm volatile("cp.async.wait_group %0;\n" ::"n"(kPages - 2) : "memory");
        __syncthreads();
        const int nt = t + kPages - 1;
        if (nt < nsl) issue(nt, nt % kPages);
        cp_async_commit();

        const float *As = ringA + page * kPage;
        const float *Bs = ringB + page * kPage;
        float4 af[2][4], bf[2][2];
#pragma unroll
        for (int q = 0; q < 4; ++q)
            af[0][q] = *reinterpret_cast<const float4 *>(As + q * 32 + tm * 4);
#pragma unroll
        for (int h = 0; h < 2; ++h)
            bf[0][h] = *reinterpret_cast<const float4 *>(Bs + h * 64 + tn * 4);
        // The slice's 32 k steps run as kBK / kUnroll passes of a loop
        // unrolled kUnroll times: fully unrolled, the FMA stream (about 70
        // KB of instructions) overflows the instruction cache (ncu at
        // 4096^3: no_instruction 0.59 stalls per issue).
#pragma unroll 1
        for (int k0 = 0; k0 < kBK; k0 += kUnroll) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int kk = k0 + u;
            const int cur = u & 1;
            if (u + 1 < kUnroll || k0 + kUnroll < kBK) {
                const float *Ak = As + (kk + 1) * kT;
                const float *Bk = Bs + (kk + 1) * kT;
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    af[cur ^ 1][q] = *reinterpret_cast<const float4 *>(Ak + q * 32 + tm * 4);
#pragma unroll
                for (int h = 0; h < 2; ++h)
                    bf[cur ^ 1][h] = *reinterpret_cast<const float4 *>(Bk + h * 64 + tn * 4);
            }
            float a[16];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[4 * q + 0] = af[cur][q].x;
                a[4 * q + 1] = af[cur][q].y;
                a[4 * q + 2] = af[cur][q].z;
                a[4 * q + 3] = af[cur][q].w;
            }
            const float2 b[4] = {make_float2(bf[cur][0].x, bf[cur][0].y),
                                 make_float2(bf[cur][0].z, bf[cur][0].w),
                                 make_float2(bf[cur][1].x, bf[cur][1].y),
                                 make_float2(bf[cur][1].z, bf[cur][1].w)};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    const int j = (i & 1) ? 3 - jj : jj;
                    if (i & 1) {
                        acc[i][j].y = fmaf(a[i], b[j].y, acc[i][j].y);
                        acc[i][j].x = fmaf(a[i], b[j].x, acc[i][j].x);
                    } else {
                        acc[i][j].x = fmaf(a[i], b[j].x, acc[i][j].x);
                        acc[i][j].y = fmaf(a[i], b[j].y, acc[i][j].y);
                    }
                }
            }
        }
        }
    }
    asm volatile("cp.async.wait_all;\n" ::: "memory");

    // ---- epilogue: C = act(alpha * acc (+ beta * C_old) (+ bias)) ----
    const float alpha = p.alpha, beta = p.beta;
    float *Cb = kExt ? p.C + bidx * p.strideC : p.C;
    const float *bias = kExt ? p.bias : nullptr;
    const int act = kExt ? p.act : kActNone;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int64_t row = row0 + (i >> 2) * 32 + tm * 4 + (i & 3);
        if (kEdge && row >= p.M) continue;
        float *crow = Cb + row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t col = col0 + h * 64 + tn * 4;
            float v[4] = {alpha * acc[i][2 * h].x, alpha * acc[i][2 * h].y,
                          alpha * acc[i][2 * h + 1].x, alpha * acc[i][2 * h + 1].y};
            float *cp = crow + col;
            if (!kEdge || col + 3 < p.N) {
                if (beta != 0.0f) {
                    const float4 old = *reinterpret_cast<const float4 *>(cp);
                    v[0] = fmaf(beta, old.x, v[0]);
                    v[1] = fmaf(beta, old.y, v[1]);
                    v[2] = fmaf(beta, old.z, v[2]);
                    v[3] = fmaf(beta, old.w, v[3]);
                }
                if (bias) {
                    const float4 bv = *reinterpret_cast<const float4 *>(bias + col);
                    v[0] += bv.x;
                    v[1] += bv.y;
                    v[2] += bv.z;
                    v[3] += bv.w;
                }
                if (act == kActGeluTanh) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) v[c] = gelu_tanh(v[c]);
                }
                *reinterpret_cast<float4 *>(cp) = make_float4(v[0], v[1], v[2], v[3]);
            } else {
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (col + c < p.N) {
                        float x = v[c];
                        if (beta != 0.0f) x = fmaf(beta, cp[c], x);
                        if (bias) x += bias[col + c];
                        if (act == kActGeluTanh) x = gelu_tanh(x);
                        cp[c] = x;
                    }
                }
            }
        }
    }
}

}  // namespace wide
}  // namespace sgemm_impl
