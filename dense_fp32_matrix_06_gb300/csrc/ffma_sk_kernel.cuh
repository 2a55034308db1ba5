// ffma_sk_kernel.cuh -- the fp32 CUDA-core GEMM as a persistent stream-K
// kernel with a deep cp.async ring (template; instantiated per operand layout
// in ffma_sk_*.cu).
//
// C_b = act(alpha * op(A_b) * op(B_b) + beta * C_b + bias), any M, N, K, any
// leading dimensions and alignment; the same arithmetic as ffma_kernel.cuh
// (8 x 8 fp32 accumulators per thread, one round-to-nearest FMA per
// accumulator per k, k ascending within a CTA's K range, boustrophedon issue
// order), scheduled differently:
//
//  * Persistent CTAs.  G CTAs (a few per SM) stay resident and split the
//    work evenly: first whole-K tiles handed out round-robin while every CTA
//    still gets one per round, then the K slices of the remaining tiles cut
//    into G equal runs in (tile, slice) order -- the stream-K decomposition
//    of Osama et al., "Stream-K: Work-centric Parallel Decomposition for
//    Dense Matrix-Matrix Multiplication on the GPU" (PPoPP 2023).  Grids of
//    fewer tiles than resident CTAs, and partial last waves, then keep every
//    SM busy to the end, where split-K into equal ranges could not.
//  * Fixed-order fix-up in a second launch.  A CTA that computed only part
//    of a tile's K range stores its partial tile in its own slot and moves
//    on; once the persistent launch is done, partial_reduce_kernel (ffma_kernel.cuh)
//    sums every contributor's partial in ascending CTA order and runs the
//    epilogue.  Nobody waits on anybody, and the sum order depends only on
//    the shape and the grid, so results are bit-identical run to run.
//  * Every operand goes through an NP-page ring of 16-byte (or, for
//    unaligned operands, 4-byte) cp.async copies, so NP - 2 slices are in
//    flight while one is computed.  An operand whose stored rows run along M
//    or N (A^T, B) lands directly in the k-major tile the FMAs read.  One
//    whose rows run along K (A, B^T) lands row by row in a raw page; each
//    thread then transposes the chunks it copied itself into one of two
//    k-major pages with an XOR swizzle that keeps the shared stores
//    conflict-free, one slice ahead of the FMAs (velog @levelstage
//    "AutoMinepp7", section "직사각형 타일링": fetch the next chunk while
//    computing, then place it in the other local-memory page; here the fetch
//    is an asynchronous copy into shared memory rather than into registers).
//  * Edges: out-of-range elements are zero-filled by the copies and C stores
//    are predicated ("Micro_gemm_4x4 - cuBLAS micro GEMM skeleton", sections
//    6 and 9; "GPU Target", section "타일링된 행렬 곱셈").
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "ffma_kernel.cuh"
#include "sgemm_internal.h"

namespace sgemm_impl {
namespace sk {

using ffma::cp_async16;
using ffma::cp_async4;
using ffma::cp_async_commit;
using ffma::gelu_tanh;
using ffma::tcol;

template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// T x T tile, K slices of BK, (T/8)^2 threads with 8 x 8 accumulators each
// (warps of 4 x 8 threads), NP-page ring.  A page holds T * BK floats; every
// thread copies kChunks 16-byte chunks of each operand per slice (two with
// BK = T/8).
template <int T, int BK, int NP>
struct Cfg {
    static constexpr int kBK = BK;
    static constexpr int kThreads = (T / 8) * (T / 8);
    static constexpr int kWarpsN = T / 64;
    static constexpr int kKG = BK / 4;                  // 4-wide k groups per slice
    static constexpr int kShift = kKG == 8 ? 2 : (kKG == 4 ? 3 : 4);   // log2(32 / kKG)
    static constexpr int kPage = T * BK;                // floats per page
    static constexpr int kChunks = kPage / 4 / kThreads;
    static constexpr int kMinBlocks = T == 128 ? 2 : 8; // resident CTAs per SM
    static_assert(T == 128 || T == 64, "tile is 128 or 64");
    static_assert(BK == T / 8 || BK == 2 * (T / 8), "K slices of T/8 or T/4");
    static_assert(NP >= 2 && NP <= 8, "ring of 2..8 pages");
};

// Batch index and first row/column of a tile: batch-major, then a grouped
// raster over kGroupM tile rows within a batch (L2 reuse of A and B panels).
template <int T, bool kExt>
__device__ __forceinline__ void tile_coords(const SkArgs &p, int64_t tile, int64_t *bidx,
                                            int64_t *row0, int64_t *col0) {
    int64_t b = 0, t_in = tile;
    if constexpr (kExt) {
        const int64_t per_batch = int64_t(p.tiles_m) * p.tiles_n;
        b = tile / per_batch;
        t_in = tile - b * per_batch;
    }
    const int64_t per_group = int64_t(kGroupM) * p.tiles_n;
    const int64_t group = t_in / per_group;
    const int64_t first_m = group * kGroupM;
    const int64_t gm = min(int64_t(p.tiles_m) - first_m, int64_t(kGroupM));
    const int64_t in_group = t_in - group * per_group;
    *bidx = b;
    *row0 = (first_m + in_group % gm) * T;
    *col0 = (in_group / gm) * T;
}

template <int T, int BKT, int NP, bool kTransA, bool kTransB, bool kVec, bool kExt>
__global__ void __launch_bounds__(Cfg<T, BKT, NP>::kThreads, Cfg<T, BKT, NP>::kMinBlocks)
ffma_sk_kernel(const SkArgs p) {
    using Cf = Cfg<T, BKT, NP>;
    constexpr int BK = Cf::kBK, NT = Cf::kThreads, KG = Cf::kKG, SH = Cf::kShift;
    constexpr int PG = Cf::kPage, CH = Cf::kChunks;
    // an operand whose stored rows run along K is staged: raw ring + transpose
    constexpr bool kStA = !kTransA;
    constexpr bool kStB = kTransB;
    constexpr bool kStaged = kStA || kStB;
    static_assert(!kStaged || NP >= 3, "a staged operand needs a ring of three pages or more");
    // k step of slice t's FMAs at which slice t+1 is staged.  Measured on
    // GB300 (1024^3 .. 4096^3): halfway, at the first k step, after the
    // last one, with or without skipping the last slice's staging -- all
    // within 2 %.
    constexpr int kStageAt = BK / 2;

    extern __shared__ __align__(16) float smem[];
    float *const ringA = smem;                        // NP pages
    float *const ringB = smem + NP * PG;              // NP pages
    float *const compA = smem + 2 * NP * PG;          // 2 pages when A is staged
    float *const compB = compA + (kStA ? 2 * PG : 0); // 2 pages when B is staged

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tm = (warp / Cf::kWarpsN) * 4 + (lane >> 3);   // 0..T/8-1
    const int tn = (warp % Cf::kWarpsN) * 8 + (lane & 7);    // 0..T/8-1

    // The segment loop's state lives in shared memory: thread 0 advances it
    // between two barriers, so none of it occupies registers across the
    // main loop.
    __shared__ long long s_it;      // next stream-K slice of this CTA's run
    __shared__ long long s_tile;    // current segment: tile, slices [s_k0, s_k1)
    __shared__ int s_round, s_k0, s_k1, s_first, s_done;
    if (tid == 0) {
        s_round = 0;
        s_it = (long long)(int64_t(blockIdx.x) * p.sk_iters / gridDim.x);
    }

    for (;;) {
        __syncthreads();   // everyone is done with the previous segment
        if (tid == 0) {
            // ---- next segment: (tile, slices [k0, k1)) ----
            const int G = gridDim.x, g = blockIdx.x;
            const int64_t U = p.sk_iters;
            const int64_t b_g = int64_t(g + 1) * U / G;   // end of this CTA's run
            const int64_t it = s_it;
            s_done = 0;
            if (s_round < p.dp_rounds) {
                s_tile = (long long)(int64_t(s_round) * G + g);
                s_k0 = 0;
                s_k1 = p.kt;
                s_first = 0;
                ++s_round;
            } else if (it < b_g) {
                const int64_t lt = it / p.kt;
                const int k0 = int(it - lt * p.kt);
                const int64_t left = b_g - it;
                const int k1 = left < int64_t(p.kt - k0) ? k0 + int(left) : p.kt;
                s_tile = (long long)(int64_t(p.dp_rounds) * G + lt);
                s_k0 = k0;
                s_k1 = k1;
                s_first = it == int64_t(g) * U / G;
                s_it = (long long)(it + (k1 - k0));
            } else {
                s_done = 1;
            }
        }
        __syncthreads();
        if (s_done) {
            // the reduction launch may be scheduled once every CTA is here
            asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
            break;
        }

        const int nsl = s_k1 - s_k0;
        // operand pointers and bounds for this segment (recomputed after the
        // main loop where needed, so they do not stay live across it)
        const float *a_src, *b_src;   // chunk h = 0 of the slice; chunk h sits at a fixed offset
        int a_lim, b_lim;     // direct: valid columns (0..4); staged: rows left from chunk 0's
        int a_krem, b_krem;   // K left after chunk 0's first k, at slice 0
        {
            int64_t bidx, row0, col0;
            tile_coords<T, kExt>(p, s_tile, &bidx, &row0, &col0);
            const float *Ab = kExt ? p.A + bidx * p.strideA : p.A;
            const float *Bb = kExt ? p.B + bidx * p.strideB : p.B;
            const int64_t kbeg = int64_t(s_k0) * BK;
            const int64_t kend = min(p.K, int64_t(s_k1) * BK);
            // chunk c = tid + h * NT of a page.  Direct page [BK][T]: k row
            // c / (T/4), columns 4 (c % (T/4)) ..; raw page [T][BK]: row c / KG,
            // k columns 4 (c % KG) ..
            if constexpr (kTransA) {
                const int kr = tid / (T / 4), m = (tid % (T / 4)) * 4;
                const int64_t left = p.M - (row0 + m);
                a_lim = left <= 0 ? 0 : (left >= 4 ? 4 : int(left));
                a_krem = int(kend - kbeg - kr);
                a_src = Ab + (kbeg + kr) * p.lda + (a_lim ? row0 + m : 0);
            } else {
                const int m = tid / KG, kc = (tid % KG) * 4;
                const int64_t left = p.M - (row0 + m);
                a_lim = left <= 0 ? 0 : (left >= T ? T : int(left));
                a_krem = int(kend - kbeg - kc);
                a_src = Ab + (a_lim ? row0 + m : 0) * p.lda + kbeg + kc;
            }
            if constexpr (!kTransB) {
                const int kr = tid / (T / 4), n = (tid % (T / 4)) * 4;
                const int64_t left = p.N - (col0 + n);
                b_lim = left <= 0 ? 0 : (left >= 4 ? 4 : int(left));
                b_krem = int(kend - kbeg - kr);
                b_src = Bb + (kbeg + kr) * p.ldb + (b_lim ? col0 + n : 0);
            } else {
                const int n = tid / KG, kc = (tid % KG) * 4;
                const int64_t left = p.N - (col0 + n);
                b_lim = left <= 0 ? 0 : (left >= T ? T : int(left));
                b_krem = int(kend - kbeg - kc);
                b_src = Bb + (b_lim ? col0 + n : 0) * p.ldb + kbeg + kc;
            }
        }

        // one operand's chunks of slice t into page `dst`.  Direct: chunk h
        // is h * NT / (T/4) k rows further on; staged: h * NT / KG rows
        // further on (a row the matrix may not have: lim counts them).
        auto copy_op = [&](float *dst, const float *src, int lim, int krem, int64_t ld,
                           bool direct, int t, const float *dummy) {
            const int64_t slice_stride = direct ? int64_t(BK) * ld : BK;
            const int64_t h_stride = direct ? int64_t(NT / (T / 4)) * ld : int64_t(NT / KG) * ld;
            const int kleft = krem - t * BK;
            const float *s0 = src + int64_t(t) * slice_stride;
#pragma unroll
            for (int h = 0; h < CH; ++h) {
                int n;
                if (direct) {
                    n = kleft - h * (NT / (T / 4)) > 0 ? lim : 0;
                } else {
                    n = lim > h * (NT / KG) ? (kleft <= 0 ? 0 : (kleft >= 4 ? 4 : kleft)) : 0;
                }
                const float *s = s0 + h * h_stride;
                float *d = dst + (tid + h * NT) * 4;
                if constexpr (kVec) {
                    cp_async16(d, n > 0 ? s : dummy, n * 4);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool ok = e < n;
                        cp_async4(d + e, ok ? s + e : dummy, ok ? 4 : 0);
                    }
                }
            }
        };
        auto issue = [&](int t, int page) {
            copy_op(ringA + page * PG, a_src, a_lim, a_krem, p.lda, kTransA, t, p.A);
            copy_op(ringB + page * PG, b_src, b_lim, b_krem, p.ldb, !kTransB, t, p.B);
        };
        // the chunks this thread copied into raw page `raw`, transposed into
        // the k-major page `comp` (columns XOR-swizzled by the k group)
        auto transpose = [&](const float *raw, float *comp) {
#pragma unroll
            for (int h = 0; h < CH; ++h) {
                const int c = tid + h * NT;
                const int x = c / KG, kc = (c % KG) * 4;
                const float4 v = *reinterpret_cast<const float4 *>(raw + c * 4);
                comp[(kc + 0) * T + tcol<true, KG, SH>(kc, x)] = v.x;
                comp[(kc + 1) * T + tcol<true, KG, SH>(kc, x)] = v.y;
                comp[(kc + 2) * T + tcol<true, KG, SH>(kc, x)] = v.z;
                comp[(kc + 3) * T + tcol<true, KG, SH>(kc, x)] = v.w;
            }
        };

        float2 acc[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

        // ---- pipeline ----
#pragma unroll
        for (int q = 0; q < NP - 1; ++q) {
            if (q < nsl) issue(q, q);
            cp_async_commit();   // one group per slice, empty ones included
        }
        if constexpr (kStaged) {
            cp_async_wait<NP - 2>();   // this thread's copies of slice 0
            if (nsl > 0) {
                if constexpr (kStA) transpose(ringA, compA);
                if constexpr (kStB) transpose(ringB, compB);
            }
        }
        int q_comp = 0;            // ring page of slice t
        int q_issue = NP - 1;      // ring page of slice t + NP - 1
        for (int t = 0; t < nsl; ++t) {
            // staged: slice t+1 must have landed (it is transposed during t);
            // direct only: slice t
            if constexpr (kStaged)
                cp_async_wait<NP - 3 >= 0 ? NP - 3 : 0>();
            else
                cp_async_wait<NP - 2>();
            __syncthreads();
            if (t + NP - 1 < nsl) issue(t + NP - 1, q_issue);
            cp_async_commit();
            if (++q_issue == NP) q_issue = 0;

            const float *As = kStA ? compA + (t & 1) * PG : ringA + q_comp * PG;
            const float *Bs = kStB ? compB + (t & 1) * PG : ringB + q_comp * PG;
            const int q_next = q_comp + 1 == NP ? 0 : q_comp + 1;
            float4 af[2][2], bf[2][2];
            af[0][0] = *reinterpret_cast<const float4 *>(As + tcol<kStA, KG, SH>(0, tm * 4));
            af[0][1] = *reinterpret_cast<const float4 *>(As + tcol<kStA, KG, SH>(0, T / 2 + tm * 4));
            bf[0][0] = *reinterpret_cast<const float4 *>(Bs + tcol<kStB, KG, SH>(0, tn * 4));
            bf[0][1] = *reinterpret_cast<const float4 *>(Bs + tcol<kStB, KG, SH>(0, T / 2 + tn * 4));
#pragma unroll
            for (int kk = 0; kk < BK; ++kk) {
                const int cur = kk & 1;
                if (kk + 1 < BK) {
                    const int k = kk + 1;
                    af[cur ^ 1][0] = *reinterpret_cast<const float4 *>(
                        As + k * T + tcol<kStA, KG, SH>(k, tm * 4));
                    af[cur ^ 1][1] = *reinterpret_cast<const float4 *>(
                        As + k * T + tcol<kStA, KG, SH>(k, T / 2 + tm * 4));
                    bf[cur ^ 1][0] = *reinterpret_cast<const float4 *>(
                        Bs + k * T + tcol<kStB, KG, SH>(k, tn * 4));
                    bf[cur ^ 1][1] = *reinterpret_cast<const float4 *>(
                        Bs + k * T + tcol<kStB, KG, SH>(k, T / 2 + tn * 4));
                }
                if (kk == kStageAt && t + 1 < nsl) {
                    // stage slice t+1 part way through slice t's FMAs
                    if constexpr (kStA) transpose(ringA + q_next * PG, compA + ((t + 1) & 1) * PG);
                    if constexpr (kStB) transpose(ringB + q_next * PG, compB + ((t + 1) & 1) * PG);
                }
                const float a[8] = {af[cur][0].x, af[cur][0].y, af[cur][0].z, af[cur][0].w,
                                    af[cur][1].x, af[cur][1].y, af[cur][1].z, af[cur][1].w};
                const float2 b[4] = {make_float2(bf[cur][0].x, bf[cur][0].y),
                                     make_float2(bf[cur][0].z, bf[cur][0].w),
                                     make_float2(bf[cur][1].x, bf[cur][1].y),
                                     make_float2(bf[cur][1].z, bf[cur][1].w)};
                // boustrophedon order: every two consecutive FMAs share a
                // source operand (odd rows run right to left)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
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
            q_comp = q_next;
        }
        cp_async_wait<0>();   // no copy of this segment outlives it

        // ---- a segment that is not a whole tile: its partial tile goes to
        // this CTA's slot (2g for its run's first segment, 2g + 1 for its
        // last) and partial_reduce_kernel sums the slots afterwards ----
        if (s_k0 != 0 || s_k1 != p.kt) {
            float4 *mine = reinterpret_cast<float4 *>(p.partials) +
                           size_t(2 * blockIdx.x + (s_first ? 0 : 1)) * 16 * NT;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = j >> 1, hh = j & 1;
                __stcg(mine + j * NT + tid,
                       make_float4(acc[i][2 * hh].x, acc[i][2 * hh].y, acc[i][2 * hh + 1].x,
                                   acc[i][2 * hh + 1].y));
            }
            continue;
        }

        // ---- epilogue: C = act(alpha * acc (+ beta * C_old) (+ bias)) ----
        int64_t bidx, row0, col0;
        tile_coords<T, kExt>(p, s_tile, &bidx, &row0, &col0);
        const float alpha = p.alpha, beta = p.beta;
        float *Cb = kExt ? p.C + bidx * p.strideC : p.C;
        const float *bias = kExt ? p.bias : nullptr;
        const int act = kExt ? p.act : kActNone;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = row0 + (i < 4 ? tm * 4 + i : T / 2 + tm * 4 + (i - 4));
            if (row >= p.M) continue;
            float *crow = Cb + row * p.ldc;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int64_t col = col0 + hh * (T / 2) + tn * 4;
                float v[4] = {alpha * acc[i][2 * hh].x, alpha * acc[i][2 * hh].y,
                              alpha * acc[i][2 * hh + 1].x, alpha * acc[i][2 * hh + 1].y};
                float *cp = crow + col;
                if (kVec && col + 3 < p.N) {
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
}

template <int T, int BK, int NP, bool kTransA, bool kTransB, bool kVec, bool kExt>
cudaError_t launch_sk_variant(const SkArgs &a, cudaStream_t stream) {
    auto kernel = ffma_sk_kernel<T, BK, NP, kTransA, kTransB, kVec, kExt>;
    constexpr int bytes = sk_smem_bytes(T, BK, NP, !kTransA, kTransB);
    static bool configured[64];
    const cudaError_t e =
        set_smem_once(reinterpret_cast<const void *>(kernel), bytes, configured, true);
    if (e != cudaSuccess) return e;
    kernel<<<unsigned(a.grid), Cfg<T, BK, NP>::kThreads, bytes, stream>>>(a);
    const cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
    // the stream-K tiles, if any, summed by a second launch on the stream
    ffma::ReduceArgs r{a.partials, a.C, a.bias, a.M, a.N, a.ldc, a.strideC, a.alpha, a.beta,
                       a.act,      a.tiles_m, a.tiles_n, 0, 0, 0, 0, 0, 0};
    r.first_tile = int64_t(a.dp_rounds) * a.grid;
    r.tiles = a.tiles - r.first_tile;
    r.kt = a.kt;
    r.grid = a.grid;
    r.sk_iters = a.sk_iters;
    return ffma::launch_partial_reduce<T, kVec, true, kExt>(r, stream);
}

// The slice and ring each layout is built with (sk_config gives the same
// numbers to the planner): operands that both arrive by direct copies (A^T
// and B) take K slices of T/4 in a three-page ring (96 KiB per 128-wide CTA);
// a staged operand keeps K slices of T/8 in a four-page ring (80 or 96 KiB
// per 128-wide CTA), two CTAs per SM either way.
template <bool kTransA, bool kTransB, bool kVec, bool kExt>
cudaError_t launch_sk_tile(const SkArgs &a, int tile, int bk, int pages, cudaStream_t stream) {
    constexpr bool kDirect = kTransA && !kTransB;
    if (tile == 128) {
        if (bk != sk_config_bk(128, kDirect) || pages != sk_config_pages(128, kDirect))
            return cudaErrorInvalidValue;
        return launch_sk_variant<128, kDirect ? 32 : 16, kDirect ? 3 : 4, kTransA, kTransB,
                                 kVec, kExt>(a, stream);
    }
    if (tile != 64 || bk != sk_config_bk(64, kDirect) || pages != sk_config_pages(64, kDirect))
        return cudaErrorInvalidValue;
    return launch_sk_variant<64, 8, 4, kTransA, kTransB, kVec, kExt>(a, stream);
}

}  // namespace sk
}  // namespace sgemm_impl
