// ffma_kernel.cuh -- the fp32 CUDA-core GEMM kernel for sm_103a (template).
//
// C_b = act(alpha * op(A_b) * op(B_b) + beta * C_b + bias), row-major, any
// M, N, K, for b in [0, batch); op(X) is X or X^T (the stored matrix read
// transposed).  The plain case (batch 1, no transposes, no bias/act) is the
// method's product C = alpha*A*B + beta*C.
//
// Design (prior art on the pages, re-derived for a 152-SM Blackwell part):
//  * Square CTA tiles (TileCfg): 128 x 128 with 256 threads (the main tile)
//    or 64 x 64 with 64 threads, K slices of T/8 -- or 32 when both operands
//    arrive by row copies -- and 8 x 8 accumulators per thread
//    updated as outer products: for every k the thread reads 8 values
//    of column k of the A tile and 8 of row k of the B tile and does 64 FMAs
//    (velog @levelstage "AutoMinepp4", section "행렬곱: by 벡터의 외적": the
//    product is a sum of outer products, which keeps the accumulators in
//    registers; "Micro_gemm_4x4 - cuBLAS micro GEMM skeleton", section 8:
//    the fully unrolled FMA pattern over the micro tile).
//  * Two issue forms of the same arithmetic: scalar fma.rn.f32 or packed
//    fma.rn.f32x2, each lane of which is an ordinary round-to-nearest fp32
//    FMA, so every accumulator sees exactly the same sequence of roundings
//    either way and the two give bit-identical C.  The packed form halves
//    the instruction stream; the planner picks it where the kernel stays
//    within its 128-register budget (the direct-copy kernel, split-K and
//    64-wide plans) and scalar issue elsewhere, where the broadcast operand
//    pairs spill.
//  * The 8 x 8 block is split into four 4 x 4 quadrants T/2 rows / columns
//    apart, so one 128-bit shared load serves 4 rows (or columns) and the
//    loads of a warp are conflict-free: a warp reads 4 distinct 16-byte A
//    chunks (each broadcast to 8 lanes) and 8 distinct B chunks.
//  * The smem tiles are k-major: As[k][m], Bs[k][n].  An operand whose
//    stored rows run along M (A^T) or N (B) is copied straight into them
//    with 16-byte cp.async.  An operand whose stored rows run along K (A, or
//    B^T) is staged through registers: a warp loads 8 rows x 16 k with
//    128-bit loads and scatters them into the tile with an XOR swizzle that
//    keeps the stores conflict-free (velog @levelstage "AutoMinepp7",
//    section "직사각형 타일링": chunks are fetched into registers before the
//    compute and split into the other local-memory page after it).
//  * The FMAs of a k step run in boustrophedon order (every two consecutive
//    FMAs share a source operand), which measured faster than row order.
//  * Two smem pages: slice t+1 is in flight (registers and async copies)
//    while slice t is computed; one barrier per K slice ("Micro_gemm_4x4 -
//    cuBLAS micro GEMM skeleton", section 8, double buffering, with the
//    asynchronous copy the page suggests for Ampere and later).  Shared-
//    memory fragments are double-buffered in registers across the 16 k steps.
//  * Edges: out-of-range A/B elements load as 0 and C stores are predicated
//    on row < M, col < N ("Micro_gemm_4x4 ...", sections 6 and 9; "GPU
//    Target", section "타일링된 행렬 곱셈": out-of-range loads read as zero).
//  * Epilogue: c = alpha * acc, then c = fma(beta, C_old, c) only when
//    beta != 0 (C is not read otherwise), then + bias[col] and the tanh
//    GELU when asked ("GPU Target", GPT-2 sublayers: x @ W + b, then the
//    outlined GELU kernel), stored with 128-bit stores.
//  * Batches are an outer index of the tile grid ("GPU Target", section
//    "타일링된 행렬 곱셈": the batched variant adds a grid dimension indexed
//    by batch, used per attention head).
//  * Split-K: when the tile grid cannot fill the GPU, K is cut into split_k
//    ranges (and, opt-in, only the tiles of a partly filled last wave into
//    tail_split ranges).  Every CTA of a split tile writes its partial tile
//    to the workspace; a second launch (partial_reduce_kernel) sums each
//    tile's partials in ascending range order and runs the epilogue.  The
//    sum order is fixed, so results are deterministic run to run.  (Summing
//    inside a thread-block cluster of the tile's CTAs through distributed
//    shared memory measured slower on GB300: clusters of 3, 6 and 9 CTAs
//    leave 291, 276 and 270 of the 304 CTA slots usable, and a CTA then
//    waits for the slowest of its cluster before a latency-bound exchange;
//    1024^3 57 -> 60 us, GPT-2 MLP-down 96 -> 136 us.)
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sgemm_internal.h"

namespace sgemm_impl {
namespace ffma {

__device__ __forceinline__ float4 ldg4(const float *p) {
    return __ldg(reinterpret_cast<const float4 *>(p));
}

__device__ __forceinline__ float ldg1(const float *p) { return __ldg(p); }

__device__ __forceinline__ unsigned smem_addr(const void *p) {
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global -> shared; bytes past `src_bytes` are zero-filled
// and not read.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

// 4-byte async copy; src_bytes == 0 writes a zero without reading.
__device__ __forceinline__ void cp_async4(void *dst, const void *src, int src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_addr(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;\n" ::: "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;\n" ::: "memory");
}

// Column of tile element (k, x) inside its smem row.  For a tile filled by
// transposing register stores, bits 3..4 of x are XOR-ed with k/4: every
// aligned group of 4 columns stays contiguous (fragment reads stay 128-bit)
// and the stores of a warp -- 8 rows x 4 k groups -- hit all 32 banks.  A tile
// filled by row copies needs no swizzle.
template <bool kSwizzle, int kKG = 4, int kShift = 3>
__device__ __forceinline__ int tcol(int k, int x) {
    if constexpr (kSwizzle)
        return x ^ (((k >> 2) & (kKG - 1)) << kShift);
    else
        return x;
}

// A square CTA tile of T x T outputs with K slices of T/8: 8 x 8 accumulators
// per thread in four 4 x 4 quadrants T/2 apart, (T/8)^2 threads, warps of 4
// (M) x 8 (N) threads.  With K slices of T/8 every thread stages exactly two
// float4 of each operand per slice, whatever T is.  T = 128 is the main
// tile; T = 64 serves grids too small to fill the GPU with 128-wide tiles.
// BK may be raised above T/8 (to 32 at T = 128) when both operands arrive
// by row copies: fewer barriers and less loop overhead per FMA.  Operands
// staged through registers need BK = T/8.
template <int T, int BK = T / 8>
struct TileCfg {
    static constexpr int kT = T;
    static constexpr int kBK = BK;
    static constexpr int kThreads = (T / 8) * (T / 8);
    static constexpr int kWarpsN = T / 64;              // warps along N
    static constexpr int kKG = kBK / 4;                 // 4-wide k groups per slice
    static constexpr int kShift = kKG == 4 ? 3 : 4;     // log2(32 / kKG)
    static constexpr int kCopyRows = T / 16;            // tile rows per copy pass
    static constexpr int kCopyPasses = BK / kCopyRows;
    // Pages of T x BK per operand: two, or three for the wide K slice (both
    // operands then arrive by cp.async only, so a third page lets two slices
    // be in flight; measured at 8192^3: 66.2 against 65.2 TFLOP/s).  Above
    // 48 KiB the tiles live in dynamic shared memory.
    static constexpr int kPages = BK > T / 8 ? 3 : 2;
    static constexpr int kSmemBytes = kPages * 2 * BK * T * 4;
    static constexpr bool kDynSmem = kSmemBytes > 48 * 1024 - 64;
    static constexpr int kMinBlocks = T == 128 ? 2 : 8; // resident CTAs per SM
    static_assert(T == 128 || T == 64, "tile is 128 or 64");
};

// The tanh form of GELU used by GPT-2: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))).
__device__ __forceinline__ float gelu_tanh(float x) {
    const float k0 = 0.7978845608028654f;   // sqrt(2/pi)
    const float u = k0 * fmaf(0.044715f * x, x * x, x);
    return 0.5f * x * (1.0f + tanhf(u));
}

// The (batch, tile, K range) CTA `pid` computes, and the tile's coordinates.
struct WorkItem {
    int64_t tile;   // global tile id over all batches
    int64_t batch;
    int64_t row0, col0;
    int64_t kbeg, kend;
    int split, nsplit;
};

__device__ __forceinline__ WorkItem work_item(const GemmArgs &p, int64_t pid, int tile) {
    WorkItem w;
    const int64_t lead = p.tail_start * p.split_k;
    int64_t kps;
    if (pid < lead) {
        w.tile = pid / p.split_k;
        w.split = int(pid - w.tile * p.split_k);
        w.nsplit = p.split_k;
        kps = p.k_per_split;
    } else {
        const int64_t j = pid - lead;
        w.tile = p.tail_start + j / p.tail_split;
        w.split = int(j % p.tail_split);
        w.nsplit = p.tail_split;
        kps = p.tail_k_per_split;
    }
    const int64_t per_batch = int64_t(p.tiles_m) * p.tiles_n;
    w.batch = w.tile / per_batch;
    const int64_t t = w.tile - w.batch * per_batch;
    // grouped raster over kGroupM tile rows (L2 reuse of A and B panels)
    const int64_t per_group = int64_t(kGroupM) * p.tiles_n;
    const int64_t group = t / per_group;
    const int64_t first_m = group * kGroupM;
    const int64_t gm = min(int64_t(p.tiles_m) - first_m, int64_t(kGroupM));
    const int64_t in_group = t - group * per_group;
    w.row0 = (first_m + in_group % gm) * tile;
    w.col0 = (in_group / gm) * tile;
    w.kbeg = int64_t(w.split) * kps;
    w.kend = min(p.K, w.kbeg + kps);
    return w;
}

// Batch and first row/column of global tile `tile` (the grouped raster of
// work_item), for the stream-K segments.
__device__ __forceinline__ WorkItem tile_item(const GemmArgs &p, int64_t tile, int tsize) {
    WorkItem w;
    w.tile = tile;
    const int64_t per_batch = int64_t(p.tiles_m) * p.tiles_n;
    w.batch = tile / per_batch;
    const int64_t t = tile - w.batch * per_batch;
    const int64_t per_group = int64_t(kGroupM) * p.tiles_n;
    const int64_t group = t / per_group;
    const int64_t first_m = group * kGroupM;
    const int64_t gm = min(int64_t(p.tiles_m) - first_m, int64_t(kGroupM));
    const int64_t in_group = t - group * per_group;
    w.row0 = (first_m + in_group % gm) * tsize;
    w.col0 = (in_group / gm) * tsize;
    w.kbeg = w.kend = 0;
    w.split = 0;
    w.nsplit = 1;
    return w;
}

// kExt: batches, bias and activation are compiled in (sgemm_ex); the plain
// product (sgemm) is built without them, which leaves it more registers.
// kSched = 1: a persistent stream-K launch -- each CTA loops over the
// segments (tile, K slices) of its share of the work, with the same main
// loop; a segment that is not a whole tile leaves its partial tile in the
// workspace, and partial_reduce_kernel sums them in ascending CTA order after the
// launch (see ffma_sk_kernel.cuh for the decomposition).  Measured on GB300
// with the A^T plan, the persistent loop issues a little worse than the
// one-tile-per-CTA grid (2048^3 with one whole tile per CTA: 351 against
// 338 us); summing the partials inside the persistent kernel cost far more
// (391 us, ncu at 4096^3: issue slots 75.9 % against 90.0 % busy, dispatch
// stalls 0.56 against 0.28 per issue), which is why the sum is a second
// launch.
template <int kTile, bool kPacked, bool kVec, bool kEdge, bool kSplit, bool kTransA,
          bool kTransB, bool kExt, int kBKT = kTile / 8, int kSched = 0>
__global__ void __launch_bounds__(TileCfg<kTile, kBKT>::kThreads,
                                  TileCfg<kTile, kBKT>::kMinBlocks)
ffma_gemm_kernel(const GemmArgs p) {
    using TC = TileCfg<kTile, kBKT>;
    constexpr int T = TC::kT, BK = TC::kBK, NT = TC::kThreads, KG = TC::kKG, SH = TC::kShift;
    static_assert(BK == T / 8 || (kTransA && !kTransB),
                  "register-staged operands need K slices of T/8");
    // A tile: As[k][m]; swizzled when filled by transposing stores (A not transposed)
    // B tile: Bs[k][n]; swizzled when filled by transposing stores (B transposed)
    constexpr bool kSwzA = !kTransA;
    constexpr bool kSwzB = kTransB;
    // Static tile pages (a one-row stand-in when the tiles are too large for
    // static shared memory and live in the dynamic block instead).
    constexpr int kStaticBK = TC::kDynSmem ? 1 : BK;
    __shared__ __align__(16) float sa[2][kStaticBK][T];
    __shared__ __align__(16) float sb[2][kStaticBK][T];
    extern __shared__ __align__(16) float dyn_smem[];
    constexpr int NP = TC::kPages;
    static_assert(NP == 2 || TC::kDynSmem, "three pages only for the dynamic layout");
    float (&As)[NP][BK][T] = *reinterpret_cast<float(*)[NP][BK][T]>(
        TC::kDynSmem ? dyn_smem : &sa[0][0][0]);
    float (&Bs)[NP][BK][T] = *reinterpret_cast<float(*)[NP][BK][T]>(
        TC::kDynSmem ? dyn_smem + NP * BK * T : &sb[0][0][0]);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // A^T plans follow the transpose pass as its programmatic dependent: wait
    // until that grid has completed and its writes are visible (a no-op when
    // the launch has no such dependency)
    if constexpr (kTransA) asm volatile("griddepcontrol.wait;\n" ::: "memory");

    // stream-K segment state (kSched = 1), advanced by thread 0 between two
    // barriers so it occupies no registers across the main loop
    __shared__ long long s_sk_it, s_sk_tile;
    __shared__ int s_sk_round, s_sk_k0, s_sk_k1, s_sk_first, s_sk_done;
    if constexpr (kSched == 1) {
        if (tid == 0) {
            s_sk_round = 0;
            s_sk_it = (long long)(int64_t(blockIdx.x) * p.sk_iters / gridDim.x);
        }
    }

    for (;;) {   // one pass unless kSched == 1
    // ---- (batch, tile, K range) of this CTA; recomputed after the main loop
    // so none of it stays live in registers across it ----
    int64_t row0, col0, kbeg, kend;
    const float *Ab;
    const float *Bb;
    if constexpr (kSched == 0) {
        const WorkItem w = work_item(p, blockIdx.x, T);
        row0 = w.row0;
        col0 = w.col0;
        kbeg = w.kbeg;
        kend = w.kend;
        Ab = kExt ? p.A + w.batch * p.strideA : p.A;
        Bb = kExt ? p.B + w.batch * p.strideB : p.B;
    } else {
        __syncthreads();   // everyone is done with the previous segment
        if (tid == 0) {
            const int G = gridDim.x, g = blockIdx.x;
            const int64_t U = p.sk_iters;
            const int64_t b_g = int64_t(g + 1) * U / G;   // end of this CTA's run
            const int64_t it = s_sk_it;
            s_sk_done = 0;
            if (s_sk_round < p.dp_rounds) {
                s_sk_tile = (long long)(int64_t(s_sk_round) * G + g);
                s_sk_k0 = 0;
                s_sk_k1 = p.sk_kt;
                s_sk_first = 0;
                ++s_sk_round;
            } else if (it < b_g) {
                const int64_t lt = it / p.sk_kt;
                const int k0 = int(it - lt * p.sk_kt);
                const int64_t left = b_g - it;
                const int k1 = left < int64_t(p.sk_kt - k0) ? k0 + int(left) : p.sk_kt;
                s_sk_tile = (long long)(int64_t(p.dp_rounds) * G + lt);
                s_sk_k0 = k0;
                s_sk_k1 = k1;
                s_sk_first = it == int64_t(g) * U / G;
                s_sk_it = (long long)(it + (k1 - k0));
            } else {
                s_sk_done = 1;
            }
        }
        __syncthreads();
        if (s_sk_done) {
            // the reduction launch may be scheduled once every CTA is here
            asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
            break;
        }
        const WorkItem w = tile_item(p, s_sk_tile, T);
        row0 = w.row0;
        col0 = w.col0;
        kbeg = int64_t(s_sk_k0) * BK;
        kend = min(p.K, int64_t(s_sk_k1) * BK);
        Ab = kExt ? p.A + w.batch * p.strideA : p.A;
        Bb = kExt ? p.B + w.batch * p.strideB : p.B;
    }
    const int nslices = kend > kbeg ? int((kend - kbeg + BK - 1) / BK) : 0;

    // ---- compute mapping: warp = 4 (M) x 8 (N) threads ----
    const int tm = (warp / TC::kWarpsN) * 4 + (lane >> 3);   // 0..T/8-1
    const int tn = (warp % TC::kWarpsN) * 8 + (lane & 7);    // 0..T/8-1

    // ---- load mapping ----
    // transposing operand (rows along K): rows r and r + T/2 of the tile, k
    // group kc (4 consecutive k): a warp reads 32/KG rows x KG*16 bytes a load.
    const int t_row = tid / KG;              // 0..T/2-1
    const int t_kc = tid % KG;               // 0..KG-1
    // copied operand (rows along M or N): tile rows k and k + T/16, 4 elements
    // at c_col.
    const int c_row = tid / (T / 4);         // 0..T/16-1
    const int c_col = (tid % (T / 4)) * 4;   // 0..T-4

    // A
    bool a_ok[2];
    const float *a_ptr[2];
    if constexpr (!kTransA) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t r = row0 + t_row + (T / 2) * h;
            a_ok[h] = !kEdge || r < p.M;
            a_ptr[h] = Ab + (a_ok[h] ? r : 0) * p.lda + kbeg + t_kc * 4;
        }
    } else {
        a_ok[0] = a_ok[1] = true;
        a_ptr[0] = Ab + (kbeg + c_row) * p.lda + row0 + c_col;
        a_ptr[1] = a_ptr[0];
    }
    // B
    bool b_ok[2];
    const float *b_ptr[2];
    if constexpr (kTransB) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t n = col0 + t_row + (T / 2) * h;
            b_ok[h] = !kEdge || n < p.N;
            b_ptr[h] = Bb + (b_ok[h] ? n : 0) * p.ldb + kbeg + t_kc * 4;
        }
    } else {
        b_ok[0] = b_ok[1] = true;
        b_ptr[0] = Bb + (kbeg + c_row) * p.ldb + col0 + c_col;
        b_ptr[1] = b_ptr[0];
    }

    float4 ra[2], rb[2];

    // rows along K -> registers (zero outside the matrix and outside [kbeg, kend))
    auto fetch_t = [&](int t, const bool (&ok)[2], const float *const (&ptr)[2], float4 (&r)[2]) {
        const int64_t koff = int64_t(t) * BK;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const float *src = ptr[h] + koff;
            if constexpr (!kEdge) {
                r[h] = ldg4(src);
            } else {
                const int64_t k = kbeg + koff + t_kc * 4;
                if (kVec && ok[h] && k + 3 < kend) {
                    r[h] = ldg4(src);
                } else {
                    r[h].x = (ok[h] && k + 0 < kend) ? ldg1(src + 0) : 0.0f;
                    r[h].y = (ok[h] && k + 1 < kend) ? ldg1(src + 1) : 0.0f;
                    r[h].z = (ok[h] && k + 2 < kend) ? ldg1(src + 2) : 0.0f;
                    r[h].w = (ok[h] && k + 3 < kend) ? ldg1(src + 3) : 0.0f;
                }
            }
        }
    };
    // registers -> tile rows k..k+3, transposed and swizzled
    auto stash_t = [&](float (*S)[T], const float4 (&r)[2]) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int x = t_row + (T / 2) * h;
            const int k = t_kc * 4;
            S[k + 0][tcol<true, KG, SH>(k, x)] = r[h].x;
            S[k + 1][tcol<true, KG, SH>(k, x)] = r[h].y;
            S[k + 2][tcol<true, KG, SH>(k, x)] = r[h].z;
            S[k + 3][tcol<true, KG, SH>(k, x)] = r[h].w;
        }
    };
    // rows along M/N -> tile, async copies (zero-filled outside); `lim` is M or N
    auto copy_c = [&](int t, float (*S)[T], const float *base, int64_t ld, int64_t x0,
                      int64_t lim, const float *dummy) {
        const int64_t koff = int64_t(t) * BK;
#pragma unroll
        for (int h = 0; h < TC::kCopyPasses; ++h) {
            const float *src = base + (koff + TC::kCopyRows * h) * ld;
            float *dst = &S[c_row + TC::kCopyRows * h][c_col];
            if constexpr (!kEdge) {
                cp_async16(dst, src, 16);
            } else {
                const int64_t k = kbeg + koff + c_row + TC::kCopyRows * h;
                const int64_t c = x0 + c_col;
                const bool k_ok = k < kend;
                if constexpr (kVec) {
                    int64_t n = k_ok ? lim - c : 0;
                    n = n < 0 ? 0 : (n > 4 ? 4 : n);
                    cp_async16(dst, n > 0 ? src : dummy, int(n) * 4);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const bool ok = k_ok && c + e < lim;
                        cp_async4(dst + e, ok ? src + e : dummy, ok ? 4 : 0);
                    }
                }
            }
        }
    };

    auto issue = [&](int t, int page) {
        if constexpr (kTransA) copy_c(t, As[page], a_ptr[0], p.lda, row0, p.M, p.A);
        if constexpr (!kTransB) copy_c(t, Bs[page], b_ptr[0], p.ldb, col0, p.N, p.B);
        cp_async_commit();
        if constexpr (!kTransA) fetch_t(t, a_ok, a_ptr, ra);
        if constexpr (kTransB) fetch_t(t, b_ok, b_ptr, rb);
    };
    auto land = [&](int page) {
        if constexpr (!kTransA) stash_t(As[page], ra);
        if constexpr (kTransB) stash_t(Bs[page], rb);
        cp_async_wait_all();
    };

    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.0f, 0.0f);

    // With three pages (copies only) slices t+1 and t+2 are in flight while t
    // is computed: wait for slice t's copy group, one barrier, refill the
    // page slice t-1 used.  With two pages slice t+1 is fetched during t.
    constexpr bool kMulti = NP > 2;
    static_assert(!kMulti || (kTransA && !kTransB), "three pages need copy-only operands");
    if constexpr (kMulti) {
#pragma unroll
        for (int q = 0; q < NP - 1; ++q) {
            if (q < nslices)
                issue(q, q);
            else
                cp_async_commit();   // keep one group per slice
        }
    } else {
        if (nslices > 0) {
            issue(0, 0);
            land(0);
        }
        __syncthreads();
    }

    for (int t = 0; t < nslices; ++t) {
        int page;
        bool more;
        if constexpr (kMulti) {
            page = t % NP;
            more = false;
            asm volatile("cp.async.wait_group %0;\n" ::"n"(NP - 2) : "memory");
            __syncthreads();
            const int nt = t + NP - 1;
            if (nt < nslices)
                issue(nt, nt % NP);
            else
                cp_async_commit();
        } else {
            page = t & 1;
            more = t + 1 < nslices;
            if (more) issue(t + 1, page ^ 1);
        }

        float4 af[2][2], bf[2][2];
        af[0][0] = *reinterpret_cast<const float4 *>(&As[page][0][tcol<kSwzA, KG, SH>(0, tm * 4)]);
        af[0][1] = *reinterpret_cast<const float4 *>(
            &As[page][0][tcol<kSwzA, KG, SH>(0, T / 2 + tm * 4)]);
        bf[0][0] = *reinterpret_cast<const float4 *>(&Bs[page][0][tcol<kSwzB, KG, SH>(0, tn * 4)]);
        bf[0][1] = *reinterpret_cast<const float4 *>(
            &Bs[page][0][tcol<kSwzB, KG, SH>(0, T / 2 + tn * 4)]);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const int cur = kk & 1;
            if (kk + 1 < BK) {
                af[cur ^ 1][0] = *reinterpret_cast<const float4 *>(
                    &As[page][kk + 1][tcol<kSwzA, KG, SH>(kk + 1, tm * 4)]);
                af[cur ^ 1][1] = *reinterpret_cast<const float4 *>(
                    &As[page][kk + 1][tcol<kSwzA, KG, SH>(kk + 1, T / 2 + tm * 4)]);
                bf[cur ^ 1][0] = *reinterpret_cast<const float4 *>(
                    &Bs[page][kk + 1][tcol<kSwzB, KG, SH>(kk + 1, tn * 4)]);
                bf[cur ^ 1][1] = *reinterpret_cast<const float4 *>(
                    &Bs[page][kk + 1][tcol<kSwzB, KG, SH>(kk + 1, T / 2 + tn * 4)]);
            }
            const float a[8] = {af[cur][0].x, af[cur][0].y, af[cur][0].z, af[cur][0].w,
                                af[cur][1].x, af[cur][1].y, af[cur][1].z, af[cur][1].w};
            const float2 b[4] = {make_float2(bf[cur][0].x, bf[cur][0].y),
                                 make_float2(bf[cur][0].z, bf[cur][0].w),
                                 make_float2(bf[cur][1].x, bf[cur][1].y),
                                 make_float2(bf[cur][1].z, bf[cur][1].w)};
            if constexpr (kPacked) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
                }
            } else {
                // Boustrophedon order over the 8 x 8 block: along row i the
                // FMAs share a[i]; odd rows run right to left (column pairs
                // and the two columns of a pair reversed), so the last FMA of
                // a row and the first of the next share b[j].  Every two
                // consecutive FMAs thus share a source operand, which the
                // operand reuse path can serve; measured on GB300 this order
                // is 1-2 % faster than plain row order and 5-8 % faster than
                // column order.  The order of the k steps, and so every
                // accumulator's rounding sequence, is unchanged.
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
        }
        if constexpr (!kMulti) {
            if (more) land(page ^ 1);
            __syncthreads();
        }
    }

    // ---- stream-K: a segment that is not a whole tile leaves its partial
    // tile in this CTA's slot (2g for its run's first segment, 2g + 1 for
    // its last) and moves on; partial_reduce_kernel sums the slots afterwards ----
    if constexpr (kSched == 1) {
        if (s_sk_k0 != 0 || s_sk_k1 != p.sk_kt) {
            float4 *mine = reinterpret_cast<float4 *>(p.partials) +
                           size_t(2 * blockIdx.x + (s_sk_first ? 0 : 1)) * 16 * NT;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = j >> 1, h = j & 1;
                __stcg(mine + j * NT + tid,
                       make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                   acc[i][2 * h + 1].y));
            }
            continue;
        }
    }

    // ---- split-K: a CTA of a split tile leaves its partial tile in its
    // slot (the tile's ranges own consecutive slots) and is done;
    // partial_reduce_kernel sums each tile's slots in range order ----
    if constexpr (kSplit && kSched == 0) {
        // the reduction launch may be scheduled once every CTA is here
        asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
        const WorkItem w = work_item(p, blockIdx.x, T);
        if (w.nsplit > 1) {
            float4 *mine = reinterpret_cast<float4 *>(p.partials) +
                           size_t(int64_t(blockIdx.x) - p.part_base) * 16 * NT;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = j >> 1, h = j & 1;
                __stcg(mine + j * NT + tid,
                       make_float4(acc[i][2 * h].x, acc[i][2 * h].y, acc[i][2 * h + 1].x,
                                   acc[i][2 * h + 1].y));
            }
            return;
        }
    }

    // ---- epilogue: C = act(alpha * acc (+ beta * C_old) (+ bias)) ----
    const float alpha = p.alpha, beta = p.beta;
    float *Cb = p.C;
    if (kExt && p.batch > 1) {
        if constexpr (kSched == 1)
            Cb += tile_item(p, s_sk_tile, T).batch * p.strideC;
        else
            Cb += work_item(p, blockIdx.x, T).batch * p.strideC;
    }
    const float *bias = kExt ? p.bias : nullptr;
    const int act = kExt ? p.act : kActNone;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = row0 + (i < 4 ? tm * 4 + i : T / 2 + tm * 4 + (i - 4));
        if (kEdge && row >= p.M) continue;
        float *crow = Cb + row * p.ldc;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t col = col0 + h * (T / 2) + tn * 4;
            float v[4] = {alpha * acc[i][2 * h].x, alpha * acc[i][2 * h].y,
                          alpha * acc[i][2 * h + 1].x, alpha * acc[i][2 * h + 1].y};
            float *cp = crow + col;
            if (!kEdge || (kVec && col + 3 < p.N)) {
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
    if constexpr (kSched == 0) break;
    }   // segment loop
}

// What the reduction of partial tiles needs of a launch (filled from
// GemmArgs or SkArgs by the product kernels' launchers).
struct ReduceArgs {
    const float *partials;   // partial tiles of (T/8)^2 * 16 float4 each
    float *C;
    const float *bias;
    int64_t M, N, ldc, strideC;
    float alpha, beta;
    int32_t act;
    int32_t tiles_m, tiles_n;
    int64_t first_tile;      // global id of the first tile reduced
    int64_t tiles;           // tiles reduced: first_tile .. first_tile + tiles - 1
    // split-K (split > 1): tile first_tile + i sums slots i*split .. i*split + split - 1
    int32_t split;
    // stream-K (split == 0): the sk_iters K slices of the tiles, kt per tile,
    // were cut into `grid` equal runs; run g left its first segment in slot
    // 2g and its last in slot 2g + 1
    int32_t kt;
    int32_t grid;
    int64_t sk_iters;
};

// The second half of a split-K or stream-K launch: for every tile whose K
// range several CTAs shared, the sum of their partial tiles in K order and
// the same epilogue as the product kernels.  Split-K: the tile's ranges in
// ascending order.  Stream-K: the first contributor's slot (2g, or 2g + 1
// when the tile does not start its run), then slot 2h of each later CTA h,
// which holds that run's first segment.  Four CTAs per tile, each a quarter
// of the accumulator rows with the product kernels' thread mapping, so a
// thread reads back exactly the values one product thread stored; all of a
// thread's loads of one contributor are in flight together.  A stream-K
// tile that one CTA computed whole was stored by the product kernel; its
// CTAs return at once.
//
// Summing in a second launch rather than in the product kernel's last CTA
// to arrive keeps the product kernels' main loops as fast as the plain
// grid's (measured on GB300, persistent stream-K with the A^T plan at
// 2048^3: 324 us against 342 with the sum in the persistent kernel; ncu at
// 4096^3 put the in-kernel version's issue slots at 75.9 % busy against
// 90.0 %, with twice the dispatch stalls), and the reduction runs on every
// SM at once instead of on one CTA per tile after all the others.
template <int kTile, bool kVec, bool kEdge, bool kExt>
__global__ void __launch_bounds__(TileCfg<kTile>::kThreads) partial_reduce_kernel(const ReduceArgs p) {
    using TC = TileCfg<kTile>;
    constexpr int T = TC::kT, NT = TC::kThreads;
    const int64_t i_tile = blockIdx.x >> 2;  // tile among those reduced
    const int q = blockIdx.x & 3;            // accumulator rows 2q, 2q + 1
    int64_t slot0, c_lo, c_hi, stride, base;  // slots: slot0, then base + stride * c
    if (p.split > 1) {
        slot0 = i_tile * p.split;
        base = slot0;
        stride = 1;
        c_lo = 1;
        c_hi = p.split - 1;
    } else {
        const int64_t G = p.grid, U = p.sk_iters;
        const int64_t x0 = i_tile * p.kt;    // the tile's first slice
        // contributors: CTA h's run starts at slice h*U/G, so the first is
        // the largest h with h*U/G <= x0, the last the largest with
        // h*U/G <= x0 + kt - 1
        const int64_t g_first = ((x0 + 1) * G - 1) / U;
        const int64_t g_last = ((x0 + p.kt) * G - 1) / U;
        if (g_first == g_last) return;
        slot0 = 2 * g_first + ((g_first * U) / G == x0 ? 0 : 1);
        base = 0;
        stride = 2;
        c_lo = g_first + 1;
        c_hi = g_last;
    }

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int tm = (warp / TC::kWarpsN) * 4 + (lane >> 3);
    const int tn = (warp % TC::kWarpsN) * 8 + (lane & 7);

    // the tile's batch and origin: batch-major, grouped raster within a batch
    const int64_t tile = p.first_tile + i_tile;
    const int64_t per_batch = int64_t(p.tiles_m) * p.tiles_n;
    const int64_t bidx = tile / per_batch;
    const int64_t t_in = tile - bidx * per_batch;
    const int64_t per_group = int64_t(kGroupM) * p.tiles_n;
    const int64_t first_m = (t_in / per_group) * kGroupM;
    const int64_t gm = min(int64_t(p.tiles_m) - first_m, int64_t(kGroupM));
    const int64_t in_group = t_in - (t_in / per_group) * per_group;
    const int64_t row0 = (first_m + in_group % gm) * T;
    const int64_t col0 = (in_group / gm) * T;

    float *Cb = kExt ? p.C + bidx * p.strideC : p.C;
    const float *bias = kExt ? p.bias : nullptr;
    const int act = kExt ? p.act : kActNone;
    const float alpha = p.alpha, beta = p.beta;

    // Everything above ran while the product kernel may still be running
    // (programmatic dependent launch); from here on its partial tiles are
    // complete and visible.  The old C values the product kernel never
    // touches are fetched first, beside the partials.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    float4 old[4];
    bool whole[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = (4 * q + j) >> 1, h = j & 1;
        const int64_t row = row0 + (i < 4 ? tm * 4 + i : T / 2 + tm * 4 + (i - 4));
        const int64_t col = col0 + h * (T / 2) + tn * 4;
        whole[j] = !kEdge || (row < p.M && kVec && col + 3 < p.N);
        old[j] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (beta != 0.0f && whole[j])
            old[j] = *reinterpret_cast<const float4 *>(Cb + row * p.ldc + col);
    }
    // partial sums in contributor order, four contributors' loads in flight
    const float4 *part = reinterpret_cast<const float4 *>(p.partials) + (4 * q) * NT + tid;
    float4 s[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] = __ldcg(part + size_t(slot0) * 16 * NT + j * NT);
    for (int64_t c0 = c_lo; c0 <= c_hi; c0 += 4) {
        float4 v[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u <= c_hi) {
                const float4 *src = part + size_t(base + stride * (c0 + u)) * 16 * NT;
#pragma unroll
                for (int j = 0; j < 4; ++j) v[u][j] = __ldcg(src + j * NT);
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (c0 + u <= c_hi) {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    s[j].x += v[u][j].x;
                    s[j].y += v[u][j].y;
                    s[j].z += v[u][j].z;
                    s[j].w += v[u][j].w;
                }
            }
        }
    }

#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int i = (4 * q + j) >> 1, h = j & 1;
        const int64_t row = row0 + (i < 4 ? tm * 4 + i : T / 2 + tm * 4 + (i - 4));
        if (kEdge && row >= p.M) continue;
        const int64_t col = col0 + h * (T / 2) + tn * 4;
        float *cp = Cb + row * p.ldc + col;
        float v[4] = {alpha * s[j].x, alpha * s[j].y, alpha * s[j].z, alpha * s[j].w};
        if (whole[j]) {
            if (beta != 0.0f) {
                v[0] = fmaf(beta, old[j].x, v[0]);
                v[1] = fmaf(beta, old[j].y, v[1]);
                v[2] = fmaf(beta, old[j].z, v[2]);
                v[3] = fmaf(beta, old[j].w, v[3]);
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

// Launches partial_reduce_kernel over r.tiles tiles (nothing when there
// are none).
// It is launched as a programmatic dependent of the product kernel: its
// CTAs may be scheduled once every product CTA has passed its main loop, and
// they wait (griddepcontrol.wait, released by the hardware when the product
// grid has completed and its writes are visible) before reading a partial.
template <int kTile, bool kVec, bool kEdge, bool kExt>
cudaError_t launch_partial_reduce(const ReduceArgs &r, cudaStream_t stream) {
    if (r.tiles <= 0 || (r.split <= 1 && r.sk_iters <= 0)) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(4 * r.tiles), 1, 1);
    cfg.blockDim = dim3(TileCfg<kTile>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, partial_reduce_kernel<kTile, kVec, kEdge, kExt>, r);
}

// `pdl`: launch as a programmatic dependent of the previous kernel on the
// stream (the transpose pass of an A^T plan; the kernel waits for it).
template <int kTile, bool kPacked, bool kVec, bool kEdge, bool kSplit, bool kTransA,
          bool kTransB, bool kExt, int kBKT = kTile / 8, int kSched = 0>
cudaError_t launch_variant(const GemmArgs &a, cudaStream_t stream, int64_t sk_grid = 0,
                           bool pdl = false) {
    using TC = TileCfg<kTile, kBKT>;
    auto kernel = ffma_gemm_kernel<kTile, kPacked, kVec, kEdge, kSplit, kTransA, kTransB, kExt,
                                   kBKT, kSched>;
    int dyn = 0;
    if constexpr (TC::kDynSmem) {
        static bool configured[64];
        dyn = TC::kSmemBytes;
        const cudaError_t e =
            set_smem_once(reinterpret_cast<const void *>(kernel), dyn, configured);
        if (e != cudaSuccess) return e;
    }
    const int64_t tiles = int64_t(a.tiles_m) * a.tiles_n * a.batch;
    const dim3 grid(kSched == 1 ? unsigned(sk_grid)
                                : unsigned(a.tail_start * a.split_k +
                                           (tiles - a.tail_start) * a.tail_split),
                    1, 1);
    if (pdl) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(TC::kThreads, 1, 1);
        cfg.dynamicSmemBytes = size_t(dyn);
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, a);
        if (e != cudaSuccess) return e;
    } else {
        kernel<<<grid, TC::kThreads, dyn, stream>>>(a);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    // split or stream-K tiles, if any, are summed by a second launch
    ReduceArgs r{a.partials, a.C, a.bias, a.M, a.N, a.ldc, a.strideC, a.alpha, a.beta, a.act,
                 a.tiles_m, a.tiles_n, 0, 0, 0, 0, 0, 0};
    if constexpr (kSched == 1) {
        r.first_tile = int64_t(a.dp_rounds) * sk_grid;
        r.tiles = tiles - r.first_tile;
        r.kt = a.sk_kt;
        r.grid = int32_t(sk_grid);
        r.sk_iters = a.sk_iters;
        return launch_partial_reduce<kTile, kVec, kEdge, kExt>(r, stream);
    } else if constexpr (kSplit) {
        if (a.split_k > 1) {
            r.first_tile = 0;
            r.tiles = tiles;
            r.split = a.split_k;
        } else {
            r.first_tile = a.tail_start;
            r.tiles = tiles - a.tail_start;
            r.split = a.tail_split;
        }
        return launch_partial_reduce<kTile, kVec, kEdge, kExt>(r, stream);
    }
    return cudaSuccess;
}

// All (vec, edge, split) variants of one tile, layout and issue form.
template <int kTile, bool kPacked, bool kTransA, bool kTransB, bool kExt>
cudaError_t launch_layout(const GemmArgs &a, bool vec, bool edge, cudaStream_t stream) {
    const bool split = a.split_k > 1 || a.tail_split > 1;
    if (!edge) {
        // full tiles are only planned on the vector path
        return split
                   ? launch_variant<kTile, kPacked, true, false, true, kTransA, kTransB, kExt>(a, stream)
                   : launch_variant<kTile, kPacked, true, false, false, kTransA, kTransB, kExt>(
                         a, stream);
    }
    if (vec)
        return split
                   ? launch_variant<kTile, kPacked, true, true, true, kTransA, kTransB, kExt>(a, stream)
                   : launch_variant<kTile, kPacked, true, true, false, kTransA, kTransB, kExt>(a, stream);
    return split
               ? launch_variant<kTile, kPacked, false, true, true, kTransA, kTransB, kExt>(a, stream)
               : launch_variant<kTile, kPacked, false, true, false, kTransA, kTransB, kExt>(a, stream);
}

}  // namespace ffma
}  // namespace sgemm_impl
