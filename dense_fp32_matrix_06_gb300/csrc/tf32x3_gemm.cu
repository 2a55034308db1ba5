// tf32x3_gemm.cu -- the separately reported tensor-core mode: fp32 GEMM from
// three TF32 tensor-core products (split precision), on sm_103a tcgen05.
//
// C = alpha * A * B + beta * C with A = A_hi + A_lo, B = B_hi + B_lo, where
// x_hi is x rounded to TF32 (10 explicit mantissa bits, round to nearest
// even) and x_lo = x - x_hi (exact in fp32) rounded to TF32 as well.  Then
//     A*B ~= A_lo*B_hi + A_hi*B_lo + A_hi*B_hi
// (the dropped A_lo*B_lo term is ~2^-22 of |A||B|), each product on the
// tensor cores with fp32 accumulation in tensor memory.  The pages have no
// tensor-core path; the computation is the same dense contraction as the
// FFMA kernel, so the tensor cores are its natural home on this chip.
//
// Pipeline:
//  1. split kernels: A (M x K) -> A_hi, A_lo (M x Kp, K-major);
//     B (K x N) -> B_hi^T, B_lo^T (N x Kp, K-major, transposed through smem
//     tiles), Kp = K rounded up to 4 so TMA row strides are 16-byte multiples.
//  2. mma kernel, one 128 x BN output tile per CTA, 128 threads:
//     warp 0 lane 0 issues TMA loads (128-byte swizzled boxes of 32 fp32 of K)
//     of the four operand tiles into a STAGES-deep smem ring; warp 1 owns the
//     tensor-memory allocation and lane 0 issues tcgen05.mma.kind::tf32
//     (M=128, N=BN, K=8) three times per 8-wide K step, committing each stage
//     back to its producer barrier; then all four warps read the accumulator
//     out of TMEM (tcgen05.ld 32x32b) and apply alpha/beta.
//  Every mbarrier wait is bounded by a time limit; on expiry the thread sets
//  the device error word, the epilogue stores nothing, in-flight copies are
//  waited for (bounded) and the TMEM is freed before the CTA exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <utility>

#include "sgemm_internal.h"

namespace sgemm_impl {

// Device error word of the tensor-core mode (bit 0: a bounded wait expired).
static __device__ unsigned g_tc_error;

namespace {

constexpr int kTcBM = 128;
constexpr int kTcBK = 32;            // fp32 elements per 128-byte swizzle row
constexpr int kTcThreads = 128;

// ---------------------------------------------------------------------------
// split into TF32 hi/lo parts
// ---------------------------------------------------------------------------

// Nearest TF32 value (ties to even) of a finite fp32 x; inf/NaN pass through.
// Written with selects rather than early returns so that the many
// conversions a thread does stay one basic block the compiler can interleave.
__device__ __forceinline__ float tf32_round(float x) {
    const uint32_t u = __float_as_uint(x);
    const uint32_t r = (u + 0x00000fffu + ((u >> 13) & 1u)) & 0xffffe000u;
    const bool special = (u & 0x7f800000u) == 0x7f800000u;   // inf or NaN: unchanged
    const bool overflow = (r & 0x7f800000u) == 0x7f800000u;  // finite rounded to inf: truncate
    const uint32_t t = overflow ? (u & 0xffffe000u) : r;
    return __uint_as_float(special ? u : t);
}

__device__ __forceinline__ void split2(float x, float &hi, float &lo) {
    hi = tf32_round(x);
    lo = tf32_round(x - hi);
}

// X (rows x cols, row stride ldx) -> hi, lo (rows x cols, row stride ldo).
__global__ void split_rows_kernel(const float *__restrict__ X, int64_t rows, int64_t cols,
                                  int64_t ldx, float *__restrict__ hi, float *__restrict__ lo,
                                  int64_t ldo) {
    // the kernel after it may be scheduled as soon as every CTA has started
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t total = rows * cols;
    for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = e / cols, c = e - r * cols;
        float h, l;
        split2(X[r * ldx + c], h, l);
        hi[r * ldo + c] = h;
        lo[r * ldo + c] = l;
    }
}

// B (K x N, row stride ldb) -> hiT, loT (N x K, row stride ldo): 32 x 32 tiles
// through padded smem so both the reads and the writes are coalesced.
__global__ void split_transpose_kernel(const float *__restrict__ B, int64_t K, int64_t N,
                                       int64_t ldb, float *__restrict__ hiT,
                                       float *__restrict__ loT, int64_t ldo) {
    __shared__ float th[32][33];
    __shared__ float tl[32][33];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t k0 = int64_t(blockIdx.y) * 32, n0 = int64_t(blockIdx.x) * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;   // 32 x 8
    for (int i = ty; i < 32; i += 8) {
        const int64_t k = k0 + i, n = n0 + tx;
        float h = 0.0f, l = 0.0f;
        if (k < K && n < N) split2(B[k * ldb + n], h, l);
        th[i][tx] = h;
        tl[i][tx] = l;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int64_t n = n0 + i, k = k0 + tx;
        if (n < N && k < K) {
            hiT[n * ldo + k] = th[tx][i];
            loT[n * ldo + k] = tl[tx][i];
        }
    }
    // Launched as a programmatic dependent of A's split pass (which it does
    // not read), it completes only after that pass has: the product after it
    // then sees both.  A no-op otherwise.
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// The same with 64 x 64 tiles and 128-bit global accesses, for B 16-byte
// aligned with ldb % 4 == 0 (ldo is a multiple of 4 and the outputs are
// 256-byte aligned): 256 threads each load four float4 along n and store four
// float4 of each output along k.  Rows of the tiles are padded by one float.
__global__ void __launch_bounds__(256)
split_transpose64_kernel(const float *__restrict__ B, int64_t K, int64_t N, int64_t ldb,
                         float *__restrict__ hiT, float *__restrict__ loT, int64_t ldo) {
    __shared__ float th[64][65];
    __shared__ float tl[64][65];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t k0 = int64_t(blockIdx.y) * 64, n0 = int64_t(blockIdx.x) * 64;
    const int t = threadIdx.x;
    const int c4 = (t & 15) * 4;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (t >> 4) + 16 * i;   // tile row (k)
        const int64_t k = k0 + r, n = n0 + c4;
        float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (k < K) {
            if (n + 3 < N) {
                v = __ldg(reinterpret_cast<const float4 *>(B + k * ldb + n));
            } else {
                const float *src = B + k * ldb;
                v.x = n + 0 < N ? src[n + 0] : 0.0f;
                v.y = n + 1 < N ? src[n + 1] : 0.0f;
                v.z = n + 2 < N ? src[n + 2] : 0.0f;
                v.w = n + 3 < N ? src[n + 3] : 0.0f;
            }
        }
        float h, l;
        split2(v.x, h, l);
        th[r][c4 + 0] = h;
        tl[r][c4 + 0] = l;
        split2(v.y, h, l);
        th[r][c4 + 1] = h;
        tl[r][c4 + 1] = l;
        split2(v.z, h, l);
        th[r][c4 + 2] = h;
        tl[r][c4 + 2] = l;
        split2(v.w, h, l);
        th[r][c4 + 3] = h;
        tl[r][c4 + 3] = l;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = (t >> 4) + 16 * i;   // tile column (n) = output row
        const int64_t n = n0 + r, k = k0 + c4;
        if (n < N && k < K) {
            // k .. k+3 stay inside the output row (ldo >= K rounded up to 4);
            // entries past K are zeros
            *reinterpret_cast<float4 *>(hiT + n * ldo + k) =
                make_float4(th[c4][r], th[c4 + 1][r], th[c4 + 2][r], th[c4 + 3][r]);
            *reinterpret_cast<float4 *>(loT + n * ldo + k) =
                make_float4(tl[c4][r], tl[c4 + 1][r], tl[c4 + 2][r], tl[c4 + 3][r]);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // as in split_transpose_kernel
}

// ---------------------------------------------------------------------------
// PTX wrappers (mbarrier, TMA, tcgen05)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ float4 lds128(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait until the phase of parity `parity` of `bar` has completed, for at most
// `limit_ns`.  On expiry set the error word and return false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) {
            atomicOr(&g_tc_error, 1u);
            return false;
        }
    }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int32_t c0,
                                            int32_t c1, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
        : "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes in 8-row (1024-byte) swizzle atoms laid out back to back.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = 0;
    d |= uint64_t((addr & 0x3FFFFu) >> 4);       // start address
    d |= uint64_t(16 >> 4) << 16;                // leading byte offset (unused here)
    d |= uint64_t(1024 >> 4) << 32;              // stride byte offset: next 8-row group
    d |= uint64_t(1) << 46;                      // descriptor version
    d |= uint64_t(2) << 61;                      // 128-byte swizzle
    return d;
}

// Instruction descriptor: D fp32, A and B tf32, both K-major, M = 128, N = bn.
__host__ __device__ constexpr uint32_t tf32_idesc(int bn) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(bn >> 3) << 17) |
           (uint32_t(kTcBM >> 4) << 24);
}

__device__ __forceinline__ void mma_tf32(uint32_t tmem_d, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, "
        "[%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

struct TcArgs {
    float *C;
    int64_t M, N, K, ldc;
    float alpha, beta;
    int32_t tiles_m, tiles_n;
    uint64_t limit_ns;     // bound on every mbarrier wait
    int32_t inject_stall;  // 1: the producer issues nothing (exercises the bounded waits)
    // Work decomposition: tiles [0, tail_start) are cut into `split` K ranges
    // of kb_per_split blocks, tiles [tail_start, tiles) into `tail_split`
    // ranges of tail_kb_per_split (only the last, partly filled wave of tiles
    // is cut when split == 1).  The ranges of a tile are consecutive CTAs.
    // Split tiles only: partial slot of CTA x is x - part_base; flag of tile
    // t is counters[t - cnt_base] (set only by a range whose waits expired).
    int32_t split;
    int32_t kb_per_split;
    int32_t tail_start;
    int32_t tail_split;
    int32_t tail_kb_per_split;
    int32_t part_base;
    int32_t cnt_base;
    unsigned *counters;    // split tiles: one failure flag per tile, zero on entry and exit
    float *partials;       // split > 1: tiles * split partial tiles of 128 x BN
};

// (tile, K range) of this CTA.
struct TcWork {
    int pid;          // tile
    int sidx, ns;     // range index, ranges of the tile
    int kbps;         // K blocks per range
    int slot_first;   // partial slot of the tile's first range
    int cnt;          // flag index
};

__device__ __forceinline__ TcWork tc_work(const TcArgs &p) {
    TcWork w;
    const int x = int(blockIdx.x);
    const int lead = p.tail_start * p.split;
    if (x < lead) {
        w.pid = x / p.split;
        w.sidx = x - w.pid * p.split;
        w.ns = p.split;
        w.kbps = p.kb_per_split;
    } else {
        const int j = x - lead;
        w.pid = p.tail_start + j / p.tail_split;
        w.sidx = j % p.tail_split;
        w.ns = p.tail_split;
        w.kbps = p.tail_kb_per_split;
    }
    w.slot_first = x - w.sidx - p.part_base;
    w.cnt = w.pid - p.cnt_base;
    return w;
}

template <int BN, int STAGES>
struct TcSmem {
    static constexpr int kABytes = kTcBM * kTcBK * 4;          // 16 KiB
    static constexpr int kBBytes = BN * kTcBK * 4;
    static constexpr int kStageBytes = 2 * kABytes + 2 * kBBytes;
    static constexpr int kBarOffset = STAGES * kStageBytes;
    // full[STAGES], empty[STAGES], done, then the TMEM address slot
    static constexpr int kBytes = kBarOffset + (2 * STAGES + 1) * 8 + 8;
    static constexpr int kDynBytes = kBytes + 1024;            // room to align to 1024
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kTcThreads, 1)
tf32x3_mma_kernel(const __grid_constant__ CUtensorMap map_a_hi,
                  const __grid_constant__ CUtensorMap map_a_lo,
                  const __grid_constant__ CUtensorMap map_b_hi,
                  const __grid_constant__ CUtensorMap map_b_lo, const TcArgs p) {
    using L = TcSmem<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + L::kBarOffset;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::kBarOffset + (2 * STAGES + 1) * 8);
    auto a_hi = [&](int s) { return base + s * L::kStageBytes; };
    auto a_lo = [&](int s) { return base + s * L::kStageBytes + L::kABytes; };
    auto b_hi = [&](int s) { return base + s * L::kStageBytes + 2 * L::kABytes; };
    auto b_lo = [&](int s) { return base + s * L::kStageBytes + 2 * L::kABytes + L::kBBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int s_mma_ok;

    // (tile, K range) of this CTA; grouped raster over 8 tile rows
    const TcWork work = tc_work(p);
    const int pid = work.pid;
    const int split_idx = work.sidx;
    const int per_group = 8 * p.tiles_n;
    const int group = pid / per_group;
    const int first_m = group * 8;
    const int gm = min(p.tiles_m - first_m, 8);
    const int in_group = pid - group * per_group;
    const int tile_m = first_m + in_group % gm;
    const int tile_n = in_group / gm;
    const int m0 = tile_m * kTcBM;
    const int n0 = tile_n * BN;
    const int nkb_all = int((p.K + kTcBK - 1) / kTcBK);
    const int kb0 = split_idx * work.kbps;
    const int nkb = max(0, min(nkb_all, kb0 + work.kbps) - kb0);   // K blocks of this CTA

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(uint32_t(BN))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // After a split pass this kernel is its programmatic dependent: the setup
    // above overlapped the pass's tail; nothing is read before it completes.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int issued = 0;   // k-blocks the producer issued (thread 0 only)
    if (warp == 0 && lane == 0) {
        // ---- TMA producer ----
        if (!p.inject_stall) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t use = uint32_t(kb / STAGES);
                if (kb >= STAGES && !mbar_wait(empty_bar(s), (use & 1u) ^ 1u, p.limit_ns)) break;
                mbar_expect_tx(full_bar(s), uint32_t(L::kStageBytes));
                const int kc = (kb0 + kb) * kTcBK;
                tma_load_2d(a_hi(s), &map_a_hi, kc, m0, full_bar(s));
                tma_load_2d(a_lo(s), &map_a_lo, kc, m0, full_bar(s));
                tma_load_2d(b_hi(s), &map_b_hi, kc, n0, full_bar(s));
                tma_load_2d(b_lo(s), &map_b_lo, kc, n0, full_bar(s));
                issued = kb + 1;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        constexpr uint32_t idesc = tf32_idesc(BN);
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % STAGES;
            const uint32_t use = uint32_t(kb / STAGES);
            if (!mbar_wait(full_bar(s), use & 1u, p.limit_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTcBK / 8; ++kk) {
                const uint32_t koff = uint32_t(kk) * 32u;   // 8 fp32 = 32 bytes along K
                const uint64_t ah = sw128_desc(a_hi(s) + koff), al = sw128_desc(a_lo(s) + koff);
                const uint64_t bh = sw128_desc(b_hi(s) + koff), bl = sw128_desc(b_lo(s) + koff);
                mma_tf32(tmem, al, bh, idesc, (kb | kk) != 0 ? 1u : 0u);
                mma_tf32(tmem, ah, bl, idesc, 1u);
                mma_tf32(tmem, ah, bh, idesc, 1u);
            }
            mma_commit(empty_bar(s));   // stage s is free once these MMAs finish
        }
        s_mma_ok = ok ? 1 : 0;
        // arrives once every MMA issued above has finished (at once if none were)
        mma_commit(done_bar);
    }
    __syncwarp();
    __syncthreads();   // both roles have finished issuing; s_mma_ok is visible

    // ---- epilogue: TMEM -> registers -> C ----
    const bool have = mbar_wait(done_bar, 0u, p.limit_ns);
    tc_fence_after();
    const bool clean = have && s_mma_ok != 0;
    const int64_t row = int64_t(m0) + warp * 32 + lane;
    const bool row_ok = row < p.M;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) && (p.ldc % 4 == 0);
    float *crow = p.C + (row_ok ? row : 0) * p.ldc;

    // alpha/beta on 32 consecutive columns of this thread's row
    auto store32 = [&](int c0, const float (&v)[32]) {
        const int64_t col = int64_t(n0) + c0;
        if (vec && col + 32 <= p.N) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 o = make_float4(p.alpha * v[4 * q], p.alpha * v[4 * q + 1],
                                       p.alpha * v[4 * q + 2], p.alpha * v[4 * q + 3]);
                float4 *dst = reinterpret_cast<float4 *>(crow + col + 4 * q);
                if (p.beta != 0.0f) {
                    const float4 old = *dst;
                    o.x = fmaf(p.beta, old.x, o.x);
                    o.y = fmaf(p.beta, old.y, o.y);
                    o.z = fmaf(p.beta, old.z, o.z);
                    o.w = fmaf(p.beta, old.w, o.w);
                }
                *dst = o;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (col + j < p.N) {
                    float o = p.alpha * v[j];
                    if (p.beta != 0.0f) o = fmaf(p.beta, crow[col + j], o);
                    crow[col + j] = o;
                }
            }
        }
    };

    if (work.ns == 1) {
        if (__all_sync(0xffffffffu, clean)) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
                if (row_ok) store32(c0, v);
            }
        }
    } else {
        // partial tile of this K range: slot blockIdx.x, row-major 128 x BN;
        // tc_reduce_kernel sums the tile's ranges after this launch
        const size_t slot = size_t(kTcBM) * BN;
        float *mine = p.partials + (size_t(work.slot_first) + size_t(split_idx)) * slot +
                      size_t(warp * 32 + lane) * BN;
        if (__all_sync(0xffffffffu, clean)) {
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 32) {
                float v[32];
                if (nkb > 0) {
                    tmem_ld32(tmem + (uint32_t(warp * 32) << 16) + uint32_t(c0), v);
                } else {   // an empty K range contributes zeros (TMEM was never written)
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    __stcg(reinterpret_cast<float4 *>(mine + c0 + 4 * q),
                           make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
            }
        } else if (threadIdx.x == 0) {
            p.counters[work.cnt] = 1u;   // a wait expired: the tile is not stored
        }
    }
    // the reduction launch may be scheduled once every CTA is here
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane == 0) {
        // copies still in flight (only after an expired wait) land before exit
        for (int kb = (issued > STAGES ? issued - STAGES : 0); kb < issued; ++kb)
            mbar_wait(full_bar(kb % STAGES), uint32_t(kb / STAGES) & 1u, p.limit_ns);
    }
    if (warp == 1 && lane == 0 && !have) mbar_wait(done_bar, 0u, p.limit_ns);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(uint32_t(BN))
                     : "memory");
    }
}

// ---------------------------------------------------------------------------
// Fused variant: A's split happens in shared memory.
//
// A is K-major as stored, so its tile arrives by TMA as raw fp32 in exactly
// the swizzled layout the MMA reads.  The raw tile lands in the A_lo slot of
// the stage; four converter warps (threads 128..255) read it, write
// A_hi = tf32(x) into the A_hi slot and overwrite the slot with
// A_lo = tf32(x - A_hi) -- same offsets, no address arithmetic -- then fence
// the generic-proxy writes for the tensor cores' async-proxy reads and arrive
// on the stage's `conv` barrier, which the MMA issuer waits on instead of the
// TMA barrier.  B must be K-major for the MMA, i.e. transposed from its
// stored layout, so it arrives already split (B_hi^T, B_lo^T, packed once).
// All eight warps share the epilogue: warp w reads TMEM lanes
// 32*(w%4)..+31, warps 0-3 the left half of the columns, 4-7 the right half.
// ---------------------------------------------------------------------------

constexpr int kFusedThreads = 256;

template <int BN, int STAGES>
struct FusedSmem {
    static constexpr int kABytes = kTcBM * kTcBK * 4;          // 16 KiB
    static constexpr int kBBytes = BN * kTcBK * 4;
    static constexpr int kASlots = 3;                           // A ring: [A_hi][A_lo]
    static constexpr int kASlotBytes = 2 * kABytes;
    static constexpr int kBStageBytes = 2 * kBBytes;            // B ring: [B_hi][B_lo]
    static constexpr int kBOffset = kASlots * kASlotBytes;
    static constexpr int kBarOffset = kBOffset + STAGES * kBStageBytes;
    // afull[A], aconv[A], aempty[A], bfull[S], bempty[S], done, then the TMEM slot
    static constexpr int kNumBars = 3 * kASlots + 2 * STAGES + 1;
    static constexpr int kBytes = kBarOffset + kNumBars * 8 + 8;
    static constexpr int kDynBytes = kBytes + 1024;
};

template <int BN, int STAGES>
__global__ void __launch_bounds__(kFusedThreads, 1)
tf32x3_fused_kernel(const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_b_hi,
                    const __grid_constant__ CUtensorMap map_b_lo, const TcArgs p) {
    using L = FusedSmem<BN, STAGES>;
    constexpr int NA = L::kASlots;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gbase = smem_raw + (base - raw);
    const uint32_t bar0 = base + L::kBarOffset;
    auto afull_bar = [&](int r) { return bar0 + 8u * r; };
    auto aconv_bar = [&](int r) { return bar0 + 8u * (NA + r); };
    auto aempty_bar = [&](int r) { return bar0 + 8u * (2 * NA + r); };
    auto bfull_bar = [&](int s) { return bar0 + 8u * (3 * NA + s); };
    auto bempty_bar = [&](int s) { return bar0 + 8u * (3 * NA + STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (3 * NA + 2 * STAGES);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + L::kBarOffset + L::kNumBars * 8);
    auto a_hi = [&](int r) { return base + r * L::kASlotBytes; };
    auto a_lo = [&](int r) { return base + r * L::kASlotBytes + L::kABytes; };
    auto b_hi = [&](int s) { return base + L::kBOffset + s * L::kBStageBytes; };
    auto b_lo = [&](int s) { return base + L::kBOffset + s * L::kBStageBytes + L::kBBytes; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    __shared__ int s_mma_ok;

    // (tile, K range) of this CTA; grouped raster over 8 tile rows
    const TcWork work = tc_work(p);
    const int pid = work.pid;
    const int split_idx = work.sidx;
    const int per_group = 8 * p.tiles_n;
    const int group = pid / per_group;
    const int first_m = group * 8;
    const int gm = min(p.tiles_m - first_m, 8);
    const int in_group = pid - group * per_group;
    const int tile_m = first_m + in_group % gm;
    const int tile_n = in_group / gm;
    const int m0 = tile_m * kTcBM;
    const int n0 = tile_n * BN;
    const int nkb_all = int((p.K + kTcBK - 1) / kTcBK);
    const int kb0 = split_idx * work.kbps;
    const int nkb = max(0, min(nkb_all, kb0 + work.kbps) - kb0);

    if (threadIdx.x == 0) {
        for (int r = 0; r < NA; ++r) {
            mbar_init(afull_bar(r), 1);
            mbar_init(aconv_bar(r), kFusedThreads - 128);
            mbar_init(aempty_bar(r), 1);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bfull_bar(s), 1);
            mbar_init(bempty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(tmem_slot)),
                     "r"(uint32_t(BN))
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // After a split pass this kernel is its programmatic dependent: the setup
    // above overlapped the pass's tail; nothing is read before it completes.
    asm volatile("griddepcontrol.wait;" ::: "memory");

    int issued_b = 0, issued_a = 0;   // K blocks each producer issued
    if (warp == 0 && lane == 0) {
        // ---- TMA producer of the packed B_hi / B_lo tiles ----
        if (!p.inject_stall) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int s = kb % STAGES;
                const uint32_t use = uint32_t(kb / STAGES);
                if (kb >= STAGES && !mbar_wait(bempty_bar(s), (use & 1u) ^ 1u, p.limit_ns)) break;
                mbar_expect_tx(bfull_bar(s), uint32_t(2 * L::kBBytes));
                const int kc = (kb0 + kb) * kTcBK;
                tma_load_2d(b_hi(s), &map_b_hi, kc, n0, bfull_bar(s));
                tma_load_2d(b_lo(s), &map_b_lo, kc, n0, bfull_bar(s));
                issued_b = kb + 1;
            }
        }
    } else if (warp == 2 && lane == 0) {
        // ---- TMA producer of the raw fp32 A tiles, into the A_lo slot ----
        if (!p.inject_stall) {
            for (int kb = 0; kb < nkb; ++kb) {
                const int r = kb % NA;
                const uint32_t use = uint32_t(kb / NA);
                if (kb >= NA && !mbar_wait(aempty_bar(r), (use & 1u) ^ 1u, p.limit_ns)) break;
                mbar_expect_tx(afull_bar(r), uint32_t(L::kABytes));
                tma_load_2d(a_lo(r), &map_a, (kb0 + kb) * kTcBK, m0, afull_bar(r));
                issued_a = kb + 1;
            }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        constexpr uint32_t idesc = tf32_idesc(BN);
        bool ok = true;
        for (int kb = 0; kb < nkb && ok; ++kb) {
            const int s = kb % STAGES, r = kb % NA;
            const uint32_t use = uint32_t(kb / STAGES), ause = uint32_t(kb / NA);
            if (!mbar_wait(aconv_bar(r), ause & 1u, p.limit_ns) ||
                !mbar_wait(bfull_bar(s), use & 1u, p.limit_ns)) {
                ok = false;
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < kTcBK / 8; ++kk) {
                const uint32_t koff = uint32_t(kk) * 32u;
                const uint64_t ah = sw128_desc(a_hi(r) + koff), al = sw128_desc(a_lo(r) + koff);
                const uint64_t bh = sw128_desc(b_hi(s) + koff), bl = sw128_desc(b_lo(s) + koff);
                mma_tf32(tmem, al, bh, idesc, (kb | kk) != 0 ? 1u : 0u);
                mma_tf32(tmem, ah, bl, idesc, 1u);
                mma_tf32(tmem, ah, bh, idesc, 1u);
            }
            mma_commit(aempty_bar(r));   // both arrive once these MMAs have finished
            mma_commit(bempty_bar(s));
        }
        s_mma_ok = ok ? 1 : 0;
        mma_commit(done_bar);
    } else if (warp >= 4) {
        // ---- converters: the raw tile in A_lo becomes A_lo in place, plus A_hi ----
        const int c = threadIdx.x - 128;
        for (int kb = 0; kb < nkb; ++kb) {
            const int r = kb % NA;
            if (!mbar_wait(afull_bar(r), uint32_t(kb / NA) & 1u, p.limit_ns)) break;
            // 128-bit shared accesses, consecutive across the 128 threads; each
            // thread reads all its elements before writing any of them back
            constexpr int kQ = L::kABytes / 16 / 128;
            float4 x[kQ];
#pragma unroll
            for (int q = 0; q < kQ; ++q) x[q] = lds128(a_lo(r) + 16u * uint32_t(c + 128 * q));
#pragma unroll
            for (int q = 0; q < kQ; ++q) {
                float4 h, l;
                split2(x[q].x, h.x, l.x);
                split2(x[q].y, h.y, l.y);
                split2(x[q].z, h.z, l.z);
                split2(x[q].w, h.w, l.w);
                const uint32_t off = 16u * uint32_t(c + 128 * q);
                sts128(a_hi(r) + off, h);
                sts128(a_lo(r) + off, l);
            }
            // make the generic-proxy writes visible to the tensor cores
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            mbar_arrive(aconv_bar(r));
        }
    }
    __syncwarp();
    __syncthreads();   // every role has finished issuing; s_mma_ok is visible

    // ---- epilogue: TMEM -> registers -> C (or partials) ----
    const bool have = mbar_wait(done_bar, 0u, p.limit_ns);
    tc_fence_after();
    const bool clean = have && s_mma_ok != 0;
    const int lrow = (warp & 3) * 32 + lane;          // TMEM lane = row in the tile
    const int cbeg = (warp >> 2) * (BN / 2);          // this warp's column half
    const int64_t row = int64_t(m0) + lrow;
    const bool row_ok = row < p.M;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) && (p.ldc % 4 == 0);
    float *crow = p.C + (row_ok ? row : 0) * p.ldc;
    const uint32_t taddr = tmem + (uint32_t((warp & 3) * 32) << 16);

    auto store32 = [&](int c0, const float (&v)[32]) {
        const int64_t col = int64_t(n0) + c0;
        if (vec && col + 32 <= p.N) {
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                float4 o = make_float4(p.alpha * v[4 * q], p.alpha * v[4 * q + 1],
                                       p.alpha * v[4 * q + 2], p.alpha * v[4 * q + 3]);
                float4 *dst = reinterpret_cast<float4 *>(crow + col + 4 * q);
                if (p.beta != 0.0f) {
                    const float4 old = *dst;
                    o.x = fmaf(p.beta, old.x, o.x);
                    o.y = fmaf(p.beta, old.y, o.y);
                    o.z = fmaf(p.beta, old.z, o.z);
                    o.w = fmaf(p.beta, old.w, o.w);
                }
                *dst = o;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (col + j < p.N) {
                    float o = p.alpha * v[j];
                    if (p.beta != 0.0f) o = fmaf(p.beta, crow[col + j], o);
                    crow[col + j] = o;
                }
            }
        }
    };

    if (work.ns == 1) {
        if (__all_sync(0xffffffffu, clean)) {
#pragma unroll 1
            for (int c0 = cbeg; c0 < cbeg + BN / 2; c0 += 32) {
                float v[32];
                tmem_ld32(taddr + uint32_t(c0), v);
                if (row_ok) store32(c0, v);
            }
        }
    } else {
        // partial tile of this K range, row-major 128 x BN; tc_reduce_kernel
        // sums the tile's ranges after this launch
        const size_t slot = size_t(kTcBM) * BN;
        float *mine = p.partials + (size_t(work.slot_first) + size_t(split_idx)) * slot +
                      size_t(lrow) * BN;
        if (__all_sync(0xffffffffu, clean)) {
#pragma unroll 1
            for (int c0 = cbeg; c0 < cbeg + BN / 2; c0 += 32) {
                float v[32];
                if (nkb > 0) {
                    tmem_ld32(taddr + uint32_t(c0), v);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    __stcg(reinterpret_cast<float4 *>(mine + c0 + 4 * q),
                           make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]));
            }
        } else if (threadIdx.x == 0) {
            p.counters[work.cnt] = 1u;   // a wait expired: the tile is not stored
        }
    }
    // the reduction launch may be scheduled once every CTA is here
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    // copies still in flight (only after an expired wait) land before exit
    if (warp == 0 && lane == 0) {
        for (int kb = (issued_b > STAGES ? issued_b - STAGES : 0); kb < issued_b; ++kb)
            mbar_wait(bfull_bar(kb % STAGES), uint32_t(kb / STAGES) & 1u, p.limit_ns);
    }
    if (warp == 2 && lane == 0) {
        for (int kb = (issued_a > NA ? issued_a - NA : 0); kb < issued_a; ++kb)
            mbar_wait(afull_bar(kb % NA), uint32_t(kb / NA) & 1u, p.limit_ns);
    }
    if (warp == 1 && lane == 0 && !have) mbar_wait(done_bar, 0u, p.limit_ns);
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(uint32_t(BN))
                     : "memory");
    }
}

// The second launch of a split plan: for every split tile, the sum of its K
// ranges' partial tiles in ascending range order, then alpha and beta.
// Launched as a programmatic dependent of the product grid (it waits for that
// grid's completion before reading).  A tile one of whose ranges gave up a
// bounded wait carries a flag: it is not stored (C stays untouched), and the
// flag is cleared for the next call.  One CTA per tile, so the CTA that
// clears the flag is the only one that reads it; each thread takes float4s
// of the tile four at a time, all their partials' loads in flight together.
__global__ void __launch_bounds__(256) tc_reduce_kernel(const TcArgs p, int bn) {
    const int i_tile = int(blockIdx.x);                 // among the split tiles
    int pid, ns;
    if (p.split > 1) {
        pid = i_tile;
        ns = p.split;
    } else {
        pid = p.tail_start + i_tile;
        ns = p.tail_split;
    }
    // the product kernels' grouped raster over 8 tile rows
    const int per_group = 8 * p.tiles_n;
    const int group = pid / per_group;
    const int first_m = group * 8;
    const int gm = min(p.tiles_m - first_m, 8);
    const int in_group = pid - group * per_group;
    const int64_t m0 = int64_t(first_m + in_group % gm) * kTcBM;
    const int64_t n0 = int64_t(in_group / gm) * bn;

    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    __shared__ unsigned s_flag;
    unsigned *flag = p.counters + i_tile;
    if (threadIdx.x == 0) s_flag = *flag;
    __syncthreads();
    if (s_flag != 0u) {
        if (threadIdx.x == 0) *flag = 0u;
        return;
    }
    const size_t slot = size_t(kTcBM) * bn;
    const float *part = p.partials + size_t(i_tile) * size_t(ns) * slot;
    const bool vec = ((reinterpret_cast<uintptr_t>(p.C) & 15u) == 0) && (p.ldc % 4 == 0);
    const int per_row = bn / 4;                          // float4 per tile row
    const int total = kTcBM * per_row;                   // float4 per tile (a multiple of 1024)
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int sidx = 0; sidx < ns; ++sidx) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                x[u] = __ldcg(reinterpret_cast<const float4 *>(part + size_t(sidx) * slot) +
                              base + u * blockDim.x);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                v[u].x += x[u].x;
                v[u].y += x[u].y;
                v[u].z += x[u].z;
                v[u].w += x[u].w;
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int idx = base + u * blockDim.x;
            const int64_t row = m0 + idx / per_row, col = n0 + (idx % per_row) * 4;
            if (row >= p.M || col >= p.N) continue;
            float o[4] = {p.alpha * v[u].x, p.alpha * v[u].y, p.alpha * v[u].z, p.alpha * v[u].w};
            float *cp = p.C + row * p.ldc + col;
            if (vec && col + 4 <= p.N) {
                if (p.beta != 0.0f) {
                    const float4 old = *reinterpret_cast<const float4 *>(cp);
                    o[0] = fmaf(p.beta, old.x, o[0]);
                    o[1] = fmaf(p.beta, old.y, o[1]);
                    o[2] = fmaf(p.beta, old.z, o[2]);
                    o[3] = fmaf(p.beta, old.w, o[3]);
                }
                *reinterpret_cast<float4 *>(cp) = make_float4(o[0], o[1], o[2], o[3]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (col + e < p.N) {
                        float x = o[e];
                        if (p.beta != 0.0f) x = fmaf(p.beta, cp[e], x);
                        cp[e] = x;
                    }
                }
            }
        }
    }
}

// Launches `kernel`, as a programmatic dependent of the kernel before it on
// the stream when `pdl` (its CTAs may be scheduled once every CTA of that
// kernel has started; each waits at griddepcontrol.wait before reading).
// Within one call: B's pass after A's, the product after the passes, the
// reduction after the product.  Measured on GB300 against plain launches
// (microseconds, L2 flushed, C the same bit for bit): 256^3 25.2 -> 21.2,
// 1024^3 49.8 -> 45.7, 1023x777x513 35.5 -> 32.4, GPT-2 QKV 45.7 -> 43.6,
// MLP-up 49.8 -> 45.7, MLP-down 64.1 -> 59.0; 2048^3 and above unchanged.
template <typename... KArgs, typename... Args>
cudaError_t launch_maybe_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, bool pdl, Args &&...args) {
    if (!pdl) {
        kernel<<<grid, block, smem, stream>>>(std::forward<Args>(args)...);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Launches tc_reduce_kernel for a plan's split tiles (nothing without any).
cudaError_t launch_tc_reduce(const TcArgs &a, int bn, cudaStream_t stream) {
    const int64_t tiles = int64_t(a.tiles_m) * a.tiles_n;
    const int64_t split_tiles = a.split > 1 ? tiles : (a.tail_split > 1 ? tiles - a.tail_start : 0);
    if (split_tiles <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(split_tiles), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, tc_reduce_kernel, a, bn);
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link-time
// dependency on the driver library).
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// 2-D fp32 tensor map over a K-major (rows x cols, row stride ld floats)
// matrix, box = 32 columns x box_rows rows, 128-byte swizzle, zero fill.
bool encode_kmajor(CUtensorMap *map, const float *ptr, int64_t rows, int64_t cols, int64_t ld,
                   int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
    const cuuint32_t box[2] = {cuuint32_t(kTcBK), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

template <int BN, int STAGES>
cudaError_t launch_mma(const CUtensorMap &ah, const CUtensorMap &al, const CUtensorMap &bh,
                       const CUtensorMap &bl, const TcArgs &a, cudaStream_t stream, bool pdl) {
    using L = TcSmem<BN, STAGES>;
    // the attribute is per device; set it on every call (cheap, host-side)
    static bool configured[64];
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(tf32x3_mma_kernel<BN, STAGES>),
                                  L::kDynBytes, configured);
    if (e != cudaSuccess) return e;
    const int64_t tiles = int64_t(a.tiles_m) * a.tiles_n;
    const unsigned grid = unsigned(int64_t(a.tail_start) * a.split +
                                   (tiles - a.tail_start) * a.tail_split);
    e = launch_maybe_pdl(tf32x3_mma_kernel<BN, STAGES>, dim3(grid), dim3(kTcThreads),
                         L::kDynBytes, stream, pdl, ah, al, bh, bl, a);
    return e == cudaSuccess ? launch_tc_reduce(a, BN, stream) : e;
}

template <int BN, int STAGES>
cudaError_t launch_fused(const CUtensorMap &a, const CUtensorMap &bh, const CUtensorMap &bl,
                         const TcArgs &args, cudaStream_t stream, bool pdl) {
    using L = FusedSmem<BN, STAGES>;
    static bool configured[64];
    cudaError_t e = set_smem_once(reinterpret_cast<const void *>(tf32x3_fused_kernel<BN, STAGES>),
                                  L::kDynBytes, configured);
    if (e != cudaSuccess) return e;
    const int64_t tiles = int64_t(args.tiles_m) * args.tiles_n;
    const unsigned grid = unsigned(int64_t(args.tail_start) * args.split +
                                   (tiles - args.tail_start) * args.tail_split);
    e = launch_maybe_pdl(tf32x3_fused_kernel<BN, STAGES>, dim3(grid), dim3(kFusedThreads),
                         L::kDynBytes, stream, pdl, a, bh, bl, args);
    return e == cudaSuccess ? launch_tc_reduce(args, BN, stream) : e;
}

}  // namespace

namespace {
constexpr int kTcBN = 256;
// Ring depths.  256-wide tiles fit two stages of B (with the three-slot A
// ring of the fused kernel: 224 KiB); 128-wide tiles leave room for more.
// Measured on GB300 (microseconds, two stages / deeper): the split-operand
// kernel with three stages on 1023x777x513 44.7 / 42.7; the fused kernel's
// B ring with four stages 1024^3 47.7 / 51.9, MLP-down 68.2 / 72.4, so it
// keeps two.
constexpr int kTcStages = 2;           // 256-wide tiles, both kernels
constexpr int kTcMmaStages128 = 3;     // split-operand kernel, 128-wide: 192 KiB
constexpr int kTcFusedStages128 = 2;   // fused kernel's B ring, 128-wide
static_assert(FusedSmem<128, kTcFusedStages128>::kDynBytes <= 227 * 1024, "fused ring too deep");
static_assert(TcSmem<128, kTcMmaStages128>::kDynBytes <= 227 * 1024, "split-operand ring too deep");
static_assert(FusedSmem<256, kTcStages>::kDynBytes <= 227 * 1024, "fused ring too deep");
static_assert(TcSmem<256, kTcStages>::kDynBytes <= 227 * 1024, "split-operand ring too deep");

size_t round256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

// Tile columns: 256 (the MMA's widest N), or 128 -- twice the tiles, but
// each A tile is split (in the kernel) twice as often per FLOP, so a
// 128-wide CTA does barely more than half a 256-wide one's work per unit of
// time (2048^3: 104 against 194 TFLOP/s).  128 pays only where 256-wide
// tiles fill at most half the SMs and K is short enough that split-K cannot
// make up for it.  Measured on GB300 (microseconds, 256 / 128): 256^3 27.3 /
// 25.2, 1024^3 58.0 / 47.8 (split 2), 1023x777x513 60.1 / 44.7, GPT-2 QKV
// 48.8 / 46.8, MLP-down 95.9 / 68.3; but 1024x1024x16384 232 / 331 and
// MLP-up (96 tiles) 49.8 / 72.4.  The tuning knob kKnobTf32x3Bn overrides.
int choose_tc_bn(int64_t M, int64_t N, int64_t K, int sms) {
    if (const int f = tuning(kKnobTf32x3Bn); f == 128 || f == 256) return f;
    const int64_t tiles256 = ((M + kTcBM - 1) / kTcBM) * ((N + 255) / 256);
    const int64_t nkb = (K + kTcBK - 1) / kTcBK;
    return (2 * tiles256 <= sms && nkb <= 96) ? 128 : kTcBN;
}

// K ranges per tile.  One CTA runs per SM, so a grid of fewer tiles than SMs
// leaves SMs idle; cutting K fills them but costs a partial-tile write and
// read per range plus a second pass of prologue and epilogue.  Measured on
// GB300 (forced splits 1..8): splitting paid off only when the grid filled at
// most half the SMs and every range kept >= 24 K blocks (768 of K) --
// 1024x1024x16384: 51 -> 111 TFLOP/s at 4 ranges, 1024x768x3072: 40 -> 54 at
// 3-4 -- and lost everywhere else (1024^3, GPT-2 QKV/MLP-up, 2048^3, 4096^3).
Tf32x3Plan tf32x3_plan(int64_t M, int64_t N, int64_t K, int sms) {
    Tf32x3Plan plan;
    plan.bn = choose_tc_bn(M, N, K, sms);
    const int64_t tiles = ((M + kTcBM - 1) / kTcBM) * ((N + plan.bn - 1) / plan.bn);
    const int64_t nkb = (K + kTcBK - 1) / kTcBK;
    plan.tiles = tiles;
    plan.tail_start = tiles;
    if (sms <= 0) return plan;
    {
        const int f = tuning(kKnobTf32x3Split);
        if (f >= 1 && f <= 64 && tiles <= kMaxSplitTiles) {
            plan.split = f;
            return plan;
        }
    }
    if (tiles <= kMaxSplitTiles && 2 * tiles <= sms) {
        // at least 24 K blocks a range on 256-wide tiles, 8 on 128-wide ones
        // (1024^3, 128-wide: 56.0 us unsplit, 47.8 in two ranges of 16;
        // 1023x777x513: 43.7 unsplit, 37.5 in two ranges of 9, 44.7 in three)
        int64_t sp = std::min<int64_t>(sms / tiles, nkb / (plan.bn == 128 ? 8 : 24));
        sp = std::min<int64_t>(sp, 16);
        plan.split = sp > 1 ? int(sp) : 1;
        return plan;
    }
    // Tail: with one CTA per SM, a last wave of tiles that fills at most half
    // the SMs idles the rest for a whole tile's time; cut just those tiles
    // into K ranges (all of them still fitting in one wave).
    // The tuning knob kKnobTf32x3Tail = 0 disables it, = s forces s ranges.
    const int64_t rem = tiles % sms;
    int want = 0;
    if (rem > 0 && 2 * rem <= sms) want = int(std::min<int64_t>(sms / rem, 4));
    if (const int force = tuning(kKnobTf32x3Tail); force >= 0) want = force;
    if (tiles >= sms && rem > 0 && want >= 2 && rem * want <= sms && nkb >= 8 * want) {
        plan.tail_start = tiles - rem;
        plan.tail_split = want;
    }
    return plan;
}

size_t tf32x3_packed_b_bytes(int64_t K, int64_t N) {
    const int64_t kp = (K + 3) / 4 * 4;
    return 2 * round256(size_t(N) * kp * 4);
}

bool tf32x3_fusable_a(const float *A, int64_t lda) {
    return (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && lda % 4 == 0;
}

// A is split inside the kernel (tf32x3_fused_kernel) whenever TMA can read it
// as stored; the tuning knob kKnobTf32x3FuseA = 0 forces the pre-pass instead.  Measured on
// GB300 (TFLOP/s, pre-pass / in-kernel): 8192^3 259 / 287 (271 / 300 with B
// packed once), 4096^3 201 / 231, 1024x1024x16384 112 / 138.  What made the
// in-kernel split pay was the branch-free TF32 rounding: with early returns
// the converters' 64 conversions per slice did not interleave and the kernel
// ran at 40 % of these rates.
bool tf32x3_use_fused_a(const float *A, int64_t lda) {
    if (tuning(kKnobTf32x3FuseA) == 0) return false;
    return tf32x3_fusable_a(A, lda);
}

size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K, const Tf32x3Plan &plan,
                              bool fused, bool packed_b) {
    const int64_t kp = (K + 3) / 4 * 4;
    const size_t a = fused ? 0 : 2 * round256(size_t(M) * kp * 4);
    const size_t b = packed_b ? 0 : tf32x3_packed_b_bytes(K, N);
    const size_t parts = size_t(plan.partial_slots()) * kTcBM * plan.bn * 4;
    return a + b + parts;
}

namespace {

// B split and transposed into `packed`; with `pdl` as a programmatic
// dependent of A's split pass (the kernels then complete only after it).
cudaError_t pack_b(int64_t K, int64_t N, const float *B, int64_t ldb, void *packed, bool pdl,
                   cudaStream_t stream) {
    const int64_t kp = (K + 3) / 4 * 4;
    float *b_hi = static_cast<float *>(packed);
    float *b_lo = reinterpret_cast<float *>(static_cast<char *>(packed) +
                                            round256(size_t(N) * kp * 4));
    if ((reinterpret_cast<uintptr_t>(B) & 15u) == 0 && ldb % 4 == 0) {
        const dim3 grid(unsigned((N + 63) / 64), unsigned((K + 63) / 64));
        return launch_maybe_pdl(split_transpose64_kernel, grid, dim3(256), 0, stream, pdl, B, K, N,
                                ldb, b_hi, b_lo, kp);
    }
    const dim3 tgrid(unsigned((N + 31) / 32), unsigned((K + 31) / 32));
    return launch_maybe_pdl(split_transpose_kernel, tgrid, dim3(32, 8), 0, stream, pdl, B, K, N,
                            ldb, b_hi, b_lo, kp);
}

}  // namespace

cudaError_t tf32x3_pack_b(int64_t K, int64_t N, const float *B, int64_t ldb, void *packed,
                          cudaStream_t stream) {
    return pack_b(K, N, B, ldb, packed, false, stream);
}

namespace {

TcArgs make_args(float *C, int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha,
                 float beta, unsigned *counters, float *parts, const Tf32x3Plan &plan,
                 uint64_t limit_ns, int inject_stall) {
    TcArgs a;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.ldc = ldc;
    a.alpha = alpha;
    a.beta = beta;
    a.tiles_m = int32_t((M + kTcBM - 1) / kTcBM);
    a.tiles_n = int32_t((N + plan.bn - 1) / plan.bn);
    a.limit_ns = limit_ns;
    a.inject_stall = inject_stall;
    const int64_t nkb = (K + kTcBK - 1) / kTcBK;
    a.split = plan.split > 1 ? plan.split : 1;
    a.kb_per_split = int32_t((nkb + a.split - 1) / a.split);
    a.tail_start = int32_t(plan.tail_start);
    a.tail_split = plan.tail_split > 1 ? plan.tail_split : 1;
    a.tail_kb_per_split = int32_t((nkb + a.tail_split - 1) / a.tail_split);
    // partial slots / flags only for split tiles
    a.part_base = a.split > 1 ? 0 : a.tail_start;
    a.cnt_base = a.split > 1 ? 0 : a.tail_start;
    a.counters = counters;
    a.partials = parts;
    return a;
}

}  // namespace

namespace {

// C = alpha*A*B + beta*C with B packed; `workspace` holds A's hi/lo (unless A
// is split in shared memory) followed by the split-K partials.  `after_pass`:
// the kernel before this call on the stream is this product's own B pass, so
// the fused kernel may be its programmatic dependent.  (After A's split pass,
// launched here, the split-operand kernel always is.)
cudaError_t packed_product(const float *A, int64_t lda, const void *packed_b, float *C,
                           int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                           void *workspace, unsigned *counters, const Tf32x3Plan &plan,
                           uint64_t limit_ns, int inject_stall, bool after_pass,
                           cudaStream_t stream) {
    const int64_t kp = (K + 3) / 4 * 4;
    const float *b_hi = static_cast<const float *>(packed_b);
    const float *b_lo = reinterpret_cast<const float *>(static_cast<const char *>(packed_b) +
                                                        round256(size_t(N) * kp * 4));
    char *w = static_cast<char *>(workspace);
    const bool fused = tf32x3_use_fused_a(A, lda);
    if (fused) {
        CUtensorMap am, bh, bl;
        if (!encode_kmajor(&am, A, M, K, lda, kTcBM) ||
            !encode_kmajor(&bh, b_hi, N, K, kp, plan.bn) ||
            !encode_kmajor(&bl, b_lo, N, K, kp, plan.bn))
            return cudaErrorInvalidValue;
        const TcArgs a = make_args(C, ldc, M, N, K, alpha, beta, counters,
                                   reinterpret_cast<float *>(w), plan, limit_ns, inject_stall);
        return plan.bn == 128
                   ? launch_fused<128, kTcFusedStages128>(am, bh, bl, a, stream, after_pass)
                   : launch_fused<kTcBN, kTcStages>(am, bh, bl, a, stream, after_pass);
    }
    const size_t abytes = round256(size_t(M) * kp * 4);
    float *a_hi = reinterpret_cast<float *>(w);
    float *a_lo = reinterpret_cast<float *>(w + abytes);
    float *parts = reinterpret_cast<float *>(w + 2 * abytes);
    int64_t blocks = (M * K + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    split_rows_kernel<<<unsigned(blocks), 256, 0, stream>>>(A, M, K, lda, a_hi, a_lo, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    CUtensorMap ah, al, bh, bl;
    if (!encode_kmajor(&ah, a_hi, M, K, kp, kTcBM) || !encode_kmajor(&al, a_lo, M, K, kp, kTcBM) ||
        !encode_kmajor(&bh, b_hi, N, K, kp, plan.bn) || !encode_kmajor(&bl, b_lo, N, K, kp, plan.bn))
        return cudaErrorInvalidValue;
    const TcArgs a = make_args(C, ldc, M, N, K, alpha, beta, counters, parts, plan, limit_ns,
                               inject_stall);
    return plan.bn == 128 ? launch_mma<128, kTcMmaStages128>(ah, al, bh, bl, a, stream, true)
                          : launch_mma<kTcBN, kTcStages>(ah, al, bh, bl, a, stream, true);
}

}  // namespace

cudaError_t launch_tf32x3_packed(const float *A, int64_t lda, const void *packed_b, float *C,
                                 int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha,
                                 float beta, void *workspace, unsigned *counters,
                                 const Tf32x3Plan &plan, uint64_t limit_ns, int inject_stall,
                                 cudaStream_t stream) {
    return packed_product(A, lda, packed_b, C, ldc, M, N, K, alpha, beta, workspace, counters,
                          plan, limit_ns, inject_stall, false, stream);
}

cudaError_t launch_tf32x3(const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                          void *workspace, unsigned *counters, const Tf32x3Plan &plan,
                          uint64_t limit_ns, int inject_stall, cudaStream_t stream) {
    constexpr int STAGES = kTcStages;
    const int64_t kp = (K + 3) / 4 * 4;
    char *w = static_cast<char *>(workspace);
    if (tf32x3_use_fused_a(A, lda)) {
        // B split and transposed into the workspace; A split in shared memory
        cudaError_t e = pack_b(K, N, B, ldb, w, false, stream);
        if (e != cudaSuccess) return e;
        return packed_product(A, lda, w, C, ldc, M, N, K, alpha, beta,
                              w + tf32x3_packed_b_bytes(K, N), counters, plan, limit_ns,
                              inject_stall, true, stream);
    }
    // both operands split (and B transposed) in a pre-pass
    const size_t abytes = round256(size_t(M) * kp * 4);
    const size_t bbytes = round256(size_t(N) * kp * 4);
    float *a_hi = reinterpret_cast<float *>(w);
    float *a_lo = reinterpret_cast<float *>(w + abytes);
    float *b_hi = reinterpret_cast<float *>(w + 2 * abytes);
    float *b_lo = reinterpret_cast<float *>(w + 2 * abytes + bbytes);
    float *parts = reinterpret_cast<float *>(w + 2 * abytes + 2 * bbytes);

    int64_t blocks = (M * K + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    split_rows_kernel<<<unsigned(blocks), 256, 0, stream>>>(A, M, K, lda, a_hi, a_lo, kp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // B's pass overlaps A's (it reads neither of A's outputs) and completes after it
    e = pack_b(K, N, B, ldb, w + 2 * abytes, true, stream);
    if (e != cudaSuccess) return e;

    CUtensorMap ah, al, bh, bl;
    if (!encode_kmajor(&ah, a_hi, M, K, kp, kTcBM) || !encode_kmajor(&al, a_lo, M, K, kp, kTcBM) ||
        !encode_kmajor(&bh, b_hi, N, K, kp, plan.bn) || !encode_kmajor(&bl, b_lo, N, K, kp, plan.bn))
        return cudaErrorInvalidValue;
    const TcArgs a = make_args(C, ldc, M, N, K, alpha, beta, counters, parts, plan, limit_ns,
                               inject_stall);
    return plan.bn == 128 ? launch_mma<128, kTcMmaStages128>(ah, al, bh, bl, a, stream, true)
                          : launch_mma<kTcBN, STAGES>(ah, al, bh, bl, a, stream, true);
}

cudaError_t tf32x3_read_error(unsigned *out, cudaStream_t stream) {
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_tc_error, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, stream);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    e = cudaMemcpyToSymbolAsync(g_tc_error, &zero, sizeof(unsigned), 0, cudaMemcpyHostToDevice,
                                stream);
    if (e != cudaSuccess) return e;
    return cudaStreamSynchronize(stream);
}

}  // namespace sgemm_impl
