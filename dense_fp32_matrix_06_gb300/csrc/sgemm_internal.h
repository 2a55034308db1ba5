// sgemm_internal.h -- shared between the C ABI layer and the kernel files.
// Not part of the public interface (that is include/sgemm.h).
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

namespace sgemm_impl {

// CTA tiles of the fp32 FFMA kernel: T x T outputs, K slices of T/8,
// (T/8)^2 threads, each owning an 8 x 8 block of accumulators.  T = 128 is
// the main tile (2 resident CTAs per SM); T = 64 is for grids that 128-wide
// tiles cannot fill (8 per SM).
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kBK = 16;
constexpr int kThreads = 256;
constexpr int kCtasPerSm = 2;   // resident 128-tile CTAs per SM
constexpr int kSmallTile = 64;
constexpr int kSmallCtasPerSm = 8;
// Tile rows per raster group (L2 reuse of A and B panels): a wave of 304
// 128-wide CTAs then covers 16 x 19 tiles rather than 8 x 38.  Measured at
// 8192^3 (product kernel, one launch): DRAM reads 3.27 GB with 8 rows, 3.09
// GB with 16, the same 65.9 TFLOP/s.
constexpr int kGroupM = 16;

// Workspace layout: [flag block: kCounterBytes][partial tiles][...].  The
// 3xTF32 mode keeps one flag per split tile in the block, set only by a K
// range whose bounded wait expired and cleared by the reduction (fixed size,
// so a buffer reused across plans never sees stale partial data where a
// flag is expected); the FFMA kernels leave it untouched.  Split plans stay
// within kMaxSplitTiles split tiles either way.
constexpr size_t kCounterBytes = 16384;
constexpr int64_t kMaxSplitTiles = kCounterBytes / sizeof(unsigned);
constexpr int kMaxSplit = 32;

// Sets the dynamic shared memory limit of `kernel` on the current device once
// (per kernel and device; `flags` is the caller's per-kernel table).  Setting
// it twice from racing threads is harmless.
// With `max_carveout` the kernel also asks for the largest shared-memory
// carveout, so that the CTAs a persistent grid counts on fit on every SM.
inline cudaError_t set_smem_once(const void *kernel, int bytes, bool (&flags)[64],
                                 bool max_carveout = false) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && flags[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && max_carveout)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 int(cudaSharedmemCarveoutMaxShared));
    if (e == cudaSuccess && dev >= 0 && dev < 64) flags[dev] = true;
    return e;
}

// Planner and dispatch overrides (tuning.cu; C ABI sgemm_set_tuning).  Each
// knob starts from an environment variable read once at library load; -1
// means the planner decides.  The order matches sgemm_tuning_knob.
enum Knob : int32_t {
    kKnobSplit = 0,          // split-K ranges of every tile (1..kMaxSplit)
    kKnobTail = 1,           // K ranges of the last partial wave (0/1 off, 2..)
    kKnobTile = 2,           // CTA tile 64 or 128
    kKnobKernel = 3,         // 0 scalar FMA issue, 1 packed f32x2
    kKnobTransposeA = 4,     // 0/1: transposed copy of A first
    kKnobFfmaExt = 5,        // 0/1: plain or extended instantiation for plain products
    kKnobTf32x3Split = 6,    // tensor mode: K ranges of every tile
    kKnobTf32x3Tail = 7,     // tensor mode: K ranges of the last partial wave
    kKnobTf32x3FuseA = 8,    // tensor mode: 0 forces the pre-pass split of A
    kKnobWorkspaceLimitMiB = 9,  // cap on each library-owned workspace
    kKnobSchedule = 10,      // 0 one CTA per (tile, K range), 1 persistent stream-K, 2 small-problem kernel
    kKnobSkMinSlices = 11,   // stream-K: fewest K slices per CTA run
    kKnobSkGrid = 12,        // stream-K: resident CTAs (grids of under two waves)
    kKnobTf32x3Bn = 13,      // tensor mode: tile columns 128 or 256
    kKnobCount = 14
};
int32_t tuning(Knob k);

// Epilogue activations.
constexpr int kActNone = 0;
constexpr int kActGeluTanh = 1;

// Everything a GEMM launch needs, by value.
struct GemmArgs {
    const float *A;
    const float *B;
    float *C;
    int64_t M, N, K;
    int64_t lda, ldb, ldc;
    float alpha, beta;
    // batch b reads A + b*strideA, B + b*strideB and writes C + b*strideC
    int64_t batch;
    int64_t strideA, strideB, strideC;
    const float *bias;     // length-N vector added to every row, or nullptr
    int32_t act;           // kActNone or kActGeluTanh
    // Work decomposition.  Tiles [0, tail_start) are cut into split_k K ranges
    // of k_per_split each; tiles [tail_start, tiles) into tail_split ranges of
    // tail_k_per_split.  CTA `pid` of the 1-D grid owns one (tile, range)
    // pair; the ranges of one tile are consecutive pids.
    int64_t k_per_split;       // multiple of kBK
    int64_t tail_k_per_split;  // multiple of kBK
    int64_t tail_start;
    int32_t split_k;
    int32_t tail_split;
    int32_t tiles_m, tiles_n;
    // Tiles are numbered over all batches (batch-major).
    // Split tiles only: the partial tile of CTA pid is slot pid - part_base
    // (16 x kThreads float4 per slot), summed by partial_reduce_kernel.
    int64_t part_base;
    float *partials;
    // Persistent stream-K launches of ffma_gemm_kernel (kSched = 1; G =
    // gridDim.x): whole-K tiles [0, dp_rounds * G) round-robin, then the
    // sk_iters K slices (of sk_kt per tile) of the rest in G equal runs.
    int32_t sk_kt;
    int32_t dp_rounds;
    int64_t sk_iters;
};

// Kernel ids a plan can name.
// Both kernels share the tile, the staging and the arithmetic (one
// round-to-nearest fp32 FMA per accumulator per k, same order); they differ
// only in how the FMAs are issued.
enum KernelId : int32_t {
    kKernelFfma128 = 0,    // scalar fma.rn.f32
    kKernelFfma2x128 = 1,  // packed fma.rn.f32x2 (two FMAs per instruction)
    kKernelFfma16x8 = 2,   // 16 x 8 accumulators per thread (operands copied directly)
};

// ---- persistent stream-K kernel (ffma_sk_kernel.cuh) ----
// G = gridDim.x CTAs stay resident and share the work evenly: first
// `dp_rounds` rounds of whole-K tiles handed out round-robin (tile r*G + g
// to CTA g), then the K slices of the remaining tiles, cut into G equal
// contiguous runs over (tile, slice) order.  A tile whose slices several
// CTAs share is summed in a fixed order by partial_reduce_kernel, launched
// after the persistent grid.
struct SkArgs {
    const float *A;
    const float *B;
    float *C;
    int64_t M, N, K;
    int64_t lda, ldb, ldc;
    float alpha, beta;
    int64_t batch;
    int64_t strideA, strideB, strideC;
    const float *bias;
    int32_t act;
    int32_t tiles_m, tiles_n;
    int32_t kt;           // K slices per tile
    int32_t dp_rounds;    // whole-K rounds: tiles [0, dp_rounds * G)
    int32_t grid;         // G, the CTAs launched (every stream-K run non-empty: G <= sk_iters)
    int64_t tiles;        // over all batches (batch-major)
    int64_t sk_iters;     // slices of tiles [dp_rounds * G, tiles), spread over the G CTAs
    float *partials;      // 2 * G partial tiles, summed by partial_reduce_kernel
};
constexpr int kSkMaxContrib = 16;   // most CTAs that may share one tile's K slices
// K slice and ring depth of the stream-K kernel for a tile: both operands
// copied directly (op(A) = A^T, op(B) = B): K slices of T/4 in three pages;
// otherwise (an operand staged through a raw page and transposed) K slices
// of T/8 in four pages.
constexpr int sk_config_bk(int tile, bool direct) {
    return tile == 128 && direct ? 32 : tile / 8;
}
constexpr int sk_config_pages(int tile, bool direct) {
    return tile == 128 && direct ? 3 : 4;
}
// op(A) = A^T when trans_a, op(B) = B^T when trans_b.
cudaError_t launch_ffma_sk(const SkArgs &a, int tile, int bk, int pages, bool vec, bool trans_a,
                           bool trans_b, bool ext, cudaStream_t stream);
cudaError_t launch_ffma_sk_nn(const SkArgs &a, int tile, int bk, int pages, bool vec, bool ext,
                              cudaStream_t stream);
cudaError_t launch_ffma_sk_nt(const SkArgs &a, int tile, int bk, int pages, bool vec,
                              cudaStream_t stream);
cudaError_t launch_ffma_sk_tn(const SkArgs &a, int tile, int bk, int pages, bool vec, bool ext,
                              cudaStream_t stream);
cudaError_t launch_ffma_sk_tt(const SkArgs &a, int tile, int bk, int pages, bool vec,
                              cudaStream_t stream);
// dynamic shared memory of one CTA of the stream-K kernel
constexpr int sk_smem_bytes(int tile, int bk, int pages, bool staged_a, bool staged_b) {
    return (2 * pages + (staged_a ? 2 : 0) + (staged_b ? 2 : 0)) * tile * bk * 4;
}

// op(A) = A^T when trans_a (A stored K x M), op(B) = B^T when trans_b.
// `tile` is 128 or 64 (the plan's bm).
cudaError_t launch_ffma(const GemmArgs &a, int kernel, int tile, bool vec, bool edge,
                        bool trans_a, bool trans_b, cudaStream_t stream);
// the transposed layouts, one translation unit each
cudaError_t launch_ffma_nt(const GemmArgs &a, int tile, bool vec, bool edge, cudaStream_t stream);
cudaError_t launch_ffma_tn(const GemmArgs &a, int tile, bool vec, bool edge, cudaStream_t stream);
cudaError_t launch_ffma_tt(const GemmArgs &a, int tile, bool vec, bool edge, cudaStream_t stream);
// op(A) = A^T, op(B) = B, 128-wide tiles, K slices of 32 (the product on
// transposed copies); split-K allowed; `ext` compiles in batches, bias and
// activation.
constexpr int kWideBK = 32;
// `pdl`: launch as a programmatic dependent of the previous kernel on the
// stream (the transpose pass), for grids of more CTAs than SMs.
cudaError_t launch_ffma_tn_wide(const GemmArgs &a, bool vec, bool edge, bool ext, bool pdl,
                                cudaStream_t stream);
// The same kernel as a persistent stream-K launch of `grid` CTAs (the
// stream-K fields of `a` set).
cudaError_t launch_ffma_tn_wide_sk(const GemmArgs &a, int64_t grid, bool vec, bool edge, bool ext,
                                   bool pdl, cudaStream_t stream);
// The small-problem kernel (ffma_tiny.cu): 32 x 32 tiles, the whole K range
// (at most kTinyMaxK) staged at once, K split across the CTA's 8 warps.
constexpr int64_t kTinyMaxK = 256;
cudaError_t launch_ffma_tiny(const GemmArgs &a, bool vec, cudaStream_t stream);
size_t tiny_smem_bytes(int64_t K);
// The 16 x 8 per-thread kernel (ffma_wide.cu): op(A) = A^T, op(B) = B, 128
// tiles, K slices of 32, no split.
cudaError_t launch_ffma16x8(const GemmArgs &a, bool edge, bool ext, cudaStream_t stream);
// The same two schedules with packed FMA issue (stream-K: plain products only).
cudaError_t launch_ffma_tn_wide_packed(const GemmArgs &a, bool vec, bool edge, bool ext,
                                       bool pdl, cudaStream_t stream);
cudaError_t launch_ffma_tn_wide_sk_packed(const GemmArgs &a, int64_t grid, bool vec, bool edge,
                                          bool pdl, cudaStream_t stream);
// At_b = A_b^T (K x M, row stride ldt) for b < batch, with A_b = A +
// b*stride_a and At_b = At + b*stride_t; M <= 65535 * 32, batch <= 65535.
cudaError_t launch_transpose(const float *A, int64_t M, int64_t K, int64_t lda, float *At,
                             int64_t ldt, cudaStream_t stream, int64_t batch = 1,
                             int64_t stride_a = 0, int64_t stride_t = 0);
cudaError_t launch_scale(float *C, int64_t M, int64_t N, int64_t ldc, float beta,
                         cudaStream_t stream);
cudaError_t launch_epilogue_only(float *C, int64_t M, int64_t N, int64_t ldc, int64_t strideC,
                                 int64_t batch, float beta, const float *bias, int act,
                                 cudaStream_t stream);
cudaError_t launch_ffma_probe(int64_t ctas, int64_t iters, bool packed, float *out,
                              cudaStream_t stream);
cudaError_t ffma_kernel_attributes(cudaFuncAttributes *attr);

// 3xTF32 tensor-core mode (tf32x3_gemm.cu).  K runs along grid dimension y
// of the split passes (32 rows of K per block at most).
constexpr int64_t kTf32x3MaxK = int64_t(65535) * 32;
// Work decomposition of a tensor-mode launch: either every tile cut into
// `split` K ranges (small grids), or only the tiles from tail_start on (the
// last, partly filled wave) cut into `tail_split` ranges.
struct Tf32x3Plan {
    int bn = 256;             // tile columns (tile rows are 128)
    int split = 1;
    int tail_split = 1;
    int64_t tiles = 0;
    int64_t tail_start = 0;   // == tiles when no tail is cut
    // partial tiles the workspace must hold
    int64_t partial_slots() const {
        return split > 1 ? tiles * split : (tail_split > 1 ? (tiles - tail_start) * tail_split : 0);
    }
    int64_t grid() const { return tail_start * split + (tiles - tail_start) * tail_split; }
};
Tf32x3Plan tf32x3_plan(int64_t M, int64_t N, int64_t K, int sms);
size_t tf32x3_workspace_bytes(int64_t M, int64_t N, int64_t K, const Tf32x3Plan &plan, bool fused,
                              bool packed_b);
size_t tf32x3_packed_b_bytes(int64_t K, int64_t N);
bool tf32x3_fusable_a(const float *A, int64_t lda);
bool tf32x3_use_fused_a(const float *A, int64_t lda);
cudaError_t tf32x3_pack_b(int64_t K, int64_t N, const float *B, int64_t ldb, void *packed,
                          cudaStream_t stream);
cudaError_t launch_tf32x3_packed(const float *A, int64_t lda, const void *packed_b, float *C,
                                 int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha,
                                 float beta, void *workspace, unsigned *counters,
                                 const Tf32x3Plan &plan,
                                 uint64_t limit_ns, int inject_stall, cudaStream_t stream);
cudaError_t launch_tf32x3(const float *A, int64_t lda, const float *B, int64_t ldb, float *C,
                          int64_t ldc, int64_t M, int64_t N, int64_t K, float alpha, float beta,
                          void *workspace, unsigned *counters, const Tf32x3Plan &plan,
                          uint64_t limit_ns,
                          int inject_stall, cudaStream_t stream);
// Reads and clears the mode's device error word (synchronises `stream`).
cudaError_t tf32x3_read_error(unsigned *out, cudaStream_t stream);
constexpr uint64_t kWaitLimitNs = 1000000000ull;   // 1 s bound on every device-side wait

}  // namespace sgemm_impl
