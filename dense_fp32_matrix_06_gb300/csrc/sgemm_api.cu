// sgemm_api.cu -- the C ABI: argument checks, the per-shape planner, the
// library-owned split-K workspace and the launches.
//
// The boundary follows the Python-facing matmul of velog @levelstage
// "AutoMinepp7" (section "직사각형 타일링"): check ranks and the inner
// dimension before any work and report a mismatch as an error; here the
// caller passes device pointers and leading dimensions instead of arrays, and
// errors are status codes.  The tile constants the pages tune by hand
// ("AutoMinepp7", section "세부 조정") become a per-shape choice in gemm_plan.
#include <cuda_runtime.h>

#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/sgemm.h"
#include "sgemm_internal.h"

using namespace sgemm_impl;

namespace {

thread_local int g_last_cuda_error = 0;

sgemm_status cuda_fail(cudaError_t e, sgemm_status s) {
    g_last_cuda_error = int(e);
    return s;
}

struct DeviceInfo {
    bool probed = false;
    bool supported = false;
    int sms = 0;
};

std::mutex g_dev_mu;
std::vector<DeviceInfo> g_devices;

// SM count of the current device, or 0 when the device cannot run the kernels.
sgemm_status current_device(int *dev_out, int *sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_UNSUPPORTED_DEVICE);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (int(g_devices.size()) <= dev) g_devices.resize(dev + 1);
    DeviceInfo &d = g_devices[dev];
    if (!d.probed) {
        int major = 0, minor = 0, sms = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaFuncAttributes attr;
        const bool image_ok = ffma_kernel_attributes(&attr) == cudaSuccess;
        cudaGetLastError();  // clear a sticky "no kernel image" from the probe
        d.supported = image_ok && major == 10 && minor == 3 && sms > 0;
        d.sms = sms;
        d.probed = true;
    }
    if (dev_out) *dev_out = dev;
    if (sms_out) *sms_out = d.sms;
    return d.supported ? SGEMM_OK : SGEMM_ERR_UNSUPPORTED_DEVICE;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

sgemm_status check_sizes(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                         int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_ARG;
    if (lda < (K > 1 ? K : 1)) return SGEMM_ERR_INVALID_ARG;
    if (ldb < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_ARG;
    if (ldc < (N > 1 ? N : 1)) return SGEMM_ERR_INVALID_ARG;
    // the tile grid is launched as one 1-D grid dimension
    if (ceil_div(M, kSmallTile) * ceil_div(N, kSmallTile) > int64_t(INT32_MAX))
        return SGEMM_ERR_INVALID_ARG;
    return SGEMM_OK;
}

// Split-K choice.  Estimated time in units of "one k of one CTA tile":
// waves * k_per_split, plus a per-CTA cost for writing and re-reading the
// partial tiles.  Only considered when the tile grid fills less than one wave
// of resident CTAs.
int choose_split(int64_t tiles, int64_t K, int sms, int64_t *k_per_split, int bk = kBK,
                 int cps = kCtasPerSm) {
    const int64_t slots = int64_t(sms) * cps;
    const int64_t kslices = ceil_div(K, bk);
    int best = 1;
    int64_t best_kps = kslices * bk;
    {
        const int s = tuning(kKnobSplit);
        if (s >= 1) {
            int64_t kps = ceil_div(kslices, s) * bk;
            int eff = int(ceil_div(K, kps > 0 ? kps : 1));
            if (eff < 1) eff = 1;
            if (eff > 1 && tiles > kMaxSplitTiles) eff = 1, kps = kslices * bk;
            *k_per_split = eff > 1 ? kps : kslices * bk;
            return eff;
        }
    }
    // A grid that gives 90-100 % of the SMs one tile each runs best unsplit:
    // a CTA alone on an SM runs at close to the SM's full rate (GPT-2 QKV,
    // 144 tiles on 152 SMs: 43.9 TFLOP/s unsplit, 41.8 split in two).  Past
    // one tile per SM, splitting evens the load again (MLP-up, 192 tiles:
    // 35.1 unsplit, 39.8 in three).
    if (tiles * 10 >= int64_t(sms) * 9 && tiles <= sms) {
        *k_per_split = best_kps;
        return 1;
    }
    if (tiles < slots && tiles <= kMaxSplitTiles && K >= 2 * 128) {
        double best_cost = double(ceil_div(tiles, slots)) * double(best_kps);
        for (int s = 2; s <= kMaxSplit; ++s) {
            const int64_t kps = ceil_div(kslices, s) * bk;
            if (kps < 128) break;  // keep at least 128 of K per partition
            const int eff = int(ceil_div(K, kps));
            const int64_t ctas = tiles * eff;
            const double cost = double(ceil_div(ctas, slots)) * (double(kps) + 8.0 * eff + 32.0);
            if (cost < best_cost * 0.97) {
                best_cost = cost;
                best = eff;
                best_kps = kps;
            }
        }
    }
    *k_per_split = best_kps;
    return best;
}

// Tail split (opt-in, tuning knob kKnobTail = s with s >= 2): cut only the tiles of
// the last, partly filled wave of resident CTAs into s K ranges.  Off by
// default: measured on GB300 it gains nothing (8192^3: 59.26 TFLOP/s either
// way; 4096^3: 56.35 with, 56.93 without), because with two CTAs per SM a
// CTA left alone on its SM in the last wave already runs at close to the
// whole SM's rate.  Plans with the A^T pass never take it: tried there (the
// last 144 of 8192^3's 4096 tiles in two K ranges), the split build of the
// kernel ran every wave slower (8192^3 15.89 -> 16.31 ms, 4096^3 2091 ->
// 2144 us).
void choose_tail(int64_t tiles, int64_t K, int sms, int64_t *tail_start, int *tail_split,
                 int64_t *tail_kps) {
    const int64_t slots = int64_t(sms) * kCtasPerSm;
    const int64_t kslices = ceil_div(K, kBK);
    *tail_start = tiles;
    *tail_split = 1;
    *tail_kps = kslices * kBK;
    const int want = tuning(kKnobTail);
    if (want < 2 || tiles < slots) return;
    const int64_t rem = tiles % slots;
    if (rem == 0 || rem > kMaxSplitTiles) return;
    const int64_t kps = ceil_div(kslices, want > kMaxSplit ? kMaxSplit : want) * kBK;
    const int eff = int(ceil_div(K, kps));
    if (eff < 2) return;
    *tail_start = tiles - rem;
    *tail_split = eff;
    *tail_kps = kps;
}

size_t split_workspace(int64_t tiles, int split_k, int64_t tail_start, int tail_split,
                       int tile = kBM) {
    const size_t per = size_t(tile) * tile * sizeof(float);
    if (split_k > 1) return kCounterBytes + size_t(tiles) * split_k * per;
    if (tail_split > 1) return kCounterBytes + size_t(tiles - tail_start) * tail_split * per;
    return 0;
}

// CTA tile for a shape.  64-wide tiles when 128-wide ones would waste 40 % or
// more of their area on padding (N = 64 attention products), or would fill
// under half the SMs while K is too short (<= 768) for split-K to make up
// for it; 128 otherwise.  Measured on GB300 (TFLOP/s, 64 against 128): 256^3
// 1.33 / 1.14, 1023x777x513 17.8 / 15.7, but 1024^3 28.9 / 31.5,
// 1024x768x3072 37.8 / 41.9, 1024x1024x16384 40.6 / 47.0 (with the split the
// cost model picks for each).  Split grids of 128-wide tiles that load the
// SMs unevenly are replanned afterwards (choose_balanced_small: 1024^3 then
// runs 64-wide tiles in eight exact K ranges).
// The tuning knob kKnobTile (64/128) overrides the choice for sweeps.
int choose_tile(int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
    {
        const int t = tuning(kKnobTile);
        if (t == 64 || t == 128) return t;
    }
    const int64_t per_batch = ceil_div(M, 128) * ceil_div(N, 128);
    const double used = double(M) * double(N) / (double(per_batch) * 128.0 * 128.0);
    if (used < 0.6) return kSmallTile;
    if (2 * per_batch * batch < sms && K <= 768) return kSmallTile;
    return 128;
}

// Issue form plan_core names: scalar FMAs unless the tuning knob kKnobKernel
// (0 = scalar, 1 = packed) asks otherwise.  plan_impl then moves the plans
// where packed issue measured faster to it (the direct-copy product after the
// A^T pass, split-K and 64-wide plans; see make_wide and plan_impl_base).
// Unsplit grids that stage A through registers stay scalar: there the
// broadcast operand pairs of the packed form push the kernel past 128
// registers (8192^3 with A staged: scalar 59.0 TFLOP/s, packed 54.0).
int32_t default_kernel() {
    const int k = tuning(kKnobKernel);
    if (k == kKernelFfma128 || k == kKernelFfma2x128) return k;   // (2: direct-copy plans only)
    return kKernelFfma128;
}

// ---- persistent stream-K schedule ----
constexpr int kSkMinSlicesDefault = 8; // fewest K slices in one CTA's run
constexpr int64_t kSkMaxK = int64_t(1) << 30;   // the kernel counts K in 32-bit integers

int64_t sk_slots(int tile, int sms) {
    return int64_t(sms) * (tile == kSmallTile ? kSmallCtasPerSm : kCtasPerSm);
}

// Turns plan `p` (tile, tiles_m, tiles_n already set) into a stream-K plan
// for `tiles` tiles of ceil(K / bk) slices on `sms` SMs.  With two waves of
// tiles or more, whole-K tiles go round-robin to every resident CTA until
// at most two waves' worth are left (all of them when the tiles fill whole
// waves); the K slices of what is left, or of every tile of a smaller grid,
// are split into G equal runs, G being the resident CTA count, or fewer so
// that a run keeps at least kKnobSkMinSlices slices and a tile is shared by
// at most kSkMaxContrib runs.
void plan_stream_k(gemm_plan_t &p, int64_t M, int64_t N, int64_t tiles, int64_t K, int sms,
                   bool direct) {
    const int tile = p.bm;
    const int bk = sk_config_bk(tile, direct);
    const int64_t kt = ceil_div(K, bk);
    const int64_t S = sk_slots(tile, sms);
    int64_t dp_rounds = 0, sk_tiles = tiles, G = S;
    if (tiles >= 2 * S) {
        dp_rounds = tiles / S - (tiles % S ? 1 : 0);
        sk_tiles = tiles - dp_rounds * S;
    } else {
        const int32_t knob = tuning(kKnobSkMinSlices);
        const int64_t min_sl = knob > 0 ? knob : kSkMinSlicesDefault;
        G = std::min<int64_t>(S, std::max<int64_t>(1, tiles * kt / min_sl));
        G = std::min<int64_t>(G, tiles * kSkMaxContrib);
        if (const int32_t force = tuning(kKnobSkGrid); force > 0)
            G = std::min<int64_t>({int64_t(force), tiles * kt, tiles * kSkMaxContrib});
    }
    p.schedule = 1;
    p.dp_rounds = int32_t(dp_rounds);
    p.sk_iters = sk_tiles * kt;
    p.grid_ctas = G;
    p.bk = bk;
    p.stages = sk_config_pages(tile, direct);
    p.split_k = 1;
    p.tail_split = 1;
    p.tail_start = tiles;
    p.k_per_split = kt * bk;
    p.tail_k_per_split = p.k_per_split;
    // direct 128-wide plans of whole tiles run unchecked; the others check
    // every tile (a few instructions a slice)
    p.edge = (direct && tile == 128 && p.vec && M % tile == 0 && N % tile == 0 && K % bk == 0)
                 ? 0
                 : 1;
    p.workspace_bytes =
        p.sk_iters > 0 ? kCounterBytes + size_t(2 * G) * tile * tile * sizeof(float) : 0;
}

// Persistent stream-K or one CTA per (tile, K range).  Measured on GB300
// (microseconds, L2 flushed, stream-K / split-K planned as above): the
// stream-K kernel wins where the grid is far from a whole wave and the K
// ranges are long or the problem tiny -- 256^3 on 64-wide tiles 17.1 / 19.2,
// 1024x1024x16384 (64 tiles of 128) 672 / 709 -- and loses where split-K
// already balances the GPU (1024^3 78.5 / 66.2, 1023x777x513 49.8 / 41.6,
// GPT-2 QKV 90.9 / 82.6, 2048^3 344.7 / 338.6): its main loop issues more
// instructions and stalls more in dispatch than the split-K kernel's, which
// eats what the even split gains.  The tuning knob kKnobSchedule overrides.
bool choose_stream_k(int tile, int64_t tiles, int64_t K, int sms) {
    const int32_t force = tuning(kKnobSchedule);
    if (force == 0 || force == 1 || force == 2) return force == 1;
    if (tile == kSmallTile) return 4 * tiles < sms;
    return 2 * tiles <= sms && K >= 8192;
}

// `direct`: both operands reach the kernel by direct copies (op(A) = A^T and
// op(B) = B), which lets a stream-K plan take the longer K slice.
// `force_tile` / `force_split` (0: the planner's choice) serve the balance
// rule below (choose_balanced_small).
void plan_core(int64_t M, int64_t N, int64_t K, int64_t batch, bool vec, int sms,
               gemm_plan_t *out, bool direct = false, int force_tile = 0, int force_split = 0) {
    gemm_plan_t p;
    std::memset(&p, 0, sizeof(p));
    const int tile = force_tile ? force_tile : choose_tile(M, N, K, batch, sms);
    const int bk = tile / 8;
    const int cps = tile == kSmallTile ? kSmallCtasPerSm : kCtasPerSm;
    p.mode = SGEMM_MODE_FFMA;
    p.kernel = default_kernel();
    p.bm = tile;
    p.bn = tile;
    p.bk = bk;
    p.threads = (tile / 8) * (tile / 8);
    p.stages = 2;
    p.vec = vec ? 1 : 0;
    p.tiles_m = ceil_div(M, tile);
    p.tiles_n = ceil_div(N, tile);
    const int64_t tiles = p.tiles_m * p.tiles_n * batch;
    int64_t kps = 0;
    p.split_k = (M > 0 && N > 0 && K > 0 && batch > 0)
                    ? choose_split(tiles, K, sms, &kps, bk, cps)
                    : 1;
    if (force_split > 1) {
        p.split_k = force_split;
        kps = K / force_split;
    }
    if (p.split_k == 1) kps = ceil_div(K, bk) * bk;
    p.k_per_split = kps > 0 ? kps : bk;
    int tail_split = 1;
    p.tail_start = tiles;
    p.tail_k_per_split = p.k_per_split;
    if (tile == 128 && p.split_k == 1 && M > 0 && N > 0 && K > 0)
        choose_tail(tiles, K, sms, &p.tail_start, &tail_split, &p.tail_k_per_split);
    p.tail_split = tail_split;
    const bool full = (M % tile == 0) && (N % tile == 0) && (K % bk == 0) &&
                      (p.split_k == 1 || K % p.k_per_split == 0) &&
                      (p.tail_split == 1 || K % p.tail_k_per_split == 0);
    p.edge = (p.vec && full) ? 0 : 1;
    p.grid_ctas = p.tail_start * p.split_k + (tiles - p.tail_start) * p.tail_split;
    p.workspace_bytes = split_workspace(tiles, p.split_k, p.tail_start, p.tail_split, tile);
    if (M > 0 && N > 0 && K > 0 && batch > 0 && K <= kSkMaxK &&
        choose_stream_k(tile, tiles, K, sms))
        plan_stream_k(p, M, N, tiles, K, sms, direct);
    *out = p;
}

// Transposing A first, and how the product then runs.  The kernel stages an
// operand whose stored rows run along K (A as given) through registers and
// transposing shared stores, and copies one whose rows run along M (A^T)
// straight in with cp.async, which leaves it 8 registers and ~10
// instructions per K slice lighter, lets the product run in K slices of 32
// through a three-page ring, and lets it issue its FMAs packed within 128
// registers (choose_wide_kernel).  A transpose pass costs 8*M*K bytes of HBM
// traffic, about 35/N of the product's time.
//
// Three plans compete: split-K without the pass (kTransposeNone), the pass
// and one CTA per tile or K range (kTransposeGrid), the pass and a
// persistent stream-K launch (kTransposeStreamK).  Measured on GB300 with
// packed issue (N = 768, 1024 and 2048, 32..1216 tiles of 128, K = 64..4096;
// microseconds, L2 flushed; none / grid / stream-K):
//  * the pass pays for K >= 256 from 0.45 of a wave (S = 2 CTAs per SM) on:
//    1152x2048x768, 144 tiles: 82.6 / 70.3 / 88.7; 9728x2048x512, 1216
//    tiles: 356 / 318 / 371; for K < 256 only on grids of 8 waves and more
//    (8192x8192x64: 181 / 173);
//  * for K >= 1024 it pays except on small grids: under 0.3 S at K = 1024
//    (1024^3: 57 / 57 / 63) and under 0.15 S at larger K (256x2048x2048:
//    55.9 / 56.0 / 62.0);
//  * stream-K after the pass beats the grid where the grid would put a
//    second CTA on only a few SMs, from sms to 1.25 sms tiles (2560x1024x2048,
//    160 tiles: 252 / 225 / 215); elsewhere the grid wins (2048^3: 353 /
//    316 / 320; 1792x2048x2048, 224 tiles: 277 / 260 / 286; 1024x1024x16384,
//    64 tiles split along K: 612 against 620 stream-K).
// Tuning knobs: kKnobTransposeA (0/1) forces the pass off or on,
// kKnobSchedule (0/1) the grid or stream-K after it.
enum TransposeFamily { kTransposeNone = 0, kTransposeGrid = 1, kTransposeStreamK = 2 };

// The bands above, for `tiles` 128-wide tiles (over all batches) and K.
int transpose_band(int64_t tiles, int64_t K, int sms) {
    const int64_t S = int64_t(sms) * kCtasPerSm;
    if (K < 256) return tiles >= 8 * S ? kTransposeGrid : kTransposeNone;
    if (K < 1024) return 20 * tiles >= 9 * S ? kTransposeGrid : kTransposeNone;
    if (tiles > sms && 4 * tiles <= 5 * int64_t(sms)) return kTransposeStreamK;
    if (K < 2048) return 10 * tiles >= 3 * S ? kTransposeGrid : kTransposeNone;
    return 20 * tiles >= 3 * S ? kTransposeGrid : kTransposeNone;
}

int choose_transpose_a(const gemm_plan_t &p, int64_t M, int64_t N, int64_t K, int sms) {
    const bool able = p.bm == 128 && p.tail_split == 1 && p.vec && K >= 1 &&
                      M <= int64_t(65535) * 32;
    if (!able) return kTransposeNone;
    const int64_t tiles = p.tiles_m * p.tiles_n;
    int want = N >= 768 ? transpose_band(tiles, K, sms) : int(kTransposeNone);
    const int32_t f = tuning(kKnobTransposeA);
    if (f == 0) return kTransposeNone;
    if (f == 1 && want == kTransposeNone)
        want = p.schedule == 1 ? kTransposeStreamK : kTransposeGrid;
    const int32_t sched = tuning(kKnobSchedule);
    if (want != kTransposeNone && (sched == 0 || sched == 1))
        want = sched == 1 ? kTransposeStreamK : kTransposeGrid;
    return want;
}

size_t transpose_bytes(int64_t M, int64_t K, int64_t *ld) {
    *ld = (M + 3) / 4 * 4;
    return (size_t(K) * size_t(*ld) * sizeof(float) + 255) / 256 * 256;
}

// Workspace of a transposing plan: [reserved block][partial tiles][A^T].
size_t transpose_workspace(const gemm_plan_t &p, int64_t M, int64_t K, int64_t *ld,
                           size_t *at_offset) {
    const int64_t tiles = p.tiles_m * p.tiles_n;
    const size_t tile_bytes = size_t(p.bm) * p.bm * sizeof(float);
    const size_t parts = p.schedule == 1 ? (p.sk_iters > 0 ? size_t(2 * p.grid_ctas) * tile_bytes : 0)
                         : p.split_k > 1 ? size_t(tiles) * p.split_k * tile_bytes
                                         : 0;
    *at_offset = kCounterBytes + parts;
    return *at_offset + transpose_bytes(M, K, ld);
}

// sgemm_ex's transposed copies: the bands of choose_transpose_a over all
// the batches' tiles, for each operand to be copied (A's copy costs 8*M*K
// bytes against 2*M*N*K FLOPs, so it needs N >= 768; B's needs M >= 768), on
// 128-wide one-CTA-per-(tile, K range) plans; where the bands ask for
// stream-K after the pass, sgemm_ex runs the grid after it.  With op(A) =
// A^T and op(B) = B nothing is copied: the pass is only the switch to the
// direct-copy kernel (K slices of 32).
bool ex_transpose_first(const gemm_plan_t &p, int64_t M, int64_t N, int64_t K, int64_t batch,
                        bool copy_a, bool copy_b, int sms) {
    const bool able = p.schedule == 0 && p.bm == 128 && p.tail_split == 1 && p.vec &&
                      batch <= 65535 && M <= int64_t(65535) * 32 && N <= int64_t(65535) * 32;
    const int64_t tiles = p.tiles_m * p.tiles_n * batch;
    bool want = able && (!copy_a || N >= 768) && (!copy_b || M >= 768) &&
                transpose_band(tiles, K, sms) != kTransposeNone;
    const int f = tuning(kKnobTransposeA);
    if (f == 0) want = false;
    if (f == 1) want = able;
    return want;
}

// Kernel of a plan whose operands both arrive by direct copies (op(A) = A^T
// copied first, op(B) = B): the 8 x 8 kernel with packed FMA issue
// (fma.rn.f32x2; the same roundings in the same order as scalar issue, so
// the same C bit for bit).  Without register staging of A the packed build
// stays within 128 registers, and half as many FMA instructions leave the
// issue slots room: measured on GB300 (scalar / packed), 8192^3 16.70 /
// 15.85 ms, 4096^3 2205 / 2090 us, split-K plans 1536x1024x1024 79.6 /
// 75.4 and 1792x2048x2048 270.0 / 258.7 us, stream-K 2048^3 323.3 / 320.1
// us.  The tuning knob kKnobKernel picks scalar issue (0) or the 16 x 8
// per-thread kernel (2, plans that do not split K).
int32_t choose_wide_kernel(const gemm_plan_t &q) {
    const int32_t k = tuning(kKnobKernel);
    if (k == kKernelFfma16x8 && q.split_k == 1 && q.tail_split == 1) return kKernelFfma16x8;
    if (k == kKernelFfma128) return kKernelFfma128;
    return kKernelFfma2x128;
}

// Re-plans a 128-wide one-CTA-per-(tile, K range) plan for the kernel that
// copies both operands directly (op(A) = A^T, op(B) = B): K slices of 32
// through a three-page ring, split-K chosen for that slice.
void make_wide(gemm_plan_t &q, int64_t M, int64_t N, int64_t K, int64_t batch, int sms) {
    q.bk = kWideBK;
    q.stages = 3;
    const int64_t tiles = q.tiles_m * q.tiles_n * batch;
    int64_t kps = 0;
    q.split_k = choose_split(tiles, K, sms, &kps, kWideBK, kCtasPerSm);
    q.k_per_split = q.split_k > 1 ? kps : ceil_div(K, kWideBK) * kWideBK;
    q.tail_split = 1;
    q.tail_start = tiles;
    q.tail_k_per_split = q.k_per_split;
    q.grid_ctas = tiles * q.split_k;
    q.edge = (q.vec && M % 128 == 0 && N % 128 == 0 && K % kWideBK == 0 &&
              (q.split_k == 1 || K % q.k_per_split == 0))
                 ? 0
                 : 1;
    q.workspace_bytes = split_workspace(tiles, q.split_k, q.tail_start, q.tail_split, 128);
    q.kernel = choose_wide_kernel(q);
}

// The small-problem kernel: 32 x 32 tiles with the whole K range (<= 256)
// staged in one go and split across the CTA's warps.  Chosen for products of
// at most 2^25 multiply-adds whose 32 x 32 tiles fit in one wave (three CTAs
// per SM), where the tiled kernels wait on loads and split-K round trips
// rather than compute.  Measured on GB300 (microseconds, L2 flushed, small
// kernel / tiled): 256^3 10.9 / 21.1, 512x512x128 10.9 / 17.1, 256x1024x128
// 10.9 / 19.1, 128x128x256 10.9 / 19.1; but 1024x1024x32 (1024 tiles) 13.0 /
// 10.9.  The tuning knob kKnobSchedule = 2 forces it (when K allows), 0 or 1
// rule it out.
bool choose_tiny(int64_t M, int64_t N, int64_t K, int sms) {
    if (K < 1 || K > kTinyMaxK) return false;
    const int32_t force = tuning(kKnobSchedule);
    if (force >= 0) return force == 2;
    return M * N * K <= (int64_t(1) << 25) && ceil_div(M, 32) * ceil_div(N, 32) <= 3 * sms;
}

void plan_tiny(gemm_plan_t &p, int64_t M, int64_t N, int64_t K) {
    const int64_t tiles_m = ceil_div(M, 32), tiles_n = ceil_div(N, 32);
    const int64_t kp = 8 * (ceil_div(K, 32) * 4);
    p.schedule = 2;
    p.kernel = kKernelFfma128;
    p.bm = p.bn = 32;
    p.bk = int32_t(kp);
    p.threads = 256;
    p.stages = 1;
    p.split_k = 1;
    p.tail_split = 1;
    p.tiles_m = tiles_m;
    p.tiles_n = tiles_n;
    p.tail_start = tiles_m * tiles_n;
    p.k_per_split = p.tail_k_per_split = kp;
    p.grid_ctas = tiles_m * tiles_n;
    p.edge = 1;
    p.dp_rounds = 0;
    p.sk_iters = 0;
    p.transpose_a = 0;
    p.a_t_ld = 0;
    p.workspace_bytes = 0;
}

sgemm_status plan_impl_base(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                            int64_t ldc, const void *A, const void *B, const void *C,
                            int sms, gemm_plan_t *out, bool allow_transpose) {
    // B and C decide whether a product after the A^T pass can take the vector
    // path: the copy of A is written aligned whatever A's own alignment
    const bool vec_bc = ldb % 4 == 0 && ldc % 4 == 0 && aligned16(B) && aligned16(C);
    const bool vec = vec_bc && lda % 4 == 0 && aligned16(A);
    plan_core(M, N, K, 1, vec, sms, out);
    if (M > 0 && N > 0 && choose_tiny(M, N, K, sms)) {
        plan_tiny(*out, M, N, K);
        return SGEMM_OK;
    }
    int fam = kTransposeNone;
    if (allow_transpose && M > 0 && N > 0 && K > 0 && vec_bc) {
        gemm_plan_t probe = *out;   // the bands as if A were aligned too
        probe.vec = 1;
        fam = choose_transpose_a(probe, M, N, K, sms);
    }
    if (fam != kTransposeNone) {
        // the product then runs with both operands copied by rows, in K slices of 32
        gemm_plan_t &q = *out;
        q.transpose_a = 1;
        q.vec = 1;
        if (fam == kTransposeStreamK) {
            plan_stream_k(q, M, N, q.tiles_m * q.tiles_n, K, sms, true);
            q.kernel = tuning(kKnobKernel) == kKernelFfma128 ? kKernelFfma128 : kKernelFfma2x128;
            size_t at_offset = 0;
            q.workspace_bytes = transpose_workspace(q, M, K, &q.a_t_ld, &at_offset);
            return SGEMM_OK;
        }
        q.schedule = 0;
        q.dp_rounds = 0;
        q.sk_iters = 0;
        make_wide(q, M, N, K, 1, sms);
        size_t at_offset = 0;
        q.workspace_bytes = transpose_workspace(q, M, K, &q.a_t_ld, &at_offset);
        return SGEMM_OK;
    }
    // Without the pass, split-K plans of 128-wide tiles and every 64-wide
    // plan issue their FMAs packed (fma.rn.f32x2; the same roundings in the
    // same order, so the same C bit for bit).  Measured on GB300
    // (microseconds, scalar / packed): 1024^3 58.0 / 56.0, MLP-up 108.1 /
    // 103.0, MLP-down 104.0 / 100.0; 64-wide tiles: 1023x777x513 37.5 / 34.5,
    // 768^3 74.4 / 70.3, 1000x1000x300 29.3 / 28.3.  Unsplit 128-wide grids
    // lose (GPT-2 QKV 82.6 / 105.1, 8192x8192x64 181 / 201): they stay
    // scalar.
    gemm_plan_t &q = *out;
    if (q.schedule == 0 && (q.bm == kSmallTile || q.split_k > 1) && tuning(kKnobKernel) < 0)
        q.kernel = kKernelFfma2x128;
    return SGEMM_OK;
}

// Split-K grids of 128-wide tiles that give every SM one CTA and some a
// second (between sms and 1.75 sms CTAs) leave the SMs unevenly loaded: at
// 1024^3, 64 tiles in four K ranges put two CTAs on 104 SMs and one on 48.
// 64-wide tiles in enough exact K ranges (at least 128 deep) for about 13.5
// CTAs a SM spread the same work evenly.  Measured on GB300 (microseconds,
// L2 flushed, 128-wide plan / 64-wide): 1024^3 55.9 / 51.8 (8 ranges),
// 1024x1024x2048 93.8 / 90.8 (8), 512x1024x2048 56.9 / 53.9 (16),
// 1024x1024x4096 173.7 / 169.6 (8); grids already near two CTAs a SM keep
// 128 (768x1024x1024, 288 CTAs: 44.6 against 45.7; 896x896x1536, 294 CTAs:
// 55.9 against 62.1), as do grids of one CTA a SM or fewer (GPT-2 QKV, 144
// CTAs: 72.4 against 80.6 at best).  Checked on sixteen other shapes the rule
// changes: 0 to 16 % faster, none slower.  Returns the number of K ranges, 0
// for no change.
int choose_balanced_small(const gemm_plan_t &q, int64_t M, int64_t N, int64_t K, int sms) {
    if (tuning(kKnobTile) >= 0 || tuning(kKnobSplit) >= 0 || tuning(kKnobSchedule) >= 0)
        return 0;
    if (q.bm != 128 || q.schedule != 0 || q.split_k < 2 || q.tail_split != 1) return 0;
    if (q.grid_ctas <= sms || 4 * q.grid_ctas > 7 * int64_t(sms)) return 0;
    const int64_t tiles64 = ceil_div(M, kSmallTile) * ceil_div(N, kSmallTile);
    const int64_t target = int64_t(27) * sms / 2;   // about 13.5 CTAs a SM
    int best = 0;
    int64_t best_gap = 0;
    for (int s = 2; s <= 16; ++s) {
        if (K % (int64_t(8) * s) != 0 || K / s < 128) continue;   // exact ranges of 8-slices
        const int64_t ctas = tiles64 * s;
        if (ctas < int64_t(kSmallCtasPerSm) * sms) continue;      // at least one full wave
        const int64_t gap = ctas > target ? ctas - target : target - ctas;
        if (!best || gap < best_gap) {
            best = s;
            best_gap = gap;
        }
    }
    return best;
}

sgemm_status plan_impl(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                       int64_t ldc, const void *A, const void *B, const void *C,
                       int sms, gemm_plan_t *out, bool allow_transpose = true) {
    sgemm_status st = plan_impl_base(M, N, K, lda, ldb, ldc, A, B, C, sms, out, allow_transpose);
    if (st != SGEMM_OK) return st;
    // (measured on operands that all take the 16-byte path; others keep the plan)
    const bool vec = ldb % 4 == 0 && ldc % 4 == 0 && aligned16(B) && aligned16(C) &&
                     lda % 4 == 0 && aligned16(A);
    const int s64 = vec ? choose_balanced_small(*out, M, N, K, sms) : 0;
    if (s64 > 0) {
        plan_core(M, N, K, 1, vec, sms, out, false, kSmallTile, s64);
        if (tuning(kKnobKernel) < 0) out->kernel = kKernelFfma2x128;
    }
    return SGEMM_OK;
}

// ---- library-owned workspace: one buffer per (device, stream) ----
struct Workspace {
    int dev;
    void *stream;
    void *ptr;
    size_t bytes;
};
std::mutex g_ws_mu;
std::vector<Workspace> g_ws;

sgemm_status library_workspace(int dev, cudaStream_t stream, size_t bytes, void **out) {
    std::lock_guard<std::mutex> lock(g_ws_mu);
    Workspace *w = nullptr;
    for (auto &e : g_ws)
        if (e.dev == dev && e.stream == (void *)stream) w = &e;
    if (w && w->bytes >= bytes) {
        *out = w->ptr;
        return SGEMM_OK;
    }
    // An optional cap (tuning knob kKnobWorkspaceLimitMiB) bounds what the
    // library may hold per (device, stream); a request above it fails as an
    // allocation failure would.
    const int32_t cap = tuning(kKnobWorkspaceLimitMiB);
    const size_t limit = cap >= 0 ? size_t(cap) << 20 : SIZE_MAX;
    if (bytes > limit) return cuda_fail(cudaErrorMemoryAllocation, SGEMM_ERR_ALLOC);
    size_t want = bytes + bytes / 4;
    want = (want + 0xFFFFF) & ~size_t(0xFFFFF);
    if (want > limit) want = bytes;
    void *p = nullptr;
    cudaError_t e = cudaMallocAsync(&p, want, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();   // a later launch check must not see this error
        return cuda_fail(e, SGEMM_ERR_ALLOC);
    }
    e = cudaMemsetAsync(p, 0, kCounterBytes, stream);
    if (e != cudaSuccess) {
        cudaFreeAsync(p, stream);
        return cuda_fail(e, SGEMM_ERR_ALLOC);
    }
    if (w) {
        cudaFreeAsync(w->ptr, stream);  // stream-ordered: after earlier users
        w->ptr = p;
        w->bytes = want;
    } else {
        g_ws.push_back(Workspace{dev, (void *)stream, p, want});
    }
    *out = p;
    return SGEMM_OK;
}

// `a` with the stream-K fields of `plan` filled in, for a persistent launch
// of ffma_gemm_kernel (the workspace holds the partial tiles after the counter block).
GemmArgs sk_gemm_args(const gemm_plan_t &plan, GemmArgs a, void *workspace) {
    a.sk_kt = int32_t(ceil_div(a.K, plan.bk));
    a.dp_rounds = plan.dp_rounds;
    a.sk_iters = plan.sk_iters;
    a.split_k = 1;
    a.tail_split = 1;
    a.tail_start = int64_t(plan.tiles_m) * plan.tiles_n * a.batch;
    a.k_per_split = a.tail_k_per_split = int64_t(a.sk_kt) * plan.bk;
    // the partial tiles follow the workspace's reserved counter block
    a.partials = nullptr;
    if (plan.sk_iters > 0)
        a.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes);
    return a;
}

// Launch arguments of a stream-K plan, from the operand fields of `a`.
SkArgs sk_args(const gemm_plan_t &plan, const GemmArgs &a, void *workspace) {
    SkArgs k;
    k.A = a.A;
    k.B = a.B;
    k.C = a.C;
    k.M = a.M;
    k.N = a.N;
    k.K = a.K;
    k.lda = a.lda;
    k.ldb = a.ldb;
    k.ldc = a.ldc;
    k.alpha = a.alpha;
    k.beta = a.beta;
    k.batch = a.batch;
    k.strideA = a.strideA;
    k.strideB = a.strideB;
    k.strideC = a.strideC;
    k.bias = a.bias;
    k.act = a.act;
    k.tiles_m = int32_t(plan.tiles_m);
    k.tiles_n = int32_t(plan.tiles_n);
    k.kt = int32_t(ceil_div(a.K, plan.bk));
    k.dp_rounds = plan.dp_rounds;
    k.grid = int32_t(plan.grid_ctas);
    k.tiles = plan.tiles_m * plan.tiles_n * a.batch;
    k.sk_iters = plan.sk_iters;
    k.partials = nullptr;
    if (plan.sk_iters > 0)
        k.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes);
    return k;
}

sgemm_status run(const gemm_plan_t &plan, int64_t M, int64_t N, int64_t K, float alpha,
                 const float *A, int64_t lda, const float *B, int64_t ldb, float beta,
                 float *C, int64_t ldc, void *workspace, cudaStream_t stream,
                 int sms) {
    if (M == 0 || N == 0) return SGEMM_OK;
    cudaError_t e;
    if (K == 0 || alpha == 0.0f) {
        e = launch_scale(C, M, N, ldc, beta, stream);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    GemmArgs a;
    a.A = A;
    a.B = B;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.lda = lda;
    a.ldb = ldb;
    a.ldc = ldc;
    a.alpha = alpha;
    a.beta = beta;
    a.batch = 1;
    a.strideA = a.strideB = a.strideC = 0;
    a.bias = nullptr;
    a.act = kActNone;
    a.k_per_split = plan.k_per_split;
    a.tail_k_per_split = plan.tail_k_per_split;
    a.tail_start = plan.tail_start;
    a.split_k = plan.split_k;
    a.tail_split = plan.tail_split;
    a.tiles_m = int32_t(plan.tiles_m);
    a.tiles_n = int32_t(plan.tiles_n);
    a.part_base = plan.split_k > 1 ? 0 : plan.tail_start;
    a.partials = nullptr;
    if (plan.split_k > 1 || plan.tail_split > 1)
        a.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + kCounterBytes);
    if (plan.schedule == 2) {
        e = launch_ffma_tiny(a, plan.vec != 0, stream);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    if (plan.transpose_a) {
        int64_t ld = 0;
        size_t at_offset = 0;
        transpose_workspace(plan, M, K, &ld, &at_offset);
        float *at = reinterpret_cast<float *>(static_cast<char *>(workspace) + at_offset);
        e = launch_transpose(A, M, K, lda, at, plan.a_t_ld, stream);
        if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
        a.A = at;
        a.lda = plan.a_t_ld;
        const bool packed = plan.kernel == kKernelFfma2x128;
        // the product as a programmatic dependent of the transpose pass, where
        // its grid has more CTAs than SMs (ffma_gemm_tn.cu)
        const bool pdl = plan.grid_ctas > sms;
        if (plan.schedule == 1)
            e = packed ? launch_ffma_tn_wide_sk_packed(sk_gemm_args(plan, a, workspace),
                                                       plan.grid_ctas, plan.vec != 0,
                                                       plan.edge != 0, pdl, stream)
                       : launch_ffma_tn_wide_sk(sk_gemm_args(plan, a, workspace), plan.grid_ctas,
                                                plan.vec != 0, plan.edge != 0, false, pdl, stream);
        else if (plan.kernel == kKernelFfma16x8)
            e = launch_ffma16x8(a, plan.edge != 0, false, stream);
        else if (packed)
            e = launch_ffma_tn_wide_packed(a, plan.vec != 0, plan.edge != 0, false, pdl, stream);
        else
            e = launch_ffma_tn_wide(a, plan.vec != 0, plan.edge != 0, false, pdl, stream);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    if (plan.schedule == 1) {
        const SkArgs k = sk_args(plan, a, workspace);
        e = launch_ffma_sk(k, plan.bm, plan.bk, plan.stages, plan.vec != 0, false, false, false,
                           stream);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    e = launch_ffma(a, plan.kernel, plan.bm, plan.vec != 0, plan.edge != 0, false, false, stream);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}

bool plan_matches(const gemm_plan_t &p, int64_t M, int64_t N, int64_t K, int64_t lda,
                  int64_t ldb, int64_t ldc, const void *A, const void *B, const void *C) {
    if (p.mode != SGEMM_MODE_FFMA) return false;
    if (p.schedule == 2) {
        gemm_plan_t q;
        std::memset(&q, 0, sizeof(q));
        q.mode = p.mode;
        q.vec = p.vec;
        if (K < 1 || K > kTinyMaxK || M <= 0 || N <= 0) return false;
        plan_tiny(q, M, N, K);
        const bool vec_ok = lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0 && aligned16(A) &&
                            aligned16(B) && aligned16(C);
        if (p.vec && !vec_ok) return false;
        return std::memcmp(&p, &q, sizeof(q)) == 0;
    }
    if (p.kernel != kKernelFfma128 && p.kernel != kKernelFfma2x128 &&
        p.kernel != kKernelFfma16x8)
        return false;
    if (p.kernel == kKernelFfma16x8 &&
        (!p.transpose_a || p.schedule != 0 || p.split_k != 1 || p.tail_split != 1))
        return false;
    const int t = p.bm;
    if ((t != 128 && t != kSmallTile) || p.bn != t || p.threads != (t / 8) * (t / 8))
        return false;
    if (t == kSmallTile && p.kernel == kKernelFfma16x8) return false;
    if (p.tiles_m != ceil_div(M, t) || p.tiles_n != ceil_div(N, t)) return false;
    const int64_t tiles = p.tiles_m * p.tiles_n;
    if (p.schedule != 0 && p.schedule != 1) return false;
    if (p.schedule == 1) {
        // stream-K: whole-K rounds, then every run non-empty, every tile
        // shared by few enough runs, partials inside the workspace
        const bool direct = p.transpose_a != 0;
        if (p.bk != sk_config_bk(t, direct) || p.stages != sk_config_pages(t, direct))
            return false;
        // unchecked tiles only where every tile is whole
        if (p.edge != 1 && !(p.edge == 0 && direct && t == 128 && p.vec && M % t == 0 &&
                             N % t == 0 && K % p.bk == 0))
            return false;
        if (p.split_k != 1 || p.tail_split != 1 || p.tail_start != tiles) return false;
        if (K <= 0) return p.sk_iters == 0 && p.dp_rounds == 0;
        if (K > kSkMaxK) return false;
        const int64_t kt = ceil_div(K, p.bk);
        if (p.k_per_split != kt * p.bk || p.tail_k_per_split != p.k_per_split) return false;
        const int64_t G = p.grid_ctas;
        if (G < 1 || G > INT32_MAX || p.dp_rounds < 0) return false;
        const int64_t dp_tiles = int64_t(p.dp_rounds) * G;
        if (dp_tiles > tiles) return false;
        const int64_t sk_tiles = tiles - dp_tiles;
        if (p.sk_iters != sk_tiles * kt) return false;
        if (sk_tiles > 0 && (G > p.sk_iters || sk_tiles > kMaxSplitTiles ||
                             G > sk_tiles * kSkMaxContrib))
            return false;
        if (p.vec && !(ldb % 4 == 0 && ldc % 4 == 0 && aligned16(B) && aligned16(C) &&
                       (p.transpose_a || (lda % 4 == 0 && aligned16(A)))))
            return false;
        if (p.transpose_a) {
            if (t != 128 || !p.vec || M > int64_t(65535) * 32) return false;
            int64_t ld = 0;
            size_t at_offset = 0;
            const size_t need = transpose_workspace(p, M, K, &ld, &at_offset);
            return p.a_t_ld == ld && p.workspace_bytes == need;
        }
        const size_t need =
            p.sk_iters > 0 ? kCounterBytes + size_t(2 * G) * t * t * sizeof(float) : 0;
        return p.workspace_bytes == need;
    }
    if (p.dp_rounds != 0 || p.sk_iters != 0) return false;
    if (p.bk != (p.transpose_a ? kWideBK : t / 8)) return false;
    if (p.stages != (p.transpose_a ? 3 : 2)) return false;
    if (p.split_k < 1 || p.split_k > kMaxSplit) return false;
    if (p.tail_split < 1 || p.tail_split > kMaxSplit) return false;
    if (p.tail_start < 0 || p.tail_start > tiles) return false;
    if (p.split_k > 1 && (p.tail_start != tiles || tiles > kMaxSplitTiles)) return false;
    if (p.tail_split > 1 && (t != 128 || tiles - p.tail_start > kMaxSplitTiles)) return false;
    if (p.k_per_split <= 0 || p.k_per_split % p.bk != 0) return false;
    if (p.tail_k_per_split <= 0 || p.tail_k_per_split % p.bk != 0) return false;
    if (K > 0 && ceil_div(K, p.k_per_split) != p.split_k) return false;
    if (K > 0 && p.tail_start < tiles && ceil_div(K, p.tail_k_per_split) != p.tail_split)
        return false;
    if (p.grid_ctas != p.tail_start * p.split_k + (tiles - p.tail_start) * p.tail_split)
        return false;
    // (a plan with the A^T pass reads the aligned copy of A, not A)
    const bool vec_ok = ldb % 4 == 0 && ldc % 4 == 0 && aligned16(B) && aligned16(C) &&
                        (p.transpose_a || (lda % 4 == 0 && aligned16(A)));
    if (p.vec && !vec_ok) return false;
    if (!p.edge) {
        if (!p.vec) return false;
        if (M % t || N % t || K % p.bk || (p.split_k > 1 && K % p.k_per_split) ||
            (p.tail_split > 1 && K % p.tail_k_per_split))
            return false;
    }
    if (p.transpose_a) {
        if (t != 128 || p.tail_split != 1 || !p.vec) return false;
        if (M > int64_t(65535) * 32) return false;
        int64_t ld = 0;
        size_t at_offset = 0;
        const size_t need = transpose_workspace(p, M, K, &ld, &at_offset);
        return p.a_t_ld == ld && p.workspace_bytes == need;
    }
    const size_t need = split_workspace(tiles, p.split_k, p.tail_start, p.tail_split, t);
    return p.workspace_bytes == need;
}

}  // namespace

extern "C" {

sgemm_status gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                       int64_t ldc, const void *A, const void *B, const void *C,
                       gemm_plan_t *out) {
    if (!out) return SGEMM_ERR_INVALID_ARG;
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    int sms = 0;
    s = current_device(nullptr, &sms);
    if (s != SGEMM_OK) return s;
    return plan_impl(M, N, K, lda, ldb, ldc, A, B, C, sms, out);
}

sgemm_status gemm_plan_for_sms(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldc, const void *A, const void *B, const void *C,
                               int32_t sm_count, gemm_plan_t *out) {
    if (!out || sm_count < 1) return SGEMM_ERR_INVALID_ARG;
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    return plan_impl(M, N, K, lda, ldb, ldc, A, B, C, sm_count, out);
}

sgemm_status gemm_plan_check(const gemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, const void *A,
                             const void *B, const void *C) {
    if (!plan) return SGEMM_ERR_INVALID_ARG;
    const sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    return plan_matches(*plan, M, N, K, lda, ldb, ldc, A, B, C) ? SGEMM_OK
                                                                : SGEMM_ERR_INVALID_ARG;
}

sgemm_status sgemm(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                   int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                   int64_t ldc, void *stream) {
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    s = current_device(&dev, &sms);
    if (s != SGEMM_OK) return s;
    gemm_plan_t plan;
    s = plan_impl(M, N, K, lda, ldb, ldc, A, B, C, sms, &plan);
    if (s != SGEMM_OK) return s;
    void *ws = nullptr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (plan.workspace_bytes > 0 && K > 0 && alpha != 0.0f) {
        const int last_error = g_last_cuda_error;
        s = library_workspace(dev, st, plan.workspace_bytes, &ws);
        if (s == SGEMM_ERR_ALLOC && plan.transpose_a) {
            // The transposed copy of A only makes the product faster; without
            // room for it, run the plan that reads A as stored (split-K
            // partials at most).
            s = plan_impl(M, N, K, lda, ldb, ldc, A, B, C, sms, &plan, false);
            if (s != SGEMM_OK) return s;
            ws = nullptr;
            s = plan.workspace_bytes > 0 ? library_workspace(dev, st, plan.workspace_bytes, &ws)
                                         : SGEMM_OK;
            if (s == SGEMM_OK) g_last_cuda_error = last_error;
        }
        if (s != SGEMM_OK) return s;
    }
    return run(plan, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ws, st, sms);
}

sgemm_status sgemm_with_plan(const gemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda, const float *B,
                             int64_t ldb, float beta, float *C, int64_t ldc, void *workspace,
                             size_t workspace_bytes, void *stream) {
    if (!plan) return SGEMM_ERR_INVALID_ARG;
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
    if (!plan_matches(*plan, M, N, K, lda, ldb, ldc, A, B, C)) return SGEMM_ERR_INVALID_ARG;
    if (plan->workspace_bytes > 0) {
        if (!workspace || workspace_bytes < plan->workspace_bytes) return SGEMM_ERR_WORKSPACE;
        if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SGEMM_ERR_INVALID_ARG;
    }
    int sms = 0;
    s = current_device(nullptr, &sms);
    if (s != SGEMM_OK) return s;
    return run(*plan, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace,
               static_cast<cudaStream_t>(stream), sms);
}

const char *sgemm_status_string(sgemm_status status) {
    switch (status) {
        case SGEMM_OK: return "SGEMM_OK";
        case SGEMM_ERR_INVALID_ARG: return "SGEMM_ERR_INVALID_ARG: invalid size, leading dimension, pointer or plan";
        case SGEMM_ERR_MISALIGNED: return "SGEMM_ERR_MISALIGNED: operand not 16-byte aligned for this mode";
        case SGEMM_ERR_UNSUPPORTED_DEVICE: return "SGEMM_ERR_UNSUPPORTED_DEVICE: no sm_103 device current";
        case SGEMM_ERR_LAUNCH: return "SGEMM_ERR_LAUNCH: a CUDA launch or call failed";
        case SGEMM_ERR_TIMEOUT: return "SGEMM_ERR_TIMEOUT: a bounded device-side wait gave up";
        case SGEMM_ERR_ALLOC: return "SGEMM_ERR_ALLOC: workspace allocation failed";
        case SGEMM_ERR_WORKSPACE: return "SGEMM_ERR_WORKSPACE: workspace smaller than the plan needs";
    }
    return "SGEMM_ERR_UNKNOWN";
}

int sgemm_last_cuda_error(void) { return g_last_cuda_error; }

sgemm_status sgemm_ffma_probe(int64_t ctas, int64_t iters, int32_t packed, float *out,
                              void *stream) {
    if (ctas <= 0 || ctas > INT32_MAX || iters < 0 || !out) return SGEMM_ERR_INVALID_ARG;
    sgemm_status s = current_device(nullptr, nullptr);
    if (s != SGEMM_OK) return s;
    cudaError_t e =
        launch_ffma_probe(ctas, iters, packed != 0, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// sgemm_noalloc: the same GEMM with its split-K scratch in a fixed buffer that
// lives inside the library, so the call never allocates device memory.
// ---------------------------------------------------------------------------

// The scratch buffer, laid out as a plan's workspace: the reserved counter
// block, then the partial tiles.  Every GPU that loads the library holds it
// until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SGEMM_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
std::vector<void *> g_noalloc_addr;  // device address of the buffer, per device

// Host code cannot use the array's name as a device pointer (on the host it is
// only a stand-in for the symbol), so the device address is looked up once per
// device, with that device current, and cached.
sgemm_status noalloc_scratch(int dev, void **out) {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (int(g_noalloc_addr.size()) <= dev) g_noalloc_addr.resize(dev + 1, nullptr);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) return cuda_fail(e, SGEMM_ERR_LAUNCH);
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return SGEMM_OK;
}

}  // namespace

extern "C" sgemm_status sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                                      const float *A, int64_t lda, const float *B, int64_t ldb,
                                      float beta, float *C, int64_t ldc, void *stream) {
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    s = current_device(&dev, &sms);
    if (s != SGEMM_OK) return s;
    gemm_plan_t plan;
    // no transposed copy of A: it would need M x K floats of scratch
    s = plan_impl(M, N, K, lda, ldb, ldc, A, B, C, sms, &plan, false);
    if (s != SGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    void *ws = nullptr;
    if (plan.workspace_bytes > 0 && K > 0 && alpha != 0.0f) {
        if (plan.workspace_bytes > size_t(SGEMM_NOALLOC_SCRATCH_BYTES)) return SGEMM_ERR_WORKSPACE;
        s = noalloc_scratch(dev, &ws);
        if (s != SGEMM_OK) return s;
        // The buffer keeps whatever the previous call left, which is fine:
        // every partial tile is written before it is read back.
    }
    return run(plan, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, ws, st, sms);
}

// ---------------------------------------------------------------------------
// 3xTF32 tensor-core mode
// ---------------------------------------------------------------------------

namespace {

sgemm_status tf32x3_run(int64_t M, int64_t N, int64_t K, float alpha, const float *A,
                        int64_t lda, const float *B, int64_t ldb, float beta, float *C,
                        int64_t ldc, uint64_t limit_ns, int inject_stall, void *stream) {
    sgemm_status s = check_sizes(M, N, K, lda, ldb, ldc);
    if (s != SGEMM_OK) return s;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || K > kTf32x3MaxK) return SGEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    s = current_device(&dev, &sms);
    if (s != SGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0 || alpha == 0.0f) {
        e = launch_scale(C, M, N, ldc, beta, st);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    const Tf32x3Plan plan = tf32x3_plan(M, N, K, sms);
    // The per-stream workspace starts with the split-K tile counters, which
    // stay zero between calls; the hi/lo operands and partials follow.
    void *ws = nullptr;
    s = library_workspace(
        dev, st,
        kCounterBytes + tf32x3_workspace_bytes(M, N, K, plan, tf32x3_use_fused_a(A, lda), false),
        &ws);
    if (s != SGEMM_OK) return s;
    e = launch_tf32x3(A, lda, B, ldb, C, ldc, M, N, K, alpha, beta,
                      static_cast<char *>(ws) + kCounterBytes, static_cast<unsigned *>(ws), plan,
                      limit_ns, inject_stall, st);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}

}  // namespace

extern "C" sgemm_status sgemm_tf32x3(int64_t M, int64_t N, int64_t K, float alpha,
                                     const float *A, int64_t lda, const float *B, int64_t ldb,
                                     float beta, float *C, int64_t ldc, void *stream) {
    return tf32x3_run(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, kWaitLimitNs, 0, stream);
}

extern "C" sgemm_status sgemm_device_status(void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_UNSUPPORTED_DEVICE;
    unsigned word = 0;
    const cudaError_t e = tf32x3_read_error(&word, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
    return word ? SGEMM_ERR_TIMEOUT : SGEMM_OK;
}

extern "C" sgemm_status sgemm_tf32x3_stall_selftest(int64_t M, int64_t N, int64_t K,
                                                    const float *A, int64_t lda, const float *B,
                                                    int64_t ldb, float *C, int64_t ldc,
                                                    int64_t limit_us, void *stream) {
    if (limit_us <= 0 || limit_us > 1000000 || K <= 0) return SGEMM_ERR_INVALID_ARG;
    sgemm_status s = sgemm_device_status(stream);   // start from a clear record
    if (s != SGEMM_OK && s != SGEMM_ERR_TIMEOUT) return s;
    s = tf32x3_run(M, N, K, 1.0f, A, lda, B, ldb, 0.0f, C, ldc, uint64_t(limit_us) * 1000ull, 1,
                   stream);
    if (s != SGEMM_OK) return s;
    return sgemm_device_status(stream);
}

// ---------------------------------------------------------------------------
// sgemm_ex: batched, transposed-operand, fused bias/GELU form of the product
// ---------------------------------------------------------------------------

extern "C" sgemm_status sgemm_ex(int32_t op_a, int32_t op_b, int64_t M, int64_t N, int64_t K,
                                 float alpha, const float *A, int64_t lda, int64_t stride_a,
                                 const float *B, int64_t ldb, int64_t stride_b, float beta,
                                 float *C, int64_t ldc, int64_t stride_c, int64_t batch,
                                 const float *bias, int32_t act, void *stream) {
    if (op_a != SGEMM_OP_N && op_a != SGEMM_OP_T) return SGEMM_ERR_INVALID_ARG;
    if (op_b != SGEMM_OP_N && op_b != SGEMM_OP_T) return SGEMM_ERR_INVALID_ARG;
    if (act != SGEMM_ACT_NONE && act != SGEMM_ACT_GELU_TANH) return SGEMM_ERR_INVALID_ARG;
    if (M < 0 || N < 0 || K < 0 || batch < 0) return SGEMM_ERR_INVALID_ARG;
    const bool ta = op_a == SGEMM_OP_T, tb = op_b == SGEMM_OP_T;
    // leading dimension >= the stored row length
    if (lda < std::max<int64_t>(1, ta ? M : K)) return SGEMM_ERR_INVALID_ARG;
    if (ldb < std::max<int64_t>(1, tb ? K : N)) return SGEMM_ERR_INVALID_ARG;
    if (ldc < std::max<int64_t>(1, N)) return SGEMM_ERR_INVALID_ARG;
    if (stride_a < 0 || stride_b < 0 || stride_c < 0) return SGEMM_ERR_INVALID_ARG;
    // the outputs of different batches may not overlap
    if (batch > 1 && stride_c < (M > 0 ? (M - 1) * ldc + N : 0)) return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0 || batch == 0) return SGEMM_OK;
    if (ceil_div(M, kSmallTile) * ceil_div(N, kSmallTile) > int64_t(INT32_MAX) / batch)
        return SGEMM_ERR_INVALID_ARG;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    if (K > 0 && alpha != 0.0f && (!A || !B)) return SGEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    sgemm_status s = current_device(&dev, &sms);
    if (s != SGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0 || alpha == 0.0f) {
        e = launch_epilogue_only(C, M, N, ldc, stride_c, batch, beta, bias, act, st);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    const bool vec = lda % 4 == 0 && ldb % 4 == 0 && ldc % 4 == 0 && stride_a % 4 == 0 &&
                     stride_b % 4 == 0 && stride_c % 4 == 0 && aligned16(A) && aligned16(B) &&
                     aligned16(C) && aligned16(bias);
    gemm_plan_t plan;
    plan_core(M, N, K, batch, vec, sms, &plan, ta && !tb);
    const bool ext = batch > 1 || bias != nullptr || act != SGEMM_ACT_NONE;
    // packed issue without the pass: 64-wide and split-K plans of plain op
    // N, N products (as sgemm); the other layouts and the fused epilogue
    // stage A or B^T through registers with scalar issue
    if (ta || tb || ext) plan.kernel = kKernelFfma128;
    else if (plan.schedule == 0 && (plan.bm == kSmallTile || plan.split_k > 1) &&
             tuning(kKnobKernel) < 0)
        plan.kernel = kKernelFfma2x128;
    // Large grids: the operands whose stored rows run along K (A as given,
    // B^T) are first copied transposed into the workspace, so the product
    // runs with both operands copied directly, in K slices of 32 -- what
    // sgemm does for A.  Layout: [reserved block][partial tiles][A^T][B].
    // (op T/N needs no copy, only the longer K slice.)
    const bool copy_a = !ta, copy_b = tb;
    const bool pre = ex_transpose_first(plan, M, N, K, batch, copy_a, copy_b, sms);
    int64_t lda_t = 0, ldb_t = 0, sa_t = 0, sb_t = 0;
    size_t a_off = 0, b_off = 0;
    if (pre) {
        make_wide(plan, M, N, K, batch, sms);
        size_t off = std::max<size_t>(plan.workspace_bytes, kCounterBytes);
        if (copy_a) {
            lda_t = (M + 3) / 4 * 4;
            sa_t = stride_a ? K * lda_t : 0;
            a_off = off;
            off += (size_t(stride_a ? batch : 1) * K * lda_t * sizeof(float) + 255) / 256 * 256;
        }
        if (copy_b) {
            ldb_t = (N + 3) / 4 * 4;
            sb_t = stride_b ? K * ldb_t : 0;
            b_off = off;
            off += (size_t(stride_b ? batch : 1) * K * ldb_t * sizeof(float) + 255) / 256 * 256;
        }
        plan.workspace_bytes = off;
    }
    void *ws = nullptr;
    if (plan.workspace_bytes > 0) {
        s = library_workspace(dev, st, plan.workspace_bytes, &ws);
        if (s != SGEMM_OK) return s;
    }
    GemmArgs a;
    a.A = A;
    a.B = B;
    a.C = C;
    a.M = M;
    a.N = N;
    a.K = K;
    a.lda = lda;
    a.ldb = ldb;
    a.ldc = ldc;
    a.alpha = alpha;
    a.beta = beta;
    a.batch = batch;
    a.strideA = stride_a;
    a.strideB = stride_b;
    a.strideC = stride_c;
    a.bias = bias;
    a.act = act;
    a.k_per_split = plan.k_per_split;
    a.tail_k_per_split = plan.tail_k_per_split;
    a.tail_start = plan.tail_start;
    a.split_k = plan.split_k;
    a.tail_split = plan.tail_split;
    a.tiles_m = int32_t(plan.tiles_m);
    a.tiles_n = int32_t(plan.tiles_n);
    a.part_base = plan.split_k > 1 ? 0 : plan.tail_start;
    a.partials = nullptr;
    if (plan.workspace_bytes > 0)
        a.partials = reinterpret_cast<float *>(static_cast<char *>(ws) + kCounterBytes);
    if (plan.schedule == 1) {
        if (ta && !tb && plan.bm == 128)   // both operands direct: the split-K kernel's loop
            e = launch_ffma_tn_wide_sk(sk_gemm_args(plan, a, ws), plan.grid_ctas, plan.vec != 0,
                                       plan.edge != 0, ext, false, st);
        else
            e = launch_ffma_sk(sk_args(plan, a, ws), plan.bm, plan.bk, plan.stages,
                               plan.vec != 0, ta, tb, ext, st);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    if (pre) {
        char *base = static_cast<char *>(ws);
        if (copy_a) {
            float *at = reinterpret_cast<float *>(base + a_off);
            e = launch_transpose(A, M, K, lda, at, lda_t, st, stride_a ? batch : 1, stride_a,
                                 sa_t);
            if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
            a.A = at;
            a.lda = lda_t;
            a.strideA = sa_t;
        }
        if (copy_b) {
            float *bt = reinterpret_cast<float *>(base + b_off);
            e = launch_transpose(B, N, K, ldb, bt, ldb_t, st, stride_b ? batch : 1, stride_b,
                                 sb_t);
            if (e != cudaSuccess) return cuda_fail(e, SGEMM_ERR_LAUNCH);
            a.B = bt;
            a.ldb = ldb_t;
            a.strideB = sb_t;
        }
        e = plan.kernel == kKernelFfma16x8 ? launch_ffma16x8(a, plan.edge != 0, ext, st)
            : plan.kernel == kKernelFfma2x128
                ? launch_ffma_tn_wide_packed(a, plan.vec != 0, plan.edge != 0, ext,
                                             plan.grid_ctas > sms, st)
                : launch_ffma_tn_wide(a, plan.vec != 0, plan.edge != 0, ext, plan.grid_ctas > sms,
                                      st);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    e = launch_ffma(a, plan.kernel, plan.bm, plan.vec != 0, plan.edge != 0, ta, tb, st);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}

// ---------------------------------------------------------------------------
// 3xTF32 with B packed once
// ---------------------------------------------------------------------------

extern "C" size_t sgemm_tf32x3_packed_b_bytes(int64_t K, int64_t N) {
    if (K <= 0 || N <= 0) return 0;
    return tf32x3_packed_b_bytes(K, N);
}

extern "C" sgemm_status sgemm_tf32x3_pack_b(int64_t K, int64_t N, const float *B, int64_t ldb,
                                           void *packed, size_t packed_bytes, void *stream) {
    if (K <= 0 || N <= 0 || K > kTf32x3MaxK || N > INT32_MAX) return SGEMM_ERR_INVALID_ARG;
    if (ldb < N || !B || !packed) return SGEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(packed) & 255u) != 0) return SGEMM_ERR_MISALIGNED;
    if (packed_bytes < tf32x3_packed_b_bytes(K, N)) return SGEMM_ERR_WORKSPACE;
    sgemm_status s = current_device(nullptr, nullptr);
    if (s != SGEMM_OK) return s;
    const cudaError_t e = tf32x3_pack_b(K, N, B, ldb, packed, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}

extern "C" sgemm_status sgemm_tf32x3_packed(int64_t M, int64_t N, int64_t K, float alpha,
                                           const float *A, int64_t lda, const void *packed_b,
                                           float beta, float *C, int64_t ldc, void *stream) {
    if (M < 0 || N < 0 || K < 0 || M > INT32_MAX || N > INT32_MAX || K > kTf32x3MaxK)
        return SGEMM_ERR_INVALID_ARG;
    if (lda < std::max<int64_t>(1, K) || ldc < std::max<int64_t>(1, N))
        return SGEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return SGEMM_OK;
    if (!C) return SGEMM_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    sgemm_status s = current_device(&dev, &sms);
    if (s != SGEMM_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (K == 0 || alpha == 0.0f) {
        e = launch_scale(C, M, N, ldc, beta, st);
        return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
    }
    if (!A || !packed_b) return SGEMM_ERR_INVALID_ARG;
    if (!tf32x3_fusable_a(A, lda) || (reinterpret_cast<uintptr_t>(packed_b) & 255u) != 0)
        return SGEMM_ERR_MISALIGNED;
    const Tf32x3Plan plan = tf32x3_plan(M, N, K, sms);
    void *ws = nullptr;
    s = library_workspace(
        dev, st,
        kCounterBytes + tf32x3_workspace_bytes(M, N, K, plan, tf32x3_use_fused_a(A, lda), true),
        &ws);
    if (s != SGEMM_OK) return s;
    e = launch_tf32x3_packed(A, lda, packed_b, C, ldc, M, N, K, alpha, beta,
                             static_cast<char *>(ws) + kCounterBytes, static_cast<unsigned *>(ws),
                             plan, kWaitLimitNs, 0, st);
    return e == cudaSuccess ? SGEMM_OK : cuda_fail(e, SGEMM_ERR_LAUNCH);
}
