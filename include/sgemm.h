/*
 * sgemm.h -- C ABI of the GB300 (sm_103a) single-precision GEMM library.
 *
 * Operation (every entry point below computes it, or plans it):
 *
 *     C = alpha * A * B + beta * C
 *
 * on row-major fp32 matrices: A is M x K with leading dimension lda, B is
 * K x N with leading dimension ldb, C is M x N with leading dimension ldc.
 * Element (i, j) of C lives at C[i*ldc + j].
 *
 *   - "Micro_gemm_4x4 - cuBLAS micro GEMM skeleton", section 2 (the kernel
 *     signature: A (M,K), B (K,N), C (M,N), alpha and beta, restrict-qualified,
 *     so C may not overlap A or B) and section 9 (the final C write: when beta
 *     is 0 the old C is not read).
 *   - velog @levelstage "AutoMinepp7", section "직사각형 타일링" (the Python-facing
 *     matmul boundary: shape checks that throw on a rank or inner-dimension
 *     mismatch; here they are status codes).
 *   - "GPU Target" (MLIR tutorial), section "타일링된 행렬 곱셈" (operands are
 *     strided views; here the stride of a row is the leading dimension).
 *
 * Conventions shared by every entry point:
 *   - A, B and C are DEVICE pointers owned by the caller; the library never
 *     frees or retains them.  C must not overlap A or B.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Every call is asynchronous on that stream and never
 *     synchronises the device or the host.
 *   - Arguments are checked before anything is launched.  M, N, K < 0,
 *     lda < max(1, K), ldb < max(1, N), ldc < max(1, N), or a NULL pointer
 *     that the call would dereference -> SGEMM_ERR_INVALID_ARG, nothing
 *     launched.
 *   - Quick returns: M == 0 or N == 0 -> SGEMM_OK, no work.  K == 0 or
 *     alpha == 0 -> C = beta * C without reading A or B (beta == 0 stores
 *     zeros without reading C).
 *   - beta == 0: C is write-only; NaN or garbage in C does not propagate.
 *   - Columns j >= N of C (the padding of a row when ldc > N) are never
 *     written.
 *   - The kernels are compiled for sm_103a only; on another device the calls
 *     return SGEMM_ERR_UNSUPPORTED_DEVICE.
 *   - Arithmetic: fp32 fused multiply-add, round-to-nearest-even, no
 *     flush-to-zero.  Each C entry is summed in a fixed order, so repeated
 *     calls with the same inputs and plan give bit-identical results.
 */
#ifndef DENSE_FP32_MATRIX_06_SGEMM_H
#define DENSE_FP32_MATRIX_06_SGEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    SGEMM_OK = 0,
    SGEMM_ERR_INVALID_ARG = 1,        /* bad size, leading dimension, pointer or plan */
    SGEMM_ERR_MISALIGNED = 2,         /* a mode that needs 16-byte alignment got less */
    SGEMM_ERR_UNSUPPORTED_DEVICE = 3, /* no device, or not an sm_103 device */
    SGEMM_ERR_LAUNCH = 4,             /* a CUDA call failed; see sgemm_last_cuda_error */
    SGEMM_ERR_TIMEOUT = 5,            /* a bounded device-side wait gave up */
    SGEMM_ERR_ALLOC = 6,              /* the library's workspace could not be grown */
    SGEMM_ERR_WORKSPACE = 7           /* caller workspace smaller than the plan needs */
} sgemm_status;

/* Arithmetic mode of a plan. */
typedef enum {
    SGEMM_MODE_FFMA = 0,    /* fp32 CUDA-core FMA (the default product path) */
    SGEMM_MODE_TF32X3 = 1   /* 3xTF32 split precision on the tensor cores (sgemm_tf32x3) */
} sgemm_mode;

/* Operand forms of sgemm_ex: op(X) = X, or X^T (the stored matrix read
 * transposed). */
typedef enum { SGEMM_OP_N = 0, SGEMM_OP_T = 1 } sgemm_op;

/* Activations of sgemm_ex's fused epilogue. */
typedef enum {
    SGEMM_ACT_NONE = 0,
    SGEMM_ACT_GELU_TANH = 1  /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
} sgemm_act;

/* Size of the block at the start of every workspace that the 3xTF32 mode
 * keeps its per-tile failure flags in (zero on entry and left zero by every
 * call); the FFMA kernels leave it untouched. */
#define SGEMM_WORKSPACE_COUNTER_BYTES 16384

/* A per-shape launch configuration chosen by gemm_plan.  Plain data: the
 * caller may inspect it, keep it and pass it back to sgemm_with_plan for any
 * call with the same (M, N, K, lda, ldb, ldc) and pointers of the same
 * alignment class. */
typedef struct {
    int32_t mode;          /* sgemm_mode */
    int32_t kernel;        /* 0: scalar fp32 FMA issue, 1: packed fp32x2 FMA issue
                              (same arithmetic and summation order), 2: a 16 x 8
                              block of accumulators per thread (128 threads a CTA;
                              transpose_a plans without split-K only) */
    int32_t bm, bn, bk;    /* CTA tile (rows of C, columns of C, K slice) */
    int32_t threads;       /* threads per CTA */
    int32_t split_k;       /* K partitions of tiles [0, tail_start) (1 = none) */
    int32_t vec;           /* 1: 16-byte vector loads/stores; 0: 4-byte */
    int32_t edge;          /* 1: bounds-checked tiles; 0: all tiles full */
    int32_t tail_split;    /* K partitions of tiles [tail_start, tiles) (1 = none) */
    int64_t k_per_split;   /* K extent of one partition (a multiple of bk) */
    int64_t tiles_m, tiles_n;
    int64_t grid_ctas;     /* CTAs launched */
    size_t workspace_bytes;/* device scratch the plan needs: a
                              SGEMM_WORKSPACE_COUNTER_BYTES block, then the
                              split-K or stream-K partial tiles, then the
                              transposed copy of A when transpose_a is set; 0
                              when it has neither partials nor copy */
    int64_t tail_start;    /* first tile (in launch order) of the tail region; tiles
                              when there is none.  Only the last, partly filled wave
                              of tiles is split, so it ends sooner */
    int64_t tail_k_per_split; /* K extent of one tail partition */
    int32_t transpose_a;   /* 1: A is first transposed into the workspace (K x M, row
                              stride a_t_ld) and the product runs with A read as a
                              row-per-k operand, which is faster for large grids */
    int32_t stages;        /* shared-memory pages in the K-slice ring: 2 (one
                              slice in flight while one is computed), or 3
                              (two in flight; K slices of 32, transpose_a) */
    int64_t a_t_ld;        /* row stride of the transposed copy (floats) */
    int32_t schedule;      /* 0: one CTA per (tile, K range) as above; 1: persistent
                              stream-K: grid_ctas CTAs stay resident, take whole-K
                              tiles round-robin for dp_rounds rounds, then split the
                              K slices of the remaining tiles into grid_ctas equal
                              runs (split_k = tail_split = 1 then); 2: small
                              problems (K <= 256): 32 x 32 tiles, 256 threads, the
                              whole K range (bk, padded) staged at once and split
                              across the CTA's 8 warps, no workspace */
    int32_t dp_rounds;     /* stream-K: rounds of whole-K tiles */
    int64_t sk_iters;      /* stream-K: K slices (of bk) of the tiles after the
                              dp_rounds * grid_ctas whole-K ones */
} gemm_plan_t;

/*
 * gemm_plan -- choose the launch configuration for one shape.
 *   M, N, K, lda, ldb, ldc: as in sgemm.  A, B, C: only their addresses'
 *   alignment is looked at (they may be NULL, which counts as aligned).
 *   out: written on success.
 * Uses the current device's SM count.  Never launches or allocates.
 * Returns SGEMM_OK, SGEMM_ERR_INVALID_ARG (bad sizes, out == NULL) or
 * SGEMM_ERR_UNSUPPORTED_DEVICE.
 */
sgemm_status gemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                       int64_t ldc, const void *A, const void *B, const void *C,
                       gemm_plan_t *out);

/*
 * gemm_plan_for_sms -- gemm_plan for a GPU with `sm_count` SMs, without
 * querying a device (offline planning, and host-side tests).  The plan is
 * valid for sgemm_with_plan on a device with that many SMs.
 * Returns SGEMM_OK or SGEMM_ERR_INVALID_ARG (bad sizes, sm_count < 1,
 * out == NULL).
 */
sgemm_status gemm_plan_for_sms(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                               int64_t ldc, const void *A, const void *B, const void *C,
                               int32_t sm_count, gemm_plan_t *out);

/*
 * sgemm -- C = alpha*A*B + beta*C on `stream` (see the conventions above).
 * Plans the shape with gemm_plan.  When the plan needs workspace (split-K
 * partials, or the transposed copy of A that large full-grid plans make
 * first: 4*K*M bytes, about 256 MiB at M = K = 8192), the library uses a
 * buffer it owns, one per (device, stream), grown with stream-ordered
 * allocation (cudaMallocAsync, plus 25 % headroom) and kept until the
 * process exits; the first call on a stream, and any call that needs more
 * than the buffer holds, therefore allocates.  If that allocation fails for
 * a plan with the transposed copy, sgemm falls back to the plan that reads A
 * as stored (no copy; split-K scratch at most) and runs it.  Returns
 * SGEMM_OK or an error status (SGEMM_ERR_ALLOC when even the fallback's
 * scratch cannot be had).
 */
sgemm_status sgemm(int64_t M, int64_t N, int64_t K, float alpha,
                   const float *A, int64_t lda, const float *B, int64_t ldb,
                   float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_with_plan -- like sgemm, with a plan from gemm_plan and caller-owned
 * workspace.  `workspace` is a device buffer of at least
 * plan->workspace_bytes bytes, 256-byte aligned, used only by work queued on
 * `stream`.  Its contents need no initialisation: a call writes every
 * partial tile and every transposed element before it reads them, so one
 * buffer serves any number of calls and plans.  Calls that share a
 * workspace must not overlap on the GPU.
 * workspace may be NULL when plan->workspace_bytes == 0.
 * Returns SGEMM_ERR_WORKSPACE when workspace_bytes < plan->workspace_bytes,
 * SGEMM_ERR_INVALID_ARG when the plan does not match the arguments.
 */
sgemm_status sgemm_with_plan(const gemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                             float alpha, const float *A, int64_t lda,
                             const float *B, int64_t ldb, float beta, float *C,
                             int64_t ldc, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * gemm_plan_check -- the check sgemm_with_plan applies to its plan, without a
 * device: whether `plan` is one this library can run for these sizes and
 * these pointers' alignment (A, B, C may be NULL, which counts as aligned).
 * Every plan gemm_plan or gemm_plan_for_sms returns passes it for the same
 * arguments; a plan edited by hand may not.
 * Returns SGEMM_OK, or SGEMM_ERR_INVALID_ARG (bad sizes, plan == NULL, or a
 * plan that does not match).
 */
sgemm_status gemm_plan_check(const gemm_plan_t *plan, int64_t M, int64_t N, int64_t K,
                             int64_t lda, int64_t ldb, int64_t ldc, const void *A,
                             const void *B, const void *C);

/* Capacity of the fixed scratch buffer sgemm_noalloc uses: 64 MiB per device. */
#define SGEMM_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)

/*
 * sgemm_noalloc -- the same C = alpha*A*B + beta*C as sgemm, with the same
 * arguments, for callers that must not allocate device memory.  The pages
 * have no counterpart to this call.  It always runs the plan without the
 * transposed copy of A (that copy would need M*K floats of scratch), so its
 * results are bit-identical to sgemm's under that plan -- sgemm with the
 * tuning knob SGEMM_TUNE_TRANSPOSE_A set to 0 -- and, for shapes where sgemm
 * makes the copy, equal to sgemm's within the accuracy the conventions above
 * state rather than bit for bit.
 *
 * Who needs it: code that runs where a cudaMalloc is not allowed or not
 * safe -- an application or framework that reserved the device memory up
 * front and forbids its plugins from allocating (a library cudaMalloc would
 * then fail or fragment its pool), latency-critical loops that must not
 * allocate after start-up (cudaMalloc may synchronise the device and stall
 * other streams), and callers that have no device-memory budget to give.
 * sgemm may allocate its split-K workspace on first use per stream;
 * sgemm_noalloc takes that scratch from a fixed buffer compiled into the
 * library instead (SGEMM_NOALLOC_SCRATCH_BYTES per device, held by every
 * GPU that loads the library until the process exits).
 *
 * It calls no cudaMalloc, cudaFree or other allocating routine.  The first
 * call on each device looks up the buffer's device address (with that device
 * current) and caches it; make that first call before any stream capture.
 * Nothing in the buffer has to start at zero (a call writes each partial
 * tile before it reads it back), so a call only launches the GEMM's kernels
 * on `stream`.
 *
 * All calls on a device share the one buffer: calls that overlap on the GPU
 * (different streams without ordering between them) race and give wrong
 * results.  Order them on one stream, or with events.
 *
 * Returns SGEMM_ERR_WORKSPACE, with nothing launched, when the shape's plan
 * needs more split-K scratch than SGEMM_NOALLOC_SCRATCH_BYTES (every plan
 * gemm_plan makes for the GB300 workloads fits; forcing a large split can
 * exceed it); otherwise the statuses of sgemm.
 */
sgemm_status sgemm_noalloc(int64_t M, int64_t N, int64_t K, float alpha,
                           const float *A, int64_t lda, const float *B, int64_t ldb,
                           float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_tf32x3 -- the separately reported tensor-core mode of the same
 * product, C = alpha*A*B + beta*C, with the arguments and conventions of
 * sgemm.  The pages compute this product on CUDA cores only; this mode
 * computes it as a dense contraction on the sm_103a tensor cores:
 * A = A_hi + A_lo and B = B_hi + B_lo, x_hi = x rounded to TF32 (round to
 * nearest even), x_lo = x - x_hi rounded to TF32, and
 * C ~= alpha*(A_lo*B_hi + A_hi*B_lo + A_hi*B_hi) + beta*C with fp32
 * accumulation in tensor memory (tcgen05.mma kind::tf32, TMA-fed).
 * Accuracy: max|C - exact| / (K*max|A|*max|B| + |beta|*max|C0|) <= 1e-5;
 * exact on integer inputs whose partial sums stay below 2^24 (their lo
 * parts are zero).  Any alignment and leading dimension are accepted: B is
 * split and transposed into a library-owned workspace per call, and A is
 * split inside the kernel (or, when its layout does not allow TMA, in a
 * pre-pass into the same workspace) -- at most 8*(M+N)*ceil(K/4)*4 bytes per
 * (device, stream), grown with stream-ordered allocation.  Grids smaller
 * than half the GPU are split along K (partials in the same workspace).  M
 * and N must be below 2^31 and K at most 2,097,120 (SGEMM_ERR_INVALID_ARG
 * otherwise).  Every device-side wait gives up after 1 s: the kernel then
 * stores nothing to C and records the event, which sgemm_device_status
 * reports.  Non-finite inputs: a NaN gives NaN where fp32 arithmetic would;
 * an infinite input gives NaN where fp32 would give +-inf (the split cannot
 * carry it: inf - inf in the low part, or inf * 0 against an operand exact in
 * TF32).  sgemm follows IEEE fp32 throughout.
 */
sgemm_status sgemm_tf32x3(int64_t M, int64_t N, int64_t K, float alpha,
                          const float *A, int64_t lda, const float *B, int64_t ldb,
                          float beta, float *C, int64_t ldc, void *stream);

/*
 * 3xTF32 with B packed once.  The tensor cores read both operands K-major,
 * and B is stored K x N (N-major), so sgemm_tf32x3 transposes and splits B
 * into TF32 hi/lo parts on every call; these calls let a B that is
 * multiplied many times (weights) be packed once.  A is K-major as stored:
 * when it is 16-byte aligned with lda % 4 == 0 its split happens inside the
 * kernel's shared-memory stage (the raw fp32 tile arrives by TMA and is split
 * in place, with no pass over A in HBM); otherwise, or with the tuning knob
 * SGEMM_TUNE_TF32X3_FUSE_A set to 0, in a pre-pass.
 *
 * sgemm_tf32x3_packed_b_bytes -- size of the packed form of a K x N matrix
 *   (0 for K or N <= 0).
 * sgemm_tf32x3_pack_b -- writes the packed form of B (K x N, row-major,
 *   ldb >= N, device pointer) into `packed` (device, 256-byte aligned,
 *   packed_bytes >= sgemm_tf32x3_packed_b_bytes(K, N)), asynchronously on
 *   `stream`.  SGEMM_ERR_MISALIGNED for a misaligned `packed`,
 *   SGEMM_ERR_WORKSPACE when packed_bytes is too small.
 * sgemm_tf32x3_packed -- C = alpha*A*B + beta*C with B given in packed form
 *   (made by sgemm_tf32x3_pack_b with the same K and N).  A must be 16-byte
 *   aligned with lda % 4 == 0 (SGEMM_ERR_MISALIGNED otherwise).  Accuracy,
 *   workspace (A's hi/lo and split-K partials) and bounded waits as
 *   sgemm_tf32x3.
 */
size_t sgemm_tf32x3_packed_b_bytes(int64_t K, int64_t N);
sgemm_status sgemm_tf32x3_pack_b(int64_t K, int64_t N, const float *B, int64_t ldb,
                                 void *packed, size_t packed_bytes, void *stream);
sgemm_status sgemm_tf32x3_packed(int64_t M, int64_t N, int64_t K, float alpha,
                                 const float *A, int64_t lda, const void *packed_b,
                                 float beta, float *C, int64_t ldc, void *stream);

/*
 * sgemm_device_status -- synchronises `stream`, then reports (and clears)
 * the record of expired device-side waits of the tensor-core mode:
 * SGEMM_ERR_TIMEOUT if any wait gave up since the last call, else SGEMM_OK
 * (SGEMM_ERR_LAUNCH if a CUDA call failed).
 */
sgemm_status sgemm_device_status(void *stream);

/*
 * sgemm_tf32x3_stall_selftest -- diagnostic of the bounded waits: runs the
 * tensor-core kernel on the given buffers with its operand loads withheld,
 * so every wait expires after `limit_us` microseconds (1..1e6), and returns
 * sgemm_device_status: SGEMM_ERR_TIMEOUT when the bounds work.  C is not
 * written.  Nothing faults or hangs; the context stays usable.
 */
sgemm_status sgemm_tf32x3_stall_selftest(int64_t M, int64_t N, int64_t K,
                                         const float *A, int64_t lda, const float *B,
                                         int64_t ldb, float *C, int64_t ldc,
                                         int64_t limit_us, void *stream);

/*
 * sgemm_ex -- the general form: for b in [0, batch)
 *
 *     C_b = act(alpha * op(A_b) * op(B_b) + beta * C_b + bias)
 *
 * with A_b = A + b*stride_a, B_b = B + b*stride_b, C_b = C + b*stride_c
 * (strides in elements), op(A_b) M x K, op(B_b) K x N, C_b M x N.
 *   - op_a == SGEMM_OP_N: A_b is M x K row-major, lda >= max(1, K);
 *     op_a == SGEMM_OP_T: A_b is stored K x M row-major, lda >= max(1, M),
 *     and read transposed.  Likewise B: N -> K x N, ldb >= max(1, N);
 *     T -> stored N x K, ldb >= max(1, K).
 *   - bias: NULL, or a device vector of N floats added to every row of C
 *     after the beta term; act: SGEMM_ACT_NONE or SGEMM_ACT_GELU_TANH,
 *     applied last (both as in a GPT-2 projection, x @ W + b, and its MLP's
 *     tanh GELU: "GPU Target" (MLIR tutorial), GPT-2 sublayers and the
 *     outlined GELU kernel).
 *   - batch: the per-head batch dimension of the MLIR page's batched
 *     matmul ("타일링된 행렬 곱셈"); stride_a or stride_b may be 0 (one
 *     operand shared by every batch); the batches of C may not overlap
 *     (stride_c >= (M-1)*ldc + N when batch > 1).
 * With batch = 1, op N/N, bias NULL and act NONE this is exactly sgemm.
 * K == 0 or alpha == 0 gives C = act(beta*C + bias) without reading A or B.
 * Same conventions as sgemm otherwise (device pointers, asynchronous on
 * `stream`, beta == 0 does not read C, padding columns untouched, library
 * workspace for split-K).  Returns SGEMM_ERR_INVALID_ARG for a bad op, act,
 * size, leading dimension, stride or pointer.
 */
sgemm_status sgemm_ex(int32_t op_a, int32_t op_b, int64_t M, int64_t N, int64_t K,
                      float alpha, const float *A, int64_t lda, int64_t stride_a,
                      const float *B, int64_t ldb, int64_t stride_b, float beta, float *C,
                      int64_t ldc, int64_t stride_c, int64_t batch, const float *bias,
                      int32_t act, void *stream);

/*
 * Tuning knobs: overrides of the planner's choices, for measurement sweeps
 * and tests.  Each starts from the environment variable named beside it,
 * read once when the library is loaded (never on the call path); after that
 * only sgemm_set_tuning changes it.  The value -1 means "the planner
 * decides" (the default).  Knobs are process-wide and take effect for plans
 * made after the change; set them while no other host thread is planning.
 */
typedef enum {
    SGEMM_TUNE_SPLIT_K = 0,       /* SGEMM_FORCE_SPLIT: K ranges per tile, 1..32 */
    SGEMM_TUNE_TAIL_SPLIT = 1,    /* SGEMM_FORCE_TAIL: K ranges of the tiles of the
                                     last partial wave, 0..32 (< 2: none) */
    SGEMM_TUNE_TILE = 2,          /* SGEMM_FORCE_TILE: CTA tile 64 or 128 */
    SGEMM_TUNE_KERNEL = 3,        /* SGEMM_FORCE_KERNEL: 0 scalar, 1 packed FMA issue,
                                     2 the 16 x 8 per-thread kernel on plans that copy
                                     both operands directly and do not split K */
    SGEMM_TUNE_TRANSPOSE_A = 4,   /* SGEMM_FORCE_TRANSPOSE_A: 0 never, 1 whenever able */
    SGEMM_TUNE_FFMA_EXT = 5,      /* SGEMM_FFMA_EXT: 0/1, which compiled build of the
                                     FFMA kernel runs plain products */
    SGEMM_TUNE_TF32X3_SPLIT = 6,  /* SGEMM_TF32X3_FORCE_SPLIT: tensor mode, 1..64 */
    SGEMM_TUNE_TF32X3_TAIL = 7,   /* SGEMM_TF32X3_FORCE_TAIL: tensor mode, 0..64 */
    SGEMM_TUNE_TF32X3_FUSE_A = 8, /* SGEMM_TF32X3_FUSE_A: 0 forces A's pre-pass split */
    SGEMM_TUNE_WORKSPACE_LIMIT_MIB = 9, /* SGEMM_WORKSPACE_LIMIT_MIB: cap, in MiB, on each
                                     library-owned workspace; a larger request fails
                                     as a failed allocation would (SGEMM_ERR_ALLOC) */
    SGEMM_TUNE_SCHEDULE = 10,     /* SGEMM_SCHEDULE: 0 one CTA per (tile, K range),
                                     1 persistent stream-K, 2 the small-problem kernel
                                     where K <= 256 (see gemm_plan_t.schedule) */
    SGEMM_TUNE_SK_MIN_SLICES = 11, /* SGEMM_SK_MIN_SLICES: stream-K, fewest K slices in
                                     one CTA's run (1..2^20) */
    SGEMM_TUNE_SK_GRID = 12,      /* SGEMM_SK_GRID: stream-K, CTAs of a grid of under two
                                     waves of tiles (1..2^20) */
    SGEMM_TUNE_TF32X3_BN = 13     /* SGEMM_TF32X3_BN: tensor mode, tile columns 128 or 256 */
} sgemm_tuning_knob;

/* Sets a knob (value -1 restores the planner's choice).  Returns
 * SGEMM_ERR_INVALID_ARG for an unknown knob or a value outside its range. */
sgemm_status sgemm_set_tuning(int32_t knob, int32_t value);

/* Current value of a knob (-1: the planner decides; -2: unknown knob). */
int32_t sgemm_get_tuning(int32_t knob);

/* Static, human-readable name of a status code (never NULL). */
const char *sgemm_status_string(sgemm_status status);

/* The CUDA error code (a cudaError_t value) behind the last
 * SGEMM_ERR_LAUNCH / SGEMM_ERR_ALLOC returned on this host thread, 0 if none. */
int sgemm_last_cuda_error(void);

/*
 * sgemm_ffma_probe -- a measurement aid, not part of the GEMM: launches
 * `ctas` CTAs of 256 threads; each thread runs `iters` rounds of 64
 * independent fp32 FMAs (as 32 packed fma.rn.f32x2 when `packed` != 0, else
 * 64 scalar fma.rn.f32) and writes one float to `out` (device, ctas*256
 * floats) so the work cannot be elided.  FLOPs = ctas * 256 * iters * 128.
 * Timed by the caller, it gives the chip's attainable fp32 FMA rate.
 * Returns SGEMM_ERR_INVALID_ARG for ctas <= 0, iters < 0 or out == NULL.
 */
sgemm_status sgemm_ffma_probe(int64_t ctas, int64_t iters, int32_t packed, float *out,
                              void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_FP32_MATRIX_06_SGEMM_H */
