"""GB300 (sm_103a) single-precision GEMM: Python binding of libsgemm.so.

The binding only marshals arguments: it turns torch CUDA tensors (or raw
device addresses) and torch's current stream into the plain pointers, sizes
and leading dimensions the C ABI in ``include/sgemm.h`` takes, and turns a
status code into an exception.  Every step of the GEMM runs in the library's
CUDA kernels.  There is no fallback: if ``libsgemm.so`` is missing or cannot
run on the current device, the calls raise.

    C = alpha * A @ B + beta * C        (row-major fp32, any M, N, K)

Shape errors raise ValueError before anything is launched, mirroring the
Python-facing matmul of velog @levelstage "AutoMinepp7" (section
"직사각형 타일링"), which rejects operands that are not 2-D or whose inner
dimensions differ.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsgemm.so")

SGEMM_OK = 0
STATUS_NAMES = {
    0: "SGEMM_OK",
    1: "SGEMM_ERR_INVALID_ARG",
    2: "SGEMM_ERR_MISALIGNED",
    3: "SGEMM_ERR_UNSUPPORTED_DEVICE",
    4: "SGEMM_ERR_LAUNCH",
    5: "SGEMM_ERR_TIMEOUT",
    6: "SGEMM_ERR_ALLOC",
    7: "SGEMM_ERR_WORKSPACE",
}
WORKSPACE_COUNTER_BYTES = 16384

# Every symbol include/sgemm.h declares (checked by the tests).
EXPORTED_SYMBOLS = (
    "gemm_plan",
    "gemm_plan_for_sms",
    "gemm_plan_check",
    "sgemm",
    "sgemm_with_plan",
    "sgemm_status_string",
    "sgemm_last_cuda_error",
    "sgemm_ffma_probe",
    "sgemm_noalloc",
    "sgemm_tf32x3",
    "sgemm_device_status",
    "sgemm_tf32x3_stall_selftest",
    "sgemm_ex",
    "sgemm_tf32x3_packed_b_bytes",
    "sgemm_tf32x3_pack_b",
    "sgemm_tf32x3_packed",
    "sgemm_set_tuning",
    "sgemm_get_tuning",
)
# sgemm_tuning_knob
TUNING_KNOBS = {
    "split_k": 0,
    "tail_split": 1,
    "tile": 2,
    "kernel": 3,
    "transpose_a": 4,
    "ffma_ext": 5,
    "tf32x3_split": 6,
    "tf32x3_tail": 7,
    "tf32x3_fuse_a": 8,
    "workspace_limit_mib": 9,
    "schedule": 10,
    "sk_min_slices": 11,
    "sk_grid": 12,
    "tf32x3_bn": 13,
}
OP_N, OP_T = 0, 1
ACT_NONE, ACT_GELU_TANH = 0, 1
NOALLOC_SCRATCH_BYTES = 64 * 1024 * 1024


class SgemmError(RuntimeError):
    """A non-OK status from the C ABI."""

    def __init__(self, status: int, where: str, detail: str = ""):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, f"status {status}")
        msg = f"{where}: {name}"
        if detail:
            msg += f" ({detail})"
        super().__init__(msg)


class GemmPlan(ctypes.Structure):
    """Mirror of gemm_plan_t."""

    _fields_ = [
        ("mode", ctypes.c_int32),
        ("kernel", ctypes.c_int32),
        ("bm", ctypes.c_int32),
        ("bn", ctypes.c_int32),
        ("bk", ctypes.c_int32),
        ("threads", ctypes.c_int32),
        ("split_k", ctypes.c_int32),
        ("vec", ctypes.c_int32),
        ("edge", ctypes.c_int32),
        ("tail_split", ctypes.c_int32),
        ("k_per_split", ctypes.c_int64),
        ("tiles_m", ctypes.c_int64),
        ("tiles_n", ctypes.c_int64),
        ("grid_ctas", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_size_t),
        ("tail_start", ctypes.c_int64),
        ("tail_k_per_split", ctypes.c_int64),
        ("transpose_a", ctypes.c_int32),
        ("stages", ctypes.c_int32),
        ("a_t_ld", ctypes.c_int64),
        ("schedule", ctypes.c_int32),
        ("dp_rounds", ctypes.c_int32),
        ("sk_iters", ctypes.c_int64),
    ]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


_lock = threading.Lock()
_lib = None

_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_f32 = ctypes.c_float


def build() -> str:
    """Compile libsgemm.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build()


def load_library() -> ctypes.CDLL:
    """Load libsgemm.so; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'` "
                "(there is no CPU fallback)")
        lib = ctypes.CDLL(LIB_PATH)
        lib.gemm_plan.argtypes = [_i64, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                  ctypes.POINTER(GemmPlan)]
        lib.gemm_plan.restype = ctypes.c_int
        lib.gemm_plan_for_sms.argtypes = [_i64, _i64, _i64, _i64, _i64, _i64, _vp, _vp, _vp,
                                          ctypes.c_int32, ctypes.POINTER(GemmPlan)]
        lib.gemm_plan_for_sms.restype = ctypes.c_int
        lib.gemm_plan_check.argtypes = [ctypes.POINTER(GemmPlan), _i64, _i64, _i64, _i64, _i64,
                                        _i64, _vp, _vp, _vp]
        lib.gemm_plan_check.restype = ctypes.c_int
        lib.sgemm.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _i64, _f32, _vp, _i64, _vp]
        lib.sgemm.restype = ctypes.c_int
        lib.sgemm_with_plan.argtypes = [ctypes.POINTER(GemmPlan), _i64, _i64, _i64, _f32, _vp,
                                        _i64, _vp, _i64, _f32, _vp, _i64, _vp, ctypes.c_size_t,
                                        _vp]
        lib.sgemm_with_plan.restype = ctypes.c_int
        lib.sgemm_status_string.argtypes = [ctypes.c_int]
        lib.sgemm_status_string.restype = ctypes.c_char_p
        lib.sgemm_last_cuda_error.argtypes = []
        lib.sgemm_last_cuda_error.restype = ctypes.c_int
        lib.sgemm_ffma_probe.argtypes = [_i64, _i64, ctypes.c_int32, _vp, _vp]
        lib.sgemm_ffma_probe.restype = ctypes.c_int
        lib.sgemm_ex.argtypes = [ctypes.c_int32, ctypes.c_int32, _i64, _i64, _i64, _f32, _vp,
                                 _i64, _i64, _vp, _i64, _i64, _f32, _vp, _i64, _i64, _i64, _vp,
                                 ctypes.c_int32, _vp]
        lib.sgemm_ex.restype = ctypes.c_int
        lib.sgemm_tf32x3_packed_b_bytes.argtypes = [_i64, _i64]
        lib.sgemm_tf32x3_packed_b_bytes.restype = ctypes.c_size_t
        lib.sgemm_tf32x3_pack_b.argtypes = [_i64, _i64, _vp, _i64, _vp, ctypes.c_size_t, _vp]
        lib.sgemm_tf32x3_pack_b.restype = ctypes.c_int
        lib.sgemm_tf32x3_packed.argtypes = [_i64, _i64, _i64, _f32, _vp, _i64, _vp, _f32, _vp,
                                            _i64, _vp]
        lib.sgemm_tf32x3_packed.restype = ctypes.c_int
        lib.sgemm_noalloc.argtypes = lib.sgemm.argtypes
        lib.sgemm_noalloc.restype = ctypes.c_int
        lib.sgemm_tf32x3.argtypes = lib.sgemm.argtypes
        lib.sgemm_tf32x3.restype = ctypes.c_int
        lib.sgemm_device_status.argtypes = [_vp]
        lib.sgemm_device_status.restype = ctypes.c_int
        lib.sgemm_tf32x3_stall_selftest.argtypes = [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp,
                                                    _i64, _i64, _vp]
        lib.sgemm_tf32x3_stall_selftest.restype = ctypes.c_int
        lib.sgemm_set_tuning.argtypes = [ctypes.c_int32, ctypes.c_int32]
        lib.sgemm_set_tuning.restype = ctypes.c_int
        lib.sgemm_get_tuning.argtypes = [ctypes.c_int32]
        lib.sgemm_get_tuning.restype = ctypes.c_int32
        _lib = lib
        return lib


def _check(status: int, where: str) -> None:
    if status != SGEMM_OK:
        lib = load_library()
        detail = lib.sgemm_status_string(status).decode()
        cuda_err = lib.sgemm_last_cuda_error()
        if cuda_err:
            detail += f"; cudaError {cuda_err}"
        raise SgemmError(status, where, detail)


def status_string(status: int) -> str:
    return load_library().sgemm_status_string(int(status)).decode()


# --------------------------------------------------------------------------
# pointer-level calls (same names and argument order as the C ABI)
# --------------------------------------------------------------------------

def gemm_plan(M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
              A: int = 0, B: int = 0, C: int = 0) -> GemmPlan:
    """gemm_plan(): the launch configuration the library picks for a shape."""
    plan = GemmPlan()
    _check(load_library().gemm_plan(M, N, K, lda, ldb, ldc, A or None, B or None, C or None,
                                    ctypes.byref(plan)), "gemm_plan")
    return plan


def gemm_plan_for_sms(M: int, N: int, K: int, lda: int, ldb: int, ldc: int, A: int = 0,
                      B: int = 0, C: int = 0, sm_count: int = 152) -> GemmPlan:
    """gemm_plan_for_sms(): plan for a GPU with `sm_count` SMs, no device needed."""
    plan = GemmPlan()
    _check(load_library().gemm_plan_for_sms(M, N, K, lda, ldb, ldc, A or None, B or None,
                                            C or None, sm_count, ctypes.byref(plan)),
           "gemm_plan_for_sms")
    return plan


def gemm_plan_check(plan: GemmPlan, M: int, N: int, K: int, lda: int, ldb: int, ldc: int,
                    A: int = 0, B: int = 0, C: int = 0) -> bool:
    """gemm_plan_check(): whether sgemm_with_plan would accept `plan` for these
    sizes and pointers' alignment (no device needed)."""
    return load_library().gemm_plan_check(ctypes.byref(plan), M, N, K, lda, ldb, ldc,
                                          A or None, B or None, C or None) == 0


def sgemm_ptr(M: int, N: int, K: int, alpha: float, A: int, lda: int, B: int, ldb: int,
              beta: float, C: int, ldc: int, stream: int = 0) -> None:
    """sgemm() on raw device addresses; `stream` is a cudaStream_t value."""
    _check(load_library().sgemm(M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                C or None, ldc, stream or None), "sgemm")


def sgemm_noalloc_ptr(M: int, N: int, K: int, alpha: float, A: int, lda: int, B: int, ldb: int,
                      beta: float, C: int, ldc: int, stream: int = 0) -> None:
    """sgemm_noalloc(): the same GEMM as sgemm_ptr without allocating device
    memory (split-K scratch comes from a fixed 64 MiB buffer inside the
    library).  For callers that may not allocate, e.g. inside a framework that
    owns all device memory.  Calls that overlap on the GPU share that buffer
    and race; keep them ordered."""
    _check(load_library().sgemm_noalloc(M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                        C or None, ldc, stream or None), "sgemm_noalloc")


def sgemm_ex_ptr(op_a: int, op_b: int, M: int, N: int, K: int, alpha: float, A: int, lda: int,
                 stride_a: int, B: int, ldb: int, stride_b: int, beta: float, C: int, ldc: int,
                 stride_c: int, batch: int = 1, bias: int = 0, act: int = ACT_NONE,
                 stream: int = 0) -> None:
    """sgemm_ex(): C_b = act(alpha op(A_b) op(B_b) + beta C_b + bias), b < batch."""
    _check(load_library().sgemm_ex(op_a, op_b, M, N, K, alpha, A or None, lda, stride_a,
                                   B or None, ldb, stride_b, beta, C or None, ldc, stride_c,
                                   batch, bias or None, act, stream or None), "sgemm_ex")


def sgemm_tf32x3_ptr(M: int, N: int, K: int, alpha: float, A: int, lda: int, B: int, ldb: int,
                     beta: float, C: int, ldc: int, stream: int = 0) -> None:
    """sgemm_tf32x3(): the 3xTF32 tensor-core mode (normalised error <= 1e-5)."""
    _check(load_library().sgemm_tf32x3(M, N, K, alpha, A or None, lda, B or None, ldb, beta,
                                       C or None, ldc, stream or None), "sgemm_tf32x3")


def tf32x3_packed_b_bytes(K: int, N: int) -> int:
    """sgemm_tf32x3_packed_b_bytes(): bytes of the packed form of a K x N B."""
    return int(load_library().sgemm_tf32x3_packed_b_bytes(K, N))


def tf32x3_pack_b_ptr(K: int, N: int, B: int, ldb: int, packed: int, packed_bytes: int,
                      stream: int = 0) -> None:
    """sgemm_tf32x3_pack_b(): split and transpose B once for the tensor-core mode."""
    _check(load_library().sgemm_tf32x3_pack_b(K, N, B or None, ldb, packed or None,
                                              packed_bytes, stream or None),
           "sgemm_tf32x3_pack_b")


def sgemm_tf32x3_packed_ptr(M: int, N: int, K: int, alpha: float, A: int, lda: int,
                            packed_b: int, beta: float, C: int, ldc: int,
                            stream: int = 0) -> None:
    """sgemm_tf32x3_packed(): the tensor-core mode with a packed B."""
    _check(load_library().sgemm_tf32x3_packed(M, N, K, alpha, A or None, lda,
                                              packed_b or None, beta, C or None, ldc,
                                              stream or None), "sgemm_tf32x3_packed")


def device_status(stream: int = 0) -> int:
    """sgemm_device_status(): 0, or 5 (SGEMM_ERR_TIMEOUT) if a bounded
    device-side wait expired since the last call.  Synchronises `stream`."""
    return int(load_library().sgemm_device_status(stream or None))


def tf32x3_stall_selftest(M: int, N: int, K: int, A: int, lda: int, B: int, ldb: int, C: int,
                          ldc: int, limit_us: int, stream: int = 0) -> int:
    """sgemm_tf32x3_stall_selftest(): returns the status code (5 when the
    bounded waits expired as intended)."""
    return int(load_library().sgemm_tf32x3_stall_selftest(M, N, K, A or None, lda, B or None,
                                                           ldb, C or None, ldc, limit_us,
                                                           stream or None))


def sgemm_with_plan_ptr(plan: GemmPlan, M: int, N: int, K: int, alpha: float, A: int, lda: int,
                        B: int, ldb: int, beta: float, C: int, ldc: int, workspace: int,
                        workspace_bytes: int, stream: int = 0) -> None:
    """sgemm_with_plan() on raw device addresses."""
    _check(load_library().sgemm_with_plan(ctypes.byref(plan), M, N, K, alpha, A or None, lda,
                                          B or None, ldb, beta, C or None, ldc,
                                          workspace or None, workspace_bytes, stream or None),
           "sgemm_with_plan")


def ffma_probe(ctas: int, iters: int, out_ptr: int, packed: bool = True, stream: int = 0) -> None:
    """sgemm_ffma_probe(): FLOPs = ctas * 256 * iters * 128."""
    _check(load_library().sgemm_ffma_probe(ctas, iters, 1 if packed else 0, out_ptr or None,
                                           stream or None), "sgemm_ffma_probe")


def set_tuning(knob: str, value: int | None) -> None:
    """sgemm_set_tuning(): override one planner choice (None = the planner's)."""
    _check(load_library().sgemm_set_tuning(TUNING_KNOBS[knob], -1 if value is None else value),
           f"sgemm_set_tuning({knob})")


def get_tuning(knob: str) -> int | None:
    """sgemm_get_tuning(): the knob's override, or None when the planner decides."""
    v = int(load_library().sgemm_get_tuning(TUNING_KNOBS[knob]))
    return None if v == -1 else v


class tuning:
    """Context manager: ``with tuning(split_k=4, tile=128): ...`` sets knobs
    for the duration of the block and restores their previous values."""

    def __init__(self, **knobs: int | None):
        for k in knobs:
            if k not in TUNING_KNOBS:
                raise KeyError(f"unknown tuning knob {k!r}")
        self.knobs = knobs
        self.saved: dict[str, int | None] = {}

    def __enter__(self):
        for k, v in self.knobs.items():
            self.saved[k] = get_tuning(k)
            set_tuning(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            set_tuning(k, v)
        return False


# --------------------------------------------------------------------------
# torch-tensor convenience layer
# --------------------------------------------------------------------------

def _row_major_view(t, name: str):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D (got {t.dim()}-D)")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32 (got {t.dtype})")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    rows, cols = t.shape
    if cols > 1 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")
    ld = t.stride(0) if rows > 1 else max(cols, 1)
    if ld < max(cols, 1):
        raise ValueError(f"{name} has a row stride smaller than its width")
    return t.data_ptr(), int(ld)


def _stream_handle(stream) -> int:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def sgemm(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """C = alpha * A @ B + beta * C on torch CUDA float32 tensors.

    A (M, K) and B (K, N) may be row-strided views (stride(1) == 1, any
    stride(0) >= width).  C (M, N) is written in place; when C is None a new
    tensor is allocated (and beta must be 0).  Runs asynchronously on `stream`
    (default: torch's current stream) and returns C.
    """
    import torch
    if not isinstance(A, torch.Tensor) or not isinstance(B, torch.Tensor):
        raise TypeError("A and B must be torch tensors")
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("sgemm works on 2-D matrices only")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    elif tuple(C.shape) != (M, N):
        raise ValueError(f"C must be ({M}, {N}), got {tuple(C.shape)}")
    a_ptr, lda = _row_major_view(A, "A")
    b_ptr, ldb = _row_major_view(B, "B")
    c_ptr, ldc = _row_major_view(C, "C")
    if not (A.device == B.device == C.device):
        raise ValueError("A, B and C must be on the same device")
    lda = max(lda, K, 1)
    ldb = max(ldb, N, 1)
    ldc = max(ldc, N, 1)
    with torch.cuda.device(A.device):
        sgemm_ptr(M, N, K, float(alpha), a_ptr, lda, b_ptr, ldb, float(beta), c_ptr, ldc,
                  _stream_handle(stream))
    return C


def sgemm_tf32x3(A, B, C=None, alpha: float = 1.0, beta: float = 0.0, stream=None):
    """The 3xTF32 tensor-core mode on torch tensors (same rules as sgemm())."""
    import torch
    if A.dim() != 2 or B.dim() != 2:
        raise ValueError("sgemm_tf32x3 works on 2-D matrices only")
    M, K = A.shape
    K2, N = B.shape
    if K != K2:
        raise ValueError(f"inner dimensions differ: A is {tuple(A.shape)}, B is {tuple(B.shape)}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    a_ptr, lda = _row_major_view(A, "A")
    b_ptr, ldb = _row_major_view(B, "B")
    c_ptr, ldc = _row_major_view(C, "C")
    with torch.cuda.device(A.device):
        sgemm_tf32x3_ptr(M, N, K, float(alpha), a_ptr, max(lda, K, 1), b_ptr, max(ldb, N, 1),
                         float(beta), c_ptr, max(ldc, N, 1), _stream_handle(stream))
    return C


def matmul(A, B, bias=None, activation: str | None = None, trans_a: bool = False,
           trans_b: bool = False, alpha: float = 1.0, C=None, beta: float = 0.0, stream=None):
    """act(alpha * op(A) @ op(B) + beta * C + bias) on torch CUDA float32 tensors.

    A, B (and C) are 2-D, or 3-D with a leading batch dimension (a 2-D operand
    is shared by every batch).  trans_a / trans_b read the stored matrix
    transposed (A stored K x M, B stored N x K).  bias: a length-N vector;
    activation: None or "gelu_tanh".  Returns C.
    """
    import torch
    for name, t in (("A", A), ("B", B)):
        if not isinstance(t, torch.Tensor) or t.dim() not in (2, 3):
            raise ValueError(f"{name} must be a 2-D or 3-D torch tensor")
    batch = max(A.shape[0] if A.dim() == 3 else 1, B.shape[0] if B.dim() == 3 else 1)
    for name, t in (("A", A), ("B", B)):
        if t.dim() == 3 and t.shape[0] != batch:
            raise ValueError(f"{name} has batch {t.shape[0]}, expected {batch}")
    a2 = A if A.dim() == 2 else A[0]
    b2 = B if B.dim() == 2 else B[0]
    M, K = (a2.shape[1], a2.shape[0]) if trans_a else (a2.shape[0], a2.shape[1])
    Kb, N = (b2.shape[1], b2.shape[0]) if trans_b else (b2.shape[0], b2.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: op(A) is {M}x{K}, op(B) is {Kb}x{N}")
    if C is None:
        if beta != 0.0:
            raise ValueError("beta != 0 needs an input C")
        C = torch.empty((batch, M, N) if batch > 1 or A.dim() == 3 or B.dim() == 3 else (M, N),
                        dtype=torch.float32, device=A.device)
    c2 = C if C.dim() == 2 else C[0]
    if tuple(c2.shape) != (M, N):
        raise ValueError(f"C must be ({M}, {N}) per batch")
    a_ptr, lda = _row_major_view(a2, "A")
    b_ptr, ldb = _row_major_view(b2, "B")
    c_ptr, ldc = _row_major_view(c2, "C")
    sa = A.stride(0) if A.dim() == 3 and batch > 1 else 0
    sb = B.stride(0) if B.dim() == 3 and batch > 1 else 0
    sc = C.stride(0) if C.dim() == 3 and batch > 1 else 0
    bias_ptr = 0
    if bias is not None:
        if bias.dtype != torch.float32 or bias.numel() != N or not bias.is_contiguous():
            raise ValueError("bias must be a contiguous float32 vector of length N")
        bias_ptr = bias.data_ptr()
    act = {None: ACT_NONE, "none": ACT_NONE, "gelu_tanh": ACT_GELU_TANH}.get(activation)
    if act is None:
        raise ValueError(f"unknown activation {activation!r}")
    with torch.cuda.device(A.device):
        sgemm_ex_ptr(OP_T if trans_a else OP_N, OP_T if trans_b else OP_N, M, N, K, float(alpha),
                     a_ptr, max(lda, (M if trans_a else K), 1), sa, b_ptr,
                     max(ldb, (K if trans_b else N), 1), sb, float(beta), c_ptr, max(ldc, N, 1),
                     sc, batch, bias_ptr, act, _stream_handle(stream))
    return C


def plan_for(A, B, C) -> GemmPlan:
    """gemm_plan() for torch tensors A (M,K), B (K,N), C (M,N)."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    a_ptr, lda = _row_major_view(A, "A")
    b_ptr, ldb = _row_major_view(B, "B")
    c_ptr, ldc = _row_major_view(C, "C")
    with torch.cuda.device(A.device):
        return gemm_plan(M, N, K, max(lda, K, 1), max(ldb, N, 1), max(ldc, N, 1),
                         a_ptr, b_ptr, c_ptr)


def sgemm_with_plan(plan: GemmPlan, A, B, C, alpha: float = 1.0, beta: float = 0.0,
                    workspace=None, stream=None):
    """sgemm_with_plan() on torch tensors; `workspace` is a CUDA uint8 tensor
    of at least plan.workspace_bytes bytes (or None when that is 0); its
    contents need no initialisation."""
    import torch
    M, K = A.shape
    N = B.shape[1]
    a_ptr, lda = _row_major_view(A, "A")
    b_ptr, ldb = _row_major_view(B, "B")
    c_ptr, ldc = _row_major_view(C, "C")
    ws_ptr, ws_bytes = 0, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    with torch.cuda.device(A.device):
        sgemm_with_plan_ptr(plan, M, N, K, float(alpha), a_ptr, max(lda, K, 1), b_ptr,
                            max(ldb, N, 1), float(beta), c_ptr, max(ldc, N, 1), ws_ptr,
                            ws_bytes, _stream_handle(stream))
    return C
