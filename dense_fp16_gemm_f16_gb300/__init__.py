"""GB300-native dense fp16 GEMM, D = A·Bᵀ (fp16 in, fp32 accumulate, fp16 out).

This module is the Python binding of the C ABI declared in
``include/gemm_f16.h``: the same entry-point names, argument marshalling only.
Every step of the GEMM runs in the library's sm_103a kernels; there is no
CPU or library fallback, and every call fails loudly (``GemmError`` /
``LibraryMissing``) when the compiled library is absent or refuses the call.

Tensors may be passed as CUDA ``torch.Tensor`` objects (float16, 2-D,
row-major contiguous) or as raw device pointers (ints) with explicit sizes.
PyTorch is used for device memory and streams only.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libgemm_f16.so")

_lock = threading.Lock()
_lib = None


class Status(enum.IntEnum):
    OK = 0
    ERR_INVALID_VALUE = 1
    ERR_MISALIGNED = 2
    ERR_UNSUPPORTED_DEVICE = 3
    ERR_LAUNCH = 4
    ERR_TIMEOUT = 5
    ERR_CUDA = 6


class Variant(enum.IntEnum):
    AUTO = 0
    TILE_2CTA_256x256 = 1
    TILE_1CTA_128x128 = 2
    TILE_1CTA_128x256 = 3
    SKINNY_SPLITK = 4
    TILE_2CTA_SPLITK = 5
    SKINNY_STREAMK = 6
    TILE_2CTA_512x256 = 7
    TILE_1CTA_SPLITK = 8


class Dtype(enum.IntEnum):
    F16 = 0
    BF16 = 1
    E4M3 = 2   # 8-bit operands, bf16 D
    E5M2 = 3


class Activation(enum.IntEnum):
    NONE = 0
    RELU = 1


class Epilogue(ctypes.Structure):
    """Mirror of gemm_epilogue_t: D = act(alpha * scale_n[n] * (A Bᵀ) + beta * C + bias[n])."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("C", ctypes.c_void_p),
                ("bias", ctypes.c_void_p), ("activation", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("scale_n", ctypes.c_void_p)]


class LibraryMissing(RuntimeError):
    """The compiled CUDA library is not there (build it first)."""


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = Status(status) if status in Status._value2member_map_ else status
        super().__init__(f"{where}: {gemm_status_string(status)}")


class Plan(ctypes.Structure):
    """Mirror of gemm_plan_t."""
    _fields_ = [
        ("variant", ctypes.c_int32), ("cta_group", ctypes.c_int32), ("tile_m", ctypes.c_int32),
        ("tile_n", ctypes.c_int32), ("tile_k", ctypes.c_int32), ("stages", ctypes.c_int32),
        ("m_tiles", ctypes.c_int64), ("n_tiles", ctypes.c_int64), ("k_blocks", ctypes.c_int64),
        ("grid_ctas", ctypes.c_int32), ("smem_bytes", ctypes.c_int32), ("tmem_cols", ctypes.c_int32),
        ("max_tiles_per_cta", ctypes.c_int32), ("workspace_bytes", ctypes.c_int64),
        ("num_full_tiles", ctypes.c_int64), ("tail_split", ctypes.c_int32), ("group_m", ctypes.c_int32),
        ("k_split", ctypes.c_int32), ("reserved", ctypes.c_int32),
    ]

    def as_dict(self) -> dict:
        d = {name: getattr(self, name) for name, _ in self._fields_}
        d["variant"] = Variant(d["variant"]).name
        return d


def load():
    """Load libgemm_f16.so (once); raises LibraryMissing if it was never built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise LibraryMissing(
                f"{LIB_PATH} is missing: build it with `python -m dense_fp16_gemm_f16_gb300.build`")
        lib = ctypes.CDLL(LIB_PATH)
        p, i64 = ctypes.c_void_p, ctypes.c_int64
        lib.gemm_f16_nt.argtypes = [p, p, p, i64, i64, i64, p]
        lib.gemm_f16_nt.restype = ctypes.c_int
        lib.gemm_f16_nt_variant.argtypes = [p, p, p, i64, i64, i64, ctypes.c_int, p]
        lib.gemm_f16_nt_variant.restype = ctypes.c_int
        lib.gemm_f16_nt_check.argtypes = [p]
        lib.gemm_f16_nt_check.restype = ctypes.c_int
        lib.gemm_status_string.argtypes = [ctypes.c_int]
        lib.gemm_status_string.restype = ctypes.c_char_p
        lib.gemm_f16_nt_plan.argtypes = [i64, i64, i64, ctypes.c_int, ctypes.c_int32, ctypes.POINTER(Plan)]
        lib.gemm_f16_nt_plan.restype = ctypes.c_int
        lib.gemm_f16_nt_noalloc.argtypes = [p, p, p, i64, i64, i64, p]
        lib.gemm_f16_nt_noalloc.restype = ctypes.c_int
        lib.gemm_bf16_nt.argtypes = [p, p, p, i64, i64, i64, p]
        lib.gemm_bf16_nt.restype = ctypes.c_int
        lib.gemm_nt_ex.argtypes = [ctypes.c_int, p, p, p, i64, i64, i64, ctypes.POINTER(Epilogue), ctypes.c_int, p]
        lib.gemm_nt_ex.restype = ctypes.c_int
        lib.gemm_nt_plan_ex.argtypes = [ctypes.c_int, i64, i64, i64, ctypes.c_int, ctypes.c_int32,
                                        ctypes.POINTER(Plan)]
        lib.gemm_nt_plan_ex.restype = ctypes.c_int
        lib.gemm_selftest_timeout.argtypes = [ctypes.c_int32, p]
        lib.gemm_selftest_timeout.restype = ctypes.c_int
        _lib = lib
        return lib


def gemm_status_string(status: int) -> str:
    return load().gemm_status_string(int(status)).decode()


# ---------------------------------------------------------------- marshalling
def _is_tensor(x) -> bool:
    return hasattr(x, "data_ptr") and hasattr(x, "dtype")


def _stream_handle(stream, device=None) -> int | None:
    if stream is None:
        if device is not None:
            import torch
            return torch.cuda.current_stream(device).cuda_stream or None
        return None
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream or None
    return int(stream) or None


def _torch_types(dtype):
    """(accepted operand dtypes, D dtype) for a Dtype."""
    import torch
    if dtype == Dtype.BF16:
        return (torch.bfloat16,), torch.bfloat16
    if dtype == Dtype.E4M3:
        return (torch.float8_e4m3fn, torch.uint8), torch.bfloat16
    if dtype == Dtype.E5M2:
        return (torch.float8_e5m2, torch.uint8), torch.bfloat16
    return (torch.float16,), torch.float16


def _operands(A, B, D, M, N, K, dtype=None):
    """(a_ptr, b_ptr, d_ptr, M, N, K, device) from tensors or raw pointers."""
    if _is_tensor(A):
        ins, out = _torch_types(Dtype.F16 if dtype is None else dtype)
        for name, t in (("A", A), ("B", B), ("D", D)):
            if not _is_tensor(t):
                raise TypeError(f"{name}: mix of tensors and raw pointers")
            want = (out,) if name == "D" else ins
            if t.dtype not in want:
                raise TypeError(f"{name} must be {' or '.join(map(str, want))}, got {t.dtype}")
            if not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if t.dim() != 2 or not t.is_contiguous():
                raise ValueError(f"{name} must be a 2-D row-major contiguous tensor")
        if A.device != B.device or A.device != D.device:
            raise ValueError("A, B and D must be on the same device")
        m, k = A.shape
        n, kb = B.shape
        if kb != k or tuple(D.shape) != (m, n):
            raise ValueError(f"shapes do not match D[M,N] = A[M,K]·B[N,K]ᵀ: {tuple(A.shape)}, "
                             f"{tuple(B.shape)}, {tuple(D.shape)}")
        for name, given, actual in (("M", M, m), ("N", N, n), ("K", K, k)):
            if given is not None and given != actual:
                raise ValueError(f"{name}={given} does not match the tensors ({actual})")
        return A.data_ptr(), B.data_ptr(), D.data_ptr(), m, n, k, A.device
    if M is None or N is None or K is None:
        raise ValueError("raw pointers need explicit M, N and K")
    return int(A or 0), int(B or 0), int(D or 0), int(M), int(N), int(K), None


def _call(fn_name: str, args, device):
    lib = load()
    fn = getattr(lib, fn_name)
    if device is not None:
        import torch
        with torch.cuda.device(device):
            st = fn(*args)
    else:
        st = fn(*args)
    if st != Status.OK:
        raise GemmError(st, fn_name)


def gemm_f16_nt(A, B, D, M=None, N=None, K=None, stream=None) -> None:
    """D = A·Bᵀ on ``stream`` (default: the tensors' current stream); asynchronous."""
    a, b, d, m, n, k, dev = _operands(A, B, D, M, N, K)
    _call("gemm_f16_nt", (a or None, b or None, d or None, m, n, k, _stream_handle(stream, dev)), dev)


def gemm_f16_nt_variant(A, B, D, M=None, N=None, K=None, variant=Variant.AUTO, stream=None) -> None:
    """gemm_f16_nt with an explicit kernel choice (a ``Variant``)."""
    a, b, d, m, n, k, dev = _operands(A, B, D, M, N, K)
    _call("gemm_f16_nt_variant",
          (a or None, b or None, d or None, m, n, k, int(variant), _stream_handle(stream, dev)), dev)


def gemm_f16_nt_noalloc(A, B, D, M=None, N=None, K=None, stream=None) -> None:
    """Small-M (M <= 64) D = A·Bᵀ using only the library's fixed scratch array.

    For callers that cannot let the library call cudaMalloc (a memory pool owns
    the device, or an allocation's implicit synchronisation is not allowed at
    this point).  Calls whose GPU work overlaps share that one array and race:
    keep them ordered on one stream.  Make the first call on a device before
    any stream capture (it looks up the array's device address).
    """
    a, b, d, m, n, k, dev = _operands(A, B, D, M, N, K)
    _call("gemm_f16_nt_noalloc", (a or None, b or None, d or None, m, n, k, _stream_handle(stream, dev)), dev)


def gemm_bf16_nt(A, B, D, M=None, N=None, K=None, stream=None) -> None:
    """D = A·Bᵀ for bf16 tensors (fp32 accumulation, bf16 output); asynchronous."""
    a, b, d, m, n, k, dev = _operands(A, B, D, M, N, K, Dtype.BF16)
    _call("gemm_bf16_nt", (a or None, b or None, d or None, m, n, k, _stream_handle(stream, dev)), dev)


def _tensor_dtype(A):
    import torch
    return {torch.bfloat16: Dtype.BF16, torch.float8_e4m3fn: Dtype.E4M3,
            torch.float8_e5m2: Dtype.E5M2}.get(getattr(A, "dtype", None), Dtype.F16)


def gemm_nt_ex(A, B, D, M=None, N=None, K=None, dtype=None, alpha=1.0, beta=0.0, C=None, bias=None,
               activation=Activation.NONE, variant=Variant.AUTO, stream=None, scale_n=None) -> None:
    """D = act(alpha·scale_n[n]·A·Bᵀ + beta·C + bias[n]).

    Operands fp16, bf16, or 8-bit (E4M3 / E5M2, as torch float8 or uint8
    tensors; D, C and bias are then bf16); the dtype is taken from the tensors
    unless given (uint8 tensors need it).  ``scale_n`` is an optional float32
    [N] tensor (or device pointer) of per-column scales."""
    if dtype is None:
        dtype = _tensor_dtype(A) if _is_tensor(A) else Dtype.F16
    a, b, d, m, n, k, dev = _operands(A, B, D, M, N, K, Dtype(dtype))
    def ptr(x, what="C and bias", want=None):
        if x is None:
            return None
        if _is_tensor(x):
            want = D.dtype if want is None else want
            if x.dtype != want or not x.is_contiguous():
                raise TypeError(f"{what} must be contiguous {want}")
            return x.data_ptr()
        return int(x)
    sc = None
    if scale_n is not None:
        import torch
        sc = ptr(scale_n, "scale_n", torch.float32)
    epi = Epilogue(float(alpha), float(beta), ptr(C), ptr(bias), int(activation), 0, sc)
    _call("gemm_nt_ex", (int(dtype), a or None, b or None, d or None, m, n, k, ctypes.byref(epi), int(variant),
                         _stream_handle(stream, dev)), dev)


def gemm_f16_nt_check(stream=None, device=None) -> None:
    """Synchronise ``stream`` and raise GemmError if a kernel reported a timeout."""
    handle = _stream_handle(stream, device)
    _call("gemm_f16_nt_check", (handle,), device)


def gemm_selftest_timeout(timeout_us: int = 1000, stream=None, device=None) -> None:
    """Enqueue the failure-detection self-test: a kernel whose bounded waits run
    out and record a timeout; the next gemm_f16_nt_check raises it."""
    _call("gemm_selftest_timeout", (int(timeout_us), _stream_handle(stream, device)), device)


def gemm_f16_nt_plan(M: int, N: int, K: int, variant=Variant.AUTO, num_sms: int = 0) -> dict:
    """What a call would run (variant, tiles, grid, shared memory, workspace)."""
    plan = Plan()
    st = load().gemm_f16_nt_plan(int(M), int(N), int(K), int(variant), int(num_sms), ctypes.byref(plan))
    if st != Status.OK:
        raise GemmError(st, "gemm_f16_nt_plan")
    return plan.as_dict()


def gemm_nt_plan_ex(dtype, M: int, N: int, K: int, variant=Variant.AUTO, num_sms: int = 0) -> dict:
    """gemm_f16_nt_plan for the operand type ``dtype`` (a ``Dtype``)."""
    plan = Plan()
    st = load().gemm_nt_plan_ex(int(dtype), int(M), int(N), int(K), int(variant), int(num_sms), ctypes.byref(plan))
    if st != Status.OK:
        raise GemmError(st, "gemm_nt_plan_ex")
    return plan.as_dict()


def gemm(A, B, variant=Variant.AUTO, stream=None):
    """Convenience: allocate D with torch on A's device and return A·Bᵀ."""
    import torch
    D = torch.empty((A.shape[0], B.shape[0]), dtype=torch.float16, device=A.device)
    gemm_f16_nt_variant(A, B, D, variant=variant, stream=stream)
    return D
