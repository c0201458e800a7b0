"""CPU oracle for the dense fp16 GEMM D = A·Bᵀ.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` are the only callers.  The CUDA library and its
Python binding never import this package, and this package imports nothing
from them.

What it computes -- "Building a Tiled GEMM" (MLC, Modern GPU Programming for
MLSys), section "GEMM": ``D[m,n] = Σ_k A[m,k]·B[n,k]`` with A [M,K] and B
[N,K] row-major fp16, accumulated here in fp64 (ascending k, one accumulator)
and rounded once, directly, to fp16 with round-to-nearest-even.  The
arithmetic lives in ``gemm_oracle.c``; this module only builds it with gcc,
loads it and marshals numpy arrays.

Pins (tests/test_oracle.py): the fp16 decode/encode is checked exhaustively
and against numpy's own float64→float16 routine; the GEMM against exact int64
arithmetic on small-integer inputs, and against closed forms (all-ones,
identity B, rank-1, zero blocks).  The bf16 and 8-bit (E4M3, E5M2) decoders
are checked exhaustively against torch's conversions (tests/test_oracle_ex.py,
tests/test_oracle_fp8.py), the fused transform and the per-column scale
against exact arithmetic.  Every function here is pinned, and the tests also
build broken copies of the C file to show that each pin fails when a
plausible mistake is planted.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "gemm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libgemm_oracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-pthread"]


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C file into a shared library with gcc.

    ``-ffp-contract=off`` keeps ``acc += a*b`` as a separate multiply and
    add on every host (gcc would otherwise contract it on aarch64); the
    products are exact in fp64, so this is belt and braces.
    """
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile gemm_oracle.c into libgemm_oracle.so next to it, if stale."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(SOURCE)):
        return _LIB_PATH
    return compile_source(SOURCE, _LIB_PATH)


def default_threads() -> int:
    """Host threads the oracle uses by default: every core this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def _ptr(a) -> int | None:
    return None if a is None else a.ctypes.data


def _as_f16(x, name: str) -> np.ndarray:
    a = np.ascontiguousarray(x)
    if a.dtype != np.float16:
        raise TypeError(f"{name} must be float16, got {a.dtype}")
    return a


class Oracle:
    """One loaded copy of an oracle shared library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.oracle_f16_to_f64.argtypes = [p, p, i64]
        lib.oracle_f16_to_f64.restype = None
        lib.oracle_f64_to_f16.argtypes = [p, p, i64]
        lib.oracle_f64_to_f16.restype = None
        lib.oracle_gemm_nt_entries.argtypes = [p, p, i64, i64, i64, p, p, i64, p, p, ctypes.c_int]
        lib.oracle_gemm_nt_entries.restype = ctypes.c_int
        lib.oracle_gemm_nt_rows.argtypes = [p, p, i64, i64, i64, i64, i64, p, p, ctypes.c_int]
        lib.oracle_gemm_nt_rows.restype = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [p, p, i64]
        lib.oracle_bf16_to_f64.restype = None
        lib.oracle_f64_to_bf16.argtypes = [p, p, i64]
        lib.oracle_f64_to_bf16.restype = None
        d = ctypes.c_double
        lib.oracle_e4m3_to_f64.argtypes = [p, p, i64]
        lib.oracle_e4m3_to_f64.restype = None
        lib.oracle_e5m2_to_f64.argtypes = [p, p, i64]
        lib.oracle_e5m2_to_f64.restype = None
        lib.oracle_gemm_nt_ex.argtypes = [ctypes.c_int, p, p, i64, i64, i64, p, p, i64, i64, i64,
                                          d, d, p, p, p, ctypes.c_int, p, p, ctypes.c_int]
        lib.oracle_gemm_nt_ex.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    # -- element conversions ------------------------------------------------
    def f16_to_f64(self, h) -> np.ndarray:
        """Decode fp16 values (float16 array, or uint16 bit patterns) into float64."""
        a = np.ascontiguousarray(h)
        bits = a.view(np.uint16) if a.dtype == np.float16 else a.astype(np.uint16, copy=False)
        bits = np.ascontiguousarray(bits)
        out = np.empty(bits.shape, dtype=np.float64)
        self.lib.oracle_f16_to_f64(_ptr(bits), _ptr(out), bits.size)
        return out

    def f64_to_f16(self, x) -> np.ndarray:
        """Round float64 values to fp16 (nearest, ties to even); returns float16."""
        a = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_f16(_ptr(a), _ptr(out), a.size)
        return out.view(np.float16)

    def bf16_to_f64(self, bits) -> np.ndarray:
        """Decode bf16 bit patterns (uint16) into float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint16)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_bf16_to_f64(_ptr(b), _ptr(out), b.size)
        return out

    def f64_to_bf16(self, x) -> np.ndarray:
        """Round float64 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
        a = np.ascontiguousarray(x, dtype=np.float64)
        out = np.empty(a.shape, dtype=np.uint16)
        self.lib.oracle_f64_to_bf16(_ptr(a), _ptr(out), a.size)
        return out

    def e4m3_to_f64(self, bits) -> np.ndarray:
        """Decode E4M3 bit patterns (uint8) into float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_e4m3_to_f64(_ptr(b), _ptr(out), b.size)
        return out

    def e5m2_to_f64(self, bits) -> np.ndarray:
        """Decode E5M2 bit patterns (uint8) into float64."""
        b = np.ascontiguousarray(bits, dtype=np.uint8)
        out = np.empty(b.shape, dtype=np.float64)
        self.lib.oracle_e5m2_to_f64(_ptr(b), _ptr(out), b.size)
        return out

    # -- the GEMM -------------------------------------------------------------
    @staticmethod
    def _operands(A, B):
        A = _as_f16(A, "A")
        B = _as_f16(B, "B")
        if A.ndim != 2 or B.ndim != 2 or A.shape[1] != B.shape[1]:
            raise ValueError(f"need A [M,K] and B [N,K]; got {A.shape} and {B.shape}")
        return A, B

    def gemm_entries(self, A, B, rows, cols, nthreads: int | None = None,
                     want_sums: bool = False):
        """D[rows[i], cols[i]] for each i, as float16 (and the fp64 sums if asked)."""
        A, B = self._operands(A, B)
        M, K = A.shape
        N = B.shape[0]
        r = np.ascontiguousarray(rows, dtype=np.int64).ravel()
        c = np.ascontiguousarray(cols, dtype=np.int64).ravel()
        if r.shape != c.shape:
            raise ValueError("rows and cols must have the same length")
        out = np.empty(r.size, dtype=np.uint16)
        sums = np.empty(r.size, dtype=np.float64) if want_sums else None
        rc = self.lib.oracle_gemm_nt_entries(
            _ptr(A), _ptr(B), M, N, K, _ptr(r), _ptr(c), r.size, _ptr(sums), _ptr(out),
            nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_gemm_nt_entries rejected its arguments")
        d = out.view(np.float16)
        return (d, sums) if want_sums else d

    def gemm_rows(self, A, B, row_begin: int, row_end: int, nthreads: int | None = None,
                  want_sums: bool = False):
        """Rows [row_begin, row_end) of D as a float16 [row_end-row_begin, N] array."""
        A, B = self._operands(A, B)
        M, K = A.shape
        N = B.shape[0]
        out = np.empty((row_end - row_begin, N), dtype=np.uint16)
        sums = np.empty(out.shape, dtype=np.float64) if want_sums else None
        rc = self.lib.oracle_gemm_nt_rows(
            _ptr(A), _ptr(B), M, N, K, row_begin, row_end, _ptr(sums), _ptr(out),
            nthreads or default_threads())
        if rc != 0:
            raise ValueError("oracle_gemm_nt_rows rejected its arguments")
        d = out.view(np.float16)
        return (d, sums) if want_sums else d

    def gemm(self, A, B, nthreads: int | None = None, want_sums: bool = False):
        """The whole of D = A·Bᵀ as float16 [M, N] (for sizes the CPU finishes quickly)."""
        A, B = self._operands(A, B)
        return self.gemm_rows(A, B, 0, A.shape[0], nthreads=nthreads, want_sums=want_sums)


def default() -> Oracle:
    """The oracle built from gemm_oracle.c (built on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def f16_to_f64(h):
    return default().f16_to_f64(h)


def f64_to_f16(x):
    return default().f64_to_f16(x)


def gemm_entries(A, B, rows, cols, nthreads=None, want_sums=False):
    return default().gemm_entries(A, B, rows, cols, nthreads=nthreads, want_sums=want_sums)


def gemm_rows(A, B, row_begin, row_end, nthreads=None, want_sums=False):
    return default().gemm_rows(A, B, row_begin, row_end, nthreads=nthreads, want_sums=want_sums)


def gemm(A, B, nthreads=None, want_sums=False):
    return default().gemm(A, B, nthreads=nthreads, want_sums=want_sums)


# ---------------------------------------------------------------------------
# element type + fused epilogue:
#   D = round(act(alpha * scale_n[n] * A Bᵀ + beta * C + bias[n]))
# ---------------------------------------------------------------------------
DTYPES = {"f16": 0, "bf16": 1, "e4m3": 2, "e5m2": 3}
#: 8-bit operand types; their D, C and bias are bf16
FP8 = ("e4m3", "e5m2")


def out_dtype(dtype: str) -> str:
    """Element type of D (and C, bias) for an operand type."""
    return "f16" if dtype == "f16" else "bf16"


def _bits(x, dtype: str) -> np.ndarray:
    """Bit patterns of an array: float16 arrays for f16, uint16 for bf16,
    uint8 for the 8-bit types."""
    a = np.ascontiguousarray(x)
    if dtype == "f16":
        if a.dtype != np.float16:
            raise TypeError(f"f16 operands must be float16 arrays, got {a.dtype}")
        return a.view(np.uint16)
    if dtype in FP8:
        if a.dtype != np.uint8:
            raise TypeError(f"{dtype} operands must be uint8 bit-pattern arrays, got {a.dtype}")
        return a
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 operands must be uint16 bit-pattern arrays, got {a.dtype}")
    return a


def _gemm_ex(o: Oracle, A, B, dtype, alpha, beta, C, bias, relu, rows=None, cols=None,
             row_begin=0, row_end=None, nthreads=None, want_pre=False, scale_n=None):
    if dtype not in DTYPES:
        raise ValueError(f"dtype must be one of {sorted(DTYPES)}")
    Ab, Bb = _bits(A, dtype), _bits(B, dtype)
    if Ab.ndim != 2 or Bb.ndim != 2 or Ab.shape[1] != Bb.shape[1]:
        raise ValueError("need A [M,K] and B [N,K]")
    M, K = Ab.shape
    N = Bb.shape[0]
    od = out_dtype(dtype)
    Cb = None if C is None or beta == 0 else _bits(C, od)
    if Cb is not None and Cb.shape != (M, N):
        raise ValueError("C must be [M, N]")
    biasb = None if bias is None else _bits(bias, od)
    if biasb is not None and biasb.shape != (N,):
        raise ValueError("bias must be [N]")
    sc = None
    if scale_n is not None:
        sc = np.ascontiguousarray(scale_n)
        if sc.dtype != np.float32 or sc.shape != (N,):
            raise TypeError("scale_n must be a float32 [N] array")
    if rows is not None:
        r = np.ascontiguousarray(rows, dtype=np.int64).ravel()
        c = np.ascontiguousarray(cols, dtype=np.int64).ravel()
        shape, count = r.shape, r.size
        rp, cp = _ptr(r), _ptr(c)
        rb, re = 0, 0
    else:
        row_end = M if row_end is None else row_end
        shape, count = (row_end - row_begin, N), 0
        rp = cp = None
        rb, re = row_begin, row_end
    out = np.empty(shape, dtype=np.uint16)
    pre = np.empty(shape, dtype=np.float64) if want_pre else None
    rc = o.lib.oracle_gemm_nt_ex(DTYPES[dtype], _ptr(Ab), _ptr(Bb), M, N, K, rp, cp, count, rb, re,
                                 float(alpha), float(beta), _ptr(Cb), _ptr(biasb), _ptr(sc),
                                 1 if relu else 0, _ptr(pre), _ptr(out), nthreads or default_threads())
    if rc != 0:
        raise ValueError("oracle_gemm_nt_ex rejected its arguments")
    res = out.view(np.float16) if od == "f16" else out
    return (res, pre) if want_pre else res


def gemm_ex(A, B, dtype="f16", alpha=1.0, beta=0.0, C=None, bias=None, relu=False,
            nthreads=None, want_pre=False, oracle=None, scale_n=None):
    """Whole D (float16 for f16, uint16 bf16 bit patterns otherwise)."""
    return _gemm_ex(oracle or default(), A, B, dtype, alpha, beta, C, bias, relu,
                    nthreads=nthreads, want_pre=want_pre, scale_n=scale_n)


def gemm_ex_entries(A, B, rows, cols, dtype="f16", alpha=1.0, beta=0.0, C=None, bias=None, relu=False,
                    nthreads=None, oracle=None, scale_n=None):
    """D at the listed (row, col) entries."""
    return _gemm_ex(oracle or default(), A, B, dtype, alpha, beta, C, bias, relu, rows=rows, cols=cols,
                    nthreads=nthreads, scale_n=scale_n)


def bf16_to_f64(bits):
    return default().bf16_to_f64(bits)


def f64_to_bf16(x):
    return default().f64_to_bf16(x)


def e4m3_to_f64(bits):
    return default().e4m3_to_f64(bits)


def e5m2_to_f64(bits):
    return default().e5m2_to_f64(bits)
