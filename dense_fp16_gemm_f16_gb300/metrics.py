"""Throughput figures reported for the GEMM.

TFLOPS counts one multiply-add as two floating-point operations:
TFLOPS = 2·M·N·K / (t · 10¹²) -- "Building a Tiled GEMM" (MLC), section
"GEMM"; the Croqtile tutorial's headline table uses the same count.
"""


def flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def tflops(M: int, N: int, K: int, seconds: float) -> float:
    return flops(M, N, K) / (seconds * 1e12)


def compulsory_bytes(M: int, N: int, K: int, elem_bytes: int = 2) -> int:
    """A and B read once and D written once."""
    return elem_bytes * (M * K + N * K + M * N)


def gbs(nbytes: int, seconds: float) -> float:
    return nbytes / (seconds * 1e9)
