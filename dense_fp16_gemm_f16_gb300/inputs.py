"""Seeded synthetic operands for D = A·Bᵀ (fp16 A [M,K], fp16 B [N,K]).

This module draws numbers and nothing else: it holds none of the GEMM's
arithmetic, so both the CPU oracle and the CUDA path may take their inputs
from it.  Values are drawn in float64 from NumPy's PCG64 generator
(``numpy.random.default_rng(seed)``) and rounded to fp16 by NumPy's own
float64→float16 cast (round to nearest, ties to even).

The five named workloads follow the shapes and value distributions the pages
work with: the single 128×128 output tile with K=64 of "Building a Tiled
GEMM" (MLC), step 1; its multi-tile K-loop (steps 2 and 3); the 8192³ fp16
problem of the Croqtile tutorial ("dense GEMM fp16 from naive", headline
table); a ragged shape with no dimension a multiple of 128; and the small-
batch decode shape the blog post's "small batch" pitfall (§5.4) is about.
"Normal(0, 1/√K)" is read as standard deviation 1/√K.  B's seed is A's seed
plus 1000.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

_CHUNK = 1 << 22  # elements drawn per generator call (bounds float64 scratch)


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    dist_a: str      # "uniform" (U[-1,1]) or "normal:<sigma>" or "normal:1/sqrtK"
    dist_b: str
    seed: int        # seed of A; B uses seed + 1000

    @property
    def seed_b(self) -> int:
        return self.seed + 1000

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        """A and B read once, D written once (fp16 = 2 bytes each)."""
        return 2 * (self.M * self.K + self.N * self.K + self.M * self.N)


WORKLOADS = {
    w.name: w for w in (
        Workload("single_tile_128x128x64", 128, 128, 64, "uniform", "uniform", 1),
        Workload("multi_tile_1024x1024x2048", 1024, 1024, 2048, "uniform", "uniform", 2),
        Workload("square_8192x8192x8192", 8192, 8192, 8192, "normal:1/sqrtK", "normal:1/sqrtK", 3),
        Workload("ragged_4000x11000x4104", 4000, 11000, 4104, "uniform", "uniform", 4),
        Workload("skinny_16x8192x8192", 16, 8192, 8192, "normal:1", "normal:1/sqrtK", 5),
    )
}

#: the workload the headline throughput is quoted on
HEADLINE = "square_8192x8192x8192"


def _sigma(dist: str, K: int) -> float:
    arg = dist.split(":", 1)[1]
    if arg == "1/sqrtK":
        return 1.0 / math.sqrt(K)
    return float(arg)


def draw(rows: int, cols: int, dist: str, seed: int, K: int | None = None,
         chunk: int = _CHUNK) -> np.ndarray:
    """A C-contiguous float16 [rows, cols] array of i.i.d. draws.

    ``dist`` is "uniform" (U[-1, 1]) or "normal:<sigma>" where sigma is a
    number or "1/sqrtK".  Draws are made in chunks from one generator, which
    gives the same stream as a single call.
    """
    K = cols if K is None else K
    rng = np.random.default_rng(seed)
    total = rows * cols
    out = np.empty(total, dtype=np.float16)
    if dist == "uniform":
        gen = lambda n: rng.uniform(-1.0, 1.0, n)          # noqa: E731
    elif dist.startswith("normal:"):
        sigma = _sigma(dist, K)
        gen = lambda n: rng.normal(0.0, sigma, n)           # noqa: E731
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    for start in range(0, total, chunk):
        n = min(chunk, total - start)
        out[start:start + n] = gen(n).astype(np.float16)
    return out.reshape(rows, cols)


def operands(M: int, N: int, K: int, dist_a: str = "uniform", dist_b: str = "uniform",
             seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """(A [M,K], B [N,K]) float16, A from ``seed`` and B from ``seed + 1000``."""
    A = draw(M, K, dist_a, seed, K=K)
    B = draw(N, K, dist_b, seed + 1000, K=K)
    return A, B


def workload_operands(name: str) -> tuple[np.ndarray, np.ndarray]:
    w = WORKLOADS[name]
    return operands(w.M, w.N, w.K, w.dist_a, w.dist_b, w.seed)


def sample_entries(M: int, N: int, seed: int, n_rows: int = 8, n_cols: int = 8,
                   n_random: int = 65536, extra_rows=(), extra_cols=()):
    """Seeded (row, col) index pairs for checking a large D entry by entry.

    All of ``n_rows`` seeded rows (every column), all of ``n_cols`` seeded
    columns (every row), ``n_random`` seeded random entries, the four corners,
    and every entry of the rows/columns listed in ``extra_rows``/``extra_cols``
    (the last row and column of partial tiles, say).  Returns two int64
    arrays; pairs may repeat.
    """
    rng = np.random.default_rng(seed)
    rows = [rng.integers(0, M, n_rows), np.asarray(list(extra_rows), dtype=np.int64)]
    cols = [rng.integers(0, N, n_cols), np.asarray(list(extra_cols), dtype=np.int64)]
    sel_rows = np.unique(np.concatenate(rows).astype(np.int64))
    sel_cols = np.unique(np.concatenate(cols).astype(np.int64))
    r_parts, c_parts = [], []
    for r in sel_rows:
        r_parts.append(np.full(N, r, dtype=np.int64))
        c_parts.append(np.arange(N, dtype=np.int64))
    for c in sel_cols:
        r_parts.append(np.arange(M, dtype=np.int64))
        c_parts.append(np.full(M, c, dtype=np.int64))
    r_parts.append(rng.integers(0, M, n_random).astype(np.int64))
    c_parts.append(rng.integers(0, N, n_random).astype(np.int64))
    r_parts.append(np.array([0, 0, M - 1, M - 1], dtype=np.int64))
    c_parts.append(np.array([0, N - 1, 0, N - 1], dtype=np.int64))
    return np.concatenate(r_parts), np.concatenate(c_parts)


def _draw_f64(rows: int, cols: int, dist: str, seed: int, K: int | None = None) -> np.ndarray:
    """The float64 draws behind ``draw`` (one generator call), as [rows, cols]."""
    K = cols if K is None else K
    rng = np.random.default_rng(seed)
    n = rows * cols
    if dist == "uniform":
        x = rng.uniform(-1.0, 1.0, n)
    elif dist.startswith("normal:"):
        x = rng.normal(0.0, _sigma(dist, K), n)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return x.reshape(rows, cols)


def draw_bf16(rows: int, cols: int, dist: str, seed: int, K: int | None = None) -> np.ndarray:
    """bf16 operands as uint16 bit patterns: the same float64 draws as ``draw``,
    rounded to float32 and then to bf16 by torch (nearest, ties to even).  Any
    bf16 value is a valid input; the CPU oracle and the GPU see the same bits."""
    import torch

    x = _draw_f64(rows, cols, dist, seed, K).ravel()
    t = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).reshape(rows, cols).copy()


#: largest finite value of each 8-bit operand type
FP8_MAX = {"e4m3": 448.0, "e5m2": 57344.0}


def _torch_fp8(fmt: str):
    import torch
    if fmt == "e4m3":
        return torch.float8_e4m3fn
    if fmt == "e5m2":
        return torch.float8_e5m2
    raise ValueError(f"unknown 8-bit format {fmt!r}")


def draw_fp8(rows: int, cols: int, dist: str, seed: int, fmt: str = "e4m3", K: int | None = None,
             per_row: bool = False) -> tuple[np.ndarray, np.ndarray]:
    """8-bit operands with their fp32 scales: the same float64 draws as ``draw``,
    divided by a scale that maps their largest magnitude onto the format's
    largest finite value -- one scale for the whole array, or one per row when
    ``per_row`` -- and rounded by torch's float32 -> 8-bit conversion (nearest,
    ties to even).  This is the amax scaling of the GEMM blog post's
    quantisation step (section 4.2); values times scale approximate the draws.
    Returns (bits uint8 [rows, cols], scale float32 [rows] or [1]).  Any
    finite 8-bit value is a valid input: the CPU oracle and the GPU see the
    same bits and the same scales."""
    import torch

    x = _draw_f64(rows, cols, dist, seed, K)
    top = FP8_MAX[fmt]
    amax = np.abs(x).max(axis=1) if per_row else np.array([np.abs(x).max() if x.size else 0.0])
    scale = (amax / top).astype(np.float32)
    scale[scale == 0] = 1.0
    div = scale.astype(np.float64)[:, None] if per_row else np.float64(scale[0])
    q = torch.from_numpy((x / div).astype(np.float32)).clamp_(-top, top).to(_torch_fp8(fmt))
    return q.view(torch.uint8).numpy().copy(), scale


def operands_fp8(M: int, N: int, K: int, dist_a: str = "uniform", dist_b: str = "uniform", seed: int = 0,
                 fmt: str = "e4m3") -> tuple[np.ndarray, np.ndarray, float, np.ndarray]:
    """(A [M,K], B [N,K], a_scale, b_scale [N]) for the 8-bit GEMM: A (the
    activations) from ``seed`` with one scale, B (the weights, one output
    channel per row) from ``seed + 1000`` with one scale per row.  With D's
    fused transform ``alpha = a_scale`` and per-column scale ``b_scale`` the
    GEMM computes the dequantised product."""
    A, sa = draw_fp8(M, K, dist_a, seed, fmt, K=K)
    B, sb = draw_fp8(N, K, dist_b, seed + 1000, fmt, K=K, per_row=True)
    return A, B, float(sa[0]), sb


def operands_bf16(M: int, N: int, K: int, dist_a: str = "uniform", dist_b: str = "uniform",
                  seed: int = 0) -> tuple[np.ndarray, np.ndarray]:
    """(A [M,K], B [N,K]) bf16 bit patterns, A from ``seed`` and B from ``seed + 1000``."""
    return draw_bf16(M, K, dist_a, seed, K=K), draw_bf16(N, K, dist_b, seed + 1000, K=K)
