"""Parity at extreme sizes: a million rows, a million columns, a million K
(needs a GB300).

Tile, K-block and unit counters, TMA coordinates and the split-K ranges all
reach values far beyond the named workloads here; entries are checked
against the CPU oracle on seeded samples that always include the last rows
and columns (and the ragged edges of the last tiles).
"""
import numpy as np
import pytest

import oracle
import dense_fp16_gemm_f16_gb300 as g
from dense_fp16_gemm_f16_gb300 import build as gbuild
from dense_fp16_gemm_f16_gb300 import inputs
from gemm_check import check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gbuild.build()
    g.load()
    yield
    g.gemm_f16_nt_check(device=torch.device("cuda"))
    torch.cuda.empty_cache()


def _run(A, B, variant=g.Variant.AUTO):
    M, N = A.shape[0], B.shape[0]
    D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt_variant(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), D, variant=variant)
    g.gemm_f16_nt_check(device=D.device)
    return D


def _sampled(D, A, B, K, what, rows, cols):
    got = D[torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()].cpu().numpy()
    assert not np.any(np.isnan(got.astype(np.float64))), what
    check_close(got, oracle.gemm_entries(A, B, rows, cols), K, what)


@pytest.mark.parametrize("M", [(1 << 20) + 40])
def test_a_million_rows(M):
    N, K = 136, 72                            # K = 72: rows off 32-byte sectors, 4-CTA clusters
    A, B = inputs.operands(M, N, K, seed=81)
    D = _run(A, B)
    rows, cols = inputs.sample_entries(M, N, seed=82, n_random=32768,
                                       extra_rows=[M - 1, M - 40, M - 41, 1 << 20, (1 << 20) - 1])
    _sampled(D, A, B, K, "M = 2^20 + 40", rows, cols)


def test_a_million_columns():
    M, N, K = 64, (1 << 20) + 8, 64          # the small-M kernel over 8193 tiles of 128 columns
    A, B = inputs.operands(M, N, K, "normal:1", "uniform", seed=83)
    D = _run(A, B)
    rows, cols = inputs.sample_entries(M, N, seed=84, n_random=32768,
                                       extra_cols=[N - 1, N - 8, N - 9, 1 << 20, (1 << 20) - 1])
    _sampled(D, A, B, K, "N = 2^20 + 8", rows, cols)


def test_a_million_k_small_m():
    M, N, K = 16, 256, 1 << 20                # 16384 K blocks per tile split over all SMs
    A, B = inputs.operands(M, N, K, seed=85)
    D = _run(A, B, g.Variant.SKINNY_SPLITK)
    check_close(D.cpu().numpy(), oracle.gemm(A, B), K, "K = 2^20, small M")


@pytest.mark.parametrize("variant,pieces", [(g.Variant.TILE_2CTA_SPLITK, 4), (g.Variant.TILE_1CTA_SPLITK, 8)],
                         ids=["pairs", "single_ctas"])
def test_long_k_split(variant, pieces):
    M, N, K = 256, 264, (1 << 18) + 8         # ragged N and K; every tile's K loop split 4 or 8 ways
    plan = g.gemm_f16_nt_plan(M, N, K, variant)
    assert plan["variant"] == variant.name and plan["k_split"] == pieces, plan
    A, B = inputs.operands(M, N, K, seed=86)
    D = _run(A, B, variant)
    rows, cols = inputs.sample_entries(M, N, seed=87, n_rows=2, n_cols=2, n_random=2048,
                                       extra_rows=[M - 1], extra_cols=[N - 1, N - 8, 255, 256])
    _sampled(D, A, B, K, "K = 2^18 + 8, split pairs", rows, cols)


def test_long_k_e4m3():
    M, N, K = 16, 128, 1 << 20
    A, B, sa, sb = inputs.operands_fp8(M, N, K, seed=88, fmt="e4m3")
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.gemm_nt_ex(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), D, dtype=g.Dtype.E4M3, alpha=sa,
                 scale_n=torch.from_numpy(sb).cuda())
    g.gemm_f16_nt_check(device=D.device)
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    check_close(got, oracle.gemm_ex(A, B, "e4m3", sa, scale_n=sb), K, "K = 2^20, E4M3", dtype="bf16")
