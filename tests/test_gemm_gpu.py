"""Parity of the CUDA path with the CPU oracle, through the C ABI (needs a GB300).

Every comparison is element by element on the same seeded inputs: the full
output at sizes the oracle finishes in seconds (several tiles, ragged
tails), and at the full sizes of the named workloads -- in the launch
configuration the benchmark times (the AUTO plan) -- all of 8 seeded rows,
8 seeded columns, 65,536 seeded random entries, the corners, and the last
row/column of every partial tile.
"""
import math

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


def _dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _run(A, B, variant=g.Variant.AUTO, fill=float("nan"), stream=None):
    """D = A·Bᵀ on the GPU through the C ABI; D is pre-filled with `fill`."""
    dA, dB = _dev(A), _dev(B)
    D = torch.full((A.shape[0], B.shape[0]), fill, dtype=torch.float16, device="cuda")
    g.gemm_f16_nt_variant(dA, dB, D, variant=variant, stream=stream)
    g.gemm_f16_nt_check(stream=stream, device=D.device)
    return D.cpu().numpy()


def _full_parity(A, B, variant=g.Variant.AUTO, what=""):
    d = _run(A, B, variant)
    ref = oracle.gemm(A, B)
    return check_close(d, ref, A.shape[1], what or f"{variant.name} {A.shape[0]}x{B.shape[0]}x{A.shape[1]}")


def _edge_indices(M, tile):
    """Last index of every tile and first of the next, plus the last index."""
    idx = set()
    for t in range(tile, M + tile, tile):
        for v in (t - 1, t, t - tile // 2 - 1, t - tile // 2):
            if 0 <= v < M:
                idx.add(v)
    idx.add(M - 1)
    return sorted(idx)


# ---------------------------------------------------------------- named workloads
SMALL = ["single_tile_128x128x64", "multi_tile_1024x1024x2048"]
LARGE = ["square_8192x8192x8192", "ragged_4000x11000x4104", "skinny_16x8192x8192"]


@pytest.mark.parametrize("name", SMALL)
def test_named_workload_full_output(name):
    A, B = inputs.workload_operands(name)
    stats = _full_parity(A, B, what=name)
    assert stats["rel_fro"] < 1e-3


@pytest.mark.parametrize("name", LARGE)
def test_named_workload_sampled(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.workload_operands(name)
    plan = g.gemm_f16_nt_plan(w.M, w.N, w.K)
    d = _run(A, B)
    rows, cols = inputs.sample_entries(
        w.M, w.N, seed=w.seed + 77,
        extra_rows=_edge_indices(w.M, plan["tile_m"]) if plan["variant"] != "SKINNY_SPLITK" else range(w.M),
        extra_cols=_edge_indices(w.N, plan["tile_n"]))
    ref = oracle.gemm_entries(A, B, rows, cols)
    check_close(d[rows, cols], ref, w.K, name)
    assert not np.any(np.isnan(d)), f"{name}: unwritten output entries"


# ---------------------------------------------------------------- every variant, ragged
TILED = [g.Variant.TILE_2CTA_256x256, g.Variant.TILE_1CTA_128x128, g.Variant.TILE_1CTA_128x256,
         g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_2CTA_512x256, g.Variant.TILE_1CTA_SPLITK]
RAGGED = [(1, 8, 8), (7, 24, 40), (128, 128, 64), (129, 136, 72), (255, 264, 200),
          (300, 520, 1000), (513, 256, 4104), (640, 1000, 520)]
SKINNY = [(1, 8, 8), (5, 136, 64), (16, 128, 64), (17, 200, 72), (33, 1000, 520),
          (64, 4096, 1024), (16, 1024, 8192), (3, 65536, 64)]


@pytest.mark.parametrize("variant", TILED, ids=lambda v: v.name)
@pytest.mark.parametrize("shape", RAGGED, ids=lambda s: "x".join(map(str, s)))
def test_tiled_variants_ragged(variant, shape):
    M, N, K = shape
    A, B = inputs.operands(M, N, K, seed=1000 + M + N + K)
    _full_parity(A, B, variant)


@pytest.mark.parametrize("variant", [g.Variant.SKINNY_SPLITK, g.Variant.SKINNY_STREAMK], ids=lambda v: v.name)
@pytest.mark.parametrize("shape", SKINNY, ids=lambda s: "x".join(map(str, s)))
def test_skinny_variant_ragged(shape, variant):
    M, N, K = shape
    A, B = inputs.operands(M, N, K, "normal:1", "normal:1/sqrtK", seed=2000 + M + N + K)
    _full_parity(A, B, variant)


# shapes the column-range small-M planner gives 8, 4, 2 and 1 K pieces per
# range (clusters of that many CTAs), and one whose ranges take two rounds
SKINNY_CLUSTERS = [(16, 1024, 8192), (16, 2560, 8192), (24, 3000, 4104), (16, 8192, 4096), (33, 1000, 520),
                   (8, 24576, 256), (64, 1032, 1032), (40, 4096, 2048), (1, 8, 8192), (7, 2048, 192),
                   (1, 8192, 1024)]


def test_skinny_cluster_sizes_all_covered():
    plans = [g.gemm_f16_nt_plan(*s) for s in SKINNY_CLUSTERS]
    assert {p["k_split"] for p in plans} == {1, 2, 4, 8}, [(p["k_split"], p["n_tiles"]) for p in plans]
    assert any(p["max_tiles_per_cta"] > 1 for p in plans)
    assert all(p["variant"] == "SKINNY_SPLITK" and p["tile_n"] <= 128 for p in plans)


@pytest.mark.parametrize("shape", SKINNY_CLUSTERS, ids=lambda s: "x".join(map(str, s)))
def test_skinny_cluster_sizes(shape):
    # full output against the oracle, and the same bits on a second call
    M, N, K = shape
    A, B = inputs.operands(M, N, K, "normal:1", "normal:1/sqrtK", seed=2500 + M + N + K)
    _full_parity(A, B, g.Variant.SKINNY_SPLITK)
    d1 = _run(A, B, g.Variant.SKINNY_SPLITK)
    d2 = _run(A, B, g.Variant.SKINNY_SPLITK)
    assert np.array_equal(d1.view(np.uint16), d2.view(np.uint16))


@pytest.mark.parametrize("shape", [(300, 520, 1000), (513, 256, 4104), (1000, 1000, 640), (1024, 1024, 2048),
                                   (512, 2048, 8192), (272, 2056, 520), (1200, 1000, 1000), (1200, 704, 1400),
                                   (1100, 504, 2000), (300, 8, 4096)], ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("variant", [g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_1CTA_SPLITK], ids=lambda v: v.name)
def test_tile_split_k(shape, variant):
    # the planner really splits these (k_split > 1); ragged M, N and K included
    M, N, K = shape
    plan = g.gemm_f16_nt_plan(M, N, K, variant)
    assert plan["variant"] == variant.name and plan["k_split"] > 1, plan
    A, B = inputs.operands(M, N, K, seed=3000 + M + N + K)
    _full_parity(A, B, variant)


@pytest.mark.parametrize("variant", [g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_1CTA_SPLITK], ids=lambda v: v.name)
def test_tile_split_k_consecutive_calls(variant):
    # three calls in a row, new data each time
    for seed in (1, 2, 3):
        A, B = inputs.operands(700, 1000, 3000, seed=seed)
        _full_parity(A, B, variant, what=f"split-K seed {seed}")


@pytest.mark.parametrize("shape", [(256, 256, 8192), (130, 264, 4104), (128, 512, 16384)],
                         ids=lambda s: "x".join(map(str, s)))
def test_tile_split_k_single_ctas_up_to_8(shape):
    # few 128x256 tiles and a long K loop: clusters of up to 8 single CTAs
    M, N, K = shape
    plan = g.gemm_f16_nt_plan(M, N, K, g.Variant.TILE_1CTA_SPLITK)
    assert plan["variant"] == "TILE_1CTA_SPLITK" and plan["k_split"] >= 5, plan
    A, B = inputs.operands(M, N, K, seed=3100 + M + N + K)
    _full_parity(A, B, g.Variant.TILE_1CTA_SPLITK)


@pytest.mark.parametrize("shape", [(96, 512, 2048), (200, 304, 4104)], ids=str)
def test_all_variants_agree(shape):
    M, N, K = shape
    A, B = inputs.operands(M, N, K, seed=31)
    ref = oracle.gemm(A, B)
    for v in TILED:
        check_close(_run(A, B, v), ref, K, v.name)


# ---------------------------------------------------------------- closed forms (exact)
@pytest.mark.parametrize("variant", TILED + [g.Variant.SKINNY_SPLITK, g.Variant.SKINNY_STREAMK],
                         ids=lambda v: v.name)
def test_closed_forms_exact(variant):
    skinny = variant in (g.Variant.SKINNY_SPLITK, g.Variant.SKINNY_STREAMK)
    M = 48 if skinny else 272
    # all ones: D = K exactly (fp32 holds every partial sum exactly)
    for K in (64, 4104):
        d = _run(np.ones((M, K), np.float16), np.ones((264, K), np.float16), variant)
        assert np.all(d == K), (variant.name, K)
    # identity B: D = A bit for bit
    K = 256
    A = inputs.draw(M, K, "uniform", seed=5)
    d = _run(A, np.eye(K, dtype=np.float16), variant)
    assert np.array_equal(d.view(np.uint16), A.view(np.uint16))
    # swapping the operands transposes D
    B = inputs.draw(136, K, "uniform", seed=6)
    if skinny:
        return
    d1 = _run(A, B, variant)
    d2 = _run(B, A, variant)
    check_close(d2, d1.T, K, "transpose")


def test_special_values_propagate():
    A = np.ones((130, 64), np.float16)
    B = np.ones((136, 64), np.float16)
    A[3, 5] = np.nan
    A[7] = 256.0
    B[9] = 256.0
    d = _run(A, B, g.Variant.TILE_1CTA_128x128)
    assert np.all(np.isnan(d[3]))
    assert np.all(np.isposinf(d[7, 9:10]))       # 256*256*64 overflows fp16
    assert d[8, 8] == 64 and d[7, 8] == 256 * 64


# ---------------------------------------------------------------- determinism, streams
@pytest.mark.parametrize("name_or_shape", ["multi_tile_1024x1024x2048", (16, 1024, 8192), (40, 5000, 3000)],
                         ids=str)
def test_bitwise_deterministic(name_or_shape):
    if isinstance(name_or_shape, str):
        A, B = inputs.workload_operands(name_or_shape)
    else:
        A, B = inputs.operands(*name_or_shape, seed=77)
    d1 = _run(A, B)
    d2 = _run(A, B)
    assert np.array_equal(d1.view(np.uint16), d2.view(np.uint16))


@pytest.mark.parametrize("variant", [g.Variant.SKINNY_SPLITK, g.Variant.SKINNY_STREAMK], ids=lambda v: v.name)
def test_skinny_split_tiles_rearm_between_calls(variant):
    # every tile's K loop is split over several CTAs: the fixed-order reduction
    # (and, for the stream-K kernel, the counter reset) on consecutive calls
    for seed in (1, 2, 3):
        A, B = inputs.operands(16, 1024, 8192, "normal:1", "normal:1/sqrtK", seed=seed)
        _full_parity(A, B, variant, what=f"{variant.name} seed {seed}")


def test_side_stream():
    A, B = inputs.operands(300, 640, 512, seed=8)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        d = _run(A, B, stream=s)
    check_close(d, oracle.gemm(A, B), 512, "side stream")
    A, B = inputs.operands(16, 640, 4096, seed=9)
    with torch.cuda.stream(s):
        d = _run(A, B, stream=s)
    check_close(d, oracle.gemm(A, B), 4096, "side stream skinny")


# ---------------------------------------------------------------- edges of the contract
def test_k_zero_writes_zeros_and_empty_is_noop():
    D = torch.full((40, 24), float("nan"), dtype=torch.float16, device="cuda")
    A = torch.empty((40, 0), dtype=torch.float16, device="cuda")
    B = torch.empty((24, 0), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(A, B, D)
    g.gemm_f16_nt_check(device=D.device)
    assert torch.all(D == 0)
    D0 = torch.full((0, 24), 1.0, dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(torch.empty((0, 8), dtype=torch.float16, device="cuda"),
                  torch.ones((24, 8), dtype=torch.float16, device="cuda"), D0)


def test_device_argument_errors():
    buf = torch.zeros(1 << 20, dtype=torch.float16, device="cuda")
    base = buf.data_ptr()
    lib = g.load()
    # misaligned A (2 bytes past a 16-byte boundary)
    st = lib.gemm_f16_nt(base + 2, base + 65536, base + 131072, 64, 64, 64, None)
    assert st == g.Status.ERR_MISALIGNED
    # D aliasing B
    st = lib.gemm_f16_nt(base, base + 65536, base + 65536 + 4096, 64, 64, 64, None)
    assert st == g.Status.ERR_INVALID_VALUE
    # nothing was launched, so the device is clean
    g.gemm_f16_nt_check(device=buf.device)


def test_plan_on_device_matches_sm_count():
    p = g.gemm_f16_nt_plan(8192, 8192, 8192)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert p["variant"] == "TILE_2CTA_256x256"
    assert 2 <= p["grid_ctas"] <= sms and p["grid_ctas"] % 2 == 0
    q = g.gemm_f16_nt_plan(16, 8192, 8192)
    assert q["grid_ctas"] == sms


@pytest.mark.parametrize("shape", [(4000, 11000, 4104), (1000, 3000, 1000), (777, 520, 4104), (513, 1032, 64),
                                   (1536, 2304, 1096)], ids=lambda s: "x".join(map(str, s)))
def test_two_consumer_pairs(shape):
    # two MMA consumers per CTA sharing each staged B tile (512 x 256 per pair):
    # ragged M (a second consumer on rows past M), ragged N and K, column
    # pieces in the last round, several rounds on the single-buffered
    # accumulators; consecutive calls give the same bits
    M, N, K = shape
    plan = g.gemm_f16_nt_plan(M, N, K, g.Variant.TILE_2CTA_512x256)
    assert plan["variant"] == "TILE_2CTA_512x256" and plan["tile_m"] == 512 and plan["grid_ctas"] % 2 == 0
    A, B = inputs.operands(M, N, K, seed=5000 + M + N + K)
    if M * N * K <= 2e10:
        _full_parity(A, B, g.Variant.TILE_2CTA_512x256)
        d1 = _run(A, B, g.Variant.TILE_2CTA_512x256)
        d2 = _run(A, B, g.Variant.TILE_2CTA_512x256)
        assert np.array_equal(d1.view(np.uint16), d2.view(np.uint16)), "two-consumer result differs between calls"
    else:
        d = _run(A, B, g.Variant.TILE_2CTA_512x256)
        rows, cols = inputs.sample_entries(M, N, seed=11, extra_rows=_edge_indices(M, 256),
                                           extra_cols=_edge_indices(N, 256))
        check_close(d[rows, cols], oracle.gemm_entries(A, B, rows, cols), K, "two-consumer sampled")
        assert not np.any(np.isnan(d))
