"""Parity of the 8-bit operand path (E4M3, E5M2) with the CPU oracle (needs a GB300).

The operands come from the seeded generator's amax quantisation: A with one
fp32 scale, B with one per row (output channel), the scales reaching the GEMM
as alpha and the per-column scale of the fused transform, so D approximates
the product of the fp64 draws.  The oracle decodes the 8-bit values exactly,
sums in fp64 and rounds once to bf16; the kernels accumulate the exact 8-bit
products in fp32 on the tensor cores and round once to bf16.  The tolerance
is the bf16 one of gemm_check.py (one bf16 ulp relative, plus fp32
accumulation error growing with sqrt(K) in units of the dequantised
products, which are at most 1 here).  D is pre-filled with NaN.
"""
import numpy as np
import pytest

import oracle
import dense_fp16_gemm_f16_gb300 as g
from dense_fp16_gemm_f16_gb300 import build as gbuild
from dense_fp16_gemm_f16_gb300 import inputs
from gemm_check import bf16_bits_to_f64, check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

TILED = [g.Variant.TILE_2CTA_256x256, g.Variant.TILE_1CTA_128x128, g.Variant.TILE_1CTA_128x256,
         g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_2CTA_512x256, g.Variant.TILE_1CTA_SPLITK]
DT = {"e4m3": g.Dtype.E4M3, "e5m2": g.Dtype.E5M2}


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gbuild.build()
    g.load()
    yield
    g.gemm_f16_nt_check(device=torch.device("cuda"))


def _bf16_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _run(A, B, fmt, variant=g.Variant.AUTO, alpha=1.0, scale_n=None, beta=0.0, C=None, bias=None,
         relu=False, as_float8=False):
    dA, dB = torch.from_numpy(np.ascontiguousarray(A)).cuda(), torch.from_numpy(np.ascontiguousarray(B)).cuda()
    if as_float8:
        tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
        dA, dB = dA.view(tdt), dB.view(tdt)
    D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=torch.bfloat16, device="cuda")
    sc = None if scale_n is None else torch.from_numpy(np.ascontiguousarray(scale_n)).cuda()
    g.gemm_nt_ex(dA, dB, D, dtype=None if as_float8 else DT[fmt], alpha=alpha, beta=beta,
                 C=None if C is None else _bf16_dev(C), bias=None if bias is None else _bf16_dev(bias),
                 activation=g.Activation.RELU if relu else g.Activation.NONE, variant=variant, scale_n=sc)
    g.gemm_f16_nt_check(device=D.device)
    return D.view(torch.int16).cpu().numpy().view(np.uint16)


def _ref(A, B, fmt, sa, sb, **kw):
    return oracle.gemm_ex(A, B, fmt, sa, scale_n=sb, **kw)


# ---------------------------------------------------------------- named workloads
@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("name", ["single_tile_128x128x64", "multi_tile_1024x1024x2048"])
def test_named_workload_full_output(name, fmt):
    w = inputs.WORKLOADS[name]
    A, B, sa, sb = inputs.operands_fp8(w.M, w.N, w.K, w.dist_a, w.dist_b, seed=w.seed, fmt=fmt)
    check_close(_run(A, B, fmt, alpha=sa, scale_n=sb), _ref(A, B, fmt, sa, sb), w.K, f"{name} {fmt}",
                dtype="bf16")


# the ragged workload with K = 4112: 8-bit rows must be whole 16-byte units,
# which 4104 bytes are not
SAMPLED = {"square_8192x8192x8192": (8192, 8192, 8192), "ragged_4000x11000x4112": (4000, 11000, 4112),
           "skinny_16x8192x8192": (16, 8192, 8192)}


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("name", sorted(SAMPLED))
def test_full_size_sampled(name, fmt):
    base = inputs.WORKLOADS[name.replace("4112", "4104")]
    M, N, K = SAMPLED[name]
    A, B, sa, sb = inputs.operands_fp8(M, N, K, base.dist_a, base.dist_b, seed=base.seed, fmt=fmt)
    d = _run(A, B, fmt, alpha=sa, scale_n=sb)
    assert not np.any(np.isnan(bf16_bits_to_f64(d))), name
    rows, cols = inputs.sample_entries(M, N, seed=base.seed + 92, n_random=32768)
    ref = oracle.gemm_ex_entries(A, B, rows, cols, fmt, sa, scale_n=sb)
    check_close(d[rows, cols], ref, K, f"{name} {fmt}", dtype="bf16")


# ---------------------------------------------------------------- every kernel, ragged shapes
SHAPES = [(7, 24, 48), (129, 136, 80), (300, 520, 1008), (513, 256, 4112)]


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("variant", TILED, ids=lambda v: v.name)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_tiled_variants_ragged(variant, shape, fmt):
    M, N, K = shape
    A, B, sa, sb = inputs.operands_fp8(M, N, K, seed=6000 + M + N + K, fmt=fmt)
    check_close(_run(A, B, fmt, variant, alpha=sa, scale_n=sb), _ref(A, B, fmt, sa, sb), K,
                f"{variant.name} {fmt}", dtype="bf16")


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("shape", [(1, 8, 16), (17, 200, 80), (33, 1000, 528), (64, 256, 4112), (16, 1024, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_skinny_ragged(shape, fmt):
    M, N, K = shape
    A, B, sa, sb = inputs.operands_fp8(M, N, K, "normal:1", "normal:1/sqrtK", seed=7000 + M + N + K, fmt=fmt)
    check_close(_run(A, B, fmt, g.Variant.SKINNY_SPLITK, alpha=sa, scale_n=sb), _ref(A, B, fmt, sa, sb), K,
                f"skinny {fmt}", dtype="bf16")


# ---------------------------------------------------------------- exact cases
def _enc(x, fmt):
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    q = torch.from_numpy(np.asarray(x, np.float32)).to(tdt)
    assert np.array_equal(q.double().numpy(), np.asarray(x, np.float64))
    return q.view(torch.uint8).numpy().copy()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_integer_operands_bit_exact(fmt):
    # small integers are exact in both formats; their fp32 sums are exact, so D
    # is the single bf16 rounding of the exact sum on both sides
    rng = np.random.default_rng(31)
    for variant in TILED + [g.Variant.SKINNY_SPLITK]:
        M = 40 if variant == g.Variant.SKINNY_SPLITK else 300
        N, K = 264, 1040
        Ai, Bi = rng.integers(-4, 5, (M, K)), rng.integers(-4, 5, (N, K))
        A, B = _enc(Ai, fmt), _enc(Bi, fmt)
        s = (2.0 ** rng.integers(-3, 4, N)).astype(np.float32)
        got = _run(A, B, fmt, variant, alpha=0.5, scale_n=s)
        want = oracle.gemm_ex(A, B, fmt, 0.5, scale_n=s)
        assert np.array_equal(got, want), variant.name


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_extremes_of_the_format(fmt):
    # the largest finite values and the smallest subnormals, over a long K
    top, tiny = (448.0, 2.0 ** -9) if fmt == "e4m3" else (57344.0, 2.0 ** -16)
    M, N, K = 256, 256, 4096
    rng = np.random.default_rng(32)
    pick = rng.integers(0, 3, (M, K))
    Av = np.where(pick == 0, top, np.where(pick == 1, -top, tiny))
    Bv = np.where(rng.integers(0, 2, (N, K)) == 0, tiny, -top)
    A, B = _enc(Av, fmt), _enc(Bv, fmt)
    got = _run(A, B, fmt, g.Variant.TILE_2CTA_256x256, alpha=2.0 ** -20)
    want = oracle.gemm_ex(A, B, fmt, 2.0 ** -20)
    # the products are exact in fp32 (but sums of +-top^2 and tiny^2 terms are not):
    # the bf16 tolerance with the accumulation term in units of alpha * top^2
    check_close(got, want, K, f"extremes {fmt}", dtype="bf16", scale=2.0 ** -20 * top * top)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fused_epilogue(fmt):
    M, N, K = 520, 776, 1040
    A, B, sa, sb = inputs.operands_fp8(M, N, K, seed=33, fmt=fmt)
    C = inputs.draw_bf16(M, N, "uniform", 34)
    bias = inputs.draw_bf16(1, N, "uniform", 35).ravel()
    for variant in [g.Variant.AUTO, g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_2CTA_512x256]:
        got = _run(A, B, fmt, variant, alpha=sa * 1.5, scale_n=sb, beta=-0.75, C=C, bias=bias, relu=True)
        want = _ref(A, B, fmt, sa * 1.5, sb, beta=-0.75, C=C, bias=bias, relu=True)
        check_close(got, want, K, f"epilogue {variant.name} {fmt}", dtype="bf16", scale=1.5)
    Ms = 24
    got = _run(A[:Ms], B, fmt, g.Variant.SKINNY_SPLITK, alpha=sa, scale_n=sb, beta=2.0, C=C[:Ms], bias=bias)
    check_close(got, _ref(A[:Ms], B, fmt, sa, sb, beta=2.0, C=C[:Ms], bias=bias), K, f"skinny epilogue {fmt}",
                dtype="bf16")


def test_float8_tensors_and_uint8_agree():
    A, B, sa, sb = inputs.operands_fp8(256, 512, 2048, seed=36, fmt="e4m3")
    a = _run(A, B, "e4m3", alpha=sa, scale_n=sb)
    b = _run(A, B, "e4m3", alpha=sa, scale_n=sb, as_float8=True)
    assert np.array_equal(a, b)


def test_deterministic_across_calls():
    A, B, sa, sb = inputs.operands_fp8(1024, 2048, 8192, seed=37, fmt="e4m3")
    for variant in (g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_2CTA_512x256, g.Variant.AUTO):
        first = _run(A, B, "e4m3", variant, alpha=sa, scale_n=sb)
        assert np.array_equal(first, _run(A, B, "e4m3", variant, alpha=sa, scale_n=sb)), variant.name
    first = _run(A[:16], B, "e4m3", g.Variant.SKINNY_SPLITK, alpha=sa, scale_n=sb)
    assert np.array_equal(first, _run(A[:16], B, "e4m3", g.Variant.SKINNY_SPLITK, alpha=sa, scale_n=sb))


def test_empty_sum_with_epilogue():
    M, N = 40, 48
    C = inputs.draw_bf16(M, N, "uniform", 38)
    bias = inputs.draw_bf16(1, N, "uniform", 39).ravel()
    A = np.zeros((M, 0), np.uint8)
    B = np.zeros((N, 0), np.uint8)
    dC, db = _bf16_dev(C), _bf16_dev(bias)
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.gemm_nt_ex(torch.empty((M, 0), dtype=torch.uint8, device="cuda"),
                 torch.empty((N, 0), dtype=torch.uint8, device="cuda"), D, dtype=g.Dtype.E4M3,
                 beta=0.5, C=dC, bias=db, activation=g.Activation.RELU)
    g.gemm_f16_nt_check(device=D.device)
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.gemm_ex(A, B, "e4m3", 1.0, 0.5, C, bias, True))
