"""Parity of the bf16 path and the fused epilogue with the CPU oracle (needs a GB300).

D = act(alpha * A·Bᵀ + beta * C + bias[n]) is computed by the oracle in fp64
with one rounding to the output type; the kernels apply it in fp32 to the
fp32 accumulator before their single rounding.  Every kernel variant is run
on ragged shapes with the output pre-filled with NaN, for fp16 and bf16.
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

TILED = [g.Variant.TILE_2CTA_256x256, g.Variant.TILE_1CTA_128x128, g.Variant.TILE_1CTA_128x256,
         g.Variant.TILE_2CTA_SPLITK, g.Variant.TILE_2CTA_512x256, g.Variant.TILE_1CTA_SPLITK]


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gbuild.build()
    g.load()
    yield
    g.gemm_f16_nt_check(device=torch.device("cuda"))


def _dev(x, dtype):
    x = np.ascontiguousarray(x)
    if dtype == "bf16":
        return torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(x).cuda()


def _host(t, dtype):
    if dtype == "bf16":
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def _draw(rows, cols, dtype, seed, dist="uniform", K=None):
    if dtype == "bf16":
        return inputs.draw_bf16(rows, cols, dist, seed, K=K)
    return inputs.draw(rows, cols, dist, seed, K=K)


def _operands(M, N, K, dtype, seed, dist_a="uniform", dist_b="uniform"):
    if dtype == "bf16":
        return inputs.operands_bf16(M, N, K, dist_a, dist_b, seed=seed)
    return inputs.operands(M, N, K, dist_a, dist_b, seed=seed)


def _run_ex(A, B, dtype, variant=g.Variant.AUTO, alpha=1.0, beta=0.0, C=None, bias=None, relu=False,
            in_place=False):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    dA, dB = _dev(A, dtype), _dev(B, dtype)
    dC = None if C is None else _dev(C, dtype)
    db = None if bias is None else _dev(bias, dtype)
    if in_place:
        D = dC
    else:
        D = torch.full((A.shape[0], B.shape[0]), float("nan"), dtype=tdt, device="cuda")
    g.gemm_nt_ex(dA, dB, D, alpha=alpha, beta=beta, C=dC, bias=db,
                 activation=g.Activation.RELU if relu else g.Activation.NONE, variant=variant)
    g.gemm_f16_nt_check(device=D.device)
    return _host(D, dtype)


# ---------------------------------------------------------------- bf16, plain product
@pytest.mark.parametrize("name", ["single_tile_128x128x64", "multi_tile_1024x1024x2048"])
def test_bf16_named_workload_full_output(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.operands_bf16(w.M, w.N, w.K, w.dist_a, w.dist_b, seed=w.seed)
    dA, dB = _dev(A, "bf16"), _dev(B, "bf16")
    D = torch.full((w.M, w.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    g.gemm_bf16_nt(dA, dB, D)
    g.gemm_f16_nt_check(device=D.device)
    check_close(_host(D, "bf16"), oracle.gemm_ex(A, B, "bf16"), w.K, name, dtype="bf16")


@pytest.mark.parametrize("name", ["square_8192x8192x8192", "ragged_4000x11000x4104", "skinny_16x8192x8192"])
def test_bf16_named_workload_sampled(name):
    w = inputs.WORKLOADS[name]
    A, B = inputs.operands_bf16(w.M, w.N, w.K, w.dist_a, w.dist_b, seed=w.seed)
    d = _run_ex(A, B, "bf16")
    rows, cols = inputs.sample_entries(w.M, w.N, seed=w.seed + 91)
    ref = oracle.gemm_ex_entries(A, B, rows, cols, "bf16")
    check_close(d[rows, cols], ref, w.K, name, dtype="bf16")
    assert not np.any(np.isnan(d.view(np.uint16).astype(np.uint32) << 16).view(np.float32)), name


BF16_SHAPES = [(7, 24, 40), (129, 136, 72), (300, 520, 1000), (513, 256, 4104)]


@pytest.mark.parametrize("variant", TILED, ids=lambda v: v.name)
@pytest.mark.parametrize("shape", BF16_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_bf16_tiled_variants_ragged(variant, shape):
    M, N, K = shape
    A, B = inputs.operands_bf16(M, N, K, seed=4000 + M + N + K)
    check_close(_run_ex(A, B, "bf16", variant), oracle.gemm_ex(A, B, "bf16"), K, variant.name, dtype="bf16")


@pytest.mark.parametrize("shape", [(1, 8, 8), (17, 200, 72), (33, 1000, 520), (16, 1024, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_bf16_skinny_ragged(shape):
    M, N, K = shape
    A, B = inputs.operands_bf16(M, N, K, "normal:1", "normal:1/sqrtK", seed=5000 + M + N + K)
    check_close(_run_ex(A, B, "bf16", g.Variant.SKINNY_SPLITK), oracle.gemm_ex(A, B, "bf16"), K, "skinny",
                dtype="bf16")


def test_bf16_closed_forms_exact():
    # bf16 holds every integer up to 256 and 1 + 2^-7; fp32 sums of them are exact
    for variant in TILED + [g.Variant.SKINNY_SPLITK]:
        M = 48 if variant == g.Variant.SKINNY_SPLITK else 272
        ones_a = np.full((M, 256), 0x3F80, np.uint16)
        ones_b = np.full((264, 256), 0x3F80, np.uint16)
        assert np.all(_run_ex(ones_a, ones_b, "bf16", variant) == 0x4380), variant.name   # 256.0
        A = inputs.draw_bf16(M, 128, "uniform", seed=12)
        eye = np.where(np.eye(128, dtype=bool), 0x3F80, 0).astype(np.uint16)
        assert np.array_equal(_run_ex(A, eye, "bf16", variant), A), variant.name


# ---------------------------------------------------------------- fused epilogue
EPI_CASES = [  # alpha, beta, bias, relu
    (1.0, 1.0, True, False),
    (1.5, -0.75, True, True),
    (-2.0, 0.0, False, True),
    (0.5, 2.0, False, False),
]


def _epi_inputs(M, N, dtype, seed):
    C = _draw(M, N, dtype, seed + 1, "uniform")
    bias = _draw(1, N, dtype, seed + 2, "uniform").reshape(N)
    return C, bias


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("variant", TILED, ids=lambda v: v.name)
@pytest.mark.parametrize("shape", [(129, 136, 72), (300, 520, 1000), (513, 256, 4104)],
                         ids=lambda s: "x".join(map(str, s)))
def test_epilogue_tiled(dtype, variant, shape):
    M, N, K = shape
    seed = 6000 + M + N + K
    A, B = _operands(M, N, K, dtype, seed)
    C, bias = _epi_inputs(M, N, dtype, seed)
    for alpha, beta, with_bias, relu in EPI_CASES:
        b = bias if with_bias else None
        d = _run_ex(A, B, dtype, variant, alpha, beta, C, b, relu)
        ref = oracle.gemm_ex(A, B, dtype, alpha, beta, C, b, relu)
        check_close(d, ref, K, f"{variant.name} {dtype} a={alpha} b={beta}", dtype=dtype, scale=abs(alpha))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(5, 136, 64), (33, 1000, 520), (16, 1024, 8192), (64, 4096, 1024)],
                         ids=lambda s: "x".join(map(str, s)))
def test_epilogue_skinny(dtype, shape):
    M, N, K = shape
    seed = 7000 + M + N + K
    A, B = _operands(M, N, K, dtype, seed, "normal:1", "normal:1/sqrtK")
    C, bias = _epi_inputs(M, N, dtype, seed)
    for alpha, beta, with_bias, relu in EPI_CASES:
        b = bias if with_bias else None
        d = _run_ex(A, B, dtype, g.Variant.SKINNY_SPLITK, alpha, beta, C, b, relu)
        ref = oracle.gemm_ex(A, B, dtype, alpha, beta, C, b, relu)
        check_close(d, ref, K, f"skinny {dtype} a={alpha} b={beta}", dtype=dtype, scale=abs(alpha))


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("shape", [(1000, 1000, 640), (512, 2048, 8192), (16, 8192, 8192)],
                         ids=lambda s: "x".join(map(str, s)))
def test_epilogue_auto_plan(dtype, shape):
    # whatever the planner picks (split-K, tiled, skinny) applies the epilogue
    M, N, K = shape
    seed = 8000 + M + N + K
    A, B = _operands(M, N, K, dtype, seed)
    C, bias = _epi_inputs(M, N, dtype, seed)
    d = _run_ex(A, B, dtype, g.Variant.AUTO, 0.75, 0.5, C, bias, True)
    rows, cols = inputs.sample_entries(M, N, seed=seed)
    ref = oracle.gemm_ex_entries(A, B, rows, cols, dtype, 0.75, 0.5, C, bias, True)
    check_close(d[rows, cols], ref, K, f"auto {dtype}", dtype=dtype)


@pytest.mark.parametrize("variant", TILED + [g.Variant.SKINNY_SPLITK], ids=lambda v: v.name)
def test_epilogue_in_place(variant):
    # C == D: each element of C is read before its own output is written
    M = 40 if variant == g.Variant.SKINNY_SPLITK else 300
    N, K = 520, 1000
    A, B = inputs.operands(M, N, K, seed=9)
    C, bias = _epi_inputs(M, N, "f16", 9)
    d = _run_ex(A, B, "f16", variant, 1.0, -1.0, C.copy(), bias, False, in_place=True)
    check_close(d, oracle.gemm_ex(A, B, "f16", 1.0, -1.0, C, bias, False), K, f"in place {variant.name}")


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_epilogue_k_zero(dtype):
    # the empty sum: D = act(beta * C + bias), exactly rounded from fp32
    M, N = 70, 136
    C, bias = _epi_inputs(M, N, dtype, 11)
    A = np.zeros((M, 0), np.uint16 if dtype == "bf16" else np.float16)
    B = np.zeros((N, 0), A.dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    D = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
    g.gemm_nt_ex(torch.empty((M, 0), dtype=tdt, device="cuda"), torch.empty((N, 0), dtype=tdt, device="cuda"),
                 D, alpha=3.0, beta=-0.5, C=_dev(C, dtype), bias=_dev(bias, dtype), activation=g.Activation.RELU)
    g.gemm_f16_nt_check(device=D.device)
    ref = oracle.gemm_ex(A, B, dtype, 3.0, -0.5, C, bias, True)
    assert np.array_equal(_host(D, dtype).view(np.uint16), np.asarray(ref).view(np.uint16))


def test_identity_epilogue_is_bitwise_plain():
    # alpha = 1, beta = 0, no bias, no activation takes the plain path
    A, B = inputs.operands(300, 520, 1000, seed=12)
    d_plain = _run_ex(A, B, "f16")
    dA, dB = _dev(A, "f16"), _dev(B, "f16")
    D = torch.full((300, 520), float("nan"), dtype=torch.float16, device="cuda")
    g.gemm_f16_nt(dA, dB, D)
    g.gemm_f16_nt_check(device=D.device)
    assert np.array_equal(D.cpu().numpy().view(np.uint16), d_plain.view(np.uint16))


# ---------------------------------------------------------------- per-column scale on 16-bit operands
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("variant", TILED + [g.Variant.SKINNY_SPLITK], ids=lambda v: v.name)
def test_per_column_scale_16bit(variant, dtype):
    # scale_n is not tied to the 8-bit types: D = act(alpha * s[n] * A·Bᵀ + beta * C + bias[n])
    M = 40 if variant == g.Variant.SKINNY_SPLITK else 300
    N, K = 520, 1000
    A, B = _operands(M, N, K, dtype, seed=7100 + M)
    rng = np.random.default_rng(7200 + M)
    s = rng.uniform(0.25, 4.0, N).astype(np.float32)
    C = _draw(M, N, dtype, 7300)
    bias = _draw(1, N, dtype, 7400).reshape(N)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    dA, dB, dC, db = _dev(A, dtype), _dev(B, dtype), _dev(C, dtype), _dev(bias, dtype)
    ds = torch.from_numpy(s).cuda()
    for alpha, beta, with_bias, relu in [(1.0, 0.0, False, False), (0.5, -1.0, True, True)]:
        D = torch.full((M, N), float("nan"), dtype=tdt, device="cuda")
        g.gemm_nt_ex(dA, dB, D, alpha=alpha, beta=beta, C=dC if beta else None, bias=db if with_bias else None,
                     activation=g.Activation.RELU if relu else g.Activation.NONE, variant=variant, scale_n=ds)
        g.gemm_f16_nt_check(device=D.device)
        ref = oracle.gemm_ex(A, B, dtype, alpha, beta, C if beta else None, bias if with_bias else None, relu,
                             scale_n=s)
        check_close(_host(D, dtype), ref, K, f"scale_n {variant.name} {dtype} alpha={alpha}", dtype=dtype, scale=4.0)
