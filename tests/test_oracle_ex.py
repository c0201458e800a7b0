"""Pins for the oracle's bf16 conversions and its fused-epilogue GEMM (no GPU).

bf16 is checked against torch's own bfloat16 conversions (an independent
library routine), exhaustively where the format is small enough; the
epilogue GEMM against exact arithmetic on small-integer and power-of-two
inputs.  As for the fp16 oracle, broken copies of the C source must each
fail at least one pin.
"""
import re

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

ALL = np.arange(65536, dtype=np.uint16)
FINITE_BF16 = ALL[(ALL & 0x7F80) != 0x7F80]


def _torch_bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).double().numpy()


def _torch_f32_to_bf16(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _same_bits(a, b, nan_mask_a=None):
    return np.array_equal(np.asarray(a, np.uint16), np.asarray(b, np.uint16))


# --------------------------------------------------------------------------- bf16
def pin_bf16_decode(o):
    d = o.bf16_to_f64(ALL)
    ref = _torch_bf16_to_f64(ALL)
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(d[~np.isnan(d)], ref[~np.isnan(ref)])
    assert o.bf16_to_f64(np.array([0x3F80], np.uint16))[0] == 1.0
    assert o.bf16_to_f64(np.array([0x0001], np.uint16))[0] == 2.0 ** -133
    assert o.bf16_to_f64(np.array([0x7F7F], np.uint16))[0] == 255 * 2.0 ** 120


def pin_bf16_roundtrip(o):
    assert np.array_equal(o.f64_to_bf16(o.bf16_to_f64(FINITE_BF16)), FINITE_BF16)
    nan = ALL[((ALL & 0x7F80) == 0x7F80) & ((ALL & 0x7F) != 0)]
    back = o.f64_to_bf16(o.bf16_to_f64(nan))
    assert np.all(((back & 0x7F80) == 0x7F80) & ((back & 0x7F) != 0))


def pin_bf16_midpoints(o):
    pos = np.arange(0, 0x7F7F, dtype=np.uint16)              # h and h + 1 finite
    lo, hi = o.bf16_to_f64(pos), o.bf16_to_f64(pos + 1)
    mid = (lo + hi) / 2                                        # exact in fp64
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint16)
    assert np.array_equal(o.f64_to_bf16(mid), even)
    assert np.array_equal(o.f64_to_bf16(-mid), even | 0x8000)
    assert np.array_equal(o.f64_to_bf16(np.nextafter(mid, np.inf)), (pos + 1).astype(np.uint16))
    assert np.array_equal(o.f64_to_bf16(np.nextafter(mid, -np.inf)), pos)
    top = 255 * 2.0 ** 120
    f = o.f64_to_bf16(np.array([top, top + 2.0 ** 119 * 0.999, top + 2.0 ** 119, 2.0 ** 128, -top - 2.0 ** 119]))
    assert list(f) == [0x7F7F, 0x7F7F, 0x7F80, 0x7F80, 0xFF80]   # the tie at 255.5 * 2^120 goes up to inf


def pin_bf16_vs_torch(o, n=1_000_000, seed=3):
    rng = np.random.default_rng(seed)
    mag = np.ldexp(rng.uniform(1.0, 2.0, n), rng.integers(-140, 128, n))
    x32 = np.where(rng.integers(0, 2, n) == 1, -mag, mag).astype(np.float32)
    x32 = x32[np.isfinite(x32)]
    # values with bits below bf16 precision, exactly representable in fp32 (so
    # torch's fp32 -> bf16 rounding sees the same number the oracle sees)
    assert np.array_equal(o.f64_to_bf16(x32.astype(np.float64)), _torch_f32_to_bf16(x32))


# --------------------------------------------------------------------------- epilogue GEMM
def _exact_round(v, dtype):
    """fp16 / bf16 bits of values that are exact in fp32 (small integers and
    dyadic fractions), rounded by numpy / torch."""
    v = np.asarray(v, dtype=np.float64)
    assert np.array_equal(v.astype(np.float32).astype(np.float64), v)
    if dtype == "f16":
        return v.astype(np.float16).view(np.uint16)
    return _torch_f32_to_bf16(v.astype(np.float32))


def _ops(rng, M, N, K, dtype, lim=4):
    Ai, Bi = rng.integers(-lim, lim + 1, (M, K)), rng.integers(-lim, lim + 1, (N, K))
    Ci, bi = rng.integers(-lim, lim + 1, (M, N)), rng.integers(-lim, lim + 1, N)
    def enc(x):
        return x.astype(np.float16) if dtype == "f16" else _exact_round(x.astype(np.float64), "bf16")
    return Ai, Bi, Ci, bi, enc(Ai), enc(Bi), enc(Ci), enc(bi)


def pin_ex_integers(o, seed=8):
    rng = np.random.default_rng(seed)
    for dtype in ("f16", "bf16"):
        for (M, N, K) in [(3, 5, 7), (9, 4, 16), (6, 11, 33)]:
            Ai, Bi, Ci, bi, A, B, C, b = _ops(rng, M, N, K, dtype)
            S = (Ai @ Bi.T).astype(np.float64)
            for alpha, beta, relu in [(1.0, 0.0, False), (2.0, 1.0, False), (-0.5, -2.0, True), (0.25, 0.5, True)]:
                want = alpha * S + beta * Ci + bi[None, :]
                if relu:
                    want = np.where(want < 0, 0.0, want)
                got = oracle._gemm_ex(o, A, B, dtype, alpha, beta, C, b, relu)
                assert np.array_equal(np.asarray(got).view(np.uint16), _exact_round(want, dtype)), (dtype, M, N, K, alpha)


def pin_ex_identity_is_plain(o, seed=9):
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, (13, 40)).astype(np.float16)
    B = rng.uniform(-1, 1, (17, 40)).astype(np.float16)
    assert np.array_equal(oracle._gemm_ex(o, A, B, "f16", 1.0, 0.0, None, None, False).view(np.uint16),
                          o.gemm(A, B).view(np.uint16))


def pin_ex_single_rounding(o):
    # fp16: 1 + 2^-11 (the midpoint between 1 and 1 + 2^-10) plus a 2^-24 bias is
    # above the midpoint: once-rounded it goes up; through fp32 it would tie to 1
    A = np.array([[1.0, 2.0 ** -11]], np.float16)
    B = np.array([[1.0, 1.0]], np.float16)
    bias = np.array([2.0 ** -24], np.float16)
    assert oracle._gemm_ex(o, A, B, "f16", 1.0, 0.0, None, bias, False).view(np.uint16)[0, 0] == 0x3C01
    # bf16: 1 + 2^-8 is the midpoint between 1 and 1 + 2^-7; + 2^-40 through C
    Ab = _exact_round(np.array([[1.0, 2.0 ** -8]]), "bf16")
    Bb = _exact_round(np.array([[1.0, 1.0]]), "bf16")
    Cb = _exact_round(np.array([[2.0 ** -40]]), "bf16")
    assert oracle._gemm_ex(o, Ab, Bb, "bf16", 1.0, 1.0, Cb, None, False)[0, 0] == 0x3F81


def pin_ex_broadcast_axes(o, seed=10):
    # bias follows the column, C the element: on a non-square D each must land on its own axis
    rng = np.random.default_rng(seed)
    M, N, K = 3, 6, 4
    A = np.zeros((M, K), np.float16)
    B = np.zeros((N, K), np.float16)
    bias = np.arange(N, dtype=np.float16)
    C = (np.arange(M * N).reshape(M, N) % 7).astype(np.float16)
    D = oracle._gemm_ex(o, A, B, "f16", 1.0, 2.0, C, bias, False).astype(np.float64)
    assert np.array_equal(D, 2.0 * C.astype(np.float64) + np.arange(N)[None, :])
    D = oracle._gemm_ex(o, A, B, "f16", 1.0, 0.0, C, None, True).astype(np.float64)   # beta = 0: C unread
    assert np.all(D == 0)


EX_PINS = [pin_bf16_decode, pin_bf16_roundtrip, pin_bf16_midpoints, pin_bf16_vs_torch,
           pin_ex_integers, pin_ex_identity_is_plain, pin_ex_single_rounding, pin_ex_broadcast_axes]


@pytest.mark.parametrize("pin", EX_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_impl):
    pin(oracle_impl)


def test_entries_match_rows(oracle_impl):
    rng = np.random.default_rng(4)
    A = rng.uniform(-1, 1, (12, 50)).astype(np.float16)
    B = rng.uniform(-1, 1, (20, 50)).astype(np.float16)
    C = rng.uniform(-1, 1, (12, 20)).astype(np.float16)
    bias = rng.uniform(-1, 1, 20).astype(np.float16)
    full = oracle.gemm_ex(A, B, "f16", 1.5, -0.75, C, bias, True)
    r, c = rng.integers(0, 12, 200), rng.integers(0, 20, 200)
    ent = oracle.gemm_ex_entries(A, B, r, c, "f16", 1.5, -0.75, C, bias, True)
    assert np.array_equal(ent.view(np.uint16), full[r, c].view(np.uint16))


MUTANTS = {
    "bf16_truncating_round": ("if (rem > half || (rem == half && (n & 1))) n += 1;  /* nearest, ties to even */", ";"),
    "bf16_decode_bias": ("else v = ldexp((double)(128 + frac), expo - 134);", "else v = ldexp((double)(128 + frac), expo - 133);"),
    "bf16_flushed_subnormals": ("if (expo == 0) v = ldexp((double)frac, -133);", "if (expo == 0) v = 0.0;"),
    "beta_sign": ("if (j->C && j->beta != 0.0) v += j->beta *", "if (j->C && j->beta != 0.0) v -= j->beta *"),
    "alpha_scales_C": ("if (j->C && j->beta != 0.0) v += j->beta *", "if (j->C && j->beta != 0.0) v += j->alpha * j->beta *"),
    "bias_dropped": ("if (j->bias) v += dec_out[j->bias[n]];", ";"),
    "relu_inverted": ("if (j->act == 1 && v < 0.0) v = 0.0;", "if (j->act == 1 && v > 0.0) v = 0.0;"),
    "ex_double_rounding": ("j->out[i] = j->dtype == 0 ? f16_encode(v) : bf16_encode(v);",
                           "j->out[i] = j->dtype == 0 ? f16_encode((double)(float)v) : bf16_encode((double)(float)v);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name} no longer in the source"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.compile_source(str(path), str(tmp_path / f"libmutant_{re.sub('[^a-z0-9]', '', name)}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in EX_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"
