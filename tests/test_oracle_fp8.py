"""Pins for the oracle's 8-bit operand types and its per-column scale (no GPU).

The GEMM blog post lists FP8 in two layouts, E4M3 and E5M2 (section 2.2),
and quantises weights with one fp32 scale per output channel and activations
with one per tensor (section 4.2).  The decoders are checked exhaustively
against torch's own float8_e4m3fn / float8_e5m2 conversions (an independent
library routine) and at the values the formats' definitions fix (448 is the
bound the blog post's quantisation step scales to); the GEMM against exact
arithmetic on small integers, powers of two and sums too large for fp16.
Broken copies of the C source must each fail at least one pin.
"""
import re

import numpy as np
import pytest

import oracle

torch = pytest.importorskip("torch")

CODES = np.arange(256, dtype=np.uint8)


def _torch_decode(bits, fmt):
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    return torch.from_numpy(np.ascontiguousarray(bits)).view(tdt).double().numpy()


def _torch_encode(x, fmt):
    """8-bit bit patterns of values exact in that format."""
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    x = np.asarray(x, dtype=np.float64)
    q = torch.from_numpy(x.astype(np.float32)).to(tdt)
    assert np.array_equal(q.double().numpy(), x), "value not exact in the 8-bit format"
    return q.view(torch.uint8).numpy().copy()


def _bf16(x):
    """bf16 bits of values exact in fp32, rounded by torch (nearest, ties to even)."""
    x = np.asarray(x, dtype=np.float64)
    assert np.array_equal(x.astype(np.float32).astype(np.float64), x)
    return torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# --------------------------------------------------------------------------- decoders
def pin_e4m3_decode(o):
    d, ref = o.e4m3_to_f64(CODES), _torch_decode(CODES, "e4m3")
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(d[~np.isnan(d)], ref[~np.isnan(ref)])
    v = o.e4m3_to_f64(np.array([0x7E, 0x01, 0x08, 0x38, 0x7F, 0xFE, 0x80], np.uint8))
    assert v[0] == 448.0 and v[1] == 2.0 ** -9 and v[2] == 2.0 ** -6 and v[3] == 1.0
    assert np.isnan(v[4]) and v[5] == -448.0 and v[6] == 0.0 and np.signbit(v[6])
    assert np.isnan(d).sum() == 2                              # S.1111.111 only: no infinities


def pin_e5m2_decode(o):
    d, ref = o.e5m2_to_f64(CODES), _torch_decode(CODES, "e5m2")
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(d[~np.isnan(d)], ref[~np.isnan(ref)])
    v = o.e5m2_to_f64(np.array([0x7B, 0x7C, 0x01, 0x3C, 0x04, 0xFC], np.uint8))
    assert list(v) == [57344.0, np.inf, 2.0 ** -16, 1.0, 2.0 ** -14, -np.inf]
    assert np.isnan(d).sum() == 6


# --------------------------------------------------------------------------- GEMM
def pin_f8_integers(o, seed=21):
    rng = np.random.default_rng(seed)
    for fmt in oracle.FP8:
        for (M, N, K) in [(3, 5, 7), (9, 4, 32), (6, 11, 33)]:
            Ai, Bi = rng.integers(-4, 5, (M, K)), rng.integers(-4, 5, (N, K))
            Ci, bi = rng.integers(-4, 5, (M, N)), rng.integers(-4, 5, N)
            A, B = _torch_encode(Ai, fmt), _torch_encode(Bi, fmt)
            C, b = _bf16(Ci), _bf16(bi)
            S = (Ai @ Bi.T).astype(np.float64)
            for alpha, beta, relu in [(1.0, 0.0, False), (2.0, 1.0, False), (-0.5, -2.0, True)]:
                want = alpha * S + beta * Ci + bi[None, :]
                if relu:
                    want = np.where(want < 0, 0.0, want)
                got = oracle._gemm_ex(o, A, B, fmt, alpha, beta, C, b, relu)
                assert np.array_equal(got, _bf16(want)), (fmt, M, N, K, alpha)


def pin_f8_scale_per_column(o, seed=22):
    # a non-square D: the scale must follow the column n (the row of B)
    rng = np.random.default_rng(seed)
    M, N, K = 3, 6, 16
    Ai, Bi = rng.integers(-3, 4, (M, K)), rng.integers(-3, 4, (N, K))
    s = np.array([0.5, 3.0, 0.75, 2.0 ** -10, 5.0, 1.25], np.float32)
    S = (Ai @ Bi.T).astype(np.float64)
    for fmt in oracle.FP8:
        A, B = _torch_encode(Ai, fmt), _torch_encode(Bi, fmt)
        got = oracle._gemm_ex(o, A, B, fmt, 0.25, 0.0, None, None, False, scale_n=s)
        assert np.array_equal(got, _bf16(0.25 * s.astype(np.float64)[None, :] * S)), fmt
    # the same scale on fp16 operands
    got = oracle._gemm_ex(o, Ai.astype(np.float16), Bi.astype(np.float16), "f16", 1.0, 0.0, None, None, False,
                          scale_n=s)
    assert np.array_equal(got.astype(np.float64), (s.astype(np.float64)[None, :] * S).astype(np.float16))


def pin_f8_wide_sums(o):
    # products and sums far beyond the 8-bit range (and fp16's) come out in bf16
    K = 4
    for fmt, top in (("e4m3", 448.0), ("e5m2", 57344.0)):
        A = _torch_encode(np.full((2, K), top), fmt)
        B = _torch_encode(np.full((3, K), -top), fmt)
        got = oracle._gemm_ex(o, A, B, fmt, 1.0, 0.0, None, None, False)
        assert np.array_equal(got, _bf16(np.full((2, 3), -K * top * top))), fmt
    # the smallest subnormals: 2^-9 * 2^-9 (E4M3) and 2^-16 * 2^-16 (E5M2)
    for fmt, tiny in (("e4m3", 2.0 ** -9), ("e5m2", 2.0 ** -16)):
        A = _torch_encode(np.array([[tiny, tiny]]), fmt)
        B = _torch_encode(np.array([[tiny, 1.0]]), fmt)
        got = oracle._gemm_ex(o, A, B, fmt, 1.0, 0.0, None, None, False)
        assert np.array_equal(got, _bf16(np.array([[tiny * tiny + tiny]]))), fmt


def pin_f8_single_rounding(o):
    # 1 + 2^-8 is the midpoint between the bf16 neighbours 1 and 1 + 2^-7; a
    # 2^-40 term through C puts the exact value above it: rounded once it goes
    # up, through fp32 it would tie to 1
    for fmt in oracle.FP8:
        A = _torch_encode(np.array([[1.0, 2.0 ** -8]]), fmt)
        B = _torch_encode(np.array([[1.0, 1.0]]), fmt)
        C = _bf16(np.array([[2.0 ** -40]]))
        assert oracle._gemm_ex(o, A, B, fmt, 1.0, 1.0, C, None, False)[0, 0] == 0x3F81, fmt


def pin_f8_nan_operand(o):
    # the E4M3 NaN code (S.1111.111) and E5M2 infinities reach D
    A = np.array([[0x7F, 0x38]], np.uint8)
    B = np.array([[0x38, 0x38]], np.uint8)
    got = oracle._gemm_ex(o, A, B, "e4m3", 1.0, 0.0, None, None, False)
    assert (got[0, 0] & 0x7F80) == 0x7F80 and (got[0, 0] & 0x7F) != 0
    A = np.array([[0x7C, 0x3C]], np.uint8)
    B = np.array([[0x3C, 0x3C]], np.uint8)
    assert oracle._gemm_ex(o, A, B, "e5m2", 1.0, 0.0, None, None, False)[0, 0] == 0x7F80


FP8_PINS = [pin_e4m3_decode, pin_e5m2_decode, pin_f8_integers, pin_f8_scale_per_column, pin_f8_wide_sums,
            pin_f8_single_rounding, pin_f8_nan_operand]


@pytest.mark.parametrize("pin", FP8_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_impl):
    pin(oracle_impl)


def test_entries_match_rows(oracle_impl):
    rng = np.random.default_rng(23)
    for fmt in oracle.FP8:
        A = rng.integers(0, 256, (12, 48), dtype=np.uint8)
        B = rng.integers(0, 256, (20, 48), dtype=np.uint8)
        for X in (A, B):                                            # finite codes only
            X[~np.isfinite(_torch_decode(X, fmt))] = 0
        s = rng.uniform(0.5, 2.0, 20).astype(np.float32)
        C = _bf16(rng.integers(-8, 9, (12, 20)))
        full = oracle.gemm_ex(A, B, fmt, 0.75, 0.5, C, None, True, scale_n=s)
        r, c = rng.integers(0, 12, 200), rng.integers(0, 20, 200)
        ent = oracle.gemm_ex_entries(A, B, r, c, fmt, 0.75, 0.5, C, None, True, scale_n=s)
        assert np.array_equal(ent, full[r, c])


MUTANTS = {
    "e4m3_decode_bias": ("else v = ldexp((double)(8 + frac), expo - 10);",
                         "else v = ldexp((double)(8 + frac), expo - 9);"),
    "e4m3_no_nan": ("else if (expo == 15 && frac == 7) v = NAN;", "else if (0) v = NAN;"),
    "e4m3_flushed_subnormals": ("if (expo == 0) v = ldexp((double)frac, -9);", "if (expo == 0) v = 0.0;"),
    "e5m2_decode_bias": ("else v = ldexp((double)(4 + frac), expo - 17);",
                         "else v = ldexp((double)(4 + frac), expo - 16);"),
    "e5m2_no_infinity": ("else if (expo == 31) v = frac ? NAN : INFINITY;", "else if (expo == 31) v = NAN;"),
    "scale_ignored": ("const double scale = j->scale_n ? (double)j->scale_n[n] : 1.0;",
                      "const double scale = 1.0;"),
    "scale_by_row": ("const double scale = j->scale_n ? (double)j->scale_n[n] : 1.0;",
                     "const double scale = j->scale_n ? (double)j->scale_n[m] : 1.0;"),
    "f8_out_as_f16": ("j->out[i] = j->dtype == 0 ? f16_encode(v) : bf16_encode(v);",
                      "j->out[i] = j->dtype == 1 ? bf16_encode(v) : f16_encode(v);"),
    "f8_C_decoded_as_f16": ("const double* dec_out = j->dtype == 0 ? decode_table() : decode_bf16_table();",
                            "const double* dec_out = j->dtype == 1 ? decode_bf16_table() : decode_table();"),
    "e5m2_decoded_as_e4m3": ("j->dtype == 2 ? decode_e4m3_table() : decode_e5m2_table();",
                             "decode_e4m3_table();"),
    "f8_double_rounding": ("j->out[i] = j->dtype == 0 ? f16_encode(v) : bf16_encode(v);",
                           "j->out[i] = j->dtype == 0 ? f16_encode(v) : bf16_encode((double)(float)v);"),
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
    for pin in FP8_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"


def test_format_bounds_printed_by_the_pages(oracle_impl):
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "fp8_quantisation_bounds.txt")
    rows = [l.split() for l in open(path) if l.strip() and not l.startswith("#")]
    assert [r[0] for r in rows] == ["e4m3", "e5m2"]
    for fmt, ebits, mbits, top in rows:
        codes = np.arange(256, dtype=np.uint8)
        vals = (oracle_impl.e4m3_to_f64 if fmt == "e4m3" else oracle_impl.e5m2_to_f64)(codes)
        finite = vals[np.isfinite(vals)]
        assert finite.max() == float(top) and finite.min() == -float(top), fmt
        # the layout: 1 + ebits + mbits bits; 2^mbits values per binade above the subnormals
        assert 1 + int(ebits) + int(mbits) == 8
        one = list(vals).index(1.0)
        assert vals[one + 1] - 1.0 == 2.0 ** -int(mbits), fmt
