"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: numpy's float16
conversions (an independent library routine), exact integer arithmetic,
closed forms, and an independent double-precision matmul (torch on the CPU).
Each ``pin_*`` function raises AssertionError when the oracle under test
disagrees; ``test_planted_mistakes_are_caught`` builds broken copies of the
C source and checks that at least one pin fails for each.
"""
import os
import re

import numpy as np
import pytest

import oracle
from dense_fp16_gemm_f16_gb300 import inputs

ALL_BITS = np.arange(65536, dtype=np.uint16)
FINITE = ALL_BITS[(ALL_BITS & 0x7C00) != 0x7C00]


def _bits(x16):
    return np.ascontiguousarray(x16).view(np.uint16)


def _same_f16(a, b):
    """Bitwise equality of float16 arrays, with any NaN equal to any NaN."""
    a, b = np.asarray(a, np.float16), np.asarray(b, np.float16)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(_bits(a)[~na], _bits(b)[~nb])


# --------------------------------------------------------------------------
# pins on the fp16 decode / encode (IEEE 754 binary16)
# --------------------------------------------------------------------------
def pin_decode(o):
    d = o.f16_to_f64(ALL_BITS)
    ref = ALL_BITS.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(d), np.isnan(ref))
    assert np.array_equal(d[~np.isnan(d)], ref[~np.isnan(ref)])
    # spot values from the format definition
    assert o.f16_to_f64(np.array([0x0001], np.uint16))[0] == 2.0 ** -24
    assert o.f16_to_f64(np.array([0x0400], np.uint16))[0] == 2.0 ** -14
    assert o.f16_to_f64(np.array([0x3C00], np.uint16))[0] == 1.0
    assert o.f16_to_f64(np.array([0x7BFF], np.uint16))[0] == 65504.0
    assert o.f16_to_f64(np.array([0xFC00], np.uint16))[0] == -np.inf


def pin_roundtrip(o):
    back = o.f64_to_f16(o.f16_to_f64(FINITE))
    assert np.array_equal(_bits(back), FINITE)
    nan_bits = ALL_BITS[((ALL_BITS & 0x7C00) == 0x7C00) & ((ALL_BITS & 0x3FF) != 0)]
    assert np.all(np.isnan(o.f64_to_f16(o.f16_to_f64(nan_bits))))


def pin_midpoints(o):
    pos = np.arange(0x0000, 0x7BFF, dtype=np.uint16)        # h and h+1 both finite
    lo = pos.view(np.float16).astype(np.float64)
    hi = (pos + 1).view(np.float16).astype(np.float64)
    mid = (lo + hi) / 2                                      # exact in fp64
    even = np.where(pos % 2 == 0, pos, pos + 1).astype(np.uint16)
    assert np.array_equal(_bits(o.f64_to_f16(mid)), even)
    assert np.array_equal(_bits(o.f64_to_f16(-mid)), even | 0x8000)
    above = np.nextafter(mid, np.inf)
    below = np.nextafter(mid, -np.inf)
    assert np.array_equal(_bits(o.f64_to_f16(above)), (pos + 1).astype(np.uint16))
    assert np.array_equal(_bits(o.f64_to_f16(below)), pos)
    # top of the range: 65504 is odd (2047 * 32); the tie at 65520 goes to 65536 = inf
    f = o.f64_to_f16(np.array([65519.999, 65520.0, -65520.0, 65536.0, 1e300, 2.0 ** 16]))
    assert f[0] == 65504 and np.isposinf(f[1]) and np.isneginf(f[2])
    assert np.isposinf(f[3]) and np.isposinf(f[4]) and np.isposinf(f[5])


def pin_specials(o):
    x = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, 2.0 ** -24, 2.0 ** -25,
                  3 * 2.0 ** -26, 3 * 2.0 ** -25, 2.0 ** -25 * (1 + 2.0 ** -40), 5e-324, -5e-324,
                  1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11], dtype=np.float64)
    expect = [0x0000, 0x8000, 0x7C00, 0xFC00, None, 0x0001, 0x0000, 0x0001, 0x0002, 0x0001,
              0x0000, 0x8000, 0x3C00, 0x3C02]
    got = _bits(o.f64_to_f16(x))
    for g, e, xv in zip(got, expect, x):
        if e is None:
            assert (g & 0x7C00) == 0x7C00 and (g & 0x3FF) != 0, xv
        else:
            assert g == e, (xv, hex(g), hex(e))


def pin_encode_vs_numpy(o, n=1_000_000, seed=11):
    rng = np.random.default_rng(seed)
    mag = np.ldexp(rng.uniform(1.0, 2.0, n), rng.integers(-40, 18, n))
    x = np.where(rng.integers(0, 2, n) == 1, -mag, mag)
    # also exact fp16 midpoints and their neighbours, where the rounding rule matters
    h = rng.integers(0, 0x7BFF, 20000).astype(np.uint16)
    m = (h.view(np.float16).astype(np.float64) + (h + 1).view(np.float16).astype(np.float64)) / 2
    x = np.concatenate([x, m, np.nextafter(m, 0), np.nextafter(m, np.inf)])
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16)
    assert _same_f16(o.f64_to_f16(x), ref)


# --------------------------------------------------------------------------
# pins on the GEMM
# --------------------------------------------------------------------------
def _int_operands(rng, M, N, K, lim=8):
    Ai = rng.integers(-lim, lim + 1, (M, K))
    Bi = rng.integers(-lim, lim + 1, (N, K))
    return Ai, Bi, Ai.astype(np.float16), Bi.astype(np.float16)


def pin_bruteforce_integers(o, seed=5):
    """Small-integer fp16 inputs: the exact D is an int64 matmul."""
    rng = np.random.default_rng(seed)
    shapes = [(m, n, k) for m in range(1, 10) for n in range(1, 10) for k in range(1, 10)]
    shapes += [tuple(int(v) for v in rng.integers(1, 34, 3)) for _ in range(40)]
    for (M, N, K) in shapes:
        Ai, Bi, A, B = _int_operands(rng, M, N, K)
        exact = Ai @ Bi.T                      # |entries| <= 33*64, exact in int64
        D = o.gemm(A, B, nthreads=1)
        assert _same_f16(D, exact.astype(np.float16)), (M, N, K)


def pin_fp64_sums_vs_exact(o, seed=6):
    """fp16 values are multiples of 2^-24, so 2^48·D is an exact int64 sum for
    |a|,|b| <= 1 and K <= 4096.  The oracle's fp64 sum must sit within the
    fp64 summation bound K·2^-53·Σ|a·b| of it (fp32 accumulation would not)."""
    rng = np.random.default_rng(seed)
    for (M, N, K) in [(4, 5, 4096), (7, 3, 1000), (16, 16, 257)]:
        A = rng.uniform(-1, 1, (M, K)).astype(np.float16)
        B = rng.uniform(-1, 1, (N, K)).astype(np.float16)
        Ai = (A.astype(np.float64) * 2.0 ** 24).astype(np.int64)
        Bi = (B.astype(np.float64) * 2.0 ** 24).astype(np.int64)
        assert np.array_equal(Ai.astype(np.float64) * 2.0 ** -24, A.astype(np.float64))
        exact = Ai @ Bi.T                      # units of 2^-48, < 2^60
        absdot = np.abs(Ai) @ np.abs(Bi).T
        D, S = o.gemm(A, B, nthreads=2, want_sums=True)
        err = np.abs(S * 2.0 ** 48 - exact.astype(np.float64))
        bound = K * 2.0 ** -53 * absdot.astype(np.float64) + 1.0
        assert np.all(err <= bound), float(np.max(err / bound))
        # the fp16 result is the once-rounded fp64 sum
        assert _same_f16(D, S.astype(np.float16))


def pin_single_rounding(o):
    """D is rounded once, from the wide sum.  With a = (1, 2^-11, 2^-15) and
    b = (1, 1, 2^-15) the sum is 1 + 2^-11 + 2^-30: just above the fp16
    midpoint between 1 and 1 + 2^-10, so it rounds up to 0x3C01.  Rounding
    through fp32 first would lose the 2^-30 and land on the tie (-> 0x3C00)."""
    A = np.array([[1.0, 2.0 ** -11, 2.0 ** -15]], np.float16)
    B = np.array([[1.0, 1.0, 2.0 ** -15], [1.0, 1.0, 0.0], [-1.0, -1.0, -(2.0 ** -15)]], np.float16)
    D = o.gemm(A, B)
    assert list(_bits(D)[0]) == [0x3C01, 0x3C00, 0xBC01]


def pin_closed_forms(o, seed=7):
    rng = np.random.default_rng(seed)
    # all ones: D = K, exact in fp16 for every K used by the named workloads
    for K in (64, 2048, 4104, 8192):
        A = np.ones((3, K), np.float16)
        B = np.ones((5, K), np.float16)
        D = o.gemm(A, B)
        assert np.all(D.astype(np.float64) == K), K
    # identity B (N = K): D = A
    K = 40
    A = rng.uniform(-1, 1, (9, K)).astype(np.float16)
    D = o.gemm(A, np.eye(K, dtype=np.float16))
    assert _same_f16(D, A)
    # a permutation B: D = A with its columns permuted
    perm = rng.permutation(K)
    P = np.zeros((K, K), np.float16)
    P[np.arange(K), perm] = 1
    assert _same_f16(o.gemm(A, P), A[:, perm])
    # rank 1: A = u aᵀ, B = v bᵀ with power-of-two entries -> D = (a·b) u vᵀ
    K = 24
    pw = lambda n: (rng.choice([-1.0, 1.0], n) * np.ldexp(1.0, rng.integers(-3, 3, n)))  # noqa: E731
    u, v, a, b = pw(6), pw(7), pw(K), pw(K)
    A = np.outer(u, a).astype(np.float16)
    B = np.outer(v, b).astype(np.float16)
    assert np.array_equal(A.astype(np.float64), np.outer(u, a))
    expect = (a @ b) * np.outer(u, v)        # every term is a power of two: exact
    assert _same_f16(o.gemm(A, B), expect.astype(np.float16))
    # zero blocks zero the matching rows / columns of D; the rest is untouched
    A = rng.uniform(-1, 1, (10, 32)).astype(np.float16)
    B = rng.uniform(-1, 1, (12, 32)).astype(np.float16)
    full = o.gemm(A, B)
    A0, B0 = A.copy(), B.copy()
    A0[2:5] = 0
    B0[7:] = 0
    D0 = o.gemm(A0, B0)
    assert np.all(D0[2:5] == 0) and np.all(D0[:, 7:] == 0)
    keep = np.ones(10, bool)
    keep[2:5] = False
    assert _same_f16(D0[keep][:, :7], full[keep][:, :7])
    # swapping the roles of A and B transposes D (D = A·Bᵀ  =>  Dᵀ = B·Aᵀ)
    assert _same_f16(o.gemm(B, A), full.T)
    # an all-zero K range contributes nothing: D(A,B) == D(A[:, :16], B[:, :16])
    A1, B1 = A.copy(), B.copy()
    A1[:, 16:] = 0
    assert _same_f16(o.gemm(A1, B1), o.gemm(A[:, :16], B[:, :16]))


ALL_PINS = [pin_decode, pin_roundtrip, pin_midpoints, pin_specials, pin_encode_vs_numpy,
            pin_bruteforce_integers, pin_fp64_sums_vs_exact, pin_single_rounding,
            pin_closed_forms]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_impl):
    pin(oracle_impl)


def test_entries_rows_and_full_agree(oracle_impl):
    A, B = inputs.operands(37, 29, 70, seed=21)
    full = oracle_impl.gemm(A, B)
    rows, cols = inputs.sample_entries(37, 29, seed=3, n_rows=2, n_cols=2, n_random=300)
    ent = oracle_impl.gemm_entries(A, B, rows, cols)
    assert _same_f16(ent, full[rows, cols])
    part = oracle_impl.gemm_rows(A, B, 5, 17)
    assert _same_f16(part, full[5:17])
    # threading does not change any result
    assert _same_f16(oracle_impl.gemm(A, B, nthreads=1), oracle_impl.gemm(A, B, nthreads=7))


def test_cross_check_torch_double(oracle_impl):
    """An independent double matmul agrees to fp64 rounding (sums) and to 1 ulp (fp16)."""
    torch = pytest.importorskip("torch")
    A, B = inputs.operands(33, 65, 300, "normal:1", "normal:1/sqrtK", seed=9)
    D, S = oracle_impl.gemm(A, B, want_sums=True)
    T = (torch.from_numpy(A).double() @ torch.from_numpy(B).double().T).numpy()
    absdot = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64)).T
    assert np.all(np.abs(S - T) <= 300 * 2.0 ** -52 * absdot)
    ulp = np.abs(_bits(D).astype(np.int32) - _bits(T.astype(np.float16)).astype(np.int32))
    same_sign = np.sign(D.astype(np.float64)) == np.sign(T)
    assert np.all(ulp[same_sign] <= 1)


def test_rejects_bad_arguments(oracle_impl):
    A = np.zeros((2, 3), np.float16)
    B = np.zeros((4, 3), np.float16)
    with pytest.raises(ValueError):
        oracle_impl.gemm_entries(A, B, [2], [0])
    with pytest.raises(ValueError):
        oracle_impl.gemm_entries(A, B, [0], [4])
    with pytest.raises(ValueError):
        oracle_impl.gemm(A, np.zeros((4, 5), np.float16))
    with pytest.raises(TypeError):
        oracle_impl.gemm(A.astype(np.float32), B)


def test_empty_shapes(oracle_impl):
    # K = 0: the empty sum, D = 0 everywhere
    D = oracle_impl.gemm(np.zeros((3, 0), np.float16), np.zeros((4, 0), np.float16))
    assert D.shape == (3, 4) and np.all(D == 0) and not np.any(np.signbit(D))
    D = oracle_impl.gemm(np.zeros((0, 5), np.float16), np.zeros((4, 5), np.float16))
    assert D.shape == (0, 4)


# --------------------------------------------------------------------------
# planted mistakes: each broken copy of the C file must fail some pin
# --------------------------------------------------------------------------
MUTANTS = {
    "dropped_last_k_term": ("for (int64_t k = 0; k < K; ++k) acc +=",
                            "for (int64_t k = 0; k + 1 < K; ++k) acc +="),
    "wrong_sign": ("acc += dec[a_row[k]] * dec[b_row[k]]", "acc -= dec[a_row[k]] * dec[b_row[k]]"),
    "b_row_indexed_by_m": ("j->B + n * j->K", "j->B + m * j->K"),
    "a_and_b_swapped_row_index": ("j->A + m * j->K, j->B + n * j->K",
                                  "j->A + n * j->K, j->B + m * j->K"),
    "fp32_accumulator": ("double acc = 0.0;", "float acc = 0.0f;"),
    "ties_away_from_zero": ("(rem == half && (n & 1))", "(rem == half)"),
    "truncating_round": ("if (rem > half || (rem == half && (n & 1))) n += 1;", ";"),
    "decode_bias_off_by_one": ("expo - 25);", "expo - 24);"),
    "subnormals_flushed": ("v = ldexp((double)frac, -24);", "v = 0.0;"),
    "overflow_threshold": ("if (E >= 16) return sign | 0x7C00u;",
                           "if (E >= 15) return sign | 0x7C00u;"),
    "double_rounding_via_fp32": ("if (j->out) j->out[i] = f16_encode(acc);",
                                 "if (j->out) j->out[i] = f16_encode((double)(float)acc);"),
}


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes_are_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(oracle.SOURCE).read()
    assert old in src, f"mutation anchor for {name} no longer in the source"
    mutated = src.replace(old, new)
    if name == "double_rounding_via_fp32":
        mutated = mutated.replace("if (j->out) j->out[idx] = f16_encode(acc);",
                                  "if (j->out) j->out[idx] = f16_encode((double)(float)acc);")
    path = tmp_path / "mutant.c"
    path.write_text(mutated)
    lib = oracle.compile_source(str(path), str(tmp_path / f"libmutant_{re.sub('[^a-z]', '', name)}.so"))
    mutant = oracle.Oracle(lib)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {name!r}"
