"""The seeded input generators (no GPU)."""
import math

import numpy as np

from dense_fp16_gemm_f16_gb300 import inputs


def test_deterministic_and_chunk_independent():
    a = inputs.draw(33, 70, "normal:1/sqrtK", seed=4)
    b = inputs.draw(33, 70, "normal:1/sqrtK", seed=4, chunk=17)
    assert a.dtype == np.float16 and a.flags.c_contiguous and a.shape == (33, 70)
    assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
    c = inputs.draw(33, 70, "uniform", seed=4, chunk=5)
    assert np.array_equal(c.view(np.uint16), inputs.draw(33, 70, "uniform", seed=4).view(np.uint16))
    assert not np.array_equal(a, inputs.draw(33, 70, "normal:1/sqrtK", seed=5))


def test_values_are_rounded_fp64_draws():
    rng = np.random.default_rng(12)
    ref = rng.uniform(-1.0, 1.0, 50 * 9).astype(np.float16).reshape(50, 9)
    assert np.array_equal(inputs.draw(50, 9, "uniform", seed=12).view(np.uint16), ref.view(np.uint16))


def test_distributions():
    u = inputs.draw(256, 1024, "uniform", seed=1).astype(np.float64)
    assert u.min() >= -1 and u.max() <= 1 and abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    n = inputs.draw(256, 4096, "normal:1/sqrtK", seed=3).astype(np.float64)
    assert abs(n.std() * math.sqrt(4096) - 1) < 0.01
    s = inputs.draw(64, 4096, "normal:1", seed=5).astype(np.float64)
    assert abs(s.std() - 1) < 0.02


def test_workloads_table():
    w = inputs.WORKLOADS
    assert [(v.M, v.N, v.K) for v in w.values()] == [
        (128, 128, 64), (1024, 1024, 2048), (8192, 8192, 8192), (4000, 11000, 4104), (16, 8192, 8192)]
    assert w[inputs.HEADLINE].flops == 2 * 8192 ** 3
    assert w["skinny_16x8192x8192"].compulsory_bytes == 134_742_016
    assert w["ragged_4000x11000x4104"].compulsory_bytes == 211_120_000
    A, B = inputs.workload_operands("single_tile_128x128x64")
    assert A.shape == (128, 64) and B.shape == (128, 64)
    A2, _ = inputs.operands(128, 128, 64, seed=1)
    assert np.array_equal(A.view(np.uint16), A2.view(np.uint16))


def test_sample_entries_cover_rows_cols_corners():
    r, c = inputs.sample_entries(100, 60, seed=2, n_rows=3, n_cols=2, n_random=50,
                                 extra_rows=[99], extra_cols=[59])
    assert r.min() >= 0 and r.max() < 100 and c.min() >= 0 and c.max() < 60
    pairs = set(zip(r.tolist(), c.tolist()))
    assert {(0, 0), (0, 59), (99, 0), (99, 59)} <= pairs
    assert all((99, j) in pairs for j in range(60)) and all((i, 59) in pairs for i in range(100))


def test_fp8_operands_scaled_to_the_format():
    torch = __import__("pytest").importorskip("torch")
    for fmt, tdt in (("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)):
        A, B, sa, sb = inputs.operands_fp8(40, 24, 96, "normal:1/sqrtK", "uniform", seed=7, fmt=fmt)
        assert A.dtype == np.uint8 and A.shape == (40, 96) and B.shape == (24, 96)
        assert sb.dtype == np.float32 and sb.shape == (24,)
        A2, B2, sa2, sb2 = inputs.operands_fp8(40, 24, 96, "normal:1/sqrtK", "uniform", seed=7, fmt=fmt)
        assert np.array_equal(A, A2) and np.array_equal(B, B2) and sa == sa2 and np.array_equal(sb, sb2)
        a = torch.from_numpy(A).view(tdt).double().numpy()
        b = torch.from_numpy(B).view(tdt).double().numpy()
        top = inputs.FP8_MAX[fmt]
        assert np.all(np.isfinite(a)) and np.all(np.isfinite(b))
        assert np.abs(a).max() == top                            # the largest draw maps onto the bound
        assert np.all(np.abs(b).max(axis=1) == top)              # per row for B
        # dequantised values follow the fp64 draws to the format's precision
        x = inputs._draw_f64(40, 96, "normal:1/sqrtK", 7)
        y = inputs._draw_f64(24, 96, "uniform", 1007)
        # (half an ulp relative for normals; half the subnormal step absolute)
        rel, sub = (2.0 ** -4, 2.0 ** -10) if fmt == "e4m3" else (2.0 ** -3, 2.0 ** -17)
        sbc = sb[:, None].astype(np.float64)
        assert np.all(np.abs(a * sa - x) <= rel * np.abs(x) + sub * sa * 1.0001)
        assert np.all(np.abs(b * sbc - y) <= rel * np.abs(y) + sub * sbc * 1.0001)
