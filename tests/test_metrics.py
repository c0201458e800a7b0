"""The throughput definition, pinned to the numbers the pages print (no GPU)."""
import os

from dense_fp16_gemm_f16_gb300 import metrics

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]


def test_tflops_reproduces_the_croqtile_table():
    for kernel, ms, printed in _rows("croqtile_throughput_table.txt"):
        got = metrics.tflops(8192, 8192, 8192, float(ms) * 1e-3)
        # times are printed to ~3 significant digits: allow 0.5 %
        assert abs(got - float(printed)) <= 0.005 * float(printed) + 0.005, (kernel, got, printed)


def test_counts():
    assert metrics.flops(128, 128, 64) == 2_097_152
    assert metrics.flops(4000, 11000, 4104) == 361_152_000_000
    assert metrics.compulsory_bytes(8192, 8192, 8192) == 402_653_184
    assert metrics.compulsory_bytes(16, 8192, 8192) == 134_742_016
    assert abs(metrics.gbs(134_742_016, 20e-6) - 6737.1008) < 1e-6
