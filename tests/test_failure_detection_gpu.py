"""Device-side failure detection, made to fire without a GPU fault (needs a GB300).

Every wait in the kernels is bounded: on expiry it records GEMM_ERR_TIMEOUT
in the device status word and the kernel returns.  The library's self-test
kernel waits, with those same waits, on an mbarrier phase that never
completes and on a counter nothing increments, with a budget of a few
milliseconds; the host must then read the timeout, the word must be cleared,
and the context must still compute correct GEMMs.
"""
import time

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


def test_timeout_is_reported_cleared_and_the_context_survives():
    s = torch.cuda.Stream()
    g.gemm_f16_nt_check(stream=s)                      # start from a clean status word
    t = time.perf_counter()
    g.gemm_selftest_timeout(3000, stream=s)            # two waits of 3 ms each
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt_check(stream=s)
    elapsed = time.perf_counter() - t
    assert e.value.status == g.Status.ERR_TIMEOUT
    assert 0.005 <= elapsed < 5.0, elapsed            # both budgets ran out, and not much more
    g.gemm_f16_nt_check(stream=s)                      # the word was cleared: no error now
    # the context is intact: split-K and small-M GEMMs (which use the re-armed
    # workspace counters) still match the oracle
    for (M, N, K, variant) in [(512, 2048, 2048, g.Variant.TILE_2CTA_SPLITK),
                               (16, 2048, 4096, g.Variant.SKINNY_SPLITK), (300, 520, 1000, g.Variant.AUTO)]:
        A, B = inputs.operands(M, N, K, seed=M + N)
        D = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
        g.gemm_f16_nt_variant(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), D, variant=variant, stream=s)
        g.gemm_f16_nt_check(stream=s)
        check_close(D.cpu().numpy(), oracle.gemm(A, B), K, f"after the timeout: {variant.name}")


def test_selftest_rejects_bad_budgets():
    for bad in (0, -1, 1000001):
        with pytest.raises(g.GemmError) as e:
            g.gemm_selftest_timeout(bad)
        assert e.value.status == g.Status.ERR_INVALID_VALUE
