"""The no-allocation entry point, gemm_f16_nt_noalloc (needs a GB300).

Some callers cannot let a library call cudaMalloc: a framework or serving
engine that has given (nearly) all device memory to its own pool, or code that
must not risk the synchronisation an allocation can cause at that point.  For
them the small-M path can run on one fixed scratch array compiled into the
library instead of a workspace allocated on first use.

This file checks, through the C ABI, on two calls in a row (the second call
finds the array as the first one left it):
  - the output against the CPU oracle, element by element, with D pre-filled
    with NaN so an unwritten element fails, within the tolerance the other
    parity tests use;
  - the output against the existing entry point gemm_f16_nt on the same
    operands, within the same tolerance (gemm_f16_nt runs the column-range
    small-M kernel, the no-allocation entry the stream-K one, so the two
    paths share no kernel);
  - a problem near the array's size limit (M = 64, N = 16384: two partial-sum
    slots per CTA), and that a problem too large for the array is refused.
It sits in a file of its own, named so that pytest collects it last.
"""
import numpy as np
import pytest

import dense_fp16_gemm_f16_gb300 as g
import oracle
from dense_fp16_gemm_f16_gb300 import build as gbuild
from dense_fp16_gemm_f16_gb300 import inputs
from gemm_check import check_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    assert torch.cuda.is_available(), "this test needs a CUDA GPU"
    gbuild.build()
    return g.load()


def _both(lib, A_h, B_h):
    """(D from gemm_f16_nt_noalloc, D from gemm_f16_nt) on the same operands,
    both pre-filled with NaN."""
    M, K = A_h.shape
    N = B_h.shape[0]
    A = torch.from_numpy(A_h).cuda()
    B = torch.from_numpy(B_h).cuda()
    D_new = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    D_old = torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream or None
    assert lib.gemm_f16_nt_noalloc(A.data_ptr(), B.data_ptr(), D_new.data_ptr(), M, N, K, stream) == 0
    assert lib.gemm_f16_nt_check(stream) == 0
    assert lib.gemm_f16_nt(A.data_ptr(), B.data_ptr(), D_old.data_ptr(), M, N, K, stream) == 0
    assert lib.gemm_f16_nt_check(stream) == 0
    return D_new.cpu().numpy(), D_old.cpu().numpy()


@pytest.mark.parametrize("shape", [(16, 8192, 8192), (5, 1024, 4104), (64, 2048, 2048), (64, 16384, 2048)],
                         ids=lambda s: "x".join(map(str, s)))
def test_noalloc_matches_oracle_and_gemm_f16_nt_on_two_calls_in_a_row(lib, shape):
    M, N, K = shape
    if (M, N) == (64, 16384):
        # near the limit: two partial-sum slots per CTA fill most of the array
        plan = g.gemm_f16_nt_plan(M, N, K, g.Variant.SKINNY_STREAMK)
        assert plan["max_tiles_per_cta"] == 2
        assert plan["workspace_bytes"] <= 16 << 20
    for call in (1, 2):
        A, B = inputs.operands(M, N, K, "normal:1", "normal:1/sqrtK", seed=100 * call + M + N)
        d_new, d_old = _both(lib, A, B)
        ref = oracle.gemm(A, B)
        check_close(d_new, ref, K, f"noalloc vs oracle {M}x{N}x{K} call {call}")
        check_close(d_old, ref, K, f"gemm_f16_nt vs oracle {M}x{N}x{K} call {call}")
        check_close(d_new, d_old, K, f"noalloc vs gemm_f16_nt {M}x{N}x{K} call {call}")


def test_noalloc_refuses_what_does_not_fit(lib):
    # arguments are checked before any launch; sizes only, the pointers are not touched
    fake = 0x7F0000000000
    S = g.Status
    # M > 64: only the small-M kernel has a no-allocation form
    assert lib.gemm_f16_nt_noalloc(fake, fake + (1 << 34), fake + (2 << 34), 65, 1024, 1024, None) \
        == S.ERR_INVALID_VALUE
    # 64 rows x 2^20 columns: more partial sums than the 16 MiB array holds
    assert lib.gemm_f16_nt_noalloc(fake, fake + (1 << 34), fake + (2 << 34), 64, 1 << 20, 64, None) \
        == S.ERR_INVALID_VALUE
