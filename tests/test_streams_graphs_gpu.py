"""Concurrent streams and CUDA-graph capture of the C-ABI calls (needs a GB300).

Every call is asynchronous on its stream and keeps its split-K partials in a
workspace of that stream, so GEMMs on different streams may overlap; and the
launch path (host planning, tensor-map encoding, one cudaLaunchKernelEx with
programmatic serialisation) has nothing a stream capture forbids once a first
call has set the device up and sized the stream's workspace, so the calls can
be recorded into a CUDA graph and replayed on new contents of the same
buffers.  Results are compared with the CPU oracle.
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


@pytest.fixture(scope="module", autouse=True)
def _library():
    assert torch.cuda.is_available(), "these tests need a CUDA GPU"
    gbuild.build()
    g.load()
    yield
    g.gemm_f16_nt_check(device=torch.device("cuda"))


def _f16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bf16_host(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def test_concurrent_streams_own_workspaces():
    # split-K pair tiles on one stream and the small-M kernels on others,
    # enqueued alternately while their kernels overlap: the stream-K small-M
    # kernel keeps fp32 partials and counters in its own stream's workspace
    A1, B1 = inputs.operands(512, 2048, 2048, seed=51)
    A2, B2 = inputs.operands(16, 4096, 4096, "normal:1", "normal:1/sqrtK", seed=52)
    dA1, dB1, dA2, dB2 = _f16(A1), _f16(B1), _f16(A2), _f16(B2)
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    D1 = [torch.full((512, 2048), float("nan"), dtype=torch.float16, device="cuda") for _ in range(2)]
    D2 = [torch.full((16, 4096), float("nan"), dtype=torch.float16, device="cuda") for _ in range(2)]
    D3 = [torch.full((16, 4096), float("nan"), dtype=torch.float16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for i in range(12):
        g.gemm_f16_nt_variant(dA1, dB1, D1[i % 2], variant=g.Variant.TILE_2CTA_SPLITK, stream=s1)
        g.gemm_f16_nt_variant(dA2, dB2, D2[i % 2], variant=g.Variant.SKINNY_SPLITK, stream=s2)
        g.gemm_f16_nt_variant(dA2, dB2, D3[i % 2], variant=g.Variant.SKINNY_STREAMK, stream=s3)
    g.gemm_f16_nt_check(stream=s1)
    g.gemm_f16_nt_check(stream=s2)
    g.gemm_f16_nt_check(stream=s3)
    ref1, ref2 = oracle.gemm(A1, B1), oracle.gemm(A2, B2)
    for d in D1:
        check_close(d.cpu().numpy(), ref1, 2048, "split-K on stream 1")
    for d in D2:
        check_close(d.cpu().numpy(), ref2, 4096, "small-M on stream 2")
    for d in D3:
        check_close(d.cpu().numpy(), ref2, 4096, "stream-K small-M on stream 3")


def test_two_split_k_calls_on_unordered_streams():
    # Two split-K calls, each with as many tiles as one wave of its clusters
    # holds (all pair slots), on two streams with no ordering between them, so
    # the second grid's clusters must wait for SMs the first one holds.  Every
    # cluster sums its own tile's pieces and waits on no other cluster, so both
    # finish, match the oracle, and no wait runs out.
    M, N, K = 1024, 1024, 4096                 # 16 pair tiles, K split over each tile's cluster
    plan = g.gemm_f16_nt_plan(M, N, K, g.Variant.TILE_2CTA_SPLITK)
    assert plan["variant"] == "TILE_2CTA_SPLITK" and plan["k_split"] > 1
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 2 * plan["grid_ctas"] > sms          # together the two grids do not fit at once
    ops = [inputs.operands(M, N, K, seed=60 + i) for i in range(2)]
    dev = [(_f16(a), _f16(b)) for a, b in ops]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    Ds = [torch.full((M, N), float("nan"), dtype=torch.float16, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    for rep in range(3):
        for i in range(2):
            g.gemm_f16_nt_variant(dev[i][0], dev[i][1], Ds[i], variant=g.Variant.TILE_2CTA_SPLITK, stream=streams[i])
    for i in range(2):
        g.gemm_f16_nt_check(stream=streams[i])   # raises on a timeout
    for i, (a, b) in enumerate(ops):
        check_close(Ds[i].cpu().numpy(), oracle.gemm(a, b), K, f"split-K on unordered stream {i}")


def test_cuda_graph_capture_and_replay():
    s = torch.cuda.Stream()
    # the buffers the graph is recorded on
    shapes = {"tiled": (300, 520, 1000), "splitk": (512, 2048, 2048), "skinny": (24, 2048, 4096)}
    A = {k: torch.empty((m, kk), dtype=torch.float16, device="cuda") for k, (m, n, kk) in shapes.items()}
    B = {k: torch.empty((n, kk), dtype=torch.float16, device="cuda") for k, (m, n, kk) in shapes.items()}
    D = {k: torch.empty((m, n), dtype=torch.float16, device="cuda") for k, (m, n, kk) in shapes.items()}
    variants = {"tiled": g.Variant.AUTO, "splitk": g.Variant.TILE_2CTA_SPLITK, "skinny": g.Variant.SKINNY_SPLITK}
    M8, N8, K8 = 260, 776, 1040
    A8 = torch.empty((M8, K8), dtype=torch.uint8, device="cuda")
    B8 = torch.empty((N8, K8), dtype=torch.uint8, device="cuda")
    S8 = torch.empty((N8,), dtype=torch.float32, device="cuda")
    D8 = torch.empty((M8, N8), dtype=torch.bfloat16, device="cuda")
    alpha8 = 0.5                                                  # fixed in the recorded call
    Ce = torch.empty((300, 520), dtype=torch.float16, device="cuda")
    be = torch.empty((520,), dtype=torch.float16, device="cuda")
    De = torch.empty((300, 520), dtype=torch.float16, device="cuda")

    def calls():
        for k in shapes:
            g.gemm_f16_nt_variant(A[k], B[k], D[k], variant=variants[k], stream=s)
        g.gemm_nt_ex(A8, B8, D8, dtype=g.Dtype.E4M3, alpha=alpha8, scale_n=S8, stream=s)
        g.gemm_nt_ex(A["tiled"], B["tiled"], De, alpha=1.5, beta=-0.5, C=Ce, bias=be,
                     activation=g.Activation.RELU, stream=s)

    # a first, uncaptured run sets the device up and sizes the stream's workspace
    with torch.cuda.stream(s):
        calls()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        calls()
    for rep in range(3):
        host = {}
        for k, (m, n, kk) in shapes.items():
            dist_a = "normal:1" if k == "skinny" else "uniform"
            a, b = inputs.operands(m, n, kk, dist_a, "uniform", seed=600 + 10 * rep + len(k))
            host[k] = (a, b)
            A[k].copy_(_f16(a)); B[k].copy_(_f16(b))
            D[k].fill_(float("nan"))
        a8, b8, _, sb = inputs.operands_fp8(M8, N8, K8, seed=700 + rep, fmt="e4m3")
        A8.copy_(torch.from_numpy(a8).cuda()); B8.copy_(torch.from_numpy(b8).cuda())
        S8.copy_(torch.from_numpy(sb).cuda())
        D8.fill_(float("nan"))
        c = inputs.draw(300, 520, "uniform", 800 + rep)
        bias = inputs.draw(1, 520, "uniform", 900 + rep).reshape(520)
        Ce.copy_(_f16(c)); be.copy_(_f16(bias)); De.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        g.gemm_f16_nt_check(stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        for k, (m, n, kk) in shapes.items():
            check_close(D[k].cpu().numpy(), oracle.gemm(*host[k]), kk, f"graph replay {rep} {k}")
        check_close(_bf16_host(D8), oracle.gemm_ex(a8, b8, "e4m3", alpha8, scale_n=sb), K8,
                    f"graph replay {rep} e4m3", dtype="bf16")
        check_close(De.cpu().numpy(), oracle.gemm_ex(*host["tiled"], "f16", 1.5, -0.5, c, bias, True), 1000,
                    f"graph replay {rep} epilogue", scale=1.5)
