"""The C-ABI boundary on the host (no GPU): the library loads, exports every
entry point its header declares, rejects bad arguments before touching a
device, and plans the launch the way the pages' tiling arithmetic says."""
import ctypes
import os
import re

import pytest

import dense_fp16_gemm_f16_gb300 as g
from dense_fp16_gemm_f16_gb300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")
FAKE = 0x7F0000000000  # a 16-byte-aligned address that is never dereferenced here


@pytest.fixture(scope="module")
def lib():
    gbuild.build()
    return g.load()


def _declared_functions():
    names = []
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"GEMM_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_entry_point(lib):
    names = _declared_functions()
    assert "gemm_f16_nt" in names and len(names) >= 5
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_only_declared_symbols_are_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gbuild.LIB_PATH], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm not available")
    exported = sorted(line.split()[-1] for line in out.stdout.splitlines() if line.strip())
    assert exported == _declared_functions()


def test_status_strings(lib):
    for s in g.Status:
        text = g.gemm_status_string(s)
        assert text.startswith("GEMM_") or s == g.Status.OK
    assert "unknown" in g.gemm_status_string(99)


def _call(M, N, K, A=FAKE, B=FAKE + (1 << 32), D=FAKE + (2 << 32), variant=0):
    lib = g.load()
    return lib.gemm_f16_nt_variant(A, B, D, M, N, K, variant, None)


def test_argument_errors_are_returned_before_any_device_call(lib):
    S = g.Status
    assert _call(-1, 8, 8) == S.ERR_INVALID_VALUE
    assert _call(8, -8, 8) == S.ERR_INVALID_VALUE
    assert _call(8, 8, -8) == S.ERR_INVALID_VALUE
    assert _call(2 ** 31, 8, 8) == S.ERR_INVALID_VALUE
    assert _call(8, 8, 8, variant=9) == S.ERR_INVALID_VALUE
    assert _call(65, 8, 8, variant=g.Variant.SKINNY_SPLITK) == S.ERR_INVALID_VALUE
    assert _call(65, 8, 8, variant=g.Variant.SKINNY_STREAMK) == S.ERR_INVALID_VALUE
    # empty problems are a no-op even with NULL pointers
    assert _call(0, 8, 8, A=0, B=0, D=0) == S.OK
    assert _call(8, 0, 8, A=0, B=0, D=0) == S.OK
    # NULL pointers with work to do
    assert _call(8, 8, 8, D=0) == S.ERR_INVALID_VALUE
    assert _call(8, 8, 8, A=0) == S.ERR_INVALID_VALUE
    assert _call(8, 8, 8, B=0) == S.ERR_INVALID_VALUE
    # TMA needs 16-byte row pitches and 16-byte aligned bases
    assert _call(8, 8, 12) == S.ERR_MISALIGNED
    assert _call(8, 12, 8) == S.ERR_MISALIGNED
    assert _call(8, 8, 8, A=FAKE + 2) == S.ERR_MISALIGNED
    assert _call(8, 8, 8, D=FAKE + (2 << 32) + 8) == S.ERR_MISALIGNED
    # D overlapping an operand
    assert _call(64, 64, 64, D=FAKE + 64) == S.ERR_INVALID_VALUE
    assert _call(64, 64, 64, B=FAKE + (2 << 32) + 8192 - 16) == S.ERR_INVALID_VALUE
    # adjacent but not overlapping is fine for validation; on a machine with no
    # GPU the call then fails at the first CUDA call, with a CUDA status
    st = _call(64, 64, 64, A=FAKE, B=FAKE + 64 * 64 * 2, D=FAKE + 2 * 64 * 64 * 2)
    assert st in (S.ERR_CUDA, S.ERR_UNSUPPORTED_DEVICE, S.OK)


def _call_ex(M, N, K, dtype=0, alpha=1.0, beta=0.0, C=None, bias=None, act=0, variant=0,
             A=FAKE, B=FAKE + (1 << 32), D=FAKE + (2 << 32), epilogue=True, scale_n=None):
    lib = g.load()
    epi = g.Epilogue(alpha, beta, C, bias, act, 0, scale_n)
    return lib.gemm_nt_ex(dtype, A, B, D, M, N, K, ctypes.byref(epi) if epilogue else None, variant, None)


def test_epilogue_argument_errors_are_returned_before_any_device_call(lib):
    S = g.Status
    D = FAKE + (2 << 32)
    assert _call_ex(8, 8, 8, dtype=4) == S.ERR_INVALID_VALUE            # unknown element type
    assert _call_ex(8, 8, 8, dtype=-1, epilogue=False) == S.ERR_INVALID_VALUE
    assert _call_ex(8, 8, 8, act=2) == S.ERR_INVALID_VALUE              # unknown activation
    assert _call_ex(8, 8, 8, beta=1.0) == S.ERR_INVALID_VALUE           # beta != 0 needs C
    assert _call_ex(8, 8, 8, beta=1.0, C=FAKE + (3 << 32) + 2) == S.ERR_MISALIGNED
    assert _call_ex(8, 8, 8, bias=FAKE + (3 << 32) + 8) == S.ERR_MISALIGNED
    assert _call_ex(8, 8, 8, beta=1.0, C=D + 16) == S.ERR_INVALID_VALUE  # C partly over D
    assert _call_ex(8, 8, 8, bias=D + 32) == S.ERR_INVALID_VALUE         # bias inside D
    # beta == 0: C is never read, so a misaligned or overlapping C is no error
    assert _call_ex(0, 8, 8, beta=0.0, C=FAKE + 2) == S.OK
    # empty problems stay a no-op with an epilogue
    assert _call_ex(0, 8, 8, beta=1.0, C=FAKE, A=0, B=0, D=0) == S.OK
    assert _call_ex(8, 0, 8, dtype=1, bias=FAKE, A=0, B=0, D=0) == S.OK
    # per-column scales: 16-byte aligned, not inside D
    assert _call_ex(8, 8, 8, scale_n=FAKE + (3 << 32) + 4) == S.ERR_MISALIGNED
    assert _call_ex(8, 8, 8, scale_n=D + 64) == S.ERR_INVALID_VALUE
    # 8-bit operands: rows of K bytes must be whole 16-byte units
    for dt in (g.Dtype.E4M3, g.Dtype.E5M2):
        assert _call_ex(8, 8, 8, dtype=dt) == S.ERR_MISALIGNED
        assert _call_ex(8, 8, 40, dtype=dt, epilogue=False) == S.ERR_MISALIGNED
        assert _call_ex(8, 12, 16, dtype=dt) == S.ERR_MISALIGNED           # D (bf16) rows
        assert _call_ex(0, 8, 8, dtype=dt, A=0, B=0, D=0) == S.OK
        # D may sit right after A (M x K bytes) without overlapping it
        st = _call_ex(64, 64, 64, dtype=dt, A=FAKE, B=FAKE + 64 * 64, D=FAKE + 2 * 64 * 64, epilogue=False)
        assert st in (S.ERR_CUDA, S.ERR_UNSUPPORTED_DEVICE, S.OK)
        assert _call_ex(64, 64, 64, dtype=dt, A=FAKE, B=FAKE + 64 * 64, D=FAKE + 64 * 64 - 16,
                        epilogue=False) == S.ERR_INVALID_VALUE
    # the plain bf16 entry point shares the operand checks
    assert lib.gemm_bf16_nt(FAKE + 2, FAKE + (1 << 32), D, 8, 8, 8, None) == S.ERR_MISALIGNED
    assert lib.gemm_bf16_nt(FAKE, FAKE + (1 << 32), D, 8, 8, 12, None) == S.ERR_MISALIGNED


def test_python_binding_rejects_bad_arguments(lib):
    with pytest.raises(ValueError):
        g.gemm_f16_nt(FAKE, FAKE, FAKE)          # raw pointers without sizes
    with pytest.raises(g.GemmError) as e:
        g.gemm_f16_nt(FAKE, FAKE + 2, FAKE + (2 << 32), 8, 8, 8)
    assert e.value.status == g.Status.ERR_MISALIGNED


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [[int(v) for v in line.split()] for line in f if line.strip() and not line.startswith("#")]


def test_tile_grid_matches_the_pages_examples(lib):
    for M, N, K, mt, nt, tiles in _rows("tile_grid_examples.txt"):
        p = g.gemm_f16_nt_plan(M, N, K, g.Variant.TILE_1CTA_128x128, num_sms=152)
        assert (p["m_tiles"], p["n_tiles"], p["m_tiles"] * p["n_tiles"]) == (mt, nt, tiles)
        assert p["tile_m"] == 128 and p["tile_n"] == 128 and p["tile_k"] == 64


def test_plans_for_the_named_workloads(lib):
    P = lambda *a, **k: g.gemm_f16_nt_plan(*a, num_sms=152, **k)  # noqa: E731
    p = P(8192, 8192, 8192)
    assert p["variant"] == "TILE_2CTA_256x256" and p["cta_group"] == 2
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (32, 32, 128)
    assert p["grid_ctas"] == 152 and p["tmem_cols"] == 512
    # 1024 tiles on 76 pairs: 13 whole rounds (988 tiles), the last 36 tiles cut
    # in halves (72 pieces on 76 pairs) instead of a 14th round of 36 tiles
    assert (p["num_full_tiles"], p["tail_split"]) == (988, 2)
    # at most 12 tile rows (12 x 256 rows x 16 KB = 48 MiB of A) per group: 32 rows in 3 groups of 11
    assert p["group_m"] == 11
    p = P(4000, 11000, 4104)
    # K = 4104: rows are not whole 32-byte sectors, so two MMA consumers per CTA
    # share each staged B tile, 512 x 256 per pair, on all 152 SMs; ragged in
    # M, N and K (the last K block 8 wide)
    assert p["variant"] == "TILE_2CTA_512x256" and p["grid_ctas"] == 152 and p["tile_m"] == 512
    assert (p["m_tiles"], p["n_tiles"], p["k_blocks"]) == (8, 43, 65)
    assert (p["num_full_tiles"], p["tail_split"]) == (304, 1)           # 4 rounds of 76 + 40 tiles whole
    assert p["group_m"] == 8                                            # all of A (32 MiB) in one group
    # rows on 32-byte sectors: the pair kernel with double-buffered accumulators
    q = P(4000, 11000, 4112)
    assert q["variant"] == "TILE_2CTA_256x256"
    assert (q["m_tiles"], q["num_full_tiles"], q["tail_split"], q["group_m"]) == (16, 684, 4, 16)
    # misaligned, but under two rounds of 512 x 256 tiles: the pair kernel
    assert P(2048, 8192, 4104)["variant"] == "TILE_2CTA_256x256"
    p = P(1024, 1024, 2048)
    # 16 pair tiles but a short K loop (32 blocks): 128x256 tiles in quarters
    assert p["variant"] == "TILE_1CTA_128x256" and p["k_split"] == 1
    p = P(512, 2048, 8192)
    # 16 pair tiles and a long K loop: each tile's K loop split over a cluster of
    # 4 pairs (32 K blocks each), 16 clusters of 8 CTAs, no workspace
    assert p["variant"] == "TILE_2CTA_SPLITK" and (p["k_split"], p["grid_ctas"]) == (4, 128)
    assert p["workspace_bytes"] == 0
    p = P(1024, 1024, 2048, variant=g.Variant.TILE_2CTA_SPLITK)        # asked for explicitly: split
    assert p["variant"] == "TILE_2CTA_SPLITK" and p["k_split"] == 4
    p = P(2048, 2048, 2048)
    assert p["variant"] == "TILE_1CTA_128x256" and p["k_split"] == 1    # 64 pair tiles: no split
    p = P(1024, 4096, 4096)
    assert p["variant"] == "TILE_2CTA_256x256"                          # 64 K blocks: the pair kernel
    # split-K asked for where the tiles already fill the GPU: plain pair tiles
    p = P(8192, 8192, 8192, variant=g.Variant.TILE_2CTA_SPLITK)
    assert p["variant"] == "TILE_2CTA_256x256" and p["k_split"] == 1
    p = P(128, 128, 64)
    assert p["variant"] == "TILE_1CTA_128x128" and p["k_blocks"] == 1
    assert (p["tail_split"], p["grid_ctas"]) == (2, 2)
    p = P(16, 8192, 8192)
    # 76 column ranges of 108 columns, each range's K loop in 2 pieces (a
    # cluster of 2 CTAs): all 152 SMs, no workspace
    assert p["variant"] == "SKINNY_SPLITK" and p["tile_m"] == 16
    assert (p["n_tiles"], p["tile_n"], p["k_split"]) == (76, 108, 2)
    assert p["grid_ctas"] == 152 and p["max_tiles_per_cta"] == 1 and p["workspace_bytes"] == 0
    # the stream-K kernel on request: 64 tiles of 128 columns dealt over 152 CTAs
    q = P(16, 8192, 8192, variant=g.Variant.SKINNY_STREAMK)
    assert q["variant"] == "SKINNY_STREAMK" and q["n_tiles"] == 64
    assert q["grid_ctas"] == 152 and q["max_tiles_per_cta"] == 2
    assert q["workspace_bytes"] >= 152 * 2 * 16 * 128 * 4 + 64 * 4
    for v in g.Variant:
        if v in (g.Variant.AUTO,):
            continue
        q = P(64, 256, 1024, variant=v)
        assert q["variant"] == v.name
        assert q["smem_bytes"] <= 232448


def test_skinny_ranges_and_pieces(lib):
    P = lambda *a, **k: g.gemm_f16_nt_plan(*a, num_sms=152, **k)  # noqa: E731
    # one K block: no split; one range per column
    p = P(5, 8, 8)
    assert p["variant"] == "SKINNY_SPLITK" and p["tile_m"] == 16
    assert (p["k_split"], p["n_tiles"], p["tile_n"], p["grid_ctas"]) == (1, 8, 1, 8)
    # short K, few columns: 19 ranges of 54 columns in clusters of 8 (152 ranges of
    # 7 columns would leave the ring mostly empty: too few bytes in flight)
    p = P(33, 1024, 640)
    assert p["tile_m"] == 64 and (p["k_split"], p["n_tiles"], p["tile_n"], p["grid_ctas"]) == (8, 19, 54, 152)
    # very short K: every CTA one range of 14 columns, no split
    p = P(7, 2048, 192)
    assert (p["k_split"], p["n_tiles"], p["tile_n"], p["grid_ctas"]) == (1, 152, 14, 152)
    # narrow B slots: the ring holds 54 K blocks in flight (1 KB of B and 2 KB of A
    # each), launched as stages of 8 blocks
    assert p["stages"] == 54
    # few columns, long K: clusters of 8 pieces, 19 ranges of 54 columns
    p = P(16, 1024, 8192)
    assert (p["k_split"], p["n_tiles"], p["tile_n"], p["grid_ctas"]) == (8, 19, 54, 152)
    # many columns, short K: every CTA owns 4 ranges of 108 columns in turn
    p = P(16, 65536, 64)
    assert (p["k_split"], p["grid_ctas"], p["max_tiles_per_cta"], p["n_tiles"], p["tile_n"]) == (1, 152, 4, 608, 108)
    # ranges never exceed 128 columns, and the split never exceeds the K blocks
    for (M, N, K) in [(1, 8, 64), (64, 16384, 2048), (16, 19456, 8192), (16, 19464, 8192), (7, 2048, 192)]:
        p = P(M, N, K)
        assert p["tile_n"] <= 128 and p["n_tiles"] * p["tile_n"] >= N
        assert p["k_split"] <= p["k_blocks"] and p["grid_ctas"] <= 152
        assert p["grid_ctas"] == (p["n_tiles"] * p["k_split"] if p["k_split"] > 1 else min(p["n_tiles"], 152))


def test_tail_split_minimises_the_last_round(lib):
    # whole rounds first; the remainder is cut into 1, 2 or 4 column pieces,
    # whichever gives the shortest tail (ties keep fewer pieces)
    cases = {  # (M, N) on 76 pairs of 256x256 tiles -> (num_full, split)
        (256 * 76, 256): (76, 1),          # exactly one round
        (256 * 77, 256): (76, 4),          # one tile left: quarters
        (256 * 38, 512): (76, 1),          # 76 tiles
        (256 * 50, 256): (0, 1),           # 50 tiles: halves would still take one round
        (256 * 100, 256): (76, 2),         # 24 left: halves fit in one round (48 <= 76)
    }
    for (M, N), want in cases.items():
        p = g.gemm_f16_nt_plan(M, N, 64, g.Variant.TILE_2CTA_256x256, num_sms=152)
        assert (p["num_full_tiles"], p["tail_split"]) == want, (M, N, p)
        units = p["num_full_tiles"] + (p["m_tiles"] * p["n_tiles"] - p["num_full_tiles"]) * p["tail_split"]
        assert p["grid_ctas"] == 2 * min(units, 76)
    # 128-wide tiles are cut at most in halves (pieces stay >= 64 columns)
    p = g.gemm_f16_nt_plan(128 * 153, 128, 64, g.Variant.TILE_1CTA_128x128, num_sms=152)
    assert (p["num_full_tiles"], p["tail_split"]) == (152, 2)


def test_ksplit_choice(lib):
    P = lambda *a, **k: g.gemm_f16_nt_plan(*a, num_sms=152, **k)  # noqa: E731
    # pieces per tile: at most 4 (clusters of at most 8 CTAs), one wave of
    # clusters (152 SMs: 38 clusters of 2 pairs, 25 of 3, 19 of 4), >= 4 K blocks each
    V = g.Variant.TILE_2CTA_SPLITK
    assert P(256, 256, 64 * 64, variant=V)["k_split"] == 4
    assert P(256, 256, 64 * 12, variant=V)["k_split"] == 3
    assert P(256, 256, 64 * 7, variant=V)["k_split"] == 1                # under 4 K blocks per piece: no split
    q = P(256 * 4, 256 * 5, 64 * 64, variant=V)                           # 20 tiles: 25 clusters of 3 pairs fit
    assert q["k_split"] == 3 and q["grid_ctas"] == 2 * 20 * 3
    q = P(256 * 8, 256 * 5, 64 * 64, variant=V)                           # 40 tiles: too many for one wave
    assert q["variant"] == "TILE_2CTA_256x256" and q["k_split"] == 1
    # single CTAs: up to 8 pieces per tile (clusters of up to 8 CTAs; 152 SMs: 152 / S clusters)
    V1 = g.Variant.TILE_1CTA_SPLITK
    assert P(128, 256, 64 * 64, variant=V1)["k_split"] == 8
    assert P(128, 256, 64 * 20, variant=V1)["k_split"] == 5               # >= 4 K blocks a piece
    q = P(128 * 20, 256, 64 * 64, variant=V1)                             # 20 tiles: 21 clusters of 7 fit
    assert q["k_split"] == 7 and q["grid_ctas"] == 20 * 7 and q["cta_group"] == 1
    assert P(128 * 40, 256, 64 * 64, variant=V1)["k_split"] == 3
    q = P(128 * 160, 256, 64 * 64, variant=V1)                            # 160 tiles: no wave fits
    assert q["variant"] == "TILE_1CTA_128x256" and q["k_split"] == 1
    # AUTO below one round of pair tiles: the cheapest of unsplit column pieces on
    # single CTAs, whole pair tiles, split K over pairs or over single CTAs
    assert P(256, 256, 64 * 20)["variant"] == "TILE_1CTA_128x256"        # short K: no split
    assert P(256, 256, 64 * 128)["variant"] == "TILE_1CTA_SPLITK"        # 2 tiles, long K: 8 pieces each
    assert P(256, 256, 64 * 128)["k_split"] == 8
    assert P(1024, 2048, 64 * 80)["variant"] == "TILE_1CTA_128x256"      # 64 tiles in halves beat S = 2
    q = P(768, 2048, 64 * 96)                                             # 24 tiles: 25 clusters of 3 pairs fit
    assert q["variant"] == "TILE_2CTA_SPLITK" and q["k_split"] == 3
    assert P(2048, 2048, 64 * 128)["variant"] == "TILE_2CTA_256x256"     # 64 whole pair tiles, long K


def test_plans_for_8bit_operands(lib):
    P = lambda *a, **k: g.gemm_nt_plan_ex(g.Dtype.E4M3, *a, num_sms=152, **k)  # noqa: E731
    p = P(8192, 8192, 8192)
    # a stage is still 128-byte rows: 128 K elements, half as many K blocks
    assert p["variant"] == "TILE_2CTA_256x256" and (p["tile_k"], p["k_blocks"]) == (128, 64)
    assert (p["num_full_tiles"], p["tail_split"]) == (988, 2)
    # A rows are half as large: up to 24 tile rows per 48 MiB group, 32 rows in 2 groups of 16
    assert p["group_m"] == 16
    # 4112-byte rows are 16-byte units but not on 32-byte sectors: two
    # consumers per CTA; 33 K blocks, the last 16 wide; all of A in one group
    p = P(4000, 11000, 4112)
    assert p["variant"] == "TILE_2CTA_512x256" and p["k_blocks"] == 33 and p["group_m"] == 8
    assert P(4000, 11000, 4128)["variant"] == "TILE_2CTA_256x256"
    with pytest.raises(g.GemmError):
        P(4000, 11000, 4104)                                 # 4104-byte rows: not 16-byte units
    p = P(16, 8192, 8192)
    assert p["variant"] == "SKINNY_SPLITK" and p["k_blocks"] == 64 and (p["k_split"], p["n_tiles"]) == (2, 76)
    p = P(512, 2048, 8192)                                   # 64 K blocks: 128 column pieces beat a split
    assert p["variant"] == "TILE_1CTA_128x256" and p["tail_split"] == 4
    p = P(512, 1024, 16384)                                  # 128 K blocks: 16 single-CTA tiles in 8 pieces
    assert p["variant"] == "TILE_1CTA_SPLITK" and p["k_split"] == 8
    assert g.gemm_nt_plan_ex(g.Dtype.F16, 8192, 8192, 8192, num_sms=152) == \
        g.gemm_f16_nt_plan(8192, 8192, 8192, num_sms=152)
    assert g.gemm_nt_plan_ex(g.Dtype.E5M2, 8192, 8192, 8192, num_sms=152)["tile_k"] == 128
    with pytest.raises(g.GemmError):
        P(64, 64, 40)                                        # K bytes not a multiple of 16
    with pytest.raises(g.GemmError):
        g.gemm_nt_plan_ex(4, 64, 64, 64, num_sms=152)


def test_short_k_loops_on_single_ctas(lib):
    # pair tiles fill the GPU but each K loop is only a few blocks: 128x256 CTAs
    F16 = lambda *a: g.gemm_f16_nt_plan(*a, num_sms=152)                  # noqa: E731
    E4 = lambda *a: g.gemm_nt_plan_ex(g.Dtype.E4M3, *a, num_sms=152)      # noqa: E731
    assert F16(4096, 8192, 512)["variant"] == "TILE_1CTA_128x256"          # 8 blocks
    assert F16(6144, 6144, 768)["variant"] == "TILE_2CTA_256x256"          # 12 blocks
    assert E4(6144, 6144, 1536)["variant"] == "TILE_1CTA_128x256"          # 12 blocks of 128
    assert E4(4096, 4096, 2048)["variant"] == "TILE_2CTA_256x256"          # 16 blocks


def test_plan_errors(lib):
    with pytest.raises(g.GemmError):
        g.gemm_f16_nt_plan(-1, 8, 8, num_sms=152)
    with pytest.raises(g.GemmError):
        g.gemm_f16_nt_plan(100, 8, 8, variant=g.Variant.SKINNY_SPLITK, num_sms=152)
    with pytest.raises(g.GemmError):
        g.gemm_f16_nt_plan(100, 8, 8, variant=g.Variant.SKINNY_STREAMK, num_sms=152)
    with pytest.raises(g.GemmError):
        g.gemm_f16_nt_plan(8, 8, 9, num_sms=152)


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(g, "_lib", None)
    monkeypatch.setattr(g, "LIB_PATH", "/nonexistent/libgemm_f16.so")
    with pytest.raises(g.LibraryMissing):
        g.load()
