"""Host-side checks of the C ABI (no GPU needed): the library loads and
exports every function include/gemm_rs.h declares, arguments are rejected
before any CUDA call, and the tile order covers every rank tile once with the
8 rank tiles of a region next to each other."""
import ctypes

import pytest

from tensor_gemm_reduce_gb300 import gemm_rs as G


@pytest.fixture(scope="module")
def lib():
    from tensor_gemm_reduce_gb300 import build
    build.build_library()
    return G.load_library()


def test_exports_every_declared_symbol(lib):
    names = G.header_symbols()
    assert set(names) >= {"gemm_rs_create", "gemm_rs_run", "gemm_rs_destroy", "gemm_rs_status",
                          "gemm_rs_strerror", "gemm_rs_get_info", "gemm_rs_schedule"}
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(G._SIGS), "binding signatures and header out of sync"


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library the binding raises; nothing computes on the CPU."""
    from tensor_gemm_reduce_gb300 import build
    monkeypatch.setattr(G, "_LIB", None)
    monkeypatch.setattr(build, "LIB", str(tmp_path / "libgemm_rs.so"))
    with pytest.raises(ImportError):
        G.load_library(build_if_missing=False)
    # a plan needs the library; when it cannot be built the call raises
    def no_compiler():
        raise RuntimeError("nvcc not found")
    monkeypatch.setattr(build, "build_library", no_compiler)
    with pytest.raises(RuntimeError, match="nvcc not found"):
        G.Plan(64, 256, 512)


def _create(**kw):
    d = G._desc(kw.pop("M", 128), kw.pop("N", 256), kw.pop("K", 512), **kw)
    h = ctypes.c_void_p()
    ws = ctypes.c_size_t()
    return G.load_library().gemm_rs_create(ctypes.byref(d), ctypes.byref(h), ctypes.byref(ws))


@pytest.mark.parametrize("kw,code", [
    (dict(world=4), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(reducer_warps=6), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(reducer_warps=-1), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(unit_rows=12), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(unit_rows=64), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(grid=-2), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(mma_ctas=3), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(mma_ctas=4), G.GEMM_RS_ERR_INVALID_ARG),  # no 4-CTA (operand-sharing) tiles
    (dict(mma_ctas=5), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(chunks=-1), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(chunks=65), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(replicas=2), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(tail_waves=65), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(half_regions=-2), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(tail_waves=-1), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(op=2), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(op=G.OP_AG, replicas=8), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(op=G.OP_AG, N=264), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
    (dict(op=G.OP_AG, copy_engines=-2), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(op=G.OP_AG, copy_engines=5), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(replicas=-1), G.GEMM_RS_ERR_INVALID_ARG),
    (dict(M=100), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
    (dict(N=12), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
    (dict(K=96), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
    (dict(M=-8), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
    (dict(M=1 << 31), G.GEMM_RS_ERR_UNSUPPORTED_SHAPE),
])
def test_create_rejects_bad_arguments(lib, kw, code):
    assert _create(**kw) == code


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.gemm_rs_create(None, ctypes.byref(h), None) == G.GEMM_RS_ERR_INVALID_ARG
    d = G._desc(128, 256, 512)
    assert lib.gemm_rs_create(ctypes.byref(d), None, None) == G.GEMM_RS_ERR_INVALID_ARG
    assert lib.gemm_rs_run(None, 0, None, None, None, None, None) == G.GEMM_RS_ERR_INVALID_ARG
    assert lib.gemm_rs_status(None, None) == G.GEMM_RS_ERR_INVALID_ARG
    assert lib.gemm_rs_get_info(None, None) == G.GEMM_RS_ERR_INVALID_ARG
    assert lib.gemm_rs_destroy(None) == G.GEMM_RS_OK


def test_strerror(lib):
    for code in range(-9, 1):
        assert G.strerror(code) and G.strerror(code) != f"status {code}"
    assert G.strerror(-99) == "unknown status"


@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("half", [0, -1, 3, 4000])
@pytest.mark.parametrize("M,N,K,band", [(128, 512, 1024, 0), (392, 776, 1600, 0),
                                        (2048, 8192, 8192, 0), (8192, 8192, 28672, 0),
                                        (1000, 6144, 6144, 3), (520, 1000, 1024, 1)])
def test_schedule_covers_every_tile_once(lib, M, N, K, band, ctas, half):
    """Every rank tile exactly once: whole tiles (8 per region, ranks in
    order) first, then the last regions as half-width tiles (16 per region:
    the left halves of ranks 0..7, then the right halves), which together
    cover the same columns."""
    d = G._desc(M, N, K, band_m=band, mma_ctas=ctas, half_regions=half)
    rows = 128 * ctas
    mt, nt = (M + rows - 1) // rows, (N + 255) // 256
    regions = mt * nt
    want = max(half, 0)  # 0 (default) and -1: none
    n_half = min(want, regions) if ctas == 2 else 0     # regions in half-width tiles
    first_half = regions - n_half
    tiles = 8 * first_half + 16 * n_half
    order = [G.gemm_rs_schedule(d, i) for i in range(tiles)]
    assert len(set(order)) == tiles
    for r, m, n, h in order:
        assert 0 <= r < 8 and 0 <= m < mt and 0 <= n < nt and h in (-1, 0, 1)
    covered = {(r, m, n, c) for r, m, n, h in order for c in ((0, 1) if h < 0 else (h,))}
    assert len(covered) == 8 * regions * 2  # every rank's both column halves of every region once
    for g in range(first_half):
        blk = order[8 * g: 8 * g + 8]
        assert [b[0] for b in blk] == list(range(8)) and {b[3] for b in blk} == {-1}
        assert len({(b[1], b[2]) for b in blk}) == 1
    for k in range(n_half):
        blk = order[8 * first_half + 16 * k: 8 * first_half + 16 * (k + 1)]
        assert [b[0] for b in blk] == list(range(8)) * 2
        assert [b[3] for b in blk] == [0] * 8 + [1] * 8
        assert len({(b[1], b[2]) for b in blk}) == 1
    # half-width tiles take the regions that come last in the whole-tile order
    d_none = G._desc(M, N, K, band_m=band, mma_ctas=ctas, half_regions=-1)
    whole = [G.gemm_rs_schedule(d_none, 8 * g)[1:3] for g in range(regions)]
    assert [order[8 * g][1:3] for g in range(first_half)] == whole[:first_half]
    assert [order[8 * first_half + 16 * k][1:3] for k in range(n_half)] == whole[first_half:]
    with pytest.raises(G.GemmRSError):
        G.gemm_rs_schedule(d, tiles)


def test_schedule_band_walks_columns_inside_band(lib):
    # band of 4 tile rows: positions 0..3 are column 0, rows 0..3
    d = G._desc(1024, 1024, 1024, band_m=4, mma_ctas=1)
    regions = [G.gemm_rs_schedule(d, 8 * g)[1:3] for g in range(8 * 4)]
    assert regions[:5] == [(0, 0), (1, 0), (2, 0), (3, 0), (0, 1)]
    assert regions[16] == (4, 0)


@pytest.mark.parametrize("ctas", [1, 2])
def test_auto_band_keeps_a_rows_within_budget(lib, ctas):
    rows = 128 * ctas
    for M, K in [(2048, 8192), (8192, 28672), (32768, 16384), (512, 6144)]:
        d = G._desc(M, 1024, K, mma_ctas=ctas)
        # find the band: the first region that is in column 1
        mt = (M + rows - 1) // rows
        band = None
        for g in range(mt * 4):
            _, m, n, _ = G.gemm_rs_schedule(d, 8 * g)
            if n == 1:
                band = g
                break
        band = band if band is not None else mt
        assert 1 <= band <= mt
        assert band == mt or band * rows * K * 2 <= 32 << 20


@pytest.mark.parametrize("ctas", [1, 2])
@pytest.mark.parametrize("M,N,K", [(2048, 10240, 8192), (392, 1536, 1600), (128, 512, 1024)])
def test_ag_schedule_walks_from_own_shard(lib, M, N, K, ctas):
    """All-gather + GEMM order (mKernel page, section 4): every rank tile once,
    rank after rank; each rank starts at the tile row holding its own shard."""
    d = G._desc(M, N, K, mma_ctas=ctas, op=G.OP_AG)
    rows = 128 * ctas
    mt, nt = (M + rows - 1) // rows, (N // 8 + 255) // 256
    seen = []
    for i in range(8 * mt * nt):
        seen.append(tuple(G.gemm_rs_schedule(d, i)[:3]))
    assert len(set(seen)) == 8 * mt * nt
    per_rank = mt * nt
    for r in range(8):
        mine = seen[r * per_rank:(r + 1) * per_rank]  # ranks one after the other
        assert {t[0] for t in mine} == {r}
        assert mine[0][1] == (r * (M // 8)) // rows and mine[0][2] == 0  # own shard first


@pytest.mark.parametrize("op", [0, 1])
def test_tune_candidates_and_their_workspace(lib, op):
    """The tuner's candidate set (host only): the requested plan first, then
    the tile shape and the number of communication warps (and unit rows)
    varied, narrower tile-order bands and (reduce-scatter) tail waves; no plan
    twice; one workspace size that fits every candidate."""
    d = G._desc(1024, 2048, 4096, op=op, timeout_ns=7)
    cands, ws = G.tune_candidates(d)
    # auto band at M=1024, K=4096, 256-row tiles: 32 MiB / (256*4096*2) = 16 -> 4 tile rows
    assert len(cands) == (1 + 11 + 2 + 3 + 2 if op == 0 else 1 + 5 + 2)
    c0 = cands[0]
    assert (c0.mma_ctas, c0.reducer_warps, c0.unit_rows, c0.band_m, c0.tail_waves) == (0, 0, 0, 0, 0)
    def resolved(c):
        ctas = c.mma_ctas or 2
        return (ctas, c.reducer_warps or (5 if op == 0 else 2),  # K = 4096 <= 6144: 5 reducers
                (c.unit_rows or 8) if op == 0 else 0, c.band_m or (4 if ctas == 2 else 8),
                (c.tail_waves or 3) if op == 0 else 0,
                max(c.half_regions, 0) if (op == 0 and ctas == 2) else 0)
    assert len({resolved(c) for c in cands}) == len(cands)
    assert {c.band_m for c in cands} >= {0, 1, 2}
    if op == 0:
        assert {c.tail_waves for c in cands} >= {0, 1, 2, 6}
        assert {c.half_regions for c in cands} == {0, 5, 10}
    assert all(c.M == 1024 and c.N == 2048 and c.K == 4096 and c.op == op and c.timeout_ns == 7
               for c in cands)
    staging = 8 * 1024 * (2048 if op == 0 else 4096) * 2
    assert ws > staging
    with pytest.raises(G.GemmRSError):
        G.tune_candidates(G._desc(100, 256, 512))


def test_header_is_plain_c():
    """include/gemm_rs.h compiles as strict C99 (no C++ in the boundary)."""
    import os
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-pedantic", "-fsyntax-only", "-x", "c",
                        os.path.join(root, "include", "gemm_rs.h")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
