"""Planner logic and the C ABI, checked on the CPU (no GPU needed).

The library's host reference of the planner (topk_plan_host) runs the same decisions
as the planning kernel; these tests check the plans it builds for every workload
against the invariants the select kernel relies on. They also check that the library
loads and exports every entry point declared in include/topk_paged.h, and that host
argument checks reject bad calls before anything is enqueued.
"""
import os
import re

import numpy as np
import pytest

import workloads as W

S = pytest.importorskip("sparse_attention_indexer_gb300")
B = S.binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_ONLY_MAX_LEN = 16384  # batches of rows at most this long: register or medium path
CLUSTER_MAX_LEN = 131072     # longer ones up to this: cluster path when their clusters fit
ABOVE_MEDIUM = CLUSTER_MAX_LEN + 1  # a max_len that keeps a batch on the full planner


def cluster_size(max_len):
    """CTAs per row on the cluster path (the library's rule), 0 outside its lengths."""
    if max_len <= HEADER_ONLY_MAX_LEN or max_len > CLUSTER_MAX_LEN:
        return 0
    return 2 if max_len <= CLUSTER_MAX_LEN // 4 else 4 if max_len <= CLUSTER_MAX_LEN // 2 else 8


def header_only(rows, max_len, grid, chunk=0):
    """Whether the plan is its header alone: the register, medium or cluster path."""
    if chunk:
        return False
    cs = cluster_size(max_len)
    return max_len <= HEADER_ONLY_MAX_LEN or (cs > 0 and rows >= 1 and rows * cs <= grid)


def _lib_or_skip():
    if not os.path.exists(B.LIB_PATH):
        pytest.skip("library not built")
    return B.lib()


def header_exports():
    names = set()
    for h in ("topk_paged.h", "indexer_prologue.h", "indexer_logits.h", "hisparse_resolver.h"):
        src = open(os.path.join(ROOT, "include", h)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b((?:topk|indexer|hisparse)_[a-z_]+)\s*\(", src))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    lib = _lib_or_skip()
    names = header_exports()
    assert "topk_select_paged" in names and "topk_plan" in names
    assert "indexer_k_prologue" in names and "hisparse_resolve" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
    assert set(names) <= set(B.EXPORTS), set(names) - set(B.EXPORTS)


def parse_plan(image, rows):
    info = B.topk_layout_info(rows)
    h = image[:256].view(np.int32)
    hdr = dict(magic=int(h.view(np.uint32)[0]), rows=int(h[1]), max_len=int(h[2]), grid=int(h[3]),
               chunk=int(h[4]), waves=int(h[5]), n_single=int(h[6]), n_multi=int(h[7]),
               status=int(h[8]), plan_error=int(h[9]), n_implicit=int(h[10]),
               dyn_period=int(h[11]))
    ri = image[info["rowinfo"]:info["rowinfo"] + 16 * rows].view(np.int32).reshape(rows, 4)
    singles = image[info["singles"]:info["singles"] + 8 * rows].view(np.int32).reshape(rows, 2)
    first = image[info["first_single"]:info["first_single"] + 4 * info["max_grid"]].view(np.int32)
    units = image[info["units"]:info["groups"]].view(np.int32).reshape(-1, 8)
    return hdr, ri, singles, (first, units), info


def host_plan(lens, max_len, grid, chunk=0):
    rows = len(lens)
    n = B.topk_workspace_bytes(rows, max_len)
    image = np.zeros(n, dtype=np.uint8)
    B.topk_plan_host(np.asarray(lens, np.int32), rows, max_len, grid, chunk, image)
    return parse_plan(image, rows)


def check_plan(lens, max_len, grid, chunk=0):
    """Invariants the select kernel relies on: each multi-CTA row's chunks cover it
    exactly, sit in one wave on distinct CTAs and fit one CTA's shared memory; single
    rows fit one CTA; every single row is listed once, longest bucket first; each
    CTA without static work gets at most one single row up front; the ticket period
    counts one claim per remaining single row plus one failing claim per CTA."""
    _lib_or_skip()
    hdr, ri, singles, (first, units), info = host_plan(lens, max_len, grid, chunk)
    if header_only(len(lens), max_len, grid, chunk):
        # register path (one warp per row), medium path (one CTA per row) or cluster
        # path (one thread-block cluster per row): the plan is its header alone
        assert hdr["magic"] == 0x54504B32 and hdr["rows"] == len(lens)
        assert hdr["max_len"] == max_len and hdr["status"] == 0 and hdr["plan_error"] == 0
        assert hdr["waves"] == 0 and hdr["n_multi"] == 0 and hdr["n_single"] == len(lens)
        return hdr, None
    rows = len(lens)
    assert hdr["magic"] == 0x54504B32 and hdr["rows"] == rows and hdr["grid"] == grid
    assert hdr["plan_error"] == 0
    cap = info["chunk_cap"]
    maxg = info["max_grid"]
    waves = hdr["waves"]
    assert waves <= info["max_waves"]
    seen = {}
    busy = np.zeros(grid, bool)
    for w in range(waves):
        for cta in range(maxg):
            u = units[w * maxg + cta]
            if u[0] < 0:
                continue
            assert cta < grid
            row, s0, n, L, rank, G, group = (int(v) for v in u[:7])
            assert (row, rank) not in seen, "unit assigned twice"
            seen[(row, rank)] = (w, cta, s0, n, L, G, group)
            busy[cta] = True
    n_multi = 0
    for r in range(rows):
        L = int(lens[r])
        Lv = L if 0 <= L <= max_len else 0
        G = int(ri[r, 1])
        assert int(ri[r, 0]) == L
        if G > 1:
            n_multi += 1
            assert 0 <= int(ri[r, 2]) < hdr["n_multi"]
            parts = [seen[(r, k)] for k in range(G)]
            assert len({p[0] for p in parts}) == 1, "a multi-CTA row spans several waves"
            assert len({p[1] for p in parts}) == G
            covered = 0
            for k, (w, cta, s0, n, Lu, Gu, grp) in enumerate(parts):
                assert Lu == L and Gu == G and grp == int(ri[r, 2])
                assert 0 <= n <= cap and s0 % 16 == 0
                assert s0 == covered or n == 0
                covered = max(covered, s0 + n)
            assert covered == Lv
        else:
            assert Lv <= cap
            assert int(ri[r, 2]) == -1
    assert n_multi == hdr["n_multi"]
    assert len(seen) == sum(int(ri[r, 1]) for r in range(rows) if int(ri[r, 1]) > 1)
    single_rows = [r for r in range(rows) if int(ri[r, 1]) == 1]
    assert hdr["n_single"] == len(single_rows)
    sl = [int(x) for x in singles[:hdr["n_single"], 0]]
    assert sorted(sl) == single_rows
    assert [int(x) for x in singles[:hdr["n_single"], 1]] == [int(lens[r]) for r in sl]
    buckets = [int(np.floor(np.log2(max(1, lens[r] if 0 <= lens[r] <= max_len else 0) or 1)))
               for r in sl]
    assert buckets == sorted(buckets, reverse=True)
    free = [c for c in range(grid) if not busy[c]]
    exp_first = [-1] * grid
    for i, c in enumerate(free[:hdr["n_single"]]):
        exp_first[c] = i
    assert [int(x) for x in first[:grid]] == exp_first
    assert hdr["n_implicit"] == min(len(free), hdr["n_single"])
    assert hdr["dyn_period"] == hdr["n_single"] - hdr["n_implicit"] + grid
    return hdr, ri


@pytest.mark.parametrize("grid", [152, 148, 132])
def test_plan_verify_configs_fit_one_wave(grid):
    b = W.verify_1m()
    hdr, ri = check_plan(b.lens, b.max_len, grid)
    need = sum(-(-int(l) // B.topk_chunk_capacity()) for l in b.lens)
    if need <= grid:  # one wave whenever the rows can fit the grid at all
        assert hdr["waves"] == 1
        assert int(ri[:, 1].sum()) <= grid
    # the 80K verify batch runs on the cluster path (7 clusters of 8): header only
    b = W.verify_80k()
    hdr, ri = check_plan(b.lens, b.max_len, grid)
    assert ri is None and hdr["waves"] == 0


def test_plan_80k_spreads_rows_over_the_grid():
    """On the work-list planner (too many rows for the cluster path, or a grid too small
    for its clusters), 80K rows are split over many CTAs each."""
    b = W.verify_80k()
    lens = np.concatenate([b.lens] * 3)  # 21 rows: 168 cluster CTAs > 152
    hdr, ri = check_plan(lens, b.max_len, 152)
    assert ri is not None and all(int(g) >= 7 for g in ri[:, 1])
    hdr, ri = check_plan(b.lens, b.max_len, 48)  # 56 cluster CTAs > 48
    assert ri is not None and hdr["waves"] == 1


def test_plan_cluster_path_rule():
    """Header-only plans for batches whose clusters (2, 4 or 8 CTAs per row by max_len)
    fit the grid; the full planner for a forced chunk, more rows, or longer rows."""
    _lib_or_skip()
    for max_len, cs in ((16385, 2), (32768, 2), (32769, 4), (65536, 4), (65537, 8), (131072, 8)):
        assert cluster_size(max_len) == cs
        rows = 152 // cs
        lens = np.full(rows, max_len, np.int32)
        hdr, ri = check_plan(lens, max_len, 152)
        assert ri is None and hdr["n_single"] == rows
        hdr, ri = check_plan(np.full(rows + 1, max_len, np.int32), max_len, 152)
        assert ri is not None
        hdr, ri = check_plan(lens, max_len, 152, chunk=8192)
        assert ri is not None
    hdr, ri = check_plan(np.full(3, 131073, np.int32), 131073, 152)
    assert ri is not None
    # the limit follows the grid: C * rows CTAs at most, one per SM
    for grid in (148, 132, 37):
        for max_len, cs in ((20000, 2), (50000, 4), (100000, 8)):
            rows = grid // cs
            if rows == 0:
                continue
            hdr, ri = check_plan(np.full(rows, max_len, np.int32), max_len, grid)
            assert ri is None, (grid, max_len)
            hdr, ri = check_plan(np.full(rows + 1, max_len, np.int32), max_len, grid)
            assert ri is not None, (grid, max_len)


def test_plan_all_workloads():
    for b in [W.pr1(), W.mixed_decode(), W.adversarial(), W.prefill()] + W.tiny_rows()[:3]:
        check_plan(b.lens, b.max_len, 152)
    # the medium batches on the full planner (a max_len above the medium range)
    for b in (W.pr1(), W.prefill()):
        check_plan(b.lens, ABOVE_MEDIUM, 152)


@pytest.mark.parametrize("chunk", [16, 64, 1000, 4096, 48128])
def test_plan_forced_chunks(chunk):
    b = W.mixed_decode()
    if chunk < 4096:
        lens = np.minimum(b.lens, 40000).astype(np.int32)
        check_plan(lens[:8], 40000, 152, chunk)
    else:
        check_plan(b.lens, b.max_len, 152, chunk)


def test_plan_degenerate_lengths():
    M = ABOVE_MEDIUM
    check_plan(np.array([0, 0, 0], np.int32), M, 152)
    check_plan(np.array([-5, M + 1, 50], np.int32), M, 152)  # invalid lengths become single rows
    check_plan(np.array([], np.int32).reshape(0), M, 152)
    check_plan(np.array([-5, 101, 50], np.int32), 100, 152)  # register path: header only
    check_plan(np.array([-5, 5001, 50], np.int32), 5000, 152)  # medium path: header only
    check_plan(np.array([0, 0, 0], np.int32), 100, 152, chunk=16)  # forced: full plan
    rng = np.random.default_rng(3)
    lens = rng.integers(0, 300_000, size=400).astype(np.int32)
    check_plan(lens, 300_000, 152)


def test_plan_reports_too_many_long_rows():
    """More rows longer than one CTA's capacity than there are group states: the plan
    is marked failed (the select call then reports a plan mismatch, rows -1)."""
    _lib_or_skip()
    lens = np.full(600, 100_000, np.int32)
    hdr, *_ = host_plan(lens, 100_000, 152)
    assert hdr["plan_error"] == 1 and hdr["status"] == 32


def test_plan_many_waves():
    lens = np.full(40, 1_000_000, np.int32)
    hdr, ri = check_plan(lens, 1_000_000, 152)
    assert hdr["waves"] > 1


def test_host_argument_errors():
    _lib_or_skip()
    assert B.topk_workspace_bytes(-1, 10) == 0
    img = np.zeros(B.topk_workspace_bytes(2, 10), np.uint8)
    with pytest.raises(B.TopKError):
        B.topk_plan_host(np.array([1, 2], np.int32), 2, 10, 152, 8, img)  # chunk < 16
    with pytest.raises(B.TopKError):
        B.topk_plan_host(np.array([1, 2], np.int32), 2, 10, 0, 0, img)
    with pytest.raises(B.TopKError):
        B.topk_plan_host(np.array([1, 2], np.int32), 2, 10, 152, 0, img[:100])
    lib = B.lib()
    # select: argument checks happen before any CUDA call
    assert lib.topk_select_paged(None, 10, None, 1, 10, 0, None, 1, None, 64, None, None, 256,
                                 None) == -3   # k
    assert lib.topk_select_paged(None, 10, None, 1, 10, 4, None, 1, None, 0, None, None, 256,
                                 None) == -4   # page size
    assert lib.topk_select_paged(None, 5, None, 1, 10, 4, None, 1, None, 64, None, None, 256,
                                 None) == -5   # ld < max_len
    assert lib.topk_select_paged(None, 10, None, 1, 10, 4, None, 1, None, 64, None, None, None,
                                 None) == -1   # workspace
    assert lib.topk_select_paged(None, 10, None, -1, 10, 4, None, 1, None, 64, None, None, 256,
                                 None) == -2   # rows
    assert lib.topk_select_paged(None, 10, None, 0, 10, 4, None, 1, None, 64, None, None, 256,
                                 None) == 0    # empty batch: nothing to do
    assert lib.topk_select_paged(4, 10, 4, 1, 10, 4, 4, 1, None, 64, 4, None, 100, None) == -6
    assert lib.topk_select_paged(2, 10, 4, 1, 10, 4, 4, 1, None, 64, 4, None, 256, None) == -8
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10, -11, 1, 16, 3):
        assert B.status_str(code)


def _brute_auto_chunk(lens, max_len, grid, cap, align=16, min_auto=2048):
    """Smallest multiple of `align` >= c0 whose split rows fit the grid, by linear scan."""
    valid = [int(l) if 0 <= l <= max_len else 0 for l in lens]
    c0 = max(-(-sum(valid) // grid), min_auto)
    c0 = min(max(-(-c0 // align) * align, align), cap)

    def slots(c):
        return sum(-(-l // c) for l in valid if l > c)
    for c in range(c0, cap + 1, align):
        if slots(c) <= grid:
            return c, True
    return cap, False


@pytest.mark.parametrize("grid", [152, 132, 37])
def test_auto_chunk_is_smallest_fitting(grid):
    """The automatic chunk is the smallest multiple of 16 (>= the even split of the
    batch over the grid) at which the split rows need no more CTAs than the grid."""
    _lib_or_skip()
    cap = B.topk_chunk_capacity()
    rng = np.random.default_rng(21)
    cases = [W.verify_80k().lens, W.verify_1m().lens, W.mixed_decode().lens,
             np.array([5000, 3, 70000, 12345], np.int32),
             rng.integers(0, 200_000, size=9).astype(np.int32),
             rng.integers(0, 60_000, size=300).astype(np.int32)]
    for lens in cases:
        max_len = int(max(lens.max(), 1))
        if header_only(len(lens), max_len, grid):
            max_len = ABOVE_MEDIUM  # the same lengths on the work-list planner
        hdr, _ = check_plan(lens, max_len, grid) if grid * cap >= max_len else (None, None)
        if hdr is None:
            continue
        c, fits = _brute_auto_chunk(lens, max_len, grid, cap)
        assert hdr["chunk"] == c, (lens[:8], hdr["chunk"], c)
        if fits:
            assert hdr["waves"] <= 1
