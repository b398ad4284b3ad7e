"""GPU parity of the cluster path (batches of a few rows of 16,385..131,072 values: one
thread-block cluster of 2, 4 or 8 CTAs per row, histograms merged through distributed
shared memory) against the CPU oracle, bit-exact.

Covers every cluster size at its smallest and largest row length, rows of every length
class (all taken, just above k, full) with ragged shares (CTAs with no values), N(0,1),
fp16-grid, few-value and all-equal rows, special values, boundary bins larger than CTA
0's candidate list (refined by the cluster one key byte at a time, down to exact ties
taken in position order), top values held by one CTA, unaligned row starts, page sizes
that are and are not powers of two, a row-to-table map, slots-only output, every device
status, a plan built for other lengths, a forced-chunk plan on the same workspace (the
work-list kernel) and a batch too large for the cluster path.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import PagedTopK, binding as B  # noqa: E402
from tests._gpu import compare_with_oracle, run_gpu, to_dev  # noqa: E402


def _cluster_size(max_len):
    return 0 if max_len <= 16384 or max_len > 131072 else 2 if max_len <= 32768 else 4 if max_len <= 65536 else 8


def _rows(rng, n, max_len, kind):
    lens = rng.integers(max_len // 2, max_len + 1, n).astype(np.int32)
    lens[:6] = np.array([max_len, max_len - 1, 2049, 2048, 17, max_len // 3 + 5], np.int32)[:min(6, n)]
    if kind == "normal":
        s = rng.standard_normal((n, max_len)).astype(np.float32)
    elif kind == "fp16":
        s = rng.standard_normal((n, max_len)).astype(np.float16).astype(np.float32)
    elif kind == "few":
        s = rng.integers(-2, 3, (n, max_len)).astype(np.float32)
    else:  # all equal per row: refined down to exact ties, taken in position order
        s = np.repeat(rng.standard_normal((n, 1)).astype(np.float32), max_len, axis=1)
    return s, lens


def _batch(name, s, lens, max_len, page_size=64, seed=0, r2t=False, ld=None):
    rng = np.random.default_rng(seed)
    rows = s.shape[0]
    ld = ld or W.round_up(max_len, 4)
    sc = np.full((rows, ld), W.POISON, np.float32)
    sc[:, :max_len] = s[:, :max_len]
    for r in range(rows):
        sc[r, max(lens[r], 0):] = W.POISON
    npg = -(-max_len // page_size)
    if r2t:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(3)])
        m = rng.integers(0, 3, rows).astype(np.int32)
    else:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(rows)])
        m = None
    return W.Batch(name, sc, lens, max_len, 2048, tab, m, page_size)


def _check(b, ks, plan=None, dev=None):
    dev = dev or to_dev(b)
    core = plan
    if core is None:
        core = PagedTopK(b.rows, b.max_len)
        core.plan(dev[1])
    for k in ks:
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)


@pytest.mark.parametrize("max_len", [16385, 32768, 32769, 65536, 65537, 131072])
@pytest.mark.parametrize("kind", ["normal", "fp16", "few", "equal"])
def test_cluster_rows_every_k(max_len, kind):
    rng = np.random.default_rng(max_len + ["normal", "fp16", "few", "equal"].index(kind))
    rows = 152 // _cluster_size(max_len) if kind == "normal" and max_len in (16385, 131072) else 9
    s, lens = _rows(rng, rows, max_len, kind)
    b = _batch(f"cluster_{kind}", s, lens, max_len, seed=1)
    _check(b, (1, 7, 256, 2047, 2048))


def test_cluster_special_values_and_tails():
    rng = np.random.default_rng(5)
    L = 70001
    vals = np.array([np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, 65504.0,
                     70000.0, 2.0 ** -20, np.nan], np.float32)
    s = rng.choice(vals, size=(10, L)).astype(np.float32)
    mix = rng.random((10, L)) < 0.4
    s[mix] = rng.standard_normal(int(mix.sum())).astype(np.float32)
    s[6, 50:] = -np.inf                    # a short N(0,1) prefix, then -inf
    s[7] = np.nan                          # NaN rows with -inf every 7th position
    s[7, ::7] = -np.inf
    s[8] = np.where(np.arange(L) % 3 == 0, np.float32(-0.0), np.float32(0.0))
    s[9] = np.float32(2.5)
    lens = np.array([L, L - 1, 40001, 16385, 2049, 2048, L, L, L, L], np.int32)
    b = _batch("cluster_special", s, lens, L, seed=6)
    _check(b, (1, 2, 100, 2048))


def test_cluster_boundary_bins_over_capacity():
    """Boundary bins of 6000 distinct values in one coarse bin (refined by a key byte,
    then gathered), of 5000 and 70000 exact ties (refined through every key byte, then
    taken in position order across the CTAs), of 3000 exact ties (gathered and ranked by
    position) and of 4096 exact ties (the list's capacity)."""
    rng = np.random.default_rng(8)
    L = 100000
    base = rng.standard_normal(L).astype(np.float32)
    rows = []
    x = base.copy()
    x[rng.choice(L, 6000, replace=False)] = (np.float32(20.0) +
                                             rng.random(6000).astype(np.float32) * np.float32(0.2))
    rows.append(x)
    for n in (5000, 70000, 3000, 4096):
        y = base.copy()
        y[rng.choice(L, n, replace=False)] = np.float32(9.0)
        rows.append(y)
    z = base.copy()
    z[: L // 2] = np.float32(9.0)           # the ties sit in the first CTAs' shares only
    rows.append(z)
    s = np.stack(rows)
    b = _batch("cluster_big_bins", s, np.full(len(rows), L, np.int32), L, seed=9)
    _check(b, (1, 2, 1000, 2048))


def test_cluster_top_values_in_one_share():
    """Sorted descending (CTA 0 holds every selected value), sorted ascending (the last
    CTA does), a step at 10 % of the row, and verify_80k's rows."""
    rng = np.random.default_rng(17)
    L = 120000
    base = rng.standard_normal(L).astype(np.float32)
    step = base.copy()
    step[: L // 10] += 5.0
    s = np.stack([np.sort(base)[::-1].copy(), np.sort(base), step])
    b = _batch("cluster_sorted", s, np.array([L, L - 5, L - 17], np.int32), L, seed=18)
    _check(b, (1, 100, 2048))
    _check(W.verify_80k(), (1, 100, 2048))


@pytest.mark.parametrize("page_size", [1, 7, 64])
def test_cluster_unaligned_rows_page_sizes_row_map(page_size):
    rng = np.random.default_rng(page_size)
    s, lens = _rows(rng, 9, 50001, "normal")
    b = _batch("cluster_pages", s, lens, 50001, page_size=page_size, seed=7, r2t=True, ld=50001)
    assert b.ld % 4 != 0  # rows start at unaligned addresses: no bulk copies
    for k in (5, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)
    slots, _, st = run_gpu(b, k=300, with_pos=False)
    assert st == 0
    compare_with_oracle(b, 300, slots, None)


def test_cluster_forced_chunk_and_batch_limit():
    """A forced-chunk plan sends the same rows through the work-list kernel, and the
    next unforced plan on the same workspace back to the cluster path; 20 rows of 8 CTAs
    do not fit 152 SMs at once and take the work-list kernel."""
    rng = np.random.default_rng(23)
    s, lens = _rows(rng, 7, 90000, "normal")
    b = _batch("cluster_forced", s, lens, 90000, seed=24)
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    for chunk in (0, 8192, 0, 48128):
        core.plan(dev[1], chunk=chunk)
        _check(b, (3, 2048), plan=core, dev=dev)
    s2, lens2 = _rows(rng, 20, 90000, "fp16")
    _check(_batch("cluster_limit", s2, lens2, 90000, seed=25), (3, 2048))


def test_cluster_status_errors_and_plan_mismatch():
    rng = np.random.default_rng(2)
    L = 40000
    s = rng.standard_normal((6, L)).astype(np.float32)
    s[1, 64:128] = 50.0
    s[2, 0:64] = 50.0
    b = _batch("cluster_errs", s, np.full(6, L, np.int32), L, seed=3)
    b.block_table[1, 1] = -3        # the selected positions of row 1 map to a negative page
    b.block_table[2, 0] = 2 ** 30   # row 2's selected slots overflow int32
    slots, pos, st = run_gpu(b, k=16)
    assert st == (B.STATUS_TABLE_ENTRY | B.STATUS_SLOT_OVERFLOW), B.status_str(st)
    ref = oracle.topk_batch(b, k=16, threads=1)
    compare_with_oracle(b, 16, slots, pos, ref=ref)
    # a length above max_len (row 1), a negative one (row 4) and a table too narrow for
    # rows 0, 2, 5
    bad = W.Batch("cluster_errs2", b.scores.copy(), np.array([L, L + 1, L, 100, -3, L], np.int32),
                  L, 16, b.block_table[:, :300].copy(), None, 64)
    slots, pos, st = run_gpu(bad, k=16)
    assert st == B.STATUS_LEN | B.STATUS_TABLE_WIDTH, B.status_str(st)
    assert np.all(slots[[0, 1, 2, 4, 5]] == -1) and np.all(pos[[0, 1, 2, 4, 5]] == -1)
    sub = W.Batch("cluster_errs3", bad.scores[[3]].copy(), bad.lens[[3]].copy(), L, 16,
                  bad.block_table[[3]].copy(), None, 64)
    compare_with_oracle(sub, 16, slots[[3]], pos[[3]])
    # a plan for one more row
    scores, lens_d, table, r2t = to_dev(b)
    core = PagedTopK(b.rows + 1, b.max_len)
    core.plan(torch.cat([lens_d, lens_d[:1]]))
    out = torch.empty((b.rows, 8), dtype=torch.int32, device="cuda")
    B.topk_select_paged(scores, scores.stride(0), lens_d, b.rows, b.max_len, 8, table,
                        table.stride(0), r2t, b.page_size, out, None, core.workspace)
    assert core.status() & B.STATUS_PLAN_MISMATCH
    assert torch.all(out == -1)


def test_cluster_one_plan_many_calls():
    """One header-only plan serves calls with changing k, scores and lengths up to
    max_len."""
    rng = np.random.default_rng(31)
    s, lens = _rows(rng, 12, 60000, "normal")
    b = _batch("cluster_many", s, lens, 60000, seed=32)
    s2, _ = _rows(rng, 12, 60000, "few")
    b2 = _batch("cluster_many2", s2, lens, 60000, seed=32)
    scores, lens_d, table, r2t = to_dev(b)
    sc2 = torch.from_numpy(b2.scores).cuda()
    core = PagedTopK(b.rows, b.max_len)
    core.plan(lens_d)
    for _ in range(2):
        for k in (2048, 17):
            for bb, ss in ((b, scores), (b2, sc2)):
                slots, pos, st = run_gpu(bb, k=k, plan=core, dev_inputs=(ss, lens_d, table, r2t))
                assert st == 0
                compare_with_oracle(bb, k, slots, pos)
    short = dataclasses.replace(b, lens=(lens // 3).astype(np.int32))
    sl = torch.from_numpy(short.lens).cuda()
    slots, pos, st = run_gpu(short, k=500, plan=core, dev_inputs=(scores, sl, table, r2t))
    assert st == 0
    compare_with_oracle(short, 500, slots, pos)
