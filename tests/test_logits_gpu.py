"""GPU parity of the indexer score producer (indexer_mqa_logits: tcgen05 e4m3 MMAs,
TMA-staged operands) against the fp64 CPU oracle, and of the producer feeding
topk_select_paged.

The tensor cores accumulate the e4m3 products in fp32 and the gate sum runs in fp32,
so a score is compared with the oracle's within TOL times the magnitude
sk * sum_h |g_h| * sum_d |q_hd k_d| (an upper bound of every partial sum; fp32
rounding of D + H + 2 = 194 operations stays below 194 * 2^-24 < 2^-16 of it).
Positions a row does not score must keep their prior contents. The selection over
the produced rows is bit-exact with the oracle's selection over the same fp32 rows;
against the fp64 scores, only near-ties at the k-th boundary may differ.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W
from oracle import logits as LG

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import PagedTopK, binding as B  # noqa: E402
from tests._gpu import compare_with_oracle  # noqa: E402

TOL = 2.0 ** -16
SENTINEL = np.float32(-7.25e33)


def _dev(b):
    d = dict(q=torch.from_numpy(np.ascontiguousarray(b.q)).cuda(),
             w=torch.from_numpy(b.w).cuda(),
             lens=torch.from_numpy(b.lens).cuda(),
             gt=None if b.group_table is None else torch.from_numpy(b.group_table).cuda(),
             table=torch.from_numpy(b.block_table).cuda(),
             cache=torch.from_numpy(b.cache).cuda(),
             scale=torch.from_numpy(b.cache_scale).cuda())
    return d


def run_logits(b, dev=None, ld=None):
    dev = dev or _dev(b)
    ld = ld or W.round_up(max(b.max_len, 1), 4)
    scores = torch.full((b.rows, ld), float(SENTINEL), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.indexer_mqa_logits(dev["q"], dev["w"], dev["lens"], b.max_len, b.group_rows, dev["gt"],
                         dev["table"], b.page_size, dev["cache"], dev["scale"], scores, status)
    torch.cuda.synchronize()
    return scores.cpu().numpy(), int(status.item())


def check_rows(b, got, rows=None, positions=None):
    """Scored positions within TOL of the oracle (all, or the given sample); unscored
    positions untouched. Returns the largest |error| / magnitude seen."""
    worst = 0.0
    for t in (range(b.rows) if rows is None else rows):
        if LG.row_error(b, t):
            assert np.all(got[t] == SENTINEL), f"row {t} has a row error but was written"
            continue
        L = int(b.lens[t])
        pos = np.arange(L) if positions is None else positions[(positions < L)]
        ref, _ = LG.scores_at(b, t, pos)
        mag = LG.magnitude_at(b, t, pos)
        g = got[t, pos].astype(np.float64)
        inf = np.isinf(ref)
        assert np.array_equal(np.isinf(g), inf) and np.all(g[inf] == ref[inf]), f"row {t}: -inf"
        err = np.abs(g[~inf] - ref[~inf])
        lim = TOL * mag[~inf] + 1e-30
        bad = np.nonzero(err > lim)[0]
        assert len(bad) == 0, (f"row {t}: {len(bad)} scores off, first at position "
                               f"{pos[~inf][bad[0]]}: got {g[~inf][bad[0]]}, want {ref[~inf][bad[0]]}")
        if len(err):
            worst = max(worst, float(np.max(err / (mag[~inf] + 1e-300))))
        if positions is None:
            assert np.all(got[t, L:] == SENTINEL), f"row {t}: positions past its length written"
    return worst


@pytest.mark.parametrize("G", [1, 3, 4, 5, 7, 8])
def test_groups_and_ragged_rows(G):
    """Groups of every width class (one half, both halves), rows of several tiles with
    ragged tails, empty rows, a partial last group, shuffled table rows."""
    rng = np.random.default_rng(G)
    rows = 2 * G + 1
    lens = rng.integers(0, 1300, rows).astype(np.int32)
    lens[0], lens[1] = 1300, 0
    b = W.logits_batch(f"g{G}", 100 + G, lens, G, n_tables=rows + 2, spare_pages=4)
    got, st = run_logits(b)
    assert st == 0, st
    check_rows(b, got)


@pytest.mark.parametrize("page_size", [64, 128, 256])
def test_page_sizes(page_size):
    b = W.logits_batch(f"p{page_size}", 7, [1000, 999, 64, 65, 1], 5, page_size=page_size,
                       n_tables=3, spare_pages=2)
    got, st = run_logits(b)
    assert st == 0
    check_rows(b, got)


def test_special_gates_and_keys():
    """Zero gates give zero; negated gates negate the score; all-zero keys score zero;
    saturated codes (+-448) everywhere in one key."""
    b = W.logits_batch("special", 11, [700, 700, 700], 3)
    w = b.w.copy()
    w[1] = 0.0
    w[2] = -w[0]
    q = b.q.copy()
    q[2] = q[0]
    cache = b.cache.copy()
    s = b.block_table[0, 0] * b.page_size  # slots of positions 0.. of the group's first page
    cache[s + 3] = 0
    cache[s + 5] = 0x7E
    cache[s + 6] = 0xFE
    b = dataclasses.replace(b, w=w, q=q, cache=cache)
    got, st = run_logits(b)
    assert st == 0
    check_rows(b, got)
    assert np.all(got[1, :700] == 0.0)
    assert np.array_equal(got[2, :700], -got[0, :700])
    assert got[0, 3] == 0.0


def test_bad_pages_slots_and_rows():
    b = W.logits_batch("bad", 13, [600, 600, 600, 600, 600, 600], 2, page_size=64,
                       n_tables=5, spare_pages=1)
    tab = b.block_table.copy()
    gt = b.group_table.copy()
    tab[gt[0], 3] = -1                              # group 0: positions 192..255 have no page
    tab[gt[0], 5] = b.num_slots // b.page_size + 2  # group 0: 320..383 past the cache
    lens = b.lens.copy()
    lens[3] = b.max_len + 1                         # row 3 (group 1): too long
    gt[2] = 17                                      # group 2: no such table row
    bad = dataclasses.replace(b, block_table=tab, group_table=gt, lens=lens)
    got, st = run_logits(bad)
    assert st == (B.LOGITS_STATUS_TABLE_ENTRY | B.LOGITS_STATUS_SLOT | B.LOGITS_STATUS_LEN |
                  B.LOGITS_STATUS_TABLE_ROW), st
    _, want = LG.mqa_logits(bad)
    assert st == want
    check_rows(bad, got)
    narrow = dataclasses.replace(b, block_table=b.block_table[:, :8])  # 512 positions at most
    got, st = run_logits(narrow)
    assert st == B.LOGITS_STATUS_TABLE_WIDTH
    assert np.all(got == SENTINEL)


def test_argument_errors():
    b = W.logits_batch("args", 15, [100, 100], 2)
    d = _dev(b)
    sc = torch.zeros((2, 128), dtype=torch.float32, device="cuda")

    def call(**kw):
        a = dict(q=d["q"], w=d["w"], lens=d["lens"], max_len=b.max_len, group_rows=2,
                 group_table=None, block_table=d["table"], page_size=64, cache=d["cache"],
                 cache_scale=d["scale"], scores=sc)
        a.update(kw)
        with pytest.raises(B.LogitsError) as e:
            B.indexer_mqa_logits(**a)
        return e.value.code

    assert call(group_rows=9) == B.LOGITS_ERR_SHAPE
    assert call(page_size=32) == B.LOGITS_ERR_SHAPE
    assert call(page_size=96) == B.LOGITS_ERR_SHAPE
    assert call(max_len=200) == B.LOGITS_ERR_SHAPE  # ld 128 < max_len
    assert call(q=d["q"][:, :32]) == B.LOGITS_ERR_SHAPE  # 32 heads
    assert call(cache=d["cache"].view(-1)[8:8 + 128 * 100].view(100, 128)) == B.LOGITS_ERR_ALIGN
    wbuf = torch.zeros(2 * 64 + 4, dtype=torch.float32, device="cuda")
    assert call(w=wbuf[1:129].view(2, 64)) == B.LOGITS_ERR_ALIGN
    sbuf = torch.zeros(b.num_slots + 4, dtype=torch.float32, device="cuda")
    assert call(cache_scale=sbuf[1:1 + b.num_slots]) == B.LOGITS_ERR_ALIGN
    assert call(lens=None) == B.LOGITS_ERR_NULL


def test_verify_80k_all_positions():
    b = W.logits_verify_80k()
    got, st = run_logits(b)
    assert st == 0
    worst = check_rows(b, got)
    print(f"verify_80k: largest |error| / magnitude = {worst:.3e}")


def test_verify_1m_sampled_positions():
    """Every position of the first and last tiles and 30000 random positions per row,
    at the launch shape the benchmark times."""
    b = W.logits_verify_1m()
    got, st = run_logits(b)
    assert st == 0
    rng = np.random.default_rng(1)
    pos = np.unique(np.concatenate([np.arange(256), np.arange(b.max_len - 300, b.max_len),
                                    rng.integers(0, b.max_len, 30000)]))
    worst = check_rows(b, got, positions=pos)
    print(f"verify_1m: largest |error| / magnitude = {worst:.3e}")
    for t in range(b.rows):
        assert np.all(got[t, int(b.lens[t]):] == SENTINEL)


def test_produced_rows_feed_the_selection():
    """indexer_mqa_logits then topk_plan + topk_select_paged on the produced rows: the
    selection is bit-exact with the oracle's on the same fp32 rows, and against the
    fp64 scores every difference is a near-tie at the k-th boundary."""
    b = W.logits_verify_80k()
    dev = _dev(b)
    got, st = run_logits(b, dev)
    assert st == 0
    r2t = b.row_to_table()
    sc = got.copy()
    for t in range(b.rows):
        sc[t, int(b.lens[t]):] = W.POISON
    tb = W.Batch("produced", sc, b.lens, b.max_len, b.k, b.block_table, r2t, b.page_size)
    scores = torch.from_numpy(sc).cuda()
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev["lens"])
    out = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    pos = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    core.select(scores, dev["lens"], b.k, dev["table"], b.page_size,
                torch.from_numpy(r2t).cuda(), out_slots=out, out_pos=pos)
    torch.cuda.synchronize()
    assert core.status() == 0
    compare_with_oracle(tb, b.k, out.cpu().numpy(), pos.cpu().numpy())
    ref, _ = LG.mqa_logits(b)
    for t in range(b.rows):
        L = int(b.lens[t])
        sel = set(pos.cpu().numpy()[t].tolist())
        exact = ref[t, :L]
        order = np.lexsort((np.arange(L), -exact))
        want = set(order[:b.k].tolist())
        kth = exact[order[b.k - 1]]
        mag = LG.magnitude_at(b, t, np.arange(L))
        for p in sel ^ want:
            assert abs(exact[p] - kth) <= 2 * TOL * mag[p], f"row {t} position {p}"
