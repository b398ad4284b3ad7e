"""Pins of the indexer score-producer oracle (oracle/logits.py) to things other than
itself (no GPU needed):

* a hand-worked case under tests/golden/ (paging, groups, both signs of the per-head
  products, an all-zero key, a key scale per slot);
* mathematics that holds for any input: a zero gate gives zero; scores are linear in
  the gate and in the key scales; permuting the heads of queries and gates together
  changes nothing; and, because max(0, x) - max(0, -x) = x and
  max(0, x) + max(0, -x) = |x|, negating the queries splits every score into a
  closed form (one combined query vector against each key) and an absolute-value
  form, both computed here through slots expanded independently of the oracle;
* brute force over tiny inputs with Python floats;
* status bits and unscored positions for each kind of bad input;
* pin strength: each deliberately wrong oracle variant fails at least one pin.
"""
import dataclasses
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import logits as LG

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "logits_hand_worked.json")


def _golden_batch():
    with open(GOLDEN) as f:
        g = json.load(f)
    D, H = g["dim"], g["heads"]
    cache = np.zeros((g["num_slots"], D), np.uint8)
    for s, chans in g["cache"].items():
        for d, code in chans.items():
            cache[int(s), int(d)] = int(code, 16)
    q = np.zeros((len(g["lens"]), H, D), np.uint8)
    for t, heads in enumerate(g["q"]):
        for h, chans in enumerate(heads):
            for d, code in chans.items():
                q[t, h, int(d)] = int(code, 16)
    b = W.LogitsBatch("golden", q, np.array(g["w"], np.float32), cache,
                      np.array(g["cache_scale"], np.float32), np.array(g["lens"], np.int32),
                      g["max_len"], g["group_rows"], np.array(g["group_table"], np.int32),
                      np.array(g["block_table"], np.int32), g["page_size"], 2)
    exp = np.array([[np.nan if v is None else v for v in row] for row in g["expected"]])
    return b, exp


def _small(seed=3, lens=(37, 50, 0, 64, 19), G=2, page_size=4, heads=5, n_tables=4):
    return W.logits_batch("small", seed, lens, G, heads=heads, page_size=page_size,
                          n_tables=n_tables, spare_pages=3)


def _expanded_slots(b, t):
    """Slot of every position of row t, by expanding the table row page by page."""
    g = t // b.group_rows
    r = g if b.group_table is None else int(b.group_table[g])
    pages = b.block_table[r].astype(np.int64)
    per_page = pages[:, None] * b.page_size + np.arange(b.page_size)[None, :]
    return per_page.reshape(-1)[:int(b.lens[t])]


def _decoded(codes):
    """e4m3 values of codes, from a 256-entry table built from the bit fields."""
    table = np.empty(256)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        table[c] = -mag if s else mag
    return table[np.asarray(codes, np.int64)]


def _neg(b):
    return dataclasses.replace(b, q=(b.q ^ np.uint8(0x80)).astype(np.uint8))


def _scored(out):
    return ~np.isnan(out)


# --------------------------------------------------------------------- the pins
def check_golden(mutant=0):
    b, exp = _golden_batch()
    out, st = LG.mqa_logits(b, mutant)
    return st == 0 and np.array_equal(_scored(out), _scored(exp)) and \
        np.array_equal(out[_scored(exp)], exp[_scored(exp)])


def check_closed_forms(b, mutant=0):
    """s(q) - s(-q) against one combined query per row; s(q) + s(-q) against the
    absolute form. Both through independently expanded slots."""
    pos_out, st1 = LG.mqa_logits(b, mutant)
    neg_out, st2 = LG.mqa_logits(_neg(b), mutant)
    if st1 or st2:
        return False
    for t in range(b.rows):
        L = int(b.lens[t])
        if L == 0:
            continue
        s = _expanded_slots(b, t)
        kv = _decoded(b.cache[s])
        qv = _decoded(b.q[t])
        g = b.w[t].astype(np.float64)
        sk = b.cache_scale[s].astype(np.float64)
        combined = (g[:, None] * qv).sum(axis=0)           # sum_h g_h q_h
        diff = sk * (kv @ combined)
        absf = sk * (np.abs(kv @ qv.T) @ g)
        mag = LG.magnitude_at(b, t, np.arange(L)) + 1e-300
        if not np.all(np.abs((pos_out[t, :L] - neg_out[t, :L]) - diff) <= 1e-12 * mag):
            return False
        if not np.all(np.abs((pos_out[t, :L] + neg_out[t, :L]) - absf) <= 1e-12 * mag):
            return False
    return True


def test_golden_hand_worked():
    assert check_golden()


def test_golden_decodes():
    b, _ = _golden_batch()
    assert _decoded([0x38, 0x40, 0xB8, 0x30, 0x44, 0x48, 0xC0, 0x3C, 0x28, 0x7E]).tolist() == \
        [1.0, 2.0, -1.0, 0.5, 3.0, 4.0, -2.0, 1.5, 0.25, 448.0]
    assert np.array_equal(_decoded(b.cache), LG.e4m3_value(b.cache))


@pytest.mark.parametrize("seed", [1, 2])
def test_closed_forms(seed):
    assert check_closed_forms(_small(seed))


def test_closed_forms_workload_sample():
    """The same on a slice of the 80K verify workload's shapes (64 heads, pages of 64)."""
    b = W.logits_batch("mid", 5, np.arange(3000, 3003), 3)
    assert check_closed_forms(b)


def test_zero_gate_gives_zero():
    b = _small()
    out, st = LG.mqa_logits(dataclasses.replace(b, w=np.zeros_like(b.w)))
    assert st == 0
    sc = _scored(out)
    assert sc.sum() == int(b.lens.sum()) and np.all(out[sc] == 0.0)


def test_linear_in_gate_and_key_scale():
    b = _small(seed=7)
    rng = np.random.default_rng(8)
    w2 = (rng.standard_normal(b.w.shape) / 8).astype(np.float32)
    s1, _ = LG.mqa_logits(b)
    s2, _ = LG.mqa_logits(dataclasses.replace(b, w=w2))
    s3, _ = LG.mqa_logits(dataclasses.replace(
        b, w=2.0 * b.w.astype(np.float64) - 3.0 * w2.astype(np.float64)))
    sc = _scored(s1)
    mag = np.zeros_like(s1)
    for t in range(b.rows):
        L = int(b.lens[t])
        m1 = LG.magnitude_at(b, t, np.arange(L))
        m2 = LG.magnitude_at(dataclasses.replace(b, w=w2), t, np.arange(L))
        mag[t, :L] = 2 * m1 + 3 * m2
    assert np.all(np.abs(s3[sc] - (2 * s1[sc] - 3 * s2[sc])) <= 1e-13 * mag[sc] + 1e-300)
    s4, _ = LG.mqa_logits(dataclasses.replace(b, cache_scale=2 * b.cache_scale))
    assert np.array_equal(s4[sc], 2 * s1[sc])


def test_head_permutation():
    b = _small(seed=9)
    perm = np.random.default_rng(10).permutation(b.heads)
    s1, _ = LG.mqa_logits(b)
    s2, _ = LG.mqa_logits(dataclasses.replace(b, q=b.q[:, perm], w=b.w[:, perm]))
    sc = _scored(s1)
    assert np.allclose(s2[sc], s1[sc], rtol=1e-13, atol=1e-300)
    s3, _ = LG.mqa_logits(dataclasses.replace(b, w=b.w[:, perm]))  # gates alone moved
    assert not np.allclose(s3[sc], s1[sc], rtol=1e-6)


def test_paging_does_not_change_scores():
    """The same keys behind another page layout (a contiguous cache, identity table)
    give the same scores."""
    b = _small(seed=11, G=5, lens=(40, 33, 12, 40, 7))
    s1, _ = LG.mqa_logits(b)
    s = _expanded_slots(b, 0)  # group 0 holds every row; row 0 is the longest
    flat = dataclasses.replace(b, cache=b.cache[s], cache_scale=b.cache_scale[s],
                               block_table=np.arange(-(-40 // b.page_size), dtype=np.int32)[None, :],
                               group_table=None)
    s2, _ = LG.mqa_logits(flat)
    sc = _scored(s1)
    assert np.array_equal(sc, _scored(s2))
    assert np.allclose(s2[sc], s1[sc], rtol=1e-13, atol=1e-300)


def test_brute_force_tiny():
    b = _small(seed=12, lens=(9, 3, 6), G=2, page_size=3, heads=3, n_tables=3)
    out, st = LG.mqa_logits(b)
    assert st == 0
    for t in range(b.rows):
        g = t // b.group_rows
        r = int(b.group_table[g]) if b.group_table is not None else g
        for p in range(int(b.lens[t])):
            slot = int(b.block_table[r, p // b.page_size]) * b.page_size + p % b.page_size
            tot = 0.0
            for h in range(b.heads):
                a = 0.0
                for d in range(b.dim):
                    a += float(_decoded(b.q[t, h, d])) * float(_decoded(b.cache[slot, d]))
                tot += float(b.w[t, h]) * max(a, 0.0)
            ref = float(b.cache_scale[slot]) * tot
            assert abs(out[t, p] - ref) <= 1e-12 * abs(ref) + 1e-300


def test_sampled_positions_match_full_rows():
    b = _small(seed=13)
    full, _ = LG.mqa_logits(b)
    pos = np.array([0, 5, 17, 36])
    part, st = LG.scores_at(b, 0, pos)
    assert st == 0 and np.array_equal(part, full[0, pos])


def test_status_and_unscored_positions():
    b = _small(seed=14, lens=(20, 20, 20, 20, 20), G=1, page_size=4, n_tables=6)
    tab = b.block_table.copy()
    gt = b.group_table.copy()
    tab[gt[0], 2] = -5                            # row 0: positions 8..11 have no page
    tab[gt[1], 4] = b.num_slots // b.page_size    # row 1: positions 16..19 past the cache
    lens = b.lens.copy()
    lens[2] = b.max_len + 1                       # row 2: longer than max_len
    gt[3] = 99                                    # row 3: no such table row
    bad = dataclasses.replace(b, block_table=tab, group_table=gt, lens=lens)
    out, st = LG.mqa_logits(bad)
    assert st == LG.ERR_TABLE_ENTRY | LG.ERR_SLOT | LG.ERR_LEN | LG.ERR_TABLE_ROW
    assert np.all(out[0, 8:12] == -np.inf) and np.all(np.isfinite(out[0, :8]))
    assert np.all(out[1, 16:20] == -np.inf) and np.all(np.isfinite(out[1, :16]))
    assert np.all(np.isnan(out[2])) and np.all(np.isnan(out[3]))
    assert np.all(np.isfinite(out[4, :20]))
    narrow = dataclasses.replace(b, block_table=b.block_table[:, :4])  # 16 positions at most
    out, st = LG.mqa_logits(narrow)
    assert st == LG.ERR_TABLE_WIDTH and np.all(np.isnan(out))


def test_magnitude_bounds_the_score():
    b = _small(seed=15)
    out, _ = LG.mqa_logits(b)
    for t in range(b.rows):
        L = int(b.lens[t])
        assert np.all(np.abs(out[t, :L]) <= LG.magnitude_at(b, t, np.arange(L)) * (1 + 1e-12))


def test_workload_shapes():
    b = W.logits_verify_80k()
    assert b.rows == 7 and b.group_rows == 7 and b.heads == 64 and b.dim == 128
    assert b.lens.tolist() == list(range(80000, 80007)) and b.page_size == 64
    assert b.block_table.shape == (1, 1251) and np.all(b.block_table >= 0)
    assert len(np.unique(b.block_table)) == 1251 and b.num_slots == 1251 * 64
    for codes in (b.q, b.cache):
        assert not np.any((codes & 0x7F) == 0x7F)  # no NaN pattern
    assert np.all(b.cache_scale > 0)
    assert b.flops() == 2 * sum(range(80000, 80007)) * 64 * 128


@pytest.mark.parametrize("mutant", sorted(LG.MUTANTS))
def test_every_mutant_fails_a_pin(mutant):
    ok = check_golden(mutant) and all(check_closed_forms(_small(s), mutant) for s in (1, 2))
    assert not ok, f"mutant {mutant} ({LG.MUTANTS[mutant]}) passes every pin"
