"""Pins of the CPU oracle to things other than itself (no GPU needed).

* brute-force rank counting on the 1000 tiny tie-heavy rows (no sort at all);
* hand-worked fixtures under tests/golden/;
* closed forms: all-equal rows, len <= k, monotone rows, k = 1 argmax, identity tables;
* invariants on every synthetic workload;
* a library cross-check (std::nth_element) of the std::sort path;
* pin strength: each deliberately wrong oracle variant fails at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import workloads as W
from tests import _checks as C

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def brute_force_positions(s: np.ndarray, L: int, k: int) -> np.ndarray:
    """Position p is chosen iff #{q : q ranks before p} < k; returns the chosen
    positions in rank order. O(L^2) comparisons, no sorting."""
    x = s[:L].astype(np.float64)
    nan = np.isnan(x)
    q = np.arange(L)
    # beats[q, p]: q ranks before p
    gt = (x[:, None] > x[None, :]) & ~nan[:, None] & ~nan[None, :]
    eq = ((x[:, None] == x[None, :]) & ~nan[:, None] & ~nan[None, :]) | (nan[:, None] & nan[None, :])
    num_over_nan = (~nan[:, None]) & nan[None, :]
    beats = gt | num_over_nan | (eq & (q[:, None] < q[None, :]))
    rank = beats.sum(axis=0)
    m = min(k, L)
    out = np.full(m, -1, dtype=np.int64)
    for p in range(L):
        if rank[p] < m:
            out[rank[p]] = p
    return out


def _run(b, k=None, mutant=0, **kw):
    return oracle.topk_batch(b, k=k, mutant=mutant, **kw)


def _table_row(b, r):
    t = r if b.row_to_table is None else int(b.row_to_table[r])
    return b.block_table[t]


# ---------------------------------------------------------------- pin functions
# Each returns None when the oracle variant passes and a message when it fails,
# so the pin-strength test can run them against mutants too.

def pin_brute_force(mutant=0):
    for b in W.tiny_rows() + W.tiny_rows(seed=W.SEED_BASE + 11, page_size=8):
        slots, pos, err = _run(b, mutant=mutant)
        if err:
            return f"{b.name}: error bits {err}"
        for r in range(b.rows):
            L = int(b.lens[r])
            exp = brute_force_positions(b.scores[r], L, b.k)
            m = exp.size
            if not np.array_equal(pos[r, :m], exp) or np.any(pos[r, m:] != -1):
                return f"{b.name} row {r}: positions {pos[r, :m]} != brute force {exp}"
            es = C.slot_of(_table_row(b, r), exp, b.page_size)
            if not np.array_equal(slots[r, :m], es) or np.any(slots[r, m:] != -1):
                return f"{b.name} row {r}: slots differ from the table lookup"
    return None


def pin_golden(mutant=0):
    with open(GOLDEN) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        rows = np.array([[float(v) for v in row] for row in c["rows"]], dtype=np.float32)
        r2t = None if c["row_to_table"] is None else np.array(c["row_to_table"], np.int32)
        slots, pos, err = oracle.topk_paged(rows, np.array(c["lens"], np.int32), c["max_len"],
                                            c["k"], np.array(c["block_table"], np.int32), r2t,
                                            c["page_size"], mutant=mutant)
        if not np.array_equal(pos, np.array(c["expect_pos"])):
            return f"{c['name']}: positions {pos.tolist()} != {c['expect_pos']}"
        if not np.array_equal(slots, np.array(c["expect_slots"])):
            return f"{c['name']}: slots {slots.tolist()} != {c['expect_slots']}"
    return None


def pin_closed_forms(mutant=0):
    rng = np.random.default_rng(7)
    ps = 16
    L = 1000
    table = rng.permutation(64).astype(np.int32).reshape(1, -1)
    ident = np.arange(64, dtype=np.int32).reshape(1, -1)
    cases = []
    # all-equal row -> positions 0..k-1
    cases.append(("all_equal", np.full(L, 0.25, np.float32), 100, np.arange(100)))
    # len <= k -> every position (equal to len), sorted: here strictly decreasing
    dec = np.linspace(5, -5, L).astype(np.float32)
    cases.append(("len_le_k", dec, 2048, np.arange(L)))
    # strictly increasing -> the last k positions, largest first
    inc = np.linspace(-3, 7, L).astype(np.float32)
    cases.append(("increasing", inc, 37, np.arange(L - 1, L - 38, -1)))
    # k = 1 -> first maximum (np.argmax returns the first occurrence)
    v = rng.integers(0, 5, L).astype(np.float32)
    cases.append(("argmax", v, 1, np.array([int(np.argmax(v))])))
    # -inf tail selected only once the finite values are exhausted
    t = np.full(L, -np.inf, np.float32)
    t[:10] = np.arange(10, 0, -1)
    cases.append(("neg_inf_tail", t, 15, np.arange(15)))
    # NaNs rank below -inf
    n = np.full(L, np.nan, np.float32)
    n[500] = -np.inf
    cases.append(("nan_below_neg_inf", n, 3, np.array([500, 0, 1])))
    # signed zeros tie with each other
    z = np.where(np.arange(L) % 2 == 0, np.float32(-0.0), np.float32(0.0)).astype(np.float32)
    z[999] = -1.0
    cases.append(("signed_zeros", z, 5, np.arange(5)))
    for name, row, k, exp in cases:
        for tab, tname in ((table, "perm"), (ident, "identity")):
            slots, pos, err = oracle.topk_paged(row.reshape(1, -1), np.array([L], np.int32), L, k,
                                                tab, None, ps, mutant=mutant)
            m = min(k, L)
            if not np.array_equal(pos[0, :m], exp):
                return f"{name}: positions differ from the closed form"
            es = C.slot_of(tab[0], exp, ps)
            if not np.array_equal(slots[0, :m], es):
                return f"{name}/{tname}: slots differ"
            if tname == "identity" and not np.array_equal(slots[0, :m], exp):
                return f"{name}: identity table must give slot == position"
    return None


def pin_invariants(mutant=0, big=False):
    batches = [W.pr1(), W.mixed_decode(), W.prefill(prefixes=(2048, 5000), q=(512, 300))]
    adv = W.adversarial()
    batches += [adv]
    if big:
        batches += [W.verify_80k(), W.verify_1m()]
    for b in batches:
        ks = b.ks if b.ks else [b.k]
        for k in ks:
            slots, pos, err = _run(b, k=k, mutant=mutant, threads=8)
            if err:
                return f"{b.name}: error bits {err}"
            try:
                C.check_batch(b.scores, b.lens, k, b.block_table, b.row_to_table, b.page_size,
                              slots, pos)
                C.check_batch(b.scores, b.lens, k, b.block_table, b.row_to_table, b.page_size,
                              slots, None)
            except AssertionError as e:
                return f"{b.name} k={k}: {e}"
    return None


def pin_errors(mutant=0):
    s = np.arange(8, dtype=np.float32).reshape(1, -1)
    tab = np.array([[3, 4]], np.int32)
    # length above max_len -> row of -1 and the length bit
    slots, _, err = oracle.topk_paged(s, np.array([9], np.int32), 8, 2, tab, None, 4, mutant=mutant)
    if err != oracle.ERR_LEN or np.any(slots != -1):
        return "len > max_len not reported"
    # pages beyond the table width
    slots, _, err = oracle.topk_paged(s, np.array([8], np.int32), 8, 2, tab, None, 2, mutant=mutant)
    if err != oracle.ERR_TABLE_WIDTH or np.any(slots != -1):
        return "table width not reported"
    # a negative entry gives -1 for that entry only
    slots, pos, err = oracle.topk_paged(s, np.array([8], np.int32), 8, 8,
                                        np.array([[-1, 5]], np.int32), None, 4, mutant=mutant)
    if err != oracle.ERR_TABLE_ENTRY or list(slots[0]) != [23, 22, 21, 20, -1, -1, -1, -1]:
        return "negative table entry not reported per entry"
    # slot overflow in 32 bits
    slots, pos, err = oracle.topk_paged(s, np.array([8], np.int32), 8, 1,
                                        np.array([[0, 2**31 // 4]], np.int32), None, 4, mutant=mutant)
    if err != oracle.ERR_SLOT_OVERFLOW or slots[0, 0] != -1:
        return "slot overflow not reported"
    return None


PINS = [pin_brute_force, pin_golden, pin_closed_forms, pin_invariants, pin_errors]


# ---------------------------------------------------------------- the tests

@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_oracle_pin(pin):
    msg = pin()
    assert msg is None, msg


@pytest.mark.slow
def test_oracle_invariants_long_rows():
    msg = pin_invariants(big=True)
    assert msg is None, msg


def test_nth_element_cross_check():
    for b in ([W.pr1(), W.mixed_decode(), W.adversarial(),
               W.prefill(prefixes=(2048, 5000), q=(512, 300))] + W.tiny_rows()):
        for k in (b.ks or [b.k]):
            s1, p1, e1 = oracle.topk_batch(b, k=k, threads=4)
            s2, p2, e2 = oracle.topk_batch(b, k=k, threads=4, use_nth=True)
            assert e1 == e2
            assert np.array_equal(p1, p2), b.name
            assert np.array_equal(s1, s2), b.name


def test_thread_count_does_not_change_result():
    b = W.mixed_decode()
    a = oracle.topk_batch(b, threads=1)
    c = oracle.topk_batch(b, threads=8)
    assert np.array_equal(a[0], c[0]) and np.array_equal(a[1], c[1])


MUTANTS = {
    1: "ties to the larger position",
    2: "ascending order",
    3: "slot without the in-page offset",
    4: "one entry short",
    5: "NaN not demoted",
    6: "bitwise signed compare (-0 != +0)",
    7: "row_to_table ignored",
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS), ids=lambda m: MUTANTS[m])
def test_pin_strength(mutant):
    """A plausible mistake planted in the oracle (compiled on the CPU only) must be
    caught by at least one pin."""
    failures = [p.__name__ for p in PINS if p(mutant=mutant) is not None]
    assert failures, f"mutant {mutant} ({MUTANTS[mutant]}) passed every pin"


def test_workload_shapes():
    b = W.verify_80k()
    assert b.scores.shape == (7, 80008) and list(b.lens) == list(range(80000, 80007))
    assert b.block_table.shape == (1, 1251)
    assert sorted(b.block_table[0].tolist()) == list(range(1251))
    assert b.algorithmic_bytes() == 2_302_432
    a = W.adversarial()
    assert a.rows == 256 and a.page_size == 32 and sorted(a.ks) == [1, 64, 512, 2048]
    assert (a.lens == 0).any() and (a.lens == 32768).any()
    m = W.mixed_decode()
    assert m.lens.min() >= 1024 and m.lens.max() <= 200000
