"""Pins of the top-K resolver oracle (oracle/resolver.py) to things other than itself
(no GPU needed):

* hand-worked steps under tests/golden/ (residency, misses into free slots, a hit that
  refreshes its slot, an eviction of the least recently used slot, exhaustion);
* an independent reference that picks victims with a heap (lazy invalidation) instead
  of a sort, over multi-step sequences;
* invariants after every step: the position map and the slot map are inverse, every
  selected position reads a row holding its data, resident and foreign rows untouched,
  counts add up, no slot used at the step was evicted;
* closed forms: an all-resident selection leaves the hot state alone; a repeated
  selection hits every time and copies nothing;
* pin strength: each deliberately wrong variant fails at least one pin.
"""
import heapq
import json
import os

import numpy as np
import pytest

import workloads as W
from oracle import resolver as RV

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "resolver_hand_worked.json")


def fresh_state(b):
    R, H = b.rows, b.hot_size
    return (np.full((R, int(b.lens.max())), -1, np.int32), np.full((R, H), -1, np.int32),
            np.full((R, H), -1, np.int32))


def run_steps(b, mutant=0, steps=None):
    t2h, ht, hs = fresh_state(b)
    kv = b.kv_init.copy()
    outs = []
    for s, sel in enumerate(b.steps if steps is None else steps):
        out, counts, err = RV.resolve_step(sel, b.block_table, b.page_size, t2h, ht, hs,
                                           b.hot_rows, s, b.host_kv, b.host_base, kv, mutant)
        outs.append((out, counts, err, t2h.copy(), ht.copy(), hs.copy(), kv.copy()))
    return outs


def heap_reference(b, steps=None):
    """The same policy with a different mechanism: victims popped from a min-heap of
    (last step, slot) entries, stale entries skipped."""
    R, H = b.rows, b.hot_size
    t2h = [dict() for _ in range(R)]
    slot_tok = [[-1] * H for _ in range(R)]
    slot_step = [[-1] * H for _ in range(R)]
    heaps = [[(-1, h) for h in range(H)] for _ in range(R)]
    for hp in heaps:
        heapq.heapify(hp)
    kv = b.kv_init.copy()
    res = []
    for s, sel in enumerate(b.steps if steps is None else steps):
        out = np.full(sel.shape, -1, np.int32)
        counts = np.zeros((R, 3), np.int32)
        err = 0
        for j in range(R):
            miss = []
            for i, p in enumerate(sel[j]):
                p = int(p)
                if p < 0:
                    continue
                blk = int(b.block_table[j, p // b.page_size])
                if blk >= 0:
                    out[j, i] = blk * b.page_size + p % b.page_size
                    counts[j, 0] += 1
                elif p in t2h[j]:
                    h = t2h[j][p]
                    out[j, i] = b.hot_rows[j, h]
                    slot_step[j][h] = s
                    heapq.heappush(heaps[j], (s, h))
                    counts[j, 1] += 1
                else:
                    miss.append(i)
            for i in miss:
                p = int(sel[j, i])
                v = None
                while heaps[j]:
                    st, h = heapq.heappop(heaps[j])
                    if st == slot_step[j][h] and st < s:
                        v = h
                        break
                if v is None:
                    err |= RV.ERR_NO_VICTIM
                    continue
                old = slot_tok[j][v]
                if old >= 0:
                    del t2h[j][old]
                slot_tok[j][v] = p
                t2h[j][p] = v
                slot_step[j][v] = s
                heapq.heappush(heaps[j], (s, v))
                kv[b.hot_rows[j, v]] = b.host_kv[b.host_base[j] + p]
                out[j, i] = b.hot_rows[j, v]
                counts[j, 2] += 1
            # entries still valid but used at this step go back for the next steps
        res.append((out, counts, err, kv.copy()))
    return res


def _small(seed=0, **kw):
    a = dict(reqs=3, k=64, lens=[3000, 900, 70], tail=256, row_bytes=16, n_steps=6)
    a.update(kw)
    return W.hisparse(seed=W.SEED_BASE + 700 + seed, **a)


# ---------------------------------------------------------------- pin functions

def pin_golden(mutant=0):
    g = json.load(open(GOLDEN))
    tab = np.asarray(g["block_table"], np.int32)
    hot_rows = np.asarray(g["hot_rows"], np.int32)
    npos = g["positions_max"]
    host = np.array([[10 * p + 1, 10 * p + 2] for p in range(npos)], np.uint8)
    kv = np.full((32, 2), 255, np.uint8)
    t2h = np.full((1, npos), -1, np.int32)
    ht = np.full((1, 2), -1, np.int32)
    hs = np.full((1, 2), -1, np.int32)
    for s, st in enumerate(g["steps"]):
        out, counts, err = RV.resolve_step(np.asarray(st["positions"], np.int32), tab,
                                           g["page_size"], t2h, ht, hs, hot_rows, s, host,
                                           np.array([0], np.int64), kv, mutant)
        if out.tolist() != st["rows"] or counts.tolist() != st["counts"] or err != st["status"]:
            return f"step {s}: rows {out.tolist()} counts {counts.tolist()} status {err}"
        if ht.tolist() != st["hot_token"] or hs.tolist() != st["hot_step"]:
            return f"step {s}: hot state {ht.tolist()} {hs.tolist()}"
        for r, v in st["kv"].items():
            if kv[int(r)].tolist() != v:
                return f"step {s}: kv row {r} = {kv[int(r)].tolist()}"
    return None


def pin_heap_reference(mutant=0):
    for seed, kw in ((0, {}), (1, dict(k=40, keep=0.3)), (2, dict(k=64, keep=0.95, n_steps=10))):
        b = _small(seed, **kw)
        got = run_steps(b, mutant)
        ref = heap_reference(b)
        for s, ((o, c, e, *_, kv), (ro, rc, re, rkv)) in enumerate(zip(got, ref)):
            if not (np.array_equal(o, ro) and np.array_equal(c, rc) and e == re and
                    np.array_equal(kv, rkv)):
                return f"seed {seed} step {s}: differs from the heap reference"
    return None


def pin_invariants(mutant=0):
    b = _small(3, k=48, keep=0.6, n_steps=8)
    resident_rows = set()
    for j in range(b.rows):
        for pg in np.nonzero(b.block_table[j] >= 0)[0]:
            blk = int(b.block_table[j, pg])
            resident_rows.update(range(blk * b.page_size, (blk + 1) * b.page_size))
    hot = set(int(x) for x in b.hot_rows.ravel())
    for s, (out, counts, err, t2h, ht, hs, kv) in enumerate(run_steps(b, mutant)):
        sel = b.steps[s]
        for j in range(b.rows):
            for h in range(b.hot_size):
                p = int(ht[j, h])
                if p >= 0 and int(t2h[j, p]) != h:
                    return f"step {s}: slot {h} holds {p} but the map says {t2h[j, p]}"
            for p in np.nonzero(t2h[j] >= 0)[0]:
                if int(ht[j, t2h[j, p]]) != p:
                    return f"step {s}: position {p} maps to a slot holding {ht[j, t2h[j, p]]}"
            for i, p in enumerate(sel[j]):
                p = int(p)
                if p < 0 or out[j, i] < 0:
                    continue
                blk = int(b.block_table[j, p // b.page_size])
                want = b.kv_init[out[j, i]] if blk >= 0 else b.host_kv[b.host_base[j] + p]
                if not np.array_equal(kv[out[j, i]], want):
                    return f"step {s}: row {out[j, i]} does not hold position {p}'s data"
            if not err and int(counts[j].sum()) != int((sel[j] >= 0).sum()):
                return f"step {s}: counts {counts[j]} do not add up"
            # every selected non-resident position is still in the slot it read from: no
            # slot used at this step was evicted by a later miss of the same step
            for i, p in enumerate(sel[j]):
                p = int(p)
                if p < 0 or out[j, i] < 0 or int(b.block_table[j, p // b.page_size]) >= 0:
                    continue
                h = int(t2h[j, p])
                if h < 0 or int(b.hot_rows[j, h]) != int(out[j, i]) or int(hs[j, h]) != s:
                    return f"step {s}: position {p} lost its slot within the step"
        untouched = [r for r in range(b.kv_rows) if r not in hot]
        if not np.array_equal(kv[untouched], b.kv_init[untouched]):
            return f"step {s}: a row outside the hot buffers was written"
    return None


def pin_closed_forms(mutant=0):
    b = _small(4, k=32)
    # only resident positions: nothing moves
    sel = np.full((b.rows, 32), -1, np.int32)
    for j in range(b.rows):
        res = np.nonzero(np.repeat(b.block_table[j] >= 0, b.page_size)[:int(b.lens[j])])[0]
        sel[j, :min(32, len(res))] = res[:32]
    out = run_steps(b, mutant, steps=[sel])[0]
    if np.any(out[4] != -1) or np.any(out[1][:, 1:] != 0):
        return "an all-resident step touched the hot state"
    # the same selection twice: the second step hits everything and copies nothing
    twice = run_steps(b, mutant, steps=[b.steps[0], b.steps[0]])
    c1 = twice[1][1]
    if np.any(c1[:, 2] != 0) or not np.array_equal(c1[:, 1], twice[0][1][:, 1] + twice[0][1][:, 2]):
        return f"a repeated selection: counts {c1.tolist()}"
    if not np.array_equal(twice[1][0], twice[0][0]):
        return "a repeated selection resolved to other rows"
    return None


def pin_mtp_hand_worked(mutant=0):
    """One request, pages of 2, positions 0..7 all host-only, three hot slots (KV rows
    20, 21, 22), slot 2 last used at step 4, slots 0 and 1 never. Step 5 has two query
    rows: row 0 selects [3, 5], row 1 selects [5, 6, 7].
      row 0: 3 and 5 miss; victims are the slots unused at step 5, least recently used
        first, ties to the lower slot: 0 and 1 (step -1) -> 3 in slot 0 (row 20), 5 in
        slot 1 (row 21);
      row 1: 5 is a hit (slot 1, row 21); 6 misses and takes the only slot not used at
        step 5, slot 2 (row 22), evicting its old position 0; 7 misses with no slot
        left: -1, status 1.
    Counts over the rows: 0 resident, 1 hit, 3 copied."""
    tab = np.full((1, 4), -1, np.int32)
    host = np.array([[10 * p] for p in range(8)], np.uint8)
    kv = np.zeros((32, 1), np.uint8)
    t2h = np.full((1, 8), -1, np.int32)
    t2h[0, 0] = 2
    ht = np.array([[-1, -1, 0]], np.int32)
    hs = np.array([[-1, -1, 4]], np.int32)
    hot_rows = np.array([[20, 21, 22]], np.int32)
    pos = np.array([[[3, 5, -1], [5, 6, 7]]], np.int32)
    out, counts, err = RV.resolve_mtp_step(pos, tab, 2, t2h, ht, hs, hot_rows, 5, host,
                                           np.array([0], np.int64), kv, mutant)
    want = [[[20, 21, -1], [21, 22, -1]]]
    if out.tolist() != want or counts.tolist() != [[0, 1, 3]] or err != RV.ERR_NO_VICTIM:
        return f"rows {out.tolist()} counts {counts.tolist()} status {err}"
    if ht.tolist() != [[3, 5, 6]] or hs.tolist() != [[5, 5, 5]] or int(t2h[0, 0]) != -1:
        return f"hot state {ht.tolist()} {hs.tolist()} map of 0: {t2h[0, 0]}"
    if kv[20, 0] != 30 or kv[21, 0] != 50 or kv[22, 0] != 60:
        return f"kv rows {kv[20:23, 0].tolist()}"
    return None


def pin_mtp_invariants(mutant=0):
    """Over a sequence of generated multi-token steps: after each step, every resolved
    non-resident position of every query row is held by the slot it resolved to, used
    at this step (no row evicts a slot an earlier row used); each position missing
    before the step is copied once whatever the number of rows that select it; the slots
    used at this step are exactly those of the distinct non-resident positions."""
    b = W.hisparse_mtp(seed=W.SEED_BASE + 900, reqs=2, k=48, q_rows=3, lens=[2500, 800],
                       tail=128, row_bytes=16, n_steps=5, draft_new=0.3)
    t2h, ht, hs = (np.full((b.rows, int(b.lens.max())), -1, np.int32),
                   np.full((b.rows, b.hot_size), -1, np.int32),
                   np.full((b.rows, b.hot_size), -1, np.int32))
    kv = b.kv_init.copy()
    for s, st in enumerate(b.steps):
        before = t2h.copy()
        out, counts, err = RV.resolve_mtp_step(st, b.block_table, b.page_size, t2h, ht, hs,
                                               b.hot_rows, s, b.host_kv, b.host_base, kv, mutant)
        if err:
            return f"step {s}: status {err} (the hot buffers hold every row's positions)"
        for j in range(b.rows):
            nonres = set()
            for q in range(st.shape[1]):
                for i, p in enumerate(st[j, q]):
                    p = int(p)
                    if p < 0 or int(b.block_table[j, p // b.page_size]) >= 0:
                        continue
                    nonres.add(p)
                    h = int(t2h[j, p])
                    if h < 0 or int(b.hot_rows[j, h]) != int(out[j, q, i]) or int(hs[j, h]) != s:
                        return f"step {s}: row {q} position {p} lost its slot within the step"
                    if not np.array_equal(kv[out[j, q, i]], b.host_kv[b.host_base[j] + p]):
                        return f"step {s}: row {out[j, q, i]} does not hold position {p}"
            missing = sum(1 for p in nonres if int(before[j, p]) < 0)
            if int(counts[j, 2]) != missing:
                return f"step {s}: {counts[j, 2]} copies for {missing} missing positions"
            if int((hs[j] == s).sum()) != len(nonres):
                return f"step {s}: {(hs[j] == s).sum()} slots used for {len(nonres)} positions"
    return None


def pin_mtp_closed_form(mutant=0):
    """A step whose query rows all select the same positions resolves like one row, and
    the later rows are all hits."""
    b = _small(5, k=40)
    one = run_steps(b, mutant, steps=[b.steps[0]])[0]
    t2h, ht, hs = fresh_state(b)
    kv = b.kv_init.copy()
    pos = np.stack([b.steps[0]] * 3, axis=1)
    out, counts, err = RV.resolve_mtp_step(pos, b.block_table, b.page_size, t2h, ht, hs,
                                           b.hot_rows, 0, b.host_kv, b.host_base, kv, mutant)
    if any(not np.array_equal(out[:, q], one[0]) for q in range(3)):
        return "repeated rows resolved to other rows"
    c1 = one[1]
    if not np.array_equal(counts, c1 + np.stack([0 * c1[:, 0], 2 * (c1[:, 1] + c1[:, 2]),
                                                 0 * c1[:, 0]], axis=1) + 2 * np.stack(
            [c1[:, 0], 0 * c1[:, 0], 0 * c1[:, 0]], axis=1)):
        return f"counts {counts.tolist()} against one row's {c1.tolist()}"
    return None


PINS = [pin_golden, pin_heap_reference, pin_invariants, pin_closed_forms, pin_mtp_hand_worked,
        pin_mtp_invariants, pin_mtp_closed_form]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    msg = pin()
    assert msg is None, msg


@pytest.mark.parametrize("mutant", sorted(RV.MUTANTS), ids=lambda m: RV.MUTANTS[m])
def test_pin_strength(mutant):
    failures = []
    for p in PINS:
        try:
            if p(mutant=mutant) is not None:
                failures.append(p.__name__)
        except Exception as ex:  # a crash also counts as caught
            failures.append(f"{p.__name__}: {ex!r}")
    assert failures, f"mutant {mutant} ({RV.MUTANTS[mutant]}) passed every pin"
