"""Independent numpy checks of a top-k + paged-slot result.

These helpers restate the selection rule directly (no sorting library shared with
the oracle) so that they can pin the oracle and, later, check the CUDA path.
Rule ("Serving GLM5.2 NVFP4 Agentic Workload with SGLang", "Kernel Optimization >
TopK-V2", with the tie/padding/slot readings): p ranks before q iff s(p) > s(q), or
they are equal (IEEE, -0 == +0) and p < q; NaN ranks below every number; a row of
length L yields min(k, L) entries then -1; slot = table[p // ps] * ps + p % ps.
"""
from __future__ import annotations

import numpy as np


def _cls(x: np.ndarray) -> np.ndarray:
    return np.where(np.isnan(x), 0, 1)


def before(sa, pa, sb, pb) -> bool:
    """Scalar form of the order: does (sa, pa) rank before (sb, pb)?"""
    ca, cb = (0 if np.isnan(sa) else 1), (0 if np.isnan(sb) else 1)
    if ca != cb:
        return ca > cb
    if ca == 1 and sa != sb:
        return sa > sb
    return pa < pb


def slot_of(table_row: np.ndarray, p: np.ndarray, ps: int) -> np.ndarray:
    p = p.astype(np.int64)
    return table_row[p // ps].astype(np.int64) * ps + p % ps


def positions_from_slots(table_row: np.ndarray, L: int, ps: int, slots: np.ndarray) -> np.ndarray:
    """Invert slot -> position for an injective table (used when only slots exist)."""
    allp = np.arange(L, dtype=np.int64)
    all_slots = slot_of(table_row, allp, ps)
    order = np.argsort(all_slots, kind="stable")
    srt = all_slots[order]
    idx = np.searchsorted(srt, slots.astype(np.int64))
    idx = np.clip(idx, 0, max(L - 1, 0))
    ok = (L > 0) & (srt[idx] == slots) if L > 0 else np.zeros(slots.shape, bool)
    out = np.where(ok, order[idx], -2)
    return out


def check_row(scores_row, L, k, table_row, ps, slots_row, pos_row=None):
    """Raises AssertionError with a message if the row's result breaks a rule.
    Returns the selected positions (in output order)."""
    m = min(k, L)
    slots_row = np.asarray(slots_row)
    assert slots_row.shape == (k,), f"slot row shape {slots_row.shape} != ({k},)"
    assert np.all(slots_row[m:] == -1), "tail beyond min(k, len) is not -1"
    if pos_row is not None:
        pos_row = np.asarray(pos_row)
        assert np.all(pos_row[m:] == -1), "position tail beyond min(k, len) is not -1"
        sel = pos_row[:m].astype(np.int64)
    else:
        sel = positions_from_slots(table_row, L, ps, slots_row[:m])
    assert np.all((sel >= 0) & (sel < L)), "selected position out of [0, len)"
    assert np.unique(sel).size == m, "selected positions are not unique"
    exp_slots = slot_of(table_row, sel, ps)
    assert np.array_equal(exp_slots, slots_row[:m].astype(np.int64)), "slot != table lookup"
    if m == L or m == 0:
        return sel
    s = np.asarray(scores_row[:L], dtype=np.float32)
    mask = np.zeros(L, bool)
    mask[sel] = True
    # worst selected and best unselected under the order
    ssel, psel = s[mask], np.nonzero(mask)[0]
    sun, pun = s[~mask], np.nonzero(~mask)[0]
    csel, cun = _cls(ssel), _cls(sun)
    # worst selected: lowest class, then lowest score, then largest position
    wc = csel.min()
    cand = np.nonzero(csel == wc)[0]
    if wc == 1:
        v = ssel[cand].min()
        cand = cand[ssel[cand] == v]
    w = cand[np.argmax(psel[cand])]
    bc = cun.max()
    cand = np.nonzero(cun == bc)[0]
    if bc == 1:
        v = sun[cand].max()
        cand = cand[sun[cand] == v]
    b = cand[np.argmin(pun[cand])]
    assert before(ssel[w], psel[w], sun[b], pun[b]), (
        f"unselected ({sun[b]}, {pun[b]}) should rank before selected ({ssel[w]}, {psel[w]})")
    return sel


def check_batch(scores, lens, k, block_table, row_to_table, ps, slots, pos=None):
    rows = scores.shape[0]
    for r in range(rows):
        t = r if row_to_table is None else int(row_to_table[r])
        check_row(scores[r], int(lens[r]), k, block_table[t], ps, slots[r],
                  None if pos is None else pos[r])


def canonical(scores_row, L, pos_row, slots_row, k):
    """Sort one row's output by (score desc, position asc) for element-wise compare."""
    m = min(k, L)
    p = np.asarray(pos_row[:m], dtype=np.int64)
    s = np.asarray(scores_row, dtype=np.float32)[p]
    cls = _cls(s)
    sk = np.where(cls == 1, s, 0).astype(np.float64)
    order = np.lexsort((p, -sk, -cls))
    return p[order], np.asarray(slots_row[:m])[order]
