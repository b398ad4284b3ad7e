"""CPU oracle of the DSA indexer score producer ("MQA logits"): one fp32-valued score
per (query row, key position), computed from FP8 (e4m3) query heads, per-head gate
weights and the FP8 keys of the paged indexer KV cache with their per-token scales.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm. The product library never imports it.

Sources. "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Indexer
Prologue Fusion": the key side quantizes each key to FP8 with a per-token scale and
stores it in the paged indexer KV cache; the query side quantizes the query heads to
FP8 and applies the head-gate scaling, the gates coming from the weights projection
(one raw gate per head). Section "What's next" names the step that consumes both, the
indexer's MQA logits kernel, whose output rows are what TopK-V2 selects from. The
pages give no formula for the logits. Readings taken here:

* score(t, p) = sk(s) * sum_h g(t, h) * max(0, sum_d q(t, h, d) * k(s, d)), where
  s = slot(t, p) is the cache slot of position p in row t's request, q and k are
  the values of the e4m3 codes, sk(s) the key's scale and g(t, h) the head gate of
  row t (the query's quantization scale already folded into it, which is what the
  query path's "head-gate scaling" step produces).
* The per-head non-linearity is a reading: the pages name none, but without one the
  gated sum over heads collapses to a single query vector, so a multi-head query
  would be pointless. ReLU is taken, the plainest choice.
* slot(t, p) = table[r][p / page_size] * page_size + p % page_size with r the
  block-table row of t's group: the slot rule of the top-k path's page translation
  and of the key-path prologue's store.
* Rows come in groups of G consecutive rows that share one block-table row; each
  row scores positions [0, len(t)). Codes hold no NaN pattern (the key-path
  prologue's saturating encoder never writes one).
* Error handling, checked in this order: a row with len < 0 or len > max_len
  (ERR_LEN), whose pages do not fit the table row (ERR_TABLE_WIDTH) or whose group's
  table row does not exist (ERR_TABLE_ROW) produces nothing; a position whose page
  entry is negative (ERR_TABLE_ENTRY) or whose slot lies outside the cache
  (ERR_SLOT) scores -inf.

Arithmetic is fp64. Each query-key product of two e4m3 values is exact in fp64 and so
is the sum of D = 128 of them (at most 36 significant bits), so the dot products are
exact; the gate sum and the key scale round once per operation in fp64.
"""
from __future__ import annotations

import numpy as np

from .prologue import e4m3_value

ERR_LEN = 1
ERR_TABLE_WIDTH = 2
ERR_TABLE_ENTRY = 4
ERR_SLOT = 8
ERR_TABLE_ROW = 16

# Deliberately wrong variants, for the pin-strength test (0 = the oracle).
MUTANTS = {
    1: "no non-linearity (linear gate over heads)",
    2: "ReLU applied after the gate: max(0, g * a)",
    3: "key scale left out",
    4: "gate of head h paired with the query of head H - 1 - h",
    5: "slot = table[p % ps] * ps + p / ps (page and offset swapped)",
    6: "|a| instead of max(0, a)",
    7: "dot product over the first D / 2 channels only",
    8: "row t reads the table row of group t instead of t / G",
    9: "key scale of slot s + 1",
}


def _slots(table_row: np.ndarray, positions: np.ndarray, page_size: int, mutant: int):
    """Cache slot of each logical position through one block-table row; also the page
    entries (negative: no page)."""
    p = np.asarray(positions, np.int64)
    if mutant == 5:
        page_idx, off = p % page_size, p // page_size
    else:
        page_idx, off = p // page_size, p % page_size
    page = table_row[page_idx].astype(np.int64)
    return page * page_size + off, page


def _row_table(b, t: int, mutant: int) -> int:
    g = t if mutant == 8 else t // b.group_rows
    if b.group_table is None:
        return g
    return int(b.group_table[g]) if g < len(b.group_table) else -1


def row_error(b, t: int, mutant: int = 0) -> int:
    """Row-level status bits of query row t (0: the row is scored)."""
    L = int(b.lens[t])
    if L < 0 or L > b.max_len:
        return ERR_LEN
    if -(-L // b.page_size) > b.block_table.shape[1]:
        return ERR_TABLE_WIDTH
    r = _row_table(b, t, mutant)
    if r < 0 or r >= b.block_table.shape[0]:
        return ERR_TABLE_ROW
    return 0


def scores_at(b, t: int, positions, mutant: int = 0):
    """Scores (float64) of query row t at the given positions (each in [0, len(t))),
    and the status bits they raise. Row-level errors must be checked first."""
    positions = np.asarray(positions, np.int64)
    r = _row_table(b, t, mutant)
    slot, page = _slots(b.block_table[r], positions, b.page_size, mutant)
    bad_page = page < 0
    bad_slot = ~bad_page & ((slot < 0) | (slot >= b.num_slots))
    ok = ~(bad_page | bad_slot)
    st = (ERR_TABLE_ENTRY if bad_page.any() else 0) | (ERR_SLOT if bad_slot.any() else 0)
    out = np.full(len(positions), -np.inf, np.float64)
    s = slot[ok]
    if len(s) == 0:
        return out, st
    D = b.dim
    kv = e4m3_value(b.cache[s])                       # [n, D]
    qv = e4m3_value(b.q[t])                           # [H, D]
    if mutant == 7:
        kv, qv = kv[:, :D // 2], qv[:, :D // 2]
    g = b.w[t].astype(np.float64)                     # [H]
    if mutant == 4:
        g = g[::-1]
    a = kv @ qv.T                                     # [n, H]: per-head dot products
    if mutant == 1:
        act = a
    elif mutant == 6:
        act = np.abs(a)
    else:
        act = np.maximum(a, 0.0)
    if mutant == 2:
        gated = np.maximum(act * g[None, :], 0.0).sum(axis=1)
    else:
        gated = act @ g
    if mutant == 3:
        sk = np.ones(len(s))
    elif mutant == 9:
        sk = b.cache_scale[np.minimum(s + 1, b.num_slots - 1)].astype(np.float64)
    else:
        sk = b.cache_scale[s].astype(np.float64)
    out[ok] = sk * gated
    return out, st


def mqa_logits(b, mutant: int = 0):
    """Every score of every row: float64 [rows, max_len] with NaN at positions a row
    does not score (past its length, or the whole row on a row-level error), and the
    OR of all status bits."""
    out = np.full((b.rows, max(b.max_len, 0)), np.nan, np.float64)
    st = 0
    for t in range(b.rows):
        e = row_error(b, t, mutant)
        if e:
            st |= e
            continue
        L = int(b.lens[t])
        if L == 0:
            continue
        out[t, :L], s = scores_at(b, t, np.arange(L), mutant)
        st |= s
    return out, st


def magnitude_at(b, t: int, positions):
    """sk(s) * sum_h |g(t, h)| * sum_d |q(t, h, d) * k(s, d)| at each position: the
    scale of the rounding error of any evaluation of the score that rounds each
    product, sum and scaling step with a relative error u (the error is at most
    about (D + H + 2) u times this). Positions with an invalid page or slot give 0."""
    positions = np.asarray(positions, np.int64)
    r = _row_table(b, t, 0)
    slot, page = _slots(b.block_table[r], positions, b.page_size, 0)
    ok = (page >= 0) & (slot >= 0) & (slot < b.num_slots)
    out = np.zeros(len(positions), np.float64)
    s = slot[ok]
    if len(s):
        kv = np.abs(e4m3_value(b.cache[s]))
        qv = np.abs(e4m3_value(b.q[t]))
        out[ok] = b.cache_scale[s].astype(np.float64) * ((kv @ qv.T) @ np.abs(b.w[t].astype(np.float64)))
    return out
