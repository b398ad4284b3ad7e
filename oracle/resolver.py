"""CPU oracle of the fused top-K resolver over a paged KV cache with host-offloaded
pages and per-request hot buffers.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm. The product library never imports it.

Source: "GLM 5.3 Optimizations, Part 1: Hybrid HiSparse Offloading in vLLM", section
"How it works" (mixed residency: the block table holds real blocks and null
placeholders; one fused kernel resolves the top-K: resident tokens are read in place,
hot tokens are read and their LRU entry refreshed, a miss copies a single row from
pinned host memory into an LRU slot) and section "Composing with the rest of vLLM"
(hot buffers default to 2 x top-K rows per request).

Readings taken here (the pages sketch the policy):

* Request j's block table row maps page p // page_size to a physical block (>= 0,
  resident) or a null placeholder (< 0: the page lives in host memory only).
* A resident position p reads KV row block * page_size + p % page_size (the slot rule
  of the top-k path's page translation).
* Request j owns hot_size hot slots; slot h is the KV row hot_rows[j, h]. State per
  request: hot_token[h] (the position the slot holds, -1 free), hot_step[h] (the last
  step that used it, -1 never), token_to_hot[p] (the slot holding position p, -1 none).
* One call is one step s of every request. Request j's selected positions (distinct,
  -1 padding) are resolved in output order: resident -> its row; else held in a hot
  slot -> a hit: that slot's row, and hot_step = s; else a miss.
* Misses take victims in output order: the slots whose hot_step is below s (a slot used
  at this step is never evicted), least recently used first, ties to the lower slot
  index (never-used slots, hot_step -1, come first). Miss i takes victim i: the
  victim's old position loses its mapping, the slot maps to the miss's position,
  hot_step = s, and host row host_base[j] + p is copied into KV row hot_rows[j, v].
* A miss with no victim left (more misses than slots unused at this step) resolves to
  -1 and sets status bit 1. A position outside the table row or the position map sets
  bit 2; a host row outside the host array bit 4; a victim's KV row outside the KV
  array bit 8. Each resolves to -1; a miss that fails takes its victim position in the
  order but changes no state.
"""
from __future__ import annotations

import numpy as np

ERR_NO_VICTIM = 1
ERR_POSITION = 2
ERR_HOST_ROW = 4
ERR_KV_ROW = 8

MUTANTS = {
    1: "victims: most recently used first",
    2: "hits do not refresh the slot's step",
    3: "victim ties go to the higher slot index",
    4: "slots used at this step may be evicted",
    5: "residency looked up at page p % page_size",
    6: "the copied host row is host_base + p + 1",
    7: "the evicted position keeps its mapping",
}


def resolve_step(positions, block_table, page_size, token_to_hot, hot_token, hot_step,
                 hot_rows, step, host_kv, host_base, kv, mutant=0):
    """One step for every request (row j of `positions` is request j). Updates the hot
    state (token_to_hot, hot_token, hot_step: int32 arrays [rows, ...]) and kv (uint8
    [kv_rows, row_bytes]) in place. Returns (rows resolved int32 [rows, k], counts
    int32 [rows, 3] = resident, hits, misses, status bits)."""
    pos = np.asarray(positions, np.int64)
    R, K = pos.shape
    tab = np.asarray(block_table, np.int64)
    ps = int(page_size)
    H = hot_token.shape[1]
    out = np.full((R, K), -1, np.int32)
    counts = np.zeros((R, 3), np.int32)
    err = 0
    for j in range(R):
        misses = []
        for i in range(K):
            p = int(pos[j, i])
            if p < 0:
                continue
            pg = (p % ps) if mutant == 5 else (p // ps)
            if pg >= tab.shape[1] or p >= token_to_hot.shape[1]:
                err |= ERR_POSITION
                continue
            blk = int(tab[j, pg])
            if blk >= 0:
                out[j, i] = blk * ps + p % ps
                counts[j, 0] += 1
                continue
            h = int(token_to_hot[j, p])
            if h >= 0:
                out[j, i] = hot_rows[j, h]
                if mutant != 2:
                    hot_step[j, h] = step
                counts[j, 1] += 1
                continue
            misses.append(i)
        # victims: slots unused at this step, least recently used, ties to the lower slot
        cand = [h for h in range(H) if mutant == 4 or hot_step[j, h] < step]
        if mutant == 1:
            cand.sort(key=lambda h: (-int(hot_step[j, h]), h))
        elif mutant == 3:
            cand.sort(key=lambda h: (int(hot_step[j, h]), -h))
        else:
            cand.sort(key=lambda h: (int(hot_step[j, h]), h))
        for mi, i in enumerate(misses):
            p = int(pos[j, i])
            if mi >= len(cand):
                err |= ERR_NO_VICTIM
                continue
            hr = int(host_base[j]) + p + (1 if mutant == 6 else 0)
            if hr < 0 or hr >= host_kv.shape[0]:
                err |= ERR_HOST_ROW
                continue
            v = cand[mi]
            if int(hot_rows[j, v]) < 0 or int(hot_rows[j, v]) >= kv.shape[0]:
                err |= ERR_KV_ROW
                continue
            old = int(hot_token[j, v])
            if old >= 0 and mutant != 7:
                token_to_hot[j, old] = -1
            hot_token[j, v] = p
            token_to_hot[j, p] = v
            hot_step[j, v] = step
            kv[int(hot_rows[j, v])] = host_kv[hr]
            out[j, i] = hot_rows[j, v]
            counts[j, 2] += 1
    return out, counts, err


def resolve_mtp_step(positions, block_table, page_size, token_to_hot, hot_token, hot_step,
                     hot_rows, step, host_kv, host_base, kv, mutant=0):
    """One multi-token verify step: positions [rows, q_rows, k]; request j's query rows
    q = 0 .. q_rows - 1 (the decoded token and its draft tokens, each with its own
    top-K) share its hot state and are resolved one after another at the same step
    (reading: the pages size hot buffers for this case at (num_speculative_tokens + 2)
    x top-K, section "Composing with the rest of vLLM", and leave the order open; the
    plainest reading is that of consecutive single-row steps with one step value).
    Returns (rows resolved [rows, q_rows, k], counts [rows, 3] summed over the query
    rows, status bits)."""
    pos = np.asarray(positions, np.int64)
    R, Q, K = pos.shape
    out = np.full((R, Q, K), -1, np.int32)
    counts = np.zeros((R, 3), np.int32)
    err = 0
    for q in range(Q):
        o, c, e = resolve_step(pos[:, q, :], block_table, page_size, token_to_hot, hot_token,
                               hot_step, hot_rows, step, host_kv, host_base, kv, mutant)
        out[:, q, :] = o
        counts += c
        err |= e
    return out, counts, err
