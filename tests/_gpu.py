"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI on a
workloads.Batch and compare it with the CPU oracle element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tests import _checks as C


def to_dev(b, ld=None):
    dev = torch.device("cuda", 0)
    scores = torch.from_numpy(np.ascontiguousarray(b.scores)).to(dev)
    lens = torch.from_numpy(b.lens.astype(np.int32)).to(dev)
    table = torch.from_numpy(np.ascontiguousarray(b.block_table.astype(np.int32))).to(dev)
    r2t = None if b.row_to_table is None else torch.from_numpy(b.row_to_table.astype(np.int32)).to(dev)
    return scores, lens, table, r2t


def run_gpu(b, k=None, chunk=0, with_pos=True, guard=64, plan=None, dev_inputs=None,
            wait_ns=None, skip_cta=-1):
    """Returns (slots, pos or None, status) as numpy arrays. Output buffers carry guard
    canaries on both sides which must stay untouched."""
    from sparse_attention_indexer_gb300 import PagedTopK
    k = b.k if k is None else k
    scores, lens, table, r2t = dev_inputs if dev_inputs is not None else to_dev(b)
    rows = b.rows
    core = plan if plan is not None else PagedTopK(rows, b.max_len)
    if plan is None:
        core.plan(lens, chunk=chunk)
    n = rows * k
    sbuf = torch.full((n + 2 * guard,), -777, dtype=torch.int32, device=scores.device)
    pbuf = torch.full((n + 2 * guard,), -777, dtype=torch.int32, device=scores.device)
    out_s = sbuf[guard:guard + n].view(rows, k)
    out_p = pbuf[guard:guard + n].view(rows, k) if with_pos else None
    if wait_ns is None:
        core.select(scores, lens, k, table, b.page_size, r2t, out_slots=out_s, out_pos=out_p)
    else:
        from sparse_attention_indexer_gb300 import binding as B
        B.topk_select_paged_test(scores, scores.stride(0), lens, rows, b.max_len, k, table,
                                 table.stride(0), r2t, b.page_size, out_s, out_p, core.workspace,
                                 wait_ns, skip_cta)
    status = core.status()
    if status & 16:
        diag = core.workspace[128:160].cpu().numpy().view(np.int32)
        print(f"timeout record (kind,row,rank,seq,seen,target,cta): {diag.tolist()}")
    sb = sbuf.cpu().numpy()
    assert np.all(sb[:guard] == -777) and np.all(sb[guard + n:] == -777), "slot canary overwritten"
    pos = None
    if with_pos:
        pb = pbuf.cpu().numpy()
        assert np.all(pb[:guard] == -777) and np.all(pb[guard + n:] == -777), "pos canary overwritten"
        pos = pb[guard:guard + n].reshape(rows, k)
    return sb[guard:guard + n].reshape(rows, k), pos, status


def compare_with_oracle(b, k, slots, pos, ref=None):
    """Bit-exact comparison after sorting each GPU row by (score desc, position asc)."""
    if ref is None:
        ref = oracle.topk_batch(b, k=k, threads=8)
    rs, rp, _ = ref
    for r in range(b.rows):
        L = int(b.lens[r])
        if not (0 <= L <= b.max_len):
            assert np.all(slots[r] == -1)
            continue
        m = min(k, L)
        if pos is not None:
            gp, gs = C.canonical(b.scores[r], L, pos[r], slots[r], k)
            if not np.array_equal(gp, rp[r, :m]):
                bad = np.nonzero(gp != rp[r, :m])[0]
                raise AssertionError(f"{b.name} k={k} row {r} (len {L}): positions differ at "
                                     f"{bad[:8]}: gpu {gp[bad[:8]]} oracle {rp[r, bad[:8]]}")
            assert np.array_equal(gs, rs[r, :m]), f"{b.name} k={k} row {r}: slots differ"
            assert np.all(pos[r, m:] == -1)
        else:
            assert np.array_equal(np.sort(slots[r, :m]), np.sort(rs[r, :m])), \
                f"{b.name} k={k} row {r}: slot sets differ"
        assert np.all(slots[r, m:] == -1), f"{b.name} row {r}: padding"
    return ref
