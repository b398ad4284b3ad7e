"""The no-allocation entry point (topk_select_paged_noalloc) against the workspace
entry points (topk_plan + topk_select_paged), through the C ABI.

Collected last on purpose: it must pass both alone in a fresh process and after every
other GPU test has used the library.
"""
import numpy as np
import pytest

import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import binding as B  # noqa: E402
from tests._gpu import compare_with_oracle, run_gpu, to_dev  # noqa: E402


def _by_position(pos, slots):
    """Rows as sets: each row's (position, slot) pairs ordered by position."""
    order = np.argsort(pos, axis=1, kind="stable")
    return np.take_along_axis(pos, order, 1), np.take_along_axis(slots, order, 1)


class _Call:
    """Device inputs and outputs of one no-allocation call, all made up front."""

    def __init__(self, b, k):
        self.b, self.k = b, k
        self.scores, self.lens, self.table, self.r2t = to_dev(b)
        self.slots = torch.full((b.rows, k), -5, dtype=torch.int32, device="cuda")
        self.pos = torch.full((b.rows, k), -5, dtype=torch.int32, device="cuda")
        self.status = torch.full((1,), -1, dtype=torch.int32, device="cuda")

    def run(self):
        b = self.b
        return B.topk_select_paged_noalloc(
            self.scores, b.ld, self.lens, b.rows, b.max_len, self.k, self.table,
            b.block_table.shape[1], self.r2t, b.page_size, self.slots, self.pos, self.status)

    def result(self):
        return self.slots.cpu().numpy(), self.pos.cpu().numpy(), int(self.status.item())


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    a = W.verify_80k()                       # 7 rows of 80K: the cluster path
    c = W.adversarial(rows=B.STATIC_MAX_ROWS, max_len=32768)  # at the row limit
    m = W.mixed_decode()                     # 64 rows up to 200K: the work-list kernel
    calls = [_Call(a, a.k), _Call(c, 512), _Call(m, 2048), _Call(a, 100)]
    calls[0].run()  # first call per device does the set-up; results checked below
    torch.cuda.synchronize()
    alloc0 = torch.cuda.memory_allocated()
    reserved0 = torch.cuda.memory_reserved()
    for call in calls:
        call.slots.fill_(-5)
        call.pos.fill_(-5)
    for call in calls:  # back to back on one stream, no sync in between
        assert call.run() == 0
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc0
    assert torch.cuda.memory_reserved() == reserved0
    for i, call in enumerate(calls):
        s, p, st = call.result()
        assert st == 0, B.status_str(st)
        ref_s, ref_p, ref_st = run_gpu(call.b, k=call.k)
        assert ref_st == 0
        gp, gs = _by_position(p, s)
        rp, rs = _by_position(ref_p, ref_s)
        assert np.array_equal(gp, rp), f"call {i}: positions differ from the workspace path"
        assert np.array_equal(gs, rs), f"call {i}: slots differ from the workspace path"
        compare_with_oracle(call.b, call.k, s, p)


def test_noalloc_register_and_medium_paths():
    """Batches that the register path (rows of at most 256 values) and the medium path
    (at most 16384) take, back to back on the static scratch: their plans are the
    header alone, and the medium path's row tickets carry from call to call."""
    pr = W.pr1()
    tiny = [t for t in W.tiny_rows() if t.rows <= B.STATIC_MAX_ROWS][:2]
    assert len(tiny) == 2
    calls = [_Call(pr, pr.k), _Call(tiny[0], tiny[0].k), _Call(pr, 100), _Call(tiny[1], tiny[1].k),
             _Call(pr, 2048)]
    for call in calls:  # back to back on one stream, no sync in between
        assert call.run() == 0
    torch.cuda.synchronize()
    for i, call in enumerate(calls):
        s, p, st = call.result()
        assert st == 0, f"call {i}: " + B.status_str(st)
        compare_with_oracle(call.b, call.k, s, p)


def test_noalloc_status_reaches_the_caller_and_the_next_call_clears_it():
    """Device status bits of a call arrive in the caller's status word; the next call
    starts from a clean status. rows == 0 and status == NULL are accepted."""
    rng = np.random.default_rng(2)
    L = 6000
    s = rng.standard_normal((3, L)).astype(np.float32)
    tab = np.stack([rng.permutation(L // 64 + 1).astype(np.int32) for _ in range(3)])
    s[1, 64:128] = 50.0
    tab[1, 1] = -3  # the selected positions of row 1 map to a negative page
    bad = W.Batch("bad_entry", s, np.full(3, L, np.int32), L, 16, tab, None, 64)
    call = _Call(bad, 16)
    assert call.run() == 0
    sl, p, st = call.result()
    assert st == B.STATUS_TABLE_ENTRY, B.status_str(st)
    compare_with_oracle(bad, 16, sl, p)  # the oracle writes -1 for those entries too
    clean = _Call(W.pr1(), 2048)
    assert clean.run() == 0
    sl, p, st = clean.result()
    assert st == 0
    compare_with_oracle(clean.b, 2048, sl, p)
    # rows == 0: nothing to select; the status word is cleared
    zero = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    assert B.topk_select_paged_noalloc(None, 16, None, 0, 16, 1, None, 1, None, 64, None, None,
                                       zero) == 0
    torch.cuda.synchronize()
    assert int(zero.item()) == 0
    # status == NULL: the call still runs
    b = clean.b
    clean.slots.fill_(-5)
    clean.pos.fill_(-5)
    assert B.topk_select_paged_noalloc(clean.scores, b.ld, clean.lens, b.rows, b.max_len, 2048,
                                       clean.table, b.block_table.shape[1], clean.r2t,
                                       b.page_size, clean.slots, clean.pos, None) == 0
    sl, p, _ = clean.result()
    compare_with_oracle(b, 2048, sl, p)


def test_noalloc_rejects_rows_above_limit():
    b = W.adversarial(rows=B.STATIC_MAX_ROWS + 1, max_len=2048)
    call = _Call(b, 16)
    with pytest.raises(B.TopKError) as ei:
        call.run()
    assert ei.value.code == B.ERR_STATIC_ROWS
    torch.cuda.synchronize()
    assert torch.all(call.slots == -5) and torch.all(call.status == -1)  # nothing enqueued
    assert "TOPK_STATIC_MAX_ROWS" in B.status_str(B.ERR_STATIC_ROWS)
