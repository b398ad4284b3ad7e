"""GPU parity of rows split over many CTAs against the CPU oracle, bit-exact, and the
bounded waits of their row barriers.

Covers massive ties over many CTAs (every refinement level, then position order),
boundary bins ranked from gathered candidates in both of their forms (pairwise ranks
and radix list selection), rows much shorter than max_len next to long ones, rows of
at most k values and zero-length rows, unaligned rows with page sizes that are not
powers of two, one plan reused over many calls with changing k and score tensors, and
a row barrier whose wait runs out (a CTA that never arrives) ending the call cleanly.
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


def _batch(name, rows, L, k=2048, page_size=64, seed=0, lens=None):
    """rows: list of float32 arrays (each clipped to L); lens default L; positions past
    a row's length hold the poison value."""
    rng = np.random.default_rng(seed)
    ld = W.round_up(L, 4)
    s = np.full((len(rows), ld), W.POISON, np.float32)
    for i, x in enumerate(rows):
        s[i, :min(L, len(x))] = x[:L]
    lens = np.full(len(rows), L, np.int32) if lens is None else np.asarray(lens, np.int32)
    npg = -(-L // page_size)
    tab = np.stack([rng.permutation(npg * 2)[:npg].astype(np.int32) for _ in rows])
    return W.Batch(name, s, lens, L, k, tab, None, page_size)


def test_massive_ties_over_many_ctas():
    """All-equal rows, +/-0 mixtures, few distinct values, NaN rows with -inf every 7th
    position, a short N(0,1) prefix before -inf, and the fp16 grid, 120000 values each,
    split into chunks of 5008 (24 CTAs per row) and automatically."""
    rng = np.random.default_rng(3)
    L = 120000
    rows = [np.full(L, 2.5, np.float32),
            np.where(np.arange(L) % 3 == 0, np.float32(-0.0), np.float32(0.0)),
            rng.integers(-3, 4, L).astype(np.float32),
            np.full(L, np.nan, np.float32),
            np.concatenate([rng.standard_normal(50).astype(np.float32),
                            np.full(L - 50, -np.inf, np.float32)]),
            rng.standard_normal(L).astype(np.float16).astype(np.float32)]
    rows[3][::7] = -np.inf
    b = _batch("ties", rows, L, seed=4)
    for chunk in (0, 5008):
        dev = to_dev(b)
        core = PagedTopK(b.rows, b.max_len)
        core.plan(dev[1], chunk=chunk)
        for k in (1, 7, 1000, 2048):
            slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
            assert st == 0, B.status_str(st)
            compare_with_oracle(b, k, slots, pos)


def test_gathered_candidates_both_rankings():
    """Boundary bins of 600 exact ties and of 3000 distinct values in one coarse bin,
    spread over the CTAs of 200000-value rows."""
    rng = np.random.default_rng(8)
    L = 200000
    base = rng.standard_normal(L).astype(np.float32)
    many = base.copy()
    many[rng.choice(L, 3000, replace=False)] = (
        np.float32(20.0) + rng.random(3000).astype(np.float32) * np.float32(0.1))
    few = base.copy()
    few[rng.choice(L, 600, replace=False)] = np.float32(9.0)
    b = _batch("gather", [base, many, few], L, seed=9)
    dev = to_dev(b)
    for chunk in (0, 12000):
        core = PagedTopK(b.rows, b.max_len)
        core.plan(dev[1], chunk=chunk)
        for k in (100, 2048, 1500, 2):
            slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
            assert st == 0, B.status_str(st)
            compare_with_oracle(b, k, slots, pos)


def test_short_and_long_rows_in_one_batch():
    """Rows of 300000, 150001, 2049 values next to rows of 17, 2048 and 0 values (every
    position taken, or none), for k = 2048, 16 and 1, with and without positions."""
    rng = np.random.default_rng(12)
    L = 300000
    rows = [rng.standard_normal(L).astype(np.float32) for _ in range(6)]
    b = _batch("short", rows, L, seed=13, lens=[L, 17, 0, 2049, 150001, 2048])
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1])
    for k in (2048, 16, 1):
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)
    slots, _, st = run_gpu(b, k=2048, plan=core, dev_inputs=dev, with_pos=False)
    assert st == 0
    compare_with_oracle(b, 2048, slots, None)


@pytest.mark.parametrize("page_size", [1, 7, 64, 4096])
def test_unaligned_rows_and_page_sizes(page_size):
    rng = np.random.default_rng(21)
    L = 100003
    rows = [rng.standard_normal(L).astype(np.float32) for _ in range(4)]
    b = W.with_ld(_batch("unaligned", rows, L, page_size=page_size, seed=22), L)
    assert b.ld % 4 != 0  # rows start at unaligned addresses
    slots, pos, st = run_gpu(b, k=2048)
    assert st == 0, B.status_str(st)
    compare_with_oracle(b, 2048, slots, pos)


def test_one_plan_many_calls():
    """One plan serves many selects: k changes and score tensors change between calls."""
    b = W.verify_80k()
    scores, lens, table, r2t = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(lens)
    other = W.verify_80k(seed=99)
    s2 = torch.from_numpy(other.scores).cuda()
    b2 = dataclasses.replace(b, scores=other.scores)
    refs = {}
    for _ in range(3):
        for k in (2048, 100, 1, 777):
            for bb, ss in ((b, scores), (b2, s2)):
                slots, pos, st = run_gpu(bb, k=k, plan=core, dev_inputs=(ss, lens, table, r2t))
                assert st == 0
                key = (bb is b, k)
                if key not in refs:
                    refs[key] = oracle.topk_batch(bb, k=k, threads=8)
                compare_with_oracle(bb, k, slots, pos, ref=refs[key])


def test_expired_wait_ends_the_call_and_a_new_plan_recovers():
    """A CTA serving a row split over many CTAs never arrives at its first row barrier;
    with a 2 ms limit the other CTAs of that row give up, the call ends, the status
    reports TOPK_STATUS_TIMEOUT and the first expired wait is recorded (kind 1, that
    row). Rows served by other CTAs are exact. A new plan then gives an exact call on
    the same workspace (here an automatic one: the cluster path)."""
    from tests.test_plan_host import parse_plan
    b = W.verify_80k()
    dev = to_dev(b)
    grid = B.topk_grid_size()
    chunk = 4096  # the work-list kernel, 20 CTAs per row
    img = np.zeros(B.topk_workspace_bytes(b.rows, b.max_len), np.uint8)
    B.topk_plan_host(b.lens, b.rows, b.max_len, grid, chunk, img)
    _, _, _, (_, units), info = parse_plan(img, b.rows)
    # wave 0, CTA 1: a rank of a split row (row, s0, n, len, rank, G, group)
    skip = 1
    row_of_skip, g_of_skip = int(units[skip, 0]), int(units[skip, 5])
    assert row_of_skip >= 0 and g_of_skip >= 2
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1], chunk=chunk)
    slots, pos, st = run_gpu(b, plan=core, dev_inputs=dev, wait_ns=2_000_000, skip_cta=skip)
    assert st & B.STATUS_TIMEOUT, B.status_str(st)
    diag = core.workspace[128:160].cpu().numpy().view(np.int32)
    assert diag[0] == 1 and diag[1] == row_of_skip
    ref = oracle.topk_batch(b, threads=8)
    keep = np.array([r for r in range(b.rows) if r != row_of_skip])
    sub = dataclasses.replace(b, scores=b.scores[keep], lens=b.lens[keep],
                              row_to_table=b.row_to_table[keep])
    compare_with_oracle(sub, b.k, slots[keep], pos[keep],
                        ref=(ref[0][keep], ref[1][keep], ref[2]))
    core.plan(dev[1])
    assert core.status() == 0
    slots, pos, st = run_gpu(b, plan=core, dev_inputs=dev)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos, ref=ref)
