"""GPU parity of the fused top-K resolver (hisparse_resolve, through the C ABI) against
the CPU oracle (oracle/resolver.py), bit-exact: after every step of a multi-step
sequence, the resolved rows, the counts, the status bits, the hot state (position map,
slot map, slot steps) and the whole KV tensor must match."""
import numpy as np
import pytest

import workloads as W
from oracle import resolver as RV

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import binding as B  # noqa: E402


def run_sequence(b, hot_rows=None, steps=None):
    dev = torch.device("cuda", 0)
    hot_rows = b.hot_rows if hot_rows is None else hot_rows
    steps = b.steps if steps is None else steps
    R, H = hot_rows.shape
    map_ld = int(b.lens.max())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g_t2h = torch.full((R, map_ld), -1, dtype=torch.int32, device=dev)
    g_ht = torch.full((R, H), -1, dtype=torch.int32, device=dev)
    g_hs = torch.full((R, H), -1, dtype=torch.int32, device=dev)
    g_hot_rows, g_tab, g_base = t(hot_rows), t(b.block_table), t(b.host_base)
    g_kv = t(b.kv_init)
    host = torch.from_numpy(b.host_kv).pin_memory()
    o_t2h = np.full((R, map_ld), -1, np.int32)
    o_ht = np.full((R, H), -1, np.int32)
    o_hs = np.full((R, H), -1, np.int32)
    o_kv = b.kv_init.copy()
    for s, sel in enumerate(steps):
        k = sel.shape[1]
        out = torch.full((R, k), -9, dtype=torch.int32, device=dev)
        counts = torch.zeros((R, 3), dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        B.hisparse_resolve(t(sel), g_tab, b.page_size, g_t2h, g_ht, g_hs, g_hot_rows, s, host,
                           g_base, g_kv, out, counts=counts, status=status)
        torch.cuda.synchronize()
        o_out, o_counts, o_err = RV.resolve_step(sel, b.block_table, b.page_size, o_t2h, o_ht,
                                                 o_hs, hot_rows, s, b.host_kv, b.host_base, o_kv)
        assert int(status.item()) == o_err, f"step {s}: status {int(status.item())} != {o_err}"
        assert np.array_equal(out.cpu().numpy(), o_out), f"step {s}: resolved rows differ"
        assert np.array_equal(counts.cpu().numpy(), o_counts), f"step {s}: counts differ"
        assert np.array_equal(g_t2h.cpu().numpy(), o_t2h), f"step {s}: position map differs"
        assert np.array_equal(g_ht.cpu().numpy(), o_ht), f"step {s}: slot map differs"
        assert np.array_equal(g_hs.cpu().numpy(), o_hs), f"step {s}: slot steps differ"
        assert np.array_equal(g_kv.cpu().numpy(), o_kv), f"step {s}: KV tensor differs"
    return o_counts


def test_small_sequence():
    b = W.hisparse(seed=W.SEED_BASE + 71, reqs=4, k=512, lens=[20000, 30000, 5000, 300],
                   row_bytes=64, n_steps=6)
    run_sequence(b)


def test_low_locality_and_many_steps():
    b = W.hisparse(seed=W.SEED_BASE + 72, reqs=3, k=256, lens=[9000, 4000, 700], row_bytes=32,
                   n_steps=12, keep=0.3)
    run_sequence(b)


def test_full_size_decode_batch():
    """8 requests, k = 2048, hot buffers of 4096 rows of 656 bytes."""
    b = W.hisparse(seed=W.SEED_BASE + 73, reqs=8, k=2048, n_steps=4)
    counts = run_sequence(b)
    assert counts[:, 1].sum() > 0 and counts[:, 2].sum() > 0  # hits and misses both occur


def test_exhausted_hot_buffer():
    """Half as many slots as selected positions: misses beyond the free slots fail."""
    b = W.hisparse(seed=W.SEED_BASE + 74, reqs=2, k=128, lens=[6000, 3000], row_bytes=16,
                   n_steps=3, tail=64)
    run_sequence(b, hot_rows=b.hot_rows[:, :64].copy())


def test_positions_outside_the_table():
    b = W.hisparse(seed=W.SEED_BASE + 75, reqs=2, k=64, lens=[3000, 1000], row_bytes=16,
                   n_steps=2)
    steps = [x.copy() for x in b.steps]
    steps[1][0, 3] = b.block_table.shape[1] * b.page_size + 5  # past the table row
    steps[1][1, 0] = int(b.lens.max()) + 1                      # past the position map
    run_sequence(b, steps=steps)


def _crafted_state(b, step, spread, n_miss, n_hit, seed, never_used=0.1):
    """A hot state whose slots were last used at steps spread over [0, spread) (a
    `never_used` share never used), each used slot holding a distinct host-only position, and one
    step's selection: n_hit of the held positions and n_miss host-only positions that no
    slot holds (both in random order, -1 padded to k = n_hit + n_miss)."""
    rng = np.random.default_rng(seed)
    R, H = b.hot_rows.shape
    map_ld = int(b.lens.max())
    t2h = np.full((R, map_ld), -1, np.int32)
    ht = np.full((R, H), -1, np.int32)
    hs = np.full((R, H), -1, np.int32)
    k = n_hit + n_miss
    sel = np.full((R, k), -1, np.int32)
    for j in range(R):
        pages = np.nonzero(b.block_table[j] < 0)[0]
        host_only = (pages[:, None] * b.page_size + np.arange(b.page_size)).ravel()
        host_only = host_only[host_only < b.lens[j]]
        pick = rng.permutation(host_only)
        used = rng.random(H) >= never_used
        held = pick[:int(used.sum())]
        hs[j, used] = rng.integers(0, spread, int(used.sum()))
        ht[j, used] = held
        t2h[j, held] = np.nonzero(used)[0]
        free = pick[int(used.sum()):]
        chosen = np.concatenate([rng.choice(held, n_hit, replace=False), free[:n_miss]])
        sel[j, :chosen.size] = rng.permutation(chosen)
    return t2h, ht, hs, sel


def _one_step_from(b, state, step):
    dev = torch.device("cuda", 0)
    t2h, ht, hs, sel = state
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g_t2h, g_ht, g_hs, g_kv = t(t2h), t(ht), t(hs), t(b.kv_init)
    host = torch.from_numpy(b.host_kv).pin_memory()
    R, k = sel.shape
    out = torch.full((R, k), -9, dtype=torch.int32, device=dev)
    counts = torch.zeros((R, 3), dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.hisparse_resolve(t(sel), t(b.block_table), b.page_size, g_t2h, g_ht, g_hs, t(b.hot_rows),
                       step, host, t(b.host_base), g_kv, out, counts=counts, status=status)
    torch.cuda.synchronize()
    o_t2h, o_ht, o_hs, o_kv = t2h.copy(), ht.copy(), hs.copy(), b.kv_init.copy()
    o_out, o_counts, o_err = RV.resolve_step(sel, b.block_table, b.page_size, o_t2h, o_ht, o_hs,
                                             b.hot_rows, step, b.host_kv, b.host_base, o_kv)
    assert int(status.item()) == o_err
    assert np.array_equal(out.cpu().numpy(), o_out), "resolved rows differ"
    assert np.array_equal(counts.cpu().numpy(), o_counts), "counts differ"
    assert np.array_equal(g_t2h.cpu().numpy(), o_t2h), "position map differs"
    assert np.array_equal(g_ht.cpu().numpy(), o_ht), "slot map differs"
    assert np.array_equal(g_hs.cpu().numpy(), o_hs), "slot steps differ"
    assert np.array_equal(g_kv.cpu().numpy(), o_kv), "KV tensor differs"
    return o_counts


@pytest.mark.parametrize("n_miss,never_used", [(40, 0.1), (500, 0.0), (1500, 0.1)])
def test_victims_from_slots_last_used_over_many_steps(n_miss, never_used):
    """Slot steps spread over 40 earlier steps. 40 misses take never-used slots; 500
    misses (every slot used) take slots from the five or so oldest steps, by step and
    then slot; 1500 misses reach slots 13 steps younger than the oldest (past the
    counting order for the eight oldest step values: the general victim order)."""
    b = W.hisparse(seed=W.SEED_BASE + 76, reqs=3, k=2048, lens=[60000, 40000, 30000],
                   row_bytes=32, n_steps=1)
    state = _crafted_state(b, 40, 40, n_miss, 200, W.SEED_BASE + 77 + n_miss, never_used)
    counts = _one_step_from(b, state, 40)
    assert np.all(counts[:, 2] == n_miss) and np.all(counts[:, 1] == 200)


@pytest.mark.parametrize("n_miss,never_used", [(150, 0.0), (700, 0.0)])
def test_victims_in_a_hot_buffer_of_odd_size(n_miss, never_used):
    """1000 slots per request (the last thread's block of 8 slots is partly outside):
    150 misses take slots from the oldest few steps, 700 reach far younger ones."""
    import dataclasses
    b = W.hisparse(seed=W.SEED_BASE + 78, reqs=2, k=1024, lens=[50000, 20000], row_bytes=48,
                   n_steps=1)
    b = dataclasses.replace(b, hot_rows=np.ascontiguousarray(b.hot_rows[:, :1000]))
    state = _crafted_state(b, 30, 30, n_miss, 100, W.SEED_BASE + 79 + n_miss, never_used)
    counts = _one_step_from(b, state, 30)
    assert np.all(counts[:, 2] == n_miss) and np.all(counts[:, 1] == 100)


def run_mtp_sequence(b, hot_rows=None):
    """hisparse_resolve_mtp step by step against the oracle's multi-token step."""
    dev = torch.device("cuda", 0)
    hot_rows = b.hot_rows if hot_rows is None else hot_rows
    R, H = hot_rows.shape
    map_ld = int(b.lens.max())
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    g_t2h = torch.full((R, map_ld), -1, dtype=torch.int32, device=dev)
    g_ht = torch.full((R, H), -1, dtype=torch.int32, device=dev)
    g_hs = torch.full((R, H), -1, dtype=torch.int32, device=dev)
    g_hot_rows, g_tab, g_base = t(hot_rows), t(b.block_table), t(b.host_base)
    g_kv = t(b.kv_init)
    host = torch.from_numpy(b.host_kv).pin_memory()
    o_t2h = np.full((R, map_ld), -1, np.int32)
    o_ht = np.full((R, H), -1, np.int32)
    o_hs = np.full((R, H), -1, np.int32)
    o_kv = b.kv_init.copy()
    total = np.zeros((R, 3), np.int64)
    for s, sel in enumerate(b.steps):
        out = torch.full(sel.shape, -9, dtype=torch.int32, device=dev)
        counts = torch.zeros((R, 3), dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        B.hisparse_resolve_mtp(t(sel), g_tab, b.page_size, g_t2h, g_ht, g_hs, g_hot_rows, s, host,
                               g_base, g_kv, out, counts=counts, status=status)
        torch.cuda.synchronize()
        o_out, o_counts, o_err = RV.resolve_mtp_step(sel, b.block_table, b.page_size, o_t2h, o_ht,
                                                     o_hs, hot_rows, s, b.host_kv, b.host_base,
                                                     o_kv)
        assert int(status.item()) == o_err, f"step {s}: status {int(status.item())} != {o_err}"
        assert np.array_equal(out.cpu().numpy(), o_out), f"step {s}: resolved rows differ"
        assert np.array_equal(counts.cpu().numpy(), o_counts), f"step {s}: counts differ"
        assert np.array_equal(g_t2h.cpu().numpy(), o_t2h), f"step {s}: position map differs"
        assert np.array_equal(g_ht.cpu().numpy(), o_ht), f"step {s}: slot map differs"
        assert np.array_equal(g_hs.cpu().numpy(), o_hs), f"step {s}: slot steps differ"
        assert np.array_equal(g_kv.cpu().numpy(), o_kv), f"step {s}: KV tensor differs"
        total += o_counts
    return total


def test_mtp_verify_steps():
    """Four requests, three query rows each (the decoded token and two drafts), k = 512,
    hot buffers of (3 + 1) * 512 rows: the rows of a step share the request's hot state."""
    b = W.hisparse_mtp(seed=W.SEED_BASE + 75, reqs=4, k=512, q_rows=3,
                       lens=[20000, 30000, 5000, 900], n_steps=5)
    total = run_mtp_sequence(b)
    assert total[:, 1].sum() > 0 and total[:, 2].sum() > 0


def test_mtp_seven_rows_and_an_exhausted_buffer():
    """Seven query rows (1 + 6 drafts) at k = 256 with hot buffers of 8 * 256 rows, then
    the same with a quarter of the slots: later rows' misses run out of victims."""
    b = W.hisparse_mtp(seed=W.SEED_BASE + 76, reqs=3, k=256, q_rows=7, lens=[12000, 6000, 3000],
                       row_bytes=32, n_steps=4, draft_new=0.4)
    run_mtp_sequence(b)
    run_mtp_sequence(b, hot_rows=b.hot_rows[:, :512].copy())


def test_mtp_single_row_equals_the_plain_call():
    """q_rows = 1 is the plain call."""
    b = W.hisparse(seed=W.SEED_BASE + 77, reqs=3, k=128, lens=[5000, 2000, 700], row_bytes=16,
                   n_steps=3)
    import dataclasses
    run_mtp_sequence(dataclasses.replace(b, steps=[s[:, None, :] for s in b.steps]))


@pytest.mark.parametrize("reqs", [20, 40, 160])
def test_batches_of_every_cluster_size(reqs):
    """The requests of a batch that leaves SMs free run as clusters that share their row
    copies (8, 4 or 2 CTAs per request by the batch size and the SM count); a batch of
    more requests than SMs runs one CTA per request. 20, 40 and 160 requests take
    clusters of 4, 2 and none on a 152-SM GPU (the size is the library's choice: the
    result must not depend on it)."""
    rng = np.random.default_rng(reqs)
    lens = rng.integers(800, 6000, reqs).tolist()
    b = W.hisparse(seed=W.SEED_BASE + 80 + reqs, reqs=reqs, k=64, lens=lens, tail=256,
                   row_bytes=48, n_steps=3)
    total = run_sequence(b)
    assert total[:, 2].sum() > 0


def test_mtp_batch_of_clusters_of_four():
    """A multi-token batch of 20 requests: each query row's copies are shared by the
    request's cluster, and the cluster meets twice per row."""
    b = W.hisparse_mtp(seed=W.SEED_BASE + 79, reqs=20, k=64, q_rows=4,
                       lens=np.random.default_rng(5).integers(800, 5000, 20).tolist(),
                       tail=256, row_bytes=32, n_steps=3)
    total = run_mtp_sequence(b)
    assert total[:, 2].sum() > 0
