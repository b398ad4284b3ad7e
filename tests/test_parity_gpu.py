"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle, bit-exact.

Each GPU row is sorted by (score desc, position asc) and compared element by element
with the oracle's positions and slots; padding must be -1 and the output buffers'
guard canaries untouched. Covers every synthetic workload at full size, every k of
the tie-heavy tiny rows, path forcing (the same rows through many chunkings), plan
reuse, unaligned row strides, the error statuses and CUDA-graph replay.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import workloads as W
from tests import _checks as C

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import PagedTopK, binding as B  # noqa: E402
from tests._gpu import compare_with_oracle, run_gpu, to_dev  # noqa: E402


def test_library_loaded_and_device_supported():
    assert B.topk_grid_size() > 0
    assert B.topk_max_row_len() >= 1_000_006


def test_pr1_ref():
    b = W.pr1()
    slots, pos, st = run_gpu(b)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos)


@pytest.mark.parametrize("page_size", [64, 8])
def test_tiny_rows_every_k(page_size):
    for b in W.tiny_rows(page_size=page_size):
        slots, pos, st = run_gpu(b)
        assert st == 0
        compare_with_oracle(b, b.k, slots, pos)


def test_verify_80k():
    b = W.verify_80k()
    slots, pos, st = run_gpu(b)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos)


def test_verify_1m():
    b = W.verify_1m()
    slots, pos, st = run_gpu(b)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos)


def test_prefill_ragged():
    """Ragged prefill: two requests (prefix 2048 and 5000 tokens, 512 and 300 new
    queries), causal row lengths stepping by one, rows mapped to their request's table;
    every k class."""
    b = W.prefill(prefixes=(2048, 5000), q=(512, 300))
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1])
    for k in (1, 100, 2048):
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)


def test_mixed_decode():
    b = W.mixed_decode()
    slots, pos, st = run_gpu(b)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos)


def test_adversarial_all_k():
    b = W.adversarial()
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1])
    for k in b.ks:
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)


def _subset(b, rows):
    return dataclasses.replace(b, scores=b.scores[rows].copy(), lens=b.lens[rows].copy(),
                               block_table=b.block_table if b.row_to_table is not None
                               else b.block_table[rows].copy(),
                               row_to_table=None if b.row_to_table is None
                               else b.row_to_table[rows].copy())


@pytest.mark.parametrize("chunk", [16, 48, 256, 1024, 5000, 0, 48128])
def test_path_forcing_same_result(chunk):
    """The result must not depend on how rows are split over CTAs."""
    adv = _subset(W.adversarial(rows=48, max_len=20000), np.arange(48))
    mixed = _subset(W.mixed_decode(), np.arange(6))
    for b in (adv, mixed):
        if chunk and chunk < 1024 and b is mixed:
            continue  # would exceed the grid for 200K rows
        for k in (1, 64, 2048):
            slots, pos, st = run_gpu(b, k=k, chunk=chunk)
            assert st == 0, B.status_str(st)
            compare_with_oracle(b, k, slots, pos)


def test_forced_multi_cta_on_ties():
    """Tie-heavy rows forced onto many CTAs: all-equal, +/-0, fp16 grid, -inf tails."""
    rng = np.random.default_rng(11)
    L = 30000
    rows = []
    rows.append(np.full(L, 2.5, np.float32))
    rows.append(np.where(np.arange(L) % 3 == 0, np.float32(-0.0), np.float32(0.0)))
    rows.append(rng.standard_normal(L).astype(np.float16).astype(np.float32))
    x = rng.standard_normal(L).astype(np.float32)
    x[100:] = -np.inf
    rows.append(x)
    rows.append(rng.integers(-3, 4, L).astype(np.float32))
    y = np.full(L, np.nan, np.float32)
    y[::7] = -np.inf
    rows.append(y)
    s = np.stack(rows)
    lens = np.full(len(rows), L, np.int32)
    tab = np.stack([rng.permutation(-(-L // 64)).astype(np.int32) for _ in rows])
    b = W.Batch("ties", s, lens, L, 2048, tab, None, 64)
    for chunk in (0, 64, 1000, 4096):
        for k in (1, 7, 2048):
            slots, pos, st = run_gpu(b, k=k, chunk=chunk)
            assert st == 0
            compare_with_oracle(b, k, slots, pos)


def test_special_values():
    rng = np.random.default_rng(5)
    L = 9000
    vals = [np.float32(v) for v in (np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 3.4e38,
                                    -3.4e38, 65504.0, 70000.0, 2.0 ** -20, np.nan)]
    rows = []
    for i in range(8):
        x = rng.choice(np.array(vals, np.float32), size=L)
        x[rng.random(L) < 0.5] = rng.standard_normal(int((rng.random(L) < 0.5).sum()) or 1)[0]
        rows.append(x.astype(np.float32))
    s = np.stack(rows)
    lens = np.array([L, L - 1, L - 2, L - 3, 5000, 2049, 2048, 1], np.int32)
    tab = np.stack([rng.permutation(-(-L // 64)).astype(np.int32) for _ in rows])
    b = W.Batch("special", s, lens, L, 2048, tab, None, 64)
    # planned with a max_len above the medium range, so that a forced chunk splits rows
    wide = dataclasses.replace(W.with_ld(b, 16392), max_len=16385)
    for bb, chunk in ((b, 0), (wide, 0), (wide, 256)):
        for k in (1, 2, 2048):
            slots, pos, st = run_gpu(bb, k=k, chunk=chunk)
            assert st == 0
            compare_with_oracle(b, k, slots, pos)


def test_unaligned_row_stride():
    b = W.verify_80k()
    b = W.with_ld(_subset(b, np.arange(3)), b.max_len)  # ld = 80006: rows start unaligned
    assert b.ld % 4 != 0
    slots, pos, st = run_gpu(b)
    assert st == 0
    compare_with_oracle(b, b.k, slots, pos)
    m = _subset(W.mixed_decode(), np.arange(5))
    m = W.with_ld(m, m.max_len + 3)
    for chunk in (0, 4096):
        slots, pos, st = run_gpu(m, chunk=chunk)
        assert st == 0
        compare_with_oracle(m, m.k, slots, pos)


def test_plan_reuse_and_repeat():
    """One plan serves many calls (new scores, new k); counters are left clean."""
    b = W.verify_80k()
    scores, lens, table, r2t = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(lens)
    first = None
    for it in range(4):
        for k in (2048, 100, 1):
            slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=(scores, lens, table, r2t))
            assert st == 0
            if k == 2048:
                if first is None:
                    compare_with_oracle(b, k, slots, pos)
                    first = np.sort(slots, axis=1)
                else:
                    assert np.array_equal(np.sort(slots, axis=1), first)
    # new scores, same plan
    b2 = dataclasses.replace(b, scores=W.verify_80k(seed=99).scores)
    s2 = torch.from_numpy(b2.scores).cuda()
    slots, pos, st = run_gpu(b2, plan=core, dev_inputs=(s2, lens, table, r2t))
    assert st == 0
    compare_with_oracle(b2, b2.k, slots, pos)


def test_slots_only_output():
    b = W.mixed_decode()
    slots, _, st = run_gpu(b, with_pos=False)
    assert st == 0
    compare_with_oracle(b, b.k, slots, None)


def test_device_plan_matches_host_reference():
    from tests.test_plan_host import header_only, parse_plan
    grid = B.topk_grid_size()
    mixed = W.mixed_decode()
    few = _subset(mixed, np.arange(20))   # one-warp planner, one row per lane, both row kinds
    more = _subset(mixed, np.arange(45))  # one-warp planner, rows 32.. in each lane's second row
    # lengths alone (the plan reads nothing else): more than grid * 48128 values over
    # <= 64 rows start the search at the chunk cap, where nothing fits one wave
    import types
    rng = np.random.default_rng(44)
    spread = lambda n: np.exp(rng.uniform(np.log(16), np.log(30000), n)).astype(int).tolist()  # noqa: E731
    # many-bucket batches ranked in one pass over 2 and 3 rounds of 256 rows; and one
    # whose 530 split rows exceed the group states (plan error: every row ranked single)
    err_rows = [49_000 + 21 * i for i in range(530)] + [int(1.5 * 2 ** (4 + i % 10)) for i in range(70)]
    big = [types.SimpleNamespace(lens=np.array(l, np.int32), rows=len(l), max_len=max(l))
           for l in ([1_000_000] * 8, [300_000] * 32, [1_900_000] * 4, [7_000_000, 10],
                     [48_128 * 21] * 7, [48_127] * 32, [200_000] * 50, [48_127] * 64,
                     [3000 + 977 * i for i in range(63)], spread(500), spread(700),
                     err_rows)]
    pf = W.prefill()
    # the medium batches on the full planner (a max_len above the cluster range), and
    # on the cluster path
    wide = [types.SimpleNamespace(lens=x.lens, rows=x.rows, max_len=m) for x in (W.pr1(), pf)
            for m in (16385, 131073)]
    for b in (W.verify_80k(), W.verify_1m(), mixed, W.adversarial(), W.pr1(), few, more,
              W.tiny_rows()[0], W.tiny_rows()[15], pf, *wide, *big):
        lens = torch.from_numpy(b.lens).cuda()
        core = PagedTopK(b.rows, b.max_len)
        core.plan(lens)
        img_dev = core.workspace.cpu().numpy()
        img_host = np.zeros_like(img_dev)
        B.topk_plan_host(b.lens, b.rows, b.max_len, grid, 0, img_host)
        hd, rd, sd, (fd, ud), info = parse_plan(img_dev, b.rows)
        hh, rh, sh, (fh, uh), _ = parse_plan(img_host, b.rows)
        if header_only(b.rows, b.max_len, grid):  # register, medium or cluster path
            assert hd == hh
            continue
        if b.rows == len(err_rows) and b.max_len > 48_128:
            assert hh["plan_error"] == 1
        assert hd == hh
        assert np.array_equal(rd, rh)
        assert np.array_equal(sd[:hh["n_single"]], sh[:hh["n_single"]])
        assert np.array_equal(fd[:grid], fh[:grid])
        # the select kernel reads the first `grid` descriptors of each wave
        idx = (np.arange(hh["waves"])[:, None] * info["max_grid"] + np.arange(grid)).ravel()
        used = uh[idx, 0] >= 0
        assert np.array_equal(ud[idx, 0] >= 0, used)
        assert np.array_equal(ud[idx][used, :7], uh[idx][used, :7])


def test_status_errors():
    rng = np.random.default_rng(2)
    L = 6000
    s = rng.standard_normal((5, L)).astype(np.float32)
    tab = np.stack([rng.permutation(L // 64 + 1).astype(np.int32) for _ in range(5)])
    lens = np.array([L, L, L, L, L], np.int32)
    # row 1: negative table entry on a page holding selected positions
    s[1, 64:128] = 50.0
    tab[1, 1] = -3
    # row 2: slot overflow
    s[2, 0:64] = 50.0
    tab[2, 0] = 2 ** 30
    b = W.Batch("errs", s, lens, L, 16, tab, None, 64)
    slots, pos, st = run_gpu(b)
    assert st == (B.STATUS_TABLE_ENTRY | B.STATUS_SLOT_OVERFLOW), B.status_str(st)
    ref = oracle.topk_batch(b, threads=1)
    assert ref[2] == 4 | 8
    for r in range(5):
        gp, gs = C.canonical(s[r], L, pos[r], slots[r], b.k)
        assert np.array_equal(gp, ref[1][r]) and np.array_equal(gs, ref[0][r])
    # length above max_len and table too narrow: those rows all -1
    b2 = W.Batch("errs2", s[:3].copy(), np.array([L, L + 1, L], np.int32), L, 16,
                 tab[:3, :50].copy(), None, 64)
    slots, pos, st = run_gpu(b2)
    assert st & B.STATUS_LEN and st & B.STATUS_TABLE_WIDTH
    assert np.all(slots == -1) and np.all(pos == -1)


def test_plan_mismatch_is_reported():
    """A full plan records every row's length; a select with other lengths reports the
    mismatch. (Plans of the register, medium and cluster paths are the header alone:
    they hold no lengths, and any lengths up to max_len are served exactly.)"""
    b = dataclasses.replace(W.with_ld(W.pr1(), 131076), max_len=131073)
    scores, lens, table, r2t = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(lens)
    other = lens.clone()
    other[0] = 100
    out = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    core.select(scores, other, b.k, table, b.page_size, r2t, out_slots=out)
    st = core.status()
    assert st & B.STATUS_PLAN_MISMATCH
    assert torch.all(out[0] == -1)
    core.clear_status()
    assert core.status() == 0


def test_cuda_graph_replay():
    b = W.verify_80k()
    scores, lens, table, r2t = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    out = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    pos = torch.empty((b.rows, b.k), dtype=torch.int32, device="cuda")
    core.plan(lens)
    core.select(scores, lens, b.k, table, b.page_size, r2t, out_slots=out, out_pos=pos)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        core.plan(lens)
        core.select(scores, lens, b.k, table, b.page_size, r2t, out_slots=out, out_pos=pos)
    for _ in range(3):
        out.fill_(-5)
        g.replay()
    torch.cuda.synchronize()
    assert core.status() == 0
    compare_with_oracle(b, b.k, out.cpu().numpy(), pos.cpu().numpy())


def test_chunks_that_open_with_their_largest_values():
    """Chunk-local skew at the 1M verify shape (21 CTAs per row): every CTA's chunk
    opens with its largest values, so each CTA's own threshold bin, and the vectors it
    marks at that bin while the first barrier propagates, come from the chunk's first
    pieces. A second batch holds each row's whole top in its first chunk, so the bins
    the CTAs publish first cannot fix the threshold and the row publishes the rest."""
    rng = np.random.default_rng(23)
    L, G = 1_000_000, 21
    c = -(-(-(-L // G)) // 16) * 16  # each CTA's chunk of a 21-CTA row
    ramp = (6.0 - 12.0 * (np.arange(L + 6) % c) / c).astype(np.float32)
    lens = np.arange(L, L + 7, dtype=np.int32)
    s = np.full((7, W.round_up(L + 6, 4)), W.POISON, np.float32)
    for r in range(7):
        s[r, :lens[r]] = ramp[:lens[r]] + 0.05 * rng.standard_normal(lens[r]).astype(np.float32)
    tab = rng.permutation(-(-(L + 6) // 64)).astype(np.int32).reshape(1, -1)
    b = W.Batch("chunk_ramps", s, lens, L + 6, 2048, tab, np.zeros(7, np.int32), 64)
    for k in (1, 100, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)
    top = s.copy()
    for r in range(7):
        top[r, :lens[r]] = np.sort(s[r, :lens[r]])[::-1]
    bt = dataclasses.replace(b, name="row_top_first", scores=top)
    for k in (100, 2048):
        slots, pos, st = run_gpu(bt, k=k)
        assert st == 0, B.status_str(st)
        compare_with_oracle(bt, k, slots, pos)


def test_skewed_rows_over_many_ctas():
    """Rows whose top values are not spread evenly over the CTAs that share them:
    sorted descending (one chunk holds the whole top-k, so the bins each CTA publishes
    first cannot fix the threshold and the row publishes the rest), sorted ascending,
    a step at 10 % of the row, shuffled sorted blocks and massive ties. Single-CTA and
    multi-CTA splits, every k class."""
    rng = np.random.default_rng(17)
    L = 160000
    base = rng.standard_normal(L).astype(np.float32)
    desc = np.sort(base)[::-1].copy()
    asc = np.sort(base).copy()
    step = base.copy()
    step[: L // 10] += 5.0
    blocks = np.sort(base).reshape(40, -1)[rng.permutation(40)].ravel().copy()
    ties = rng.integers(-2, 3, L).astype(np.float32)
    s = np.stack([desc, asc, step, blocks, ties])
    lens = np.array([L, L - 5, L - 17, L, L], np.int32)
    tab = np.stack([rng.permutation(L // 64 + 1).astype(np.int32) for _ in range(5)])
    b = W.Batch("sampled", s, lens, L, 2048, tab, None, 64)
    for chunk in (16384, 20000, 48128):
        for k in (1, 100, 2048):
            slots, pos, st = run_gpu(b, k=k, chunk=chunk)
            assert st == 0, B.status_str(st)
            compare_with_oracle(b, k, slots, pos)
    # one CTA per row
    one = W.Batch("sampled1", s[:, :40000].copy(), np.full(5, 40000, np.int32), 40000, 2048,
                  tab[:, :626].copy(), None, 64)
    for k in (1, 100, 2048):
        slots, pos, st = run_gpu(one, k=k, chunk=48128)
        assert st == 0
        compare_with_oracle(one, k, slots, pos)


def test_eight_rows_of_1m_take_two_waves():
    """8 rows x 1,000,000: 168 CTAs at the largest chunk, more than one wave of the grid
    (the small-batch planner must hand these rows to the multi-wave path)."""
    rng = np.random.default_rng(W.SEED_BASE + 40)
    L = 1_000_000
    s = rng.standard_normal((8, L)).astype(np.float32)
    tab = rng.permutation(L // 64 + 1).astype(np.int32)[None, :]
    b = W.Batch("eight_1m", s, np.full(8, L, np.int32), L, 2048, tab,
                np.zeros(8, np.int32), 64)
    slots, pos, st = run_gpu(b)
    assert st == 0, B.status_str(st)
    compare_with_oracle(b, b.k, slots, pos)
