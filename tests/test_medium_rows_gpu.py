"""GPU parity of the medium-row path (batches whose rows are at most 16384 values: one
CTA per row, several CTAs per SM, exact radix selection over coarse digit, key bytes
and position) against the CPU oracle, bit-exact.

Covers rows of every length class (all taken, just above k, full), N(0,1), fp16-grid,
few-value and all-equal rows (selection down to the position levels), special values
(+/-inf, +/-0, denormals, NaN, values past the fp16 range), -inf tails and NaN rows,
unaligned row starts, page sizes that are and are not powers of two, a row-to-table
map, slots-only output, the 4096-row ragged prefill batch, one plan serving many calls
(the row tickets carry across calls), a forced-chunk plan, every device status and a
plan built for other lengths.
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


def _rows(rng, n, max_len, kind):
    lens = rng.integers(257, max_len + 1, n).astype(np.int32)
    lens[:6] = np.minimum([max_len, max_len - 1, 257, 2048, 2049, 1], max_len)[:min(6, n)]
    if kind == "normal":
        s = rng.standard_normal((n, max_len)).astype(np.float32)
    elif kind == "fp16":
        s = rng.standard_normal((n, max_len)).astype(np.float16).astype(np.float32)
    elif kind == "few":
        s = rng.integers(-2, 3, (n, max_len)).astype(np.float32)
    else:  # all equal per row: the selection reaches the position levels
        s = np.repeat(rng.standard_normal((n, 1)).astype(np.float32), max_len, axis=1)
    return s, lens


def _batch(name, s, lens, max_len, page_size=64, seed=0, r2t=False, ld=None):
    rng = np.random.default_rng(seed)
    rows = s.shape[0]
    ld = ld or W.round_up(max_len, 4)
    sc = np.full((rows, ld), W.POISON, np.float32)
    sc[:, :max_len] = s[:, :max_len]
    for r in range(rows):
        sc[r, lens[r]:] = W.POISON
    npg = -(-max_len // page_size)
    if r2t:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(3)])
        m = rng.integers(0, 3, rows).astype(np.int32)
    else:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(rows)])
        m = None
    return W.Batch(name, sc, lens, max_len, 2048, tab, m, page_size)


@pytest.mark.parametrize("max_len", [300, 4099, 12288, 16384])
@pytest.mark.parametrize("kind", ["normal", "fp16", "few", "equal"])
def test_medium_rows_every_k(max_len, kind):
    rng = np.random.default_rng(max_len + ["normal", "fp16", "few", "equal"].index(kind))
    s, lens = _rows(rng, 40, max_len, kind)
    b = _batch(f"medium_{kind}", s, lens, max_len, seed=1)
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1])
    for k in (1, 7, 255, 256, 257, 1000, 2048):
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)


def test_medium_special_values_and_tails():
    rng = np.random.default_rng(5)
    L = 9000
    vals = np.array([np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, 65504.0,
                     70000.0, 2.0 ** -20, np.nan], np.float32)
    s = rng.choice(vals, size=(10, L)).astype(np.float32)
    mix = rng.random((10, L)) < 0.4
    s[mix] = rng.standard_normal(int(mix.sum())).astype(np.float32)
    s[6, 50:] = -np.inf                    # a short N(0,1) prefix, then -inf
    s[7] = np.nan                          # NaN rows with -inf every 7th position
    s[7, ::7] = -np.inf
    s[8] = np.where(np.arange(L) % 3 == 0, np.float32(-0.0), np.float32(0.0))
    s[9] = np.float32(2.5)
    lens = np.array([L, L - 1, 8193, 4097, 2049, 2048, L, L, L, L], np.int32)
    b = _batch("medium_special", s, lens, L, seed=6)
    for k in (1, 2, 100, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)


@pytest.mark.parametrize("page_size", [1, 7, 64])
def test_medium_unaligned_rows_page_sizes_row_map(page_size):
    rng = np.random.default_rng(page_size)
    s, lens = _rows(rng, 30, 6001, "normal")
    b = _batch("medium_pages", s, lens, 6001, page_size=page_size, seed=7, r2t=True, ld=6001)
    assert b.ld % 4 != 0  # rows start at unaligned addresses
    for k in (5, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)
    slots, _, st = run_gpu(b, k=300, with_pos=False)
    assert st == 0
    compare_with_oracle(b, 300, slots, None)


def test_medium_prefill_batch():
    b = W.prefill()
    assert b.max_len <= 16384
    for k in (1, 100, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)


def test_medium_one_plan_many_calls_and_forced_chunk():
    """The row tickets carry from call to call: many calls on one plan, with changing k
    and score tensors, are all exact; a forced-chunk plan is served by the same path."""
    rng = np.random.default_rng(9)
    s, lens = _rows(rng, 700, 3000, "normal")
    b = _batch("medium_many", s, lens, 3000, seed=10)
    s2, _ = _rows(rng, 700, 3000, "fp16")
    b2 = _batch("medium_many2", s2, lens, 3000, seed=10)
    scores, lens_d, table, r2t = to_dev(b)
    sc2 = torch.from_numpy(b2.scores).cuda()
    core = PagedTopK(b.rows, b.max_len)
    core.plan(lens_d)
    refs = {}
    for it in range(3):
        for k in (2048, 17, 1):
            for bb, ss in ((b, scores), (b2, sc2)):
                slots, pos, st = run_gpu(bb, k=k, plan=core, dev_inputs=(ss, lens_d, table, r2t))
                assert st == 0
                key = (bb.name, k)
                if key not in refs:
                    refs[key] = oracle.topk_batch(bb, k=k, threads=8)
                compare_with_oracle(bb, k, slots, pos, ref=refs[key])
    core.plan(lens_d, chunk=512)
    slots, pos, st = run_gpu(b, k=100, plan=core, dev_inputs=(scores, lens_d, table, r2t))
    assert st == 0
    compare_with_oracle(b, 100, slots, pos)


def test_medium_rows_copied_ahead_with_error_and_short_rows():
    """Many more rows than CTAs: each CTA copies its next row into shared memory while
    it finishes the current one. Rows too long for the table (their copy is issued,
    then the row reports the table width and writes -1), rows no longer than k (no
    copy, every position taken) and ordinary rows are interleaved."""
    rng = np.random.default_rng(41)
    rows, L = 1500, 3000
    lens = rng.integers(50, L + 1, rows).astype(np.int32)
    s = rng.standard_normal((rows, L)).astype(np.float32)
    b = _batch("medium_copied", s, lens, L, seed=42, r2t=True)
    narrow = W.Batch(b.name, b.scores, b.lens, b.max_len, b.k, b.block_table[:, :40].copy(),
                     b.row_to_table, b.page_size)  # 2560 positions: longer rows fail
    k = 128
    slots, pos, st = run_gpu(narrow, k=k)
    bad = lens > 40 * 64
    assert bad.any() and (lens <= k).any()
    assert st == B.STATUS_TABLE_WIDTH, B.status_str(st)
    assert np.all(slots[bad] == -1) and np.all(pos[bad] == -1)
    ok = np.nonzero(~bad)[0]
    sub = W.Batch("medium_copied_ok", narrow.scores[ok].copy(), lens[ok].copy(), L, k,
                  narrow.block_table, narrow.row_to_table[ok].copy(), 64)
    compare_with_oracle(sub, k, slots[ok], pos[ok])


def test_medium_status_errors_and_plan_mismatch():
    rng = np.random.default_rng(2)
    L = 5000
    s = rng.standard_normal((6, L)).astype(np.float32)
    s[1, 64:128] = 50.0
    s[2, 0:64] = 50.0
    b = _batch("medium_errs", s, np.full(6, L, np.int32), L, seed=3)
    b.block_table[1, 1] = -3        # the selected positions of row 1 map to a negative page
    b.block_table[2, 0] = 2 ** 30   # row 2's selected slots overflow int32
    slots, pos, st = run_gpu(b, k=16)
    assert st == (B.STATUS_TABLE_ENTRY | B.STATUS_SLOT_OVERFLOW), B.status_str(st)
    ref = oracle.topk_batch(b, k=16, threads=1)
    compare_with_oracle(b, 16, slots, pos, ref=ref)
    # a length above max_len (row 1) and a table too narrow for rows 0, 2, 5
    bad = W.Batch("medium_errs2", b.scores.copy(), np.array([L, L + 1, L, 100, 0, L], np.int32),
                  L, 16, b.block_table[:, :10].copy(), None, 64)
    slots, pos, st = run_gpu(bad, k=16)
    assert st & B.STATUS_LEN and st & B.STATUS_TABLE_WIDTH, B.status_str(st)
    assert np.all(slots[[0, 1, 2, 5]] == -1) and np.all(pos[[0, 1, 2, 5]] == -1)
    sub = W.Batch("medium_errs3", bad.scores[[3, 4]].copy(), bad.lens[[3, 4]].copy(), L, 16,
                  bad.block_table[[3, 4]].copy(), None, 64)
    compare_with_oracle(sub, 16, slots[[3, 4]], pos[[3, 4]])
    # a plan for one more row
    scores, lens_d, table, r2t = to_dev(b)
    core = PagedTopK(b.rows + 1, b.max_len)
    core.plan(torch.cat([lens_d, lens_d[:1]]))
    out = torch.empty((b.rows, 8), dtype=torch.int32, device="cuda")
    B.topk_select_paged(scores, scores.stride(0), lens_d, b.rows, b.max_len, 8, table,
                        table.stride(0), r2t, b.page_size, out, None, core.workspace)
    assert core.status() & B.STATUS_PLAN_MISMATCH
    assert torch.all(out == -1)
