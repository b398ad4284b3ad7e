"""GPU parity of the register-resident path (batches whose rows are at most 256 values:
one warp per row) against the CPU oracle, bit-exact.

Covers special values (+/-inf, +/-0, denormals, NaN, values past the fp16 range), tie
heavy and all-equal rows, every length from 0 to 256 with k below, at and above it,
page sizes that are and are not powers of two, a row-to-table map, slots-only output,
every device status, a plan built for other lengths, and thousands of rows per call.
"""
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
    lens = rng.integers(0, max_len + 1, n).astype(np.int32)
    lens[:4] = [0, 1, max_len - 1, max_len][:min(4, n)]
    if kind == "normal":
        s = rng.standard_normal((n, max_len)).astype(np.float32)
    elif kind == "fp16":
        s = rng.standard_normal((n, max_len)).astype(np.float16).astype(np.float32)
    elif kind == "ties":
        s = rng.integers(-2, 3, (n, max_len)).astype(np.float32)
    else:  # all equal per row
        s = np.repeat(rng.standard_normal((n, 1)).astype(np.float32), max_len, axis=1)
    return s, lens


def _batch(name, s, lens, max_len, page_size=64, seed=0, r2t=False):
    rng = np.random.default_rng(seed)
    rows = s.shape[0]
    ld = W.round_up(max_len, 4)
    sc = np.full((rows, ld), W.POISON, np.float32)
    sc[:, :max_len] = s
    for r in range(rows):
        sc[r, lens[r]:max_len] = W.POISON
    npg = -(-max_len // page_size)
    if r2t:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(3)])
        m = rng.integers(0, 3, rows).astype(np.int32)
    else:
        tab = np.stack([rng.permutation(npg * 3)[:npg].astype(np.int32) for _ in range(rows)])
        m = None
    return W.Batch(name, sc, lens, max_len, 2048, tab, m, page_size)


@pytest.mark.parametrize("max_len", [64, 100, 256])
@pytest.mark.parametrize("kind", ["normal", "fp16", "ties", "equal"])
def test_short_rows_every_k(max_len, kind):
    rng = np.random.default_rng(max_len * 10 + ["normal", "fp16", "ties", "equal"].index(kind))
    s, lens = _rows(rng, 300, max_len, kind)
    b = _batch(f"short_{kind}", s, lens, max_len, seed=1)
    dev = to_dev(b)
    core = PagedTopK(b.rows, b.max_len)
    core.plan(dev[1])
    for k in (1, 2, 7, 63, 64, 65, 128, 200, 255, 256, 2048):
        slots, pos, st = run_gpu(b, k=k, plan=core, dev_inputs=dev)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)


def test_short_special_values():
    rng = np.random.default_rng(5)
    L = 256
    vals = np.array([np.inf, -np.inf, 0.0, -0.0, 1e-40, -1e-40, 3.4e38, -3.4e38, 65504.0,
                     70000.0, 2.0 ** -20, np.nan], np.float32)
    s = rng.choice(vals, size=(12, L)).astype(np.float32)
    mix = rng.random((12, L)) < 0.4
    s[mix] = rng.standard_normal(int(mix.sum())).astype(np.float32)
    lens = np.array([L, L - 1, 200, 129, 128, 65, 64, 33, 32, 2, 1, 0], np.int32)
    b = _batch("short_special", s, lens, L, seed=6)
    for k in (1, 2, 31, 100, 2048):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0, B.status_str(st)
        compare_with_oracle(b, k, slots, pos)


@pytest.mark.parametrize("page_size", [1, 3, 64])
def test_short_page_sizes_row_map_and_slots_only(page_size):
    rng = np.random.default_rng(page_size)
    s, lens = _rows(rng, 200, 256, "normal")
    b = _batch("short_pages", s, lens, 256, page_size=page_size, seed=7, r2t=True)
    for k in (5, 100):
        slots, pos, st = run_gpu(b, k=k)
        assert st == 0
        compare_with_oracle(b, k, slots, pos)
    slots, _, st = run_gpu(b, k=100, with_pos=False)
    assert st == 0
    compare_with_oracle(b, 100, slots, None)


def test_short_many_rows():
    rng = np.random.default_rng(9)
    s, lens = _rows(rng, 5000, 192, "fp16")
    b = _batch("short_many", s, lens, 192, seed=10)
    slots, pos, st = run_gpu(b, k=32)
    assert st == 0
    compare_with_oracle(b, 32, slots, pos)


def test_short_status_errors():
    rng = np.random.default_rng(2)
    L = 200
    s = rng.standard_normal((6, L)).astype(np.float32)
    s[1, 64:128] = 50.0
    s[2, 0:64] = 50.0
    b = _batch("short_errs", s, np.full(6, L, np.int32), L, seed=3)
    b.block_table[1, 1] = -3        # the selected positions of row 1 map to a negative page
    b.block_table[2, 0] = 2 ** 30   # row 2's selected slots overflow int32
    slots, pos, st = run_gpu(b, k=16)
    assert st == (B.STATUS_TABLE_ENTRY | B.STATUS_SLOT_OVERFLOW), B.status_str(st)
    ref = oracle.topk_batch(b, k=16, threads=1)
    assert ref[2] == 4 | 8
    compare_with_oracle(b, 16, slots, pos, ref=ref)
    # a length above max_len (row 1) and a table too narrow (every row): rows all -1
    bad = W.Batch("short_errs2", b.scores.copy(), np.array([L, L + 1, L, 10, 0, L], np.int32),
                  L, 16, b.block_table[:, :2].copy(), None, 64)
    slots, pos, st = run_gpu(bad, k=16)
    assert st & B.STATUS_LEN and st & B.STATUS_TABLE_WIDTH, B.status_str(st)
    assert np.all(slots[[0, 1, 2, 5]] == -1) and np.all(pos[[0, 1, 2, 5]] == -1)
    # rows whose pages fit the narrow table are exact
    sub = W.Batch("short_errs3", bad.scores[[3, 4]].copy(), bad.lens[[3, 4]].copy(), L, 16,
                  bad.block_table[[3, 4]].copy(), None, 64)
    compare_with_oracle(sub, 16, slots[[3, 4]], pos[[3, 4]])


def test_short_plan_mismatch():
    rng = np.random.default_rng(4)
    s, lens = _rows(rng, 20, 128, "normal")
    b = _batch("short_plan", s, lens, 128, seed=5)
    scores, lens_d, table, r2t = to_dev(b)
    core = PagedTopK(b.rows + 1, b.max_len)  # a plan for one more row
    core.plan(torch.cat([lens_d, lens_d[:1]]))
    out = torch.empty((b.rows, 8), dtype=torch.int32, device="cuda")
    B.topk_select_paged(scores, scores.stride(0), lens_d, b.rows, b.max_len, 8, table,
                        table.stride(0), r2t, b.page_size, out, None, core.workspace)
    assert core.status() & B.STATUS_PLAN_MISMATCH
    assert torch.all(out == -1)
