"""GPU parity of the indexer key-path prologue (indexer_k_prologue, through the C ABI)
against the CPU oracle (oracle/prologue.py).

What must agree: which slots are written (and that no other slot is touched), the
status bits, each token's fp32 scale (relative 4e-6: the kernel's LayerNorm runs in
fp32), and every e4m3 code. A code may differ by one step only where the oracle's
exact value r = y / scale lies next to the midpoint between the two neighbouring
codes: the kernel takes that rounding decision on its fp32 value. Its error is
relative to the token's magnitude, not to each channel (y = (x - mean) * rstd * w + b
cancels in small channels): about ten fp32 ulps of the largest |y|, i.e. 10 * 2^-24 *
448 = 2.7e-4 in units of the scale. Allowed: |r - midpoint| <= 5e-4 + 1e-5 |midpoint|.
"""
import numpy as np
import pytest

import workloads as W
from oracle import prologue as P

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from sparse_attention_indexer_gb300 import binding as B  # noqa: E402

SENTINEL_CODE = 0xAA
SENTINEL_SCALE = -7.0


def run_both(b: W.KeyBatch, cs_offset: int = 0):
    """(gpu cache, gpu scales, gpu status), (oracle cache, scales, status, y, slots).
    cs_offset > 0 places the cos/sin table that many floats into a larger buffer (an
    address without 16-byte alignment)."""
    dev = torch.device("cuda", 0)
    cs = torch.from_numpy(b.cos_sin).to(dev)
    if cs_offset:
        buf = torch.zeros(cs.numel() + cs_offset, dtype=torch.float32, device=dev)
        buf[cs_offset:] = cs.reshape(-1)
        cs = buf[cs_offset:].view(cs.shape)
    cache = torch.full((b.num_slots, b.dim), SENTINEL_CODE, dtype=torch.uint8, device=dev)
    scales = torch.full((b.num_slots,), SENTINEL_SCALE, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    B.indexer_k_prologue(torch.from_numpy(b.k_bf16.view(np.int16)).to(dev),
                         torch.from_numpy(b.ln_w).to(dev), torch.from_numpy(b.ln_b).to(dev),
                         b.eps, torch.from_numpy(b.positions).to(dev),
                         cs, b.rope_dim,
                         torch.from_numpy(b.token_table).to(dev),
                         torch.from_numpy(b.block_table).to(dev), b.page_size, cache, scales,
                         status=status)
    torch.cuda.synchronize()
    oc = np.full((b.num_slots, b.dim), SENTINEL_CODE, np.uint8)
    os_ = np.full(b.num_slots, SENTINEL_SCALE, np.float32)
    err, y, slots = P.key_prologue(b.k_bf16, b.ln_w, b.ln_b, b.eps, b.positions, b.cos_sin,
                                   b.rope_dim, b.token_table, b.block_table, b.page_size, oc, os_)
    return (cache.cpu().numpy(), scales.cpu().numpy(), int(status.item())), (oc, os_, err, y, slots)


def compare(gpu, ref, max_flip_frac=1e-3):
    gc, gs, gst = gpu
    oc, os_, ost, y, slots = ref
    assert gst == ost, f"status {gst} != oracle {ost}"
    stored = slots[slots >= 0]
    untouched = np.ones(oc.shape[0], bool)
    untouched[stored] = False
    assert np.all(gc[untouched] == SENTINEL_CODE), "a slot outside the tokens' was written"
    assert np.all(gs[untouched] == SENTINEL_SCALE), "a scale outside the tokens' was written"
    if stored.size == 0:
        return 0
    s_o = os_[stored].astype(np.float64)
    s_g = gs[stored].astype(np.float64)
    assert np.all(np.abs(s_g - s_o) <= 4e-6 * s_o), f"scale: max rel {np.max(np.abs(s_g / s_o - 1))}"
    vg = P.e4m3_value(gc[stored])
    vo = P.e4m3_value(oc[stored])
    differ = vg != vo
    n_flip = int(differ.sum())
    if n_flip:
        ok_tok = slots >= 0
        r = y[ok_tok] / s_o[:, None]
        idx = np.nonzero(differ)
        a, bval = vg[idx], vo[idx]
        mid = (a + bval) / 2
        # neighbouring codes (one step apart) and the exact value next to their midpoint
        step_ok = np.abs(gc[stored][idx].astype(np.int32) - oc[stored][idx].astype(np.int32)) == 1
        near = np.abs(r[idx] - mid) <= 5e-4 + 1e-5 * np.abs(mid)
        bad = ~(step_ok & near)
        assert not np.any(bad), (f"{int(bad.sum())} codes differ beyond a rounding tie: "
                                 f"gpu {a[bad][:4]} oracle {bval[bad][:4]} exact {r[idx][bad][:4]}")
        assert n_flip <= max_flip_frac * vg.size, f"{n_flip} rounding-tie flips of {vg.size}"
    return n_flip


def test_workload_multi_request():
    """A 16K-token prefill chunk, a 4K chunk and 7 decode tokens near position 100K."""
    b = W.key_prologue()
    compare(*run_both(b))


@pytest.mark.parametrize("rope_dim", [0, 2, 6, 24, 64, 128])
def test_rope_widths(rope_dim):
    """Rotated widths from none to all 128 channels; a lane holds channels 8h .. 8h + 7,
    so at 2 and 6 one lane rotates part of its pairs and at 24 three lanes rotate all of
    theirs while the rest rotate none."""
    b = W.key_prologue(seed=W.SEED_BASE + 60 + rope_dim, reqs=((0, 700), (5000, 300)),
                       rope_dim=rope_dim, max_pos=8192)
    compare(*run_both(b))


def test_unaligned_rope_table():
    """A cos/sin table at an address without 16-byte alignment (the header asks for
    4-byte alignment only)."""
    b = W.key_prologue(seed=W.SEED_BASE + 69, reqs=((0, 700), (5000, 300)), rope_dim=64,
                       max_pos=8192)
    compare(*run_both(b, cs_offset=1))


def test_page_sizes_and_tables():
    for ps in (1, 16, 64, 256):
        b = W.key_prologue(seed=W.SEED_BASE + 70 + ps, reqs=((0, 513), (1000, 77), (3, 1)),
                           page_size=ps, max_pos=4096)
        compare(*run_both(b))


def _crafted():
    """128-channel tokens that stress the readings: constant rows (LayerNorm gives the
    bias), all-zero rows with zero bias (amax 0: scale 1, codes 0), tiny and huge
    magnitudes (subnormal and saturating codes through the weights), exact powers of
    two, and each rejected-token case. Inputs stay below 1e19 in magnitude: the kernel
    squares them in fp32."""
    b = W.key_prologue(seed=W.SEED_BASE + 80, reqs=((0, 40), (200, 10)), max_pos=4096)
    k = b.k_bf16.view(np.uint16).copy()
    x = np.zeros((50, 128), np.float32)
    x[0] = 3.0                       # constant: y = bias
    x[1] = 0.0                       # zeros
    x[2, ::2], x[2, 1::2] = 1.0, -1.0
    x[3] = np.linspace(-1e15, 1e15, 128)  # squares stay inside fp32
    x[4] = np.linspace(-1e-30, 1e-30, 128)
    x[5, 0] = 1.0                    # one spike
    x[6] = np.ldexp(1.0, np.arange(128) % 20 - 10)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    k[:7] = bits[:7]
    w = b.ln_w.copy()
    w[:8] = [1e-4, 3e-3, 1.0, 100.0, 1e-6, 0.0, -2.0, 7.5]
    bias = b.ln_b.copy()
    bias[:] = 0.0
    bias[::5] = 0.25
    pos = b.positions.copy()
    tt = b.token_table.copy()
    pos[30] = -3                     # position error
    pos[31] = 4096                   # past the cos/sin table
    pos[32] = b.block_table.shape[1] * b.page_size  # past the table row -> table width
    tt[33] = 5                       # no such table row
    tab = b.block_table.copy()
    tab[1, 3] = -1                   # request 1's page 3 (its tokens at 200..209): negative
    return W.KeyBatch("crafted", k, w.astype(np.float32), bias.astype(np.float32), b.eps, pos,
                      b.cos_sin, b.rope_dim, tt, tab, b.page_size, b.num_slots)


def test_crafted_tokens_and_statuses():
    b = _crafted()
    gpu, ref = run_both(b)
    assert ref[2] == (P.ERR_POSITION | P.ERR_TABLE_WIDTH | P.ERR_TABLE_ROW |
                      P.ERR_TABLE_ENTRY), ref[2]
    compare(gpu, ref)


def test_slot_outside_cache():
    b = W.key_prologue(seed=W.SEED_BASE + 90, reqs=((0, 100),), max_pos=1024)
    b = W.KeyBatch(b.name, b.k_bf16, b.ln_w, b.ln_b, b.eps, b.positions, b.cos_sin, b.rope_dim,
                   b.token_table, b.block_table, b.page_size, b.num_slots - 64)
    gpu, ref = run_both(b)
    assert ref[2] == P.ERR_SLOT
    compare(gpu, ref)


def test_zero_tokens_and_row_stride():
    b = W.key_prologue(seed=W.SEED_BASE + 91, reqs=((10, 37),), max_pos=1024)
    dev = torch.device("cuda", 0)
    kk = torch.zeros((37, 136), dtype=torch.int16, device=dev)  # row stride 136 > 128
    kk[:, :128] = torch.from_numpy(b.k_bf16.view(np.int16)).to(dev)
    cache = torch.full((b.num_slots, 128), SENTINEL_CODE, dtype=torch.uint8, device=dev)
    scales = torch.full((b.num_slots,), SENTINEL_SCALE, dtype=torch.float32, device=dev)
    args = (torch.from_numpy(b.ln_w).to(dev), torch.from_numpy(b.ln_b).to(dev), b.eps,
            torch.from_numpy(b.positions).to(dev), torch.from_numpy(b.cos_sin).to(dev),
            b.rope_dim, torch.from_numpy(b.token_table).to(dev),
            torch.from_numpy(b.block_table).to(dev), b.page_size, cache, scales)
    B.indexer_k_prologue(kk[:0, :128], *args)  # zero tokens: nothing enqueued
    torch.cuda.synchronize()
    assert torch.all(cache == SENTINEL_CODE)
    B.indexer_k_prologue(kk[:, :128], *args)
    torch.cuda.synchronize()
    gpu = (cache.cpu().numpy(), scales.cpu().numpy(), 0)
    oc = np.full((b.num_slots, 128), SENTINEL_CODE, np.uint8)
    os_ = np.full(b.num_slots, SENTINEL_SCALE, np.float32)
    err, y, slots = P.key_prologue(b.k_bf16, b.ln_w, b.ln_b, b.eps, b.positions, b.cos_sin,
                                   b.rope_dim, b.token_table, b.block_table, b.page_size, oc, os_)
    compare(gpu, (oc, os_, err, y, slots))
