"""indexer_k_prologue's host-side argument checks (no GPU needed: every error is
returned before any CUDA call)."""
import os

import pytest

S = pytest.importorskip("sparse_attention_indexer_gb300")
B = S.binding


def _lib():
    if not os.path.exists(B.LIB_PATH):
        pytest.skip("library not built")
    return B.lib()


def _call(lib, **kw):
    a = dict(k=0x1000, ld=128, tokens=4, dim=128, ln_w=0x2000, ln_b=0x3000, eps=1e-6,
             positions=0x4000, cos_sin=0x5000, max_pos=16, rope_dim=64, token_table=0x6000,
             block_table=0x7000, n_tables=1, table_ld=4, page_size=64, cache=0x8000,
             cache_scale=0x9000, num_slots=256, status=None, stream=None)
    a.update(kw)
    return lib.indexer_k_prologue(*a.values())


def test_argument_errors_before_any_launch():
    lib = _lib()
    shape = B.PROLOGUE_ERR_SHAPE
    assert _call(lib, dim=64) == shape
    assert _call(lib, tokens=-1) == shape
    assert _call(lib, rope_dim=3) == shape
    assert _call(lib, rope_dim=130) == shape
    assert _call(lib, max_pos=0) == shape
    assert _call(lib, page_size=0) == shape
    assert _call(lib, n_tables=0) == shape
    assert _call(lib, table_ld=0) == shape
    assert _call(lib, num_slots=-1) == shape
    assert _call(lib, ld=100) == shape
    assert _call(lib, ld=132) == shape          # not a multiple of 8
    assert _call(lib, eps=-1.0) == shape
    assert _call(lib, eps=float("nan")) == shape
    assert _call(lib, tokens=0) == B.PROLOGUE_OK  # nothing to do
    assert _call(lib, k=None) == B.PROLOGUE_ERR_NULL
    assert _call(lib, cache_scale=None) == B.PROLOGUE_ERR_NULL
    assert _call(lib, k=0x1008) == B.PROLOGUE_ERR_ALIGN      # k needs 16 bytes
    assert _call(lib, ln_w=0x2008) == B.PROLOGUE_ERR_ALIGN   # ln_w needs 16 bytes
    assert _call(lib, cache=0x8004) == B.PROLOGUE_ERR_ALIGN
    assert _call(lib, status=0x9002) == B.PROLOGUE_ERR_ALIGN
