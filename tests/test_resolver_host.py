"""hisparse_resolve's host-side argument checks (no GPU needed: every error is returned
before any CUDA call)."""
import os

import pytest

S = pytest.importorskip("sparse_attention_indexer_gb300")
B = S.binding


def _call(**kw):
    if not os.path.exists(B.LIB_PATH):
        pytest.skip("library not built")
    a = dict(positions=0x1000, rows=2, k=16, block_table=0x2000, table_ld=4, page_size=64,
             token_to_hot=0x3000, map_ld=256, hot_token=0x4000, hot_step=0x5000,
             hot_rows=0x6000, hot_size=32, step=0, host_kv=0x7000, host_base=0x8000,
             host_rows=512, kv=0x9000, kv_rows=64, row_bytes=656, out_rows=0xA000,
             counts=None, status=None, stream=None)
    a.update(kw)
    return B.lib().hisparse_resolve(*a.values())


def test_argument_errors_before_any_launch():
    shape = -2
    for kw in (dict(rows=-1), dict(k=0), dict(k=2049), dict(hot_size=0), dict(hot_size=4097),
               dict(page_size=0), dict(table_ld=0), dict(map_ld=0), dict(step=-1),
               dict(row_bytes=8), dict(row_bytes=650), dict(kv_rows=-1), dict(host_rows=-1)):
        assert _call(**kw) == shape, kw
    assert _call(rows=0) == 0
    assert _call(positions=None) == -1
    assert _call(host_kv=None) == -1
    assert _call(kv=0x9008) == -3
    assert _call(host_kv=0x7004) == -3
    assert _call(host_base=0x8004) == -3
    assert _call(status=0x10002) == -3
