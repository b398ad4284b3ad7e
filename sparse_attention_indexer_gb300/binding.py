"""Thin Python binding of the C ABI in include/topk_paged.h.

Argument marshalling only: every step of the computation runs in the CUDA library.
Functions keep the C names and argument order; pointer arguments accept CUDA torch
tensors (their data_ptr is passed) or plain integers, and `stream` accepts a
torch.cuda.Stream, a raw handle or None (the current torch stream). If the library
is missing this module raises; there is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("TOPK_PAGED_LIB") or os.path.join(_PKG, "libtopk_paged.so")

TOPK_MAX_K = 2048
STATUS_LEN = 1
STATUS_TABLE_WIDTH = 2
STATUS_TABLE_ENTRY = 4
STATUS_SLOT_OVERFLOW = 8
STATUS_TIMEOUT = 16
STATUS_PLAN_MISMATCH = 32
STATUS_ORDER = 64
ERR_STATIC_ROWS = -12
STATIC_MAX_ROWS = 64

EXPORTS = (
    "topk_workspace_bytes", "topk_max_row_len", "topk_chunk_capacity", "topk_plan",
    "topk_plan_ex", "topk_select_paged", "topk_read_status", "topk_clear_status",
    "topk_status_str", "topk_grid_size", "topk_plan_host", "topk_layout_info",
    "topk_select_paged_noalloc", "indexer_k_prologue", "hisparse_resolve",
    "topk_select_paged_test", "indexer_mqa_logits", "hisparse_resolve_mtp",
)


class TopKError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {code} ({status_str(code)})")
        self.code = code


_lib = None

_c = ctypes
_VP = _c.c_void_p
_SIGS = {
    "topk_workspace_bytes": (_c.c_size_t, [_c.c_int, _c.c_int]),
    "topk_max_row_len": (_c.c_int64, []),
    "topk_chunk_capacity": (_c.c_int, []),
    "topk_grid_size": (_c.c_int, []),
    "topk_plan": (_c.c_int, [_VP, _c.c_int, _c.c_int, _VP, _c.c_size_t, _VP]),
    "topk_plan_ex": (_c.c_int, [_VP, _c.c_int, _c.c_int, _c.c_int, _VP, _c.c_size_t, _VP]),
    "topk_select_paged": (_c.c_int, [_VP, _c.c_int64, _VP, _c.c_int, _c.c_int, _c.c_int, _VP,
                                     _c.c_int64, _VP, _c.c_int, _VP, _VP, _VP, _VP]),
    "topk_read_status": (_c.c_int, [_VP, _VP, _c.POINTER(_c.c_int)]),
    "topk_clear_status": (_c.c_int, [_VP, _VP]),
    "topk_status_str": (_c.c_char_p, [_c.c_int]),
    "topk_plan_host": (_c.c_int, [_VP, _c.c_int, _c.c_int, _c.c_int, _c.c_int, _VP, _c.c_size_t]),
    "topk_layout_info": (_c.c_int, [_c.c_int, _c.POINTER(_c.c_int64), _c.c_int]),
    "topk_select_paged_test": (_c.c_int, [_VP, _c.c_int64, _VP, _c.c_int, _c.c_int, _c.c_int,
                                          _VP, _c.c_int64, _VP, _c.c_int, _VP, _VP, _VP, _VP,
                                          _c.c_uint64, _c.c_int]),
    "topk_select_paged_noalloc": (_c.c_int, [_VP, _c.c_int64, _VP, _c.c_int, _c.c_int, _c.c_int,
                                             _VP, _c.c_int64, _VP, _c.c_int, _VP, _VP, _VP, _VP]),
    "indexer_k_prologue": (_c.c_int, [_VP, _c.c_int64, _c.c_int, _c.c_int, _VP, _VP, _c.c_float,
                                      _VP, _VP, _c.c_int, _c.c_int, _VP, _VP, _c.c_int,
                                      _c.c_int64, _c.c_int, _VP, _VP, _c.c_int64, _VP, _VP]),
    "indexer_mqa_logits": (_c.c_int, [_VP, _VP, _c.c_int, _c.c_int, _c.c_int, _VP, _c.c_int,
                                      _c.c_int, _VP, _VP, _c.c_int, _c.c_int, _c.c_int, _VP, _VP,
                                      _c.c_int64, _VP, _c.c_int64, _VP, _VP]),
    "hisparse_resolve": (_c.c_int, [_VP, _c.c_int, _c.c_int, _VP, _c.c_int64, _c.c_int, _VP,
                                    _c.c_int64, _VP, _VP, _VP, _c.c_int, _c.c_int, _VP, _VP,
                                    _c.c_int64, _VP, _c.c_int64, _c.c_int, _VP, _VP, _VP, _VP]),
    "hisparse_resolve_mtp": (_c.c_int, [_VP, _c.c_int, _c.c_int, _c.c_int, _VP, _c.c_int64,
                                        _c.c_int, _VP, _c.c_int64, _VP, _VP, _VP, _c.c_int,
                                        _c.c_int, _VP, _VP, _c.c_int64, _VP, _c.c_int64, _c.c_int,
                                        _VP, _VP, _VP, _VP]),
}

# include/hisparse_resolver.h
RESOLVER_STATUS_NO_VICTIM = 1
RESOLVER_STATUS_POSITION = 2
RESOLVER_STATUS_HOST_ROW = 4
RESOLVER_STATUS_KV_ROW = 8

# include/indexer_prologue.h
PROLOGUE_OK = 0
PROLOGUE_ERR_NULL = -1
PROLOGUE_ERR_SHAPE = -2
PROLOGUE_ERR_ALIGN = -3
PROLOGUE_ERR_CUDA = -4
PROLOGUE_STATUS_POSITION = 1
PROLOGUE_STATUS_TABLE_WIDTH = 2
PROLOGUE_STATUS_TABLE_ENTRY = 4
PROLOGUE_STATUS_SLOT = 8
PROLOGUE_STATUS_TABLE_ROW = 16


class PrologueError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"indexer_k_prologue: {code}")
        self.code = code


def lib():
    """Loads libtopk_paged.so (built by sparse_attention_indexer_gb300.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {LIB_PATH} is missing "
                               "(run `python -c 'import __graft_entry__ as g; g.build()'`)")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(l, name)
            fn.restype = res
            fn.argtypes = args
        _lib = l
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if x.numel() > 0 and not x.is_cuda:
            raise ValueError("device pointer argument must be a CUDA tensor")
        return x.data_ptr() or None
    return int(x)


def _stream(s) -> Optional[int]:
    if s is None:
        return torch.cuda.current_stream().cuda_stream or None
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream or None
    return int(s) or None


def _check(code: int, what: str) -> int:
    if code < 0:
        raise TopKError(code, what)
    return code


def status_str(code: int) -> str:
    return lib().topk_status_str(int(code)).decode()


topk_status_str = status_str


def topk_workspace_bytes(rows: int, max_len: int) -> int:
    return int(lib().topk_workspace_bytes(int(rows), int(max_len)))


def topk_max_row_len() -> int:
    return int(_check(lib().topk_max_row_len(), "topk_max_row_len"))


def topk_chunk_capacity() -> int:
    return int(lib().topk_chunk_capacity())


def topk_grid_size() -> int:
    return int(_check(lib().topk_grid_size(), "topk_grid_size"))


def topk_plan(lens, rows: int, max_len: int, workspace, ws_bytes: int, stream=None) -> int:
    return _check(lib().topk_plan(_ptr(lens), int(rows), int(max_len), _ptr(workspace),
                                  int(ws_bytes), _stream(stream)), "topk_plan")


def topk_plan_ex(lens, rows: int, max_len: int, chunk: int, workspace, ws_bytes: int,
                 stream=None) -> int:
    return _check(lib().topk_plan_ex(_ptr(lens), int(rows), int(max_len), int(chunk),
                                     _ptr(workspace), int(ws_bytes), _stream(stream)),
                  "topk_plan_ex")


def topk_select_paged_test(scores, ld: int, lens, rows: int, max_len: int, k: int, block_table,
                           table_ld: int, row_to_table, page_size: int, out_slots, out_pos,
                           workspace, wait_ns: int, skip_cta: int, stream=None) -> int:
    """topk_select_paged with a bounded-wait limit (ns) and a CTA that skips the first
    row-barrier arrival of its units (test hooks)."""
    return _check(lib().topk_select_paged_test(
        _ptr(scores), int(ld), _ptr(lens), int(rows), int(max_len), int(k), _ptr(block_table),
        int(table_ld), _ptr(row_to_table), int(page_size), _ptr(out_slots), _ptr(out_pos),
        _ptr(workspace), _stream(stream), int(wait_ns), int(skip_cta)), "topk_select_paged_test")


def topk_select_paged(scores, ld: int, lens, rows: int, max_len: int, k: int, block_table,
                      table_ld: int, row_to_table, page_size: int, out_slots, out_pos,
                      workspace, stream=None) -> int:
    return _check(lib().topk_select_paged(
        _ptr(scores), int(ld), _ptr(lens), int(rows), int(max_len), int(k), _ptr(block_table),
        int(table_ld), _ptr(row_to_table), int(page_size), _ptr(out_slots), _ptr(out_pos),
        _ptr(workspace), _stream(stream)), "topk_select_paged")


def topk_select_paged_noalloc(scores, ld: int, lens, rows: int, max_len: int, k: int,
                              block_table, table_ld: int, row_to_table, page_size: int,
                              out_slots, out_pos, status, stream=None) -> int:
    """No workspace argument: the library's static device scratch serves the call."""
    return _check(lib().topk_select_paged_noalloc(
        _ptr(scores), int(ld), _ptr(lens), int(rows), int(max_len), int(k), _ptr(block_table),
        int(table_ld), _ptr(row_to_table), int(page_size), _ptr(out_slots), _ptr(out_pos),
        _ptr(status), _stream(stream)), "topk_select_paged_noalloc")


def topk_read_status(workspace, stream=None) -> int:
    v = ctypes.c_int(0)
    _check(lib().topk_read_status(_ptr(workspace), _stream(stream), ctypes.byref(v)),
           "topk_read_status")
    return int(v.value)


def topk_clear_status(workspace, stream=None) -> int:
    return _check(lib().topk_clear_status(_ptr(workspace), _stream(stream)), "topk_clear_status")


def topk_plan_host(lens, rows: int, max_len: int, grid: int, chunk: int, image) -> int:
    """Host reference of the planner writing into a host buffer (numpy uint8 array)."""
    import numpy as np
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    return _check(lib().topk_plan_host(lens.ctypes.data_as(ctypes.c_void_p), int(rows),
                                       int(max_len), int(grid), int(chunk),
                                       image.ctypes.data_as(ctypes.c_void_p), int(image.nbytes)),
                  "topk_plan_host")


def indexer_k_prologue(k, ln_w, ln_b, eps: float, positions, cos_sin, rope_dim: int,
                       token_table, block_table, page_size: int, cache, cache_scale,
                       status=None, stream=None) -> int:
    """indexer_k_prologue of include/indexer_prologue.h on CUDA tensors: k (bf16 or
    its int16 bits) [tokens, ld], ln_w / ln_b float32 [dim], positions / token_table
    int32 [tokens], cos_sin float32 [max_pos, rope_dim], block_table int32
    [n_tables, table_ld], cache uint8 [num_slots, dim], cache_scale float32
    [num_slots], status int32 [1] or None. Argument marshalling only."""
    tokens, ld = (int(k.shape[0]), int(k.stride(0))) if k.dim() == 2 else (0, 0)
    dim = int(k.shape[1]) if k.dim() == 2 else 0
    code = lib().indexer_k_prologue(
        _ptr(k), ld, tokens, dim, _ptr(ln_w), _ptr(ln_b), float(eps), _ptr(positions),
        _ptr(cos_sin), int(cos_sin.shape[0]), int(rope_dim), _ptr(token_table),
        _ptr(block_table), int(block_table.shape[0]), int(block_table.stride(0)), int(page_size),
        _ptr(cache), _ptr(cache_scale), int(cache.shape[0]), _ptr(status), _stream(stream))
    if code < 0:
        raise PrologueError(code)
    return code


# include/indexer_logits.h
LOGITS_ERR_NULL = -1
LOGITS_ERR_SHAPE = -2
LOGITS_ERR_ALIGN = -3
LOGITS_ERR_CUDA = -4
LOGITS_STATUS_LEN = 1
LOGITS_STATUS_TABLE_WIDTH = 2
LOGITS_STATUS_TABLE_ENTRY = 4
LOGITS_STATUS_SLOT = 8
LOGITS_STATUS_TABLE_ROW = 16
LOGITS_STATUS_TIMEOUT = 32


class LogitsError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"indexer_mqa_logits: {code}")
        self.code = code


def indexer_mqa_logits(q, w, lens, max_len: int, group_rows: int, group_table, block_table,
                       page_size: int, cache, cache_scale, scores, status=None,
                       stream=None) -> int:
    """indexer_mqa_logits of include/indexer_logits.h on CUDA tensors: q uint8 [rows,
    heads, dim], w float32 [rows, heads], lens int32 [rows], group_table int32 [groups]
    or None, block_table int32 [n_tables, table_ld], cache uint8 [num_slots, dim],
    cache_scale float32 [num_slots], scores float32 [rows, ld], status int32 [1] or
    None. Argument marshalling only."""
    rows, heads, dim = (int(x) for x in q.shape)
    code = lib().indexer_mqa_logits(
        _ptr(q), _ptr(w), rows, heads, dim, _ptr(lens), int(max_len), int(group_rows),
        _ptr(group_table), _ptr(block_table), int(block_table.shape[0]),
        int(block_table.stride(0)), int(page_size), _ptr(cache), _ptr(cache_scale),
        int(cache.shape[0]), _ptr(scores), int(scores.stride(0)), _ptr(status), _stream(stream))
    if code < 0:
        raise LogitsError(code)
    return code


class ResolverError(RuntimeError):
    def __init__(self, code: int):
        super().__init__(f"hisparse_resolve: {code}")
        self.code = code


def hisparse_resolve(positions, block_table, page_size: int, token_to_hot, hot_token,
                     hot_step, hot_rows, step: int, host_kv, host_base, kv, out_rows,
                     counts=None, status=None, stream=None) -> int:
    """hisparse_resolve of include/hisparse_resolver.h: positions / block_table /
    token_to_hot / hot_token / hot_step / hot_rows / out_rows CUDA int32 tensors, host_kv
    a pinned CPU uint8 tensor [host_rows, row_bytes], host_base CUDA int64 [rows], kv
    CUDA uint8 [kv_rows, row_bytes]. Argument marshalling only."""
    if host_kv.is_cuda or (host_kv.numel() and not host_kv.is_pinned()):
        raise ValueError("host_kv must be pinned host memory")
    rows, k = int(positions.shape[0]), int(positions.shape[1])
    code = lib().hisparse_resolve(
        _ptr(positions), rows, k, _ptr(block_table), int(block_table.stride(0)),
        int(page_size), _ptr(token_to_hot), int(token_to_hot.stride(0)), _ptr(hot_token),
        _ptr(hot_step), _ptr(hot_rows), int(hot_rows.shape[1]), int(step),
        host_kv.data_ptr() or None, _ptr(host_base), int(host_kv.shape[0]), _ptr(kv),
        int(kv.shape[0]), int(kv.shape[1]), _ptr(out_rows), _ptr(counts), _ptr(status),
        _stream(stream))
    if code < 0:
        raise ResolverError(code)
    return code


def hisparse_resolve_mtp(positions, block_table, page_size: int, token_to_hot, hot_token,
                         hot_step, hot_rows, step: int, host_kv, host_base, kv, out_rows,
                         counts=None, status=None, stream=None) -> int:
    """hisparse_resolve_mtp of include/hisparse_resolver.h: as hisparse_resolve, with
    positions and out_rows CUDA int32 [rows, q_rows, k]. Argument marshalling only."""
    if host_kv.is_cuda or (host_kv.numel() and not host_kv.is_pinned()):
        raise ValueError("host_kv must be pinned host memory")
    rows, q_rows, k = (int(x) for x in positions.shape)
    code = lib().hisparse_resolve_mtp(
        _ptr(positions), rows, q_rows, k, _ptr(block_table), int(block_table.stride(0)),
        int(page_size), _ptr(token_to_hot), int(token_to_hot.stride(0)), _ptr(hot_token),
        _ptr(hot_step), _ptr(hot_rows), int(hot_rows.shape[1]), int(step),
        host_kv.data_ptr() or None, _ptr(host_base), int(host_kv.shape[0]), _ptr(kv),
        int(kv.shape[0]), int(kv.shape[1]), _ptr(out_rows), _ptr(counts), _ptr(status),
        _stream(stream))
    if code < 0:
        raise ResolverError(code)
    return code


def topk_layout_info(rows: int):
    arr = (ctypes.c_int64 * 12)()
    _check(lib().topk_layout_info(int(rows), arr, 12), "topk_layout_info")
    keys = ("max_grid", "max_waves", "chunk_cap", "header_bytes", "rowinfo", "singles",
            "first_single", "units", "groups", "threads", "group_cap", "list_cap")
    return dict(zip(keys, [int(v) for v in arr]))
