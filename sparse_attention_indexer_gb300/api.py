"""Tensor-level front end over the C ABI: workspace ownership, plan reuse, host I/O.

Every compute step runs in the CUDA library (libtopk_paged.so); this module only
allocates device memory through torch and passes pointers, sizes and the stream.
"""
from __future__ import annotations

from typing import Optional, Tuple

import torch

from . import binding as B


class PagedTopK:
    """Top-k selection with paged slot translation for batches of up to `rows` rows
    whose valid lengths are at most `max_len`.

    plan() is called once per batch (per forward); select() once per indexer layer,
    any k in [1, 2048]. Output rows hold min(k, len) slots then -1."""

    def __init__(self, rows: int, max_len: int, device: Optional[torch.device] = None):
        if device is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.rows = int(rows)
        self.max_len = int(max_len)
        self.device = device
        self.ws_bytes = B.topk_workspace_bytes(self.rows, self.max_len)
        # torch's caching allocator returns 512-byte aligned blocks
        self.workspace = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
        assert self.workspace.data_ptr() % 256 == 0

    def plan(self, lens: torch.Tensor, chunk: int = 0, stream=None) -> None:
        """chunk forces the elements per CTA when nonzero (tests: path forcing)."""
        assert lens.dtype == torch.int32 and lens.is_cuda and lens.numel() == self.rows
        if chunk:
            B.topk_plan_ex(lens, self.rows, self.max_len, chunk, self.workspace, self.ws_bytes,
                           stream)
        else:
            B.topk_plan(lens, self.rows, self.max_len, self.workspace, self.ws_bytes, stream)

    def select(self, scores: torch.Tensor, lens: torch.Tensor, k: int, block_table: torch.Tensor,
               page_size: int, row_to_table: Optional[torch.Tensor] = None,
               out_slots: Optional[torch.Tensor] = None, out_pos: Optional[torch.Tensor] = None,
               with_pos: bool = False, stream=None) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
        assert scores.dtype == torch.float32 and scores.dim() == 2 and scores.stride(1) == 1
        assert scores.shape[0] == self.rows
        assert block_table.dtype == torch.int32 and block_table.dim() == 2
        assert block_table.stride(1) == 1
        if out_slots is None:
            out_slots = torch.empty((self.rows, k), dtype=torch.int32, device=scores.device)
        if with_pos and out_pos is None:
            out_pos = torch.empty((self.rows, k), dtype=torch.int32, device=scores.device)
        B.topk_select_paged(scores, scores.stride(0), lens, self.rows, self.max_len, k,
                            block_table, block_table.stride(0), row_to_table, page_size,
                            out_slots, out_pos, self.workspace, stream)
        return out_slots, out_pos

    def status(self, stream=None) -> int:
        return B.topk_read_status(self.workspace, stream)

    def clear_status(self, stream=None) -> None:
        B.topk_clear_status(self.workspace, stream)


class HostPagedTopK:
    """End-to-end call on host buffers: pinned host -> device copies, plan + select,
    device -> pinned host copy of the slots, all on one stream."""

    def __init__(self, rows: int, ld: int, max_len: int, k: int, n_tables: int, table_ld: int,
                 with_row_to_table: bool, device: Optional[torch.device] = None):
        self.core = PagedTopK(rows, max_len, device)
        dev = self.core.device
        self.k = int(k)
        self.scores = torch.empty((rows, ld), dtype=torch.float32, device=dev)
        self.lens = torch.empty(rows, dtype=torch.int32, device=dev)
        self.table = torch.empty((n_tables, table_ld), dtype=torch.int32, device=dev)
        self.r2t = (torch.empty(rows, dtype=torch.int32, device=dev) if with_row_to_table
                    else None)
        self.out = torch.empty((rows, k), dtype=torch.int32, device=dev)
        self.out_host = torch.empty((rows, k), dtype=torch.int32, pin_memory=True)

    def h2d_bytes(self, with_table: bool = True) -> int:
        b = self.scores.numel() * 4 + self.lens.numel() * 4
        if with_table:
            b += self.table.numel() * 4 + (self.r2t.numel() * 4 if self.r2t is not None else 0)
        return b

    def d2h_bytes(self) -> int:
        return self.out.numel() * 4

    def __call__(self, scores_h: torch.Tensor, lens_h: torch.Tensor, table_h: torch.Tensor,
                 r2t_h: Optional[torch.Tensor], page_size: int, copy_table: bool = True,
                 stream=None) -> torch.Tensor:
        self.scores.copy_(scores_h, non_blocking=True)
        self.lens.copy_(lens_h, non_blocking=True)
        if copy_table:
            self.table.copy_(table_h, non_blocking=True)
            if self.r2t is not None:
                self.r2t.copy_(r2t_h, non_blocking=True)
        self.core.plan(self.lens, stream=stream)
        self.core.select(self.scores, self.lens, self.k, self.table, page_size, self.r2t,
                         out_slots=self.out, stream=stream)
        self.out_host.copy_(self.out, non_blocking=True)
        return self.out_host
