"""GB300 (sm_103a) indexer top-k selection fused with paged KV-slot translation.

The computation lives in the CUDA library libtopk_paged.so (C ABI:
include/topk_paged.h); `binding` mirrors that ABI name for name and `api` wraps it
with torch-owned device memory and streams.
"""
from . import binding
from .api import HostPagedTopK, PagedTopK
from .binding import TopKError

__all__ = ["binding", "PagedTopK", "HostPagedTopK", "TopKError"]
