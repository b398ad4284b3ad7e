"""CPU oracle for indexer top-k selection with paged slot translation.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm. The product library never imports it.

The computation lives in ``topk_oracle.cpp`` (plain C++: a full std::sort of each
row under the tie rule, then the page-table lookup); this module compiles it with
the host compiler on first use and calls it through ctypes. See the header of the
C++ file for the definition and the readings of the source pages it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "topk_oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LOCK = threading.Lock()
_LIBS = {}

ERR_LEN = 1
ERR_TABLE_WIDTH = 2
ERR_TABLE_ENTRY = 4
ERR_SLOT_OVERFLOW = 8


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mut{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one deliberately wrong variant) into oracle/_build."""
    out = lib_path(mutant)
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(_SRC)):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _lib(mutant: int = 0):
    with _LOCK:
        if mutant not in _LIBS:
            lib = ctypes.CDLL(build(mutant))
            for fn in (lib.oracle_topk_paged, lib.oracle_topk_paged_nth):
                fn.restype = ctypes.c_int
                fn.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                               ctypes.c_int, ctypes.c_int, ctypes.c_void_p, ctypes.c_int64,
                               ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                               ctypes.c_int]
            _LIBS[mutant] = lib
        return _LIBS[mutant]


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def topk_paged(scores: np.ndarray, lens: np.ndarray, max_len: int, k: int,
               block_table: np.ndarray, row_to_table: Optional[np.ndarray], page_size: int,
               threads: int = 1, use_nth: bool = False, mutant: int = 0
               ) -> Tuple[np.ndarray, np.ndarray, int]:
    """Returns (slots[rows, k], positions[rows, k], error_bits), each row sorted by
    (score desc, position asc) and padded with -1."""
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    lens = np.ascontiguousarray(lens, dtype=np.int32)
    block_table = np.ascontiguousarray(block_table, dtype=np.int32)
    if block_table.ndim == 1:
        block_table = block_table.reshape(1, -1)
    if row_to_table is not None:
        row_to_table = np.ascontiguousarray(row_to_table, dtype=np.int32)
    rows = int(scores.shape[0])
    slots = np.empty((rows, k), dtype=np.int32)
    pos = np.empty((rows, k), dtype=np.int32)
    lib = _lib(mutant)
    fn = lib.oracle_topk_paged_nth if use_nth else lib.oracle_topk_paged
    err = fn(_ptr(scores), scores.shape[1], _ptr(lens), rows, int(max_len), int(k),
             _ptr(block_table), block_table.shape[1], _ptr(row_to_table), int(page_size),
             _ptr(slots), _ptr(pos), int(threads))
    if err < 0:
        raise ValueError("oracle rejected its arguments")
    return slots, pos, err


def topk_batch(batch, k: Optional[int] = None, **kw):
    """Convenience: run the oracle on a workloads.Batch."""
    return topk_paged(batch.scores, batch.lens, batch.max_len, batch.k if k is None else k,
                      batch.block_table, batch.row_to_table, batch.page_size, **kw)
