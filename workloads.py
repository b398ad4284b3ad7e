"""Seeded synthetic inputs for per-query top-k selection with paged slot translation.

This module only draws random numbers and lays them out as arrays (score rows,
valid lengths, block tables). It holds none of the selection or slot arithmetic,
so both the CPU oracle and the CUDA path can consume its batches without sharing
any of the method's code.

Workloads follow the indexer top-k setting of "Serving GLM5.2 NVFP4 Agentic
Workload with SGLang" (section "Kernel Optimization > TopK-V2", Fig. 4): fp32
score rows over the historical KV positions of each query, k up to 2048, KV pages
of 64 tokens ("llm-d ... GLM-5.2 on H200", KV block size). The agentic replay
corpus measured there is not available; the distributions below stand in for it.

Every batch stores scores as float32 [rows, ld] with ld >= max_len. Entries at
positions >= lens[r] are poisoned with +3e38 so that any out-of-range read would
win the selection and fail parity loudly.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

POISON = np.float32(3.0e38)
SEED_BASE = 0x5EED0000


@dataclasses.dataclass
class Batch:
    """One call's worth of inputs (k may be varied by the caller per call)."""

    name: str
    scores: np.ndarray            # float32 [rows, ld]
    lens: np.ndarray              # int32 [rows]
    max_len: int
    k: int
    block_table: np.ndarray       # int32 [n_tables, table_ld]
    row_to_table: Optional[np.ndarray]  # int32 [rows] or None (identity)
    page_size: int
    ks: Optional[List[int]] = None  # per-call k sequence, where the workload defines one

    @property
    def rows(self) -> int:
        return int(self.scores.shape[0])

    @property
    def ld(self) -> int:
        return int(self.scores.shape[1])

    def algorithmic_bytes(self, k: Optional[int] = None, with_pos: bool = False) -> int:
        """Scores read once + each distinct table's used pages once + the slot output."""
        k = self.k if k is None else k
        score_b = 4 * int(self.lens.astype(np.int64).sum())
        r2t = (np.arange(self.rows, dtype=np.int64) if self.row_to_table is None
               else self.row_to_table.astype(np.int64))
        pages = 0
        for t in np.unique(r2t):
            lmax = int(self.lens[r2t == t].max()) if self.rows else 0
            pages += -(-lmax // self.page_size)
        out_b = 4 * self.rows * k * (2 if with_pos else 1)
        return score_b + 4 * pages + out_b


def round_up(x: int, m: int) -> int:
    return -(-x // m) * m


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def _empty_scores(rows: int, ld: int) -> np.ndarray:
    s = np.empty((rows, ld), dtype=np.float32)
    s.fill(POISON)
    return s


def _shuffled_pages(rng: np.random.Generator, n: int) -> np.ndarray:
    return rng.permutation(n).astype(np.int32)


def _tables_from_pool(rng, lens, page_size, table_ld):
    """One table row per request; pages drawn without replacement from one shuffled pool.
    Unused entries are -1 (a null placeholder that must never be read)."""
    need = [-(-int(l) // page_size) for l in lens]
    pool = _shuffled_pages(rng, max(1, sum(need)))
    tab = np.full((len(lens), table_ld), -1, dtype=np.int32)
    off = 0
    for r, n in enumerate(need):
        tab[r, :n] = pool[off:off + n]
        off += n
    return tab


def pr1(seed: int = SEED_BASE + 0) -> Batch:
    """4 rows, lens {4096, 5000, 6144, 8192}, k=2048, N(0,1), page_size 64,
    block tables = a random permutation of 4*128 page ids sliced 128 per row."""
    rng = _rng(seed)
    lens = np.array([4096, 5000, 6144, 8192], dtype=np.int32)
    max_len = 8192
    s = _empty_scores(4, round_up(max_len, 4))
    for r, l in enumerate(lens):
        s[r, :l] = rng.standard_normal(l).astype(np.float32)
    perm = _shuffled_pages(rng, 512)
    tab = perm.reshape(4, 128).copy()
    return Batch("pr1_ref", s, lens, max_len, 2048, tab, None, 64)


def tiny_rows(seed: int = SEED_BASE + 10, n_rows: int = 1000, page_size: int = 64):
    """1000 tiny rows, len U[1, 64], per-row k U[1, 16], values uniform on {-2..2}
    (massive ties). Returned as one Batch per k value (k is a per-call argument)."""
    rng = _rng(seed)
    lens = rng.integers(1, 65, size=n_rows).astype(np.int32)
    ks = rng.integers(1, 17, size=n_rows)
    max_len = 64
    vals = rng.integers(-2, 3, size=(n_rows, max_len)).astype(np.float32)
    tabs = _tables_from_pool(rng, lens, page_size, -(-max_len // page_size))
    out = []
    for k in range(1, 17):
        idx = np.nonzero(ks == k)[0]
        if idx.size == 0:
            continue
        s = _empty_scores(idx.size, max_len)
        for j, r in enumerate(idx):
            s[j, :lens[r]] = vals[r, :lens[r]]
        out.append(Batch(f"tiny_k{k}", s, lens[idx].copy(), max_len, k,
                         tabs[idx].copy(), None, page_size))
    return out


def verify_80k(seed: int = SEED_BASE + 1) -> Batch:
    """bs=1 MTP target verify at 80K ISL: 7 rows with causal lengths 80000..80006,
    k=2048, N(0,1) with 1% of positions given a +3 sigma outlier, page_size 64,
    one shuffled table of 1251 pages shared by the 7 rows."""
    rng = _rng(seed)
    lens = np.arange(80000, 80007, dtype=np.int32)
    max_len = 80006
    s = _empty_scores(7, round_up(max_len, 4))
    for r, l in enumerate(lens):
        x = rng.standard_normal(l)
        x += 3.0 * (rng.random(l) < 0.01)
        s[r, :l] = x.astype(np.float32)
    tab = _shuffled_pages(rng, -(-max_len // 64)).reshape(1, -1)
    return Batch("verify_80k", s, lens, max_len, 2048, tab,
                 np.zeros(7, dtype=np.int32), 64)


def verify_1m(seed: int = SEED_BASE + 2, amplitude: float = 1.0, period: int = 1 << 18) -> Batch:
    """bs=1 MTP target verify at 1M ISL: 7 rows with lengths 1,000,000..1,000,006,
    k=2048, N(0,1) plus a slowly varying sinusoidal bias A*sin(2*pi*p/P) along
    position (A=1, P=2^18 positions), page_size 64, one shuffled table."""
    rng = _rng(seed)
    lens = np.arange(1_000_000, 1_000_007, dtype=np.int32)
    max_len = 1_000_006
    s = _empty_scores(7, round_up(max_len, 4))
    bias = amplitude * np.sin(2.0 * math.pi * np.arange(max_len) / period)
    for r, l in enumerate(lens):
        s[r, :l] = (rng.standard_normal(l) + bias[:l]).astype(np.float32)
    tab = _shuffled_pages(rng, -(-max_len // 64)).reshape(1, -1)
    return Batch("verify_1m", s, lens, max_len, 2048, tab,
                 np.zeros(7, dtype=np.int32), 64)


def mixed_decode(seed: int = SEED_BASE + 3) -> Batch:
    """Mixed decode batch: 64 requests x 1 row, lengths log-uniform in [1024, 200000],
    k=2048, N(0,1), page_size 64, a random page table per request."""
    rng = _rng(seed)
    lens = np.floor(np.exp(rng.uniform(math.log(1024), math.log(200000), size=64))).astype(np.int32)
    lens = np.clip(lens, 1024, 200000)
    max_len = 200000
    s = _empty_scores(64, round_up(max_len, 4))
    for r, l in enumerate(lens):
        s[r, :l] = rng.standard_normal(l).astype(np.float32)
    tab = _tables_from_pool(rng, lens, 64, -(-max_len // 64))
    return Batch("mixed_decode", s, lens, max_len, 2048, tab, None, 64)


ADV_KS = (1, 64, 512, 2048)


def adversarial(seed: int = SEED_BASE + 4, rows: int = 256, max_len: int = 32768) -> Batch:
    """256 rows x max_len 32768, page_size 32, 1024-page table per row from one
    shuffled pool; k drawn per call from {1, 64, 512, 2048}. Row kind = row mod 6:
    0 all-equal (cycling +/-0 alternating by position, all -0.0, all 1.5);
    1 N(0,1) rounded to the fp16 grid; 2 N(0,1) prefix then -inf up to len;
    3 len U[0, 2047] (below the largest k, some exactly 0); 4 Cauchy tan(pi(U-1/2));
    5 N(0,1) at full length. Lengths of kinds other than 3 and 5 are U[1, max_len]."""
    rng = _rng(seed)
    ps = 32
    lens = np.zeros(rows, dtype=np.int32)
    s = _empty_scores(rows, round_up(max_len, 4))
    for r in range(rows):
        kind, m = r % 6, r // 6
        if kind == 3:
            l = 0 if m % 4 == 0 else int(rng.integers(0, 2048))
        elif kind == 5:
            l = max_len
        else:
            l = int(rng.integers(1, max_len + 1))
        lens[r] = l
        if kind == 0:
            c = m % 3
            if c == 0:
                x = np.where(np.arange(l) % 2 == 0, np.float32(0.0), np.float32(-0.0))
            elif c == 1:
                x = np.full(l, -0.0, dtype=np.float32)
            else:
                x = np.full(l, 1.5, dtype=np.float32)
        elif kind == 1:
            x = rng.standard_normal(l).astype(np.float16).astype(np.float32)
        elif kind == 2:
            x = rng.standard_normal(l).astype(np.float32)
            cut = int(rng.integers(0, l + 1))
            x[cut:] = -np.inf
        elif kind == 4:
            x = np.tan(math.pi * (rng.random(l) - 0.5)).astype(np.float32)
        else:
            x = rng.standard_normal(l).astype(np.float32)
        s[r, :l] = x
    tab = _tables_from_pool(rng, [max_len] * rows, ps, max_len // ps)
    ks = [int(v) for v in rng.permutation(np.array(ADV_KS))]
    return Batch("adversarial", s, lens, max_len, ks[0], tab, None, ps, ks=ks)


def prefill(seed: int = SEED_BASE + 5, prefixes=(8192,), q=(4096,), k: int = 2048,
            page_size: int = 64) -> Batch:
    """Ragged prefill: request j has prefixes[j] cached tokens and q[j] new query tokens;
    query i of request j scores the causal prefix of length prefixes[j] + i + 1. Rows
    are the queries of all requests in order (thousands of rows whose lengths step by
    one); scores N(0,1); each request's pages come from one shuffled pool and every
    row maps to its request's table (row_to_table)."""
    rng = _rng(seed)
    lens, r2t = [], []
    for j, (pre, nq) in enumerate(zip(prefixes, q)):
        lens.extend(pre + i + 1 for i in range(nq))
        r2t.extend([j] * nq)
    lens = np.array(lens, dtype=np.int32)
    max_len = int(max(p + n for p, n in zip(prefixes, q)))
    s = _empty_scores(len(lens), round_up(max_len, 4))
    for r, l in enumerate(lens):
        s[r, :l] = rng.standard_normal(int(l)).astype(np.float32)
    req_len = np.array([p + n for p, n in zip(prefixes, q)], dtype=np.int32)
    tab = _tables_from_pool(rng, req_len, page_size, -(-max_len // page_size))
    return Batch("prefill", s, lens, max_len, k, tab, np.array(r2t, dtype=np.int32), page_size)


CONFIGS = {
    "pr1_ref": pr1,
    "verify_80k": verify_80k,
    "verify_1m": verify_1m,
    "mixed_decode": mixed_decode,
    "adversarial": adversarial,
    "prefill": prefill,
}


def with_ld(b: Batch, ld: int) -> Batch:
    """Same rows re-laid with another row stride (e.g. ld = max_len, not a multiple of 4)."""
    assert ld >= b.max_len
    s = _empty_scores(b.rows, ld)
    w = min(ld, b.ld)
    s[:, :w] = b.scores[:, :w]
    return dataclasses.replace(b, scores=s)


# ---------------------------------------------------------------- key-path prologue
@dataclasses.dataclass
class KeyBatch:
    """Inputs of one call of the indexer key-path prologue (LayerNorm, RoPE, FP8 store
    into the paged indexer KV cache) for T tokens of D channels."""

    name: str
    k_bf16: np.ndarray        # uint16 [T, D]: bfloat16 bit patterns (the wk projection's output)
    ln_w: np.ndarray          # float32 [D]
    ln_b: np.ndarray          # float32 [D]
    eps: float
    positions: np.ndarray     # int32 [T]: logical position of each token in its request
    cos_sin: np.ndarray       # float32 [max_pos, R]: cos of the R / 2 pair angles, then sines
    rope_dim: int
    token_table: np.ndarray   # int32 [T]: block-table row of each token's request
    block_table: np.ndarray   # int32 [n_req, table_ld]
    page_size: int
    num_slots: int

    @property
    def tokens(self) -> int:
        return int(self.k_bf16.shape[0])

    @property
    def dim(self) -> int:
        return int(self.k_bf16.shape[1])

    def algorithmic_bytes(self) -> int:
        """Keys, positions, token tables and each token's cos/sin row read once (the
        distinct positions' rows), each used table entry once; codes and scales
        written once."""
        T, D = self.k_bf16.shape
        rows = len(np.unique(self.positions[(self.positions >= 0) &
                                            (self.positions < self.cos_sin.shape[0])]))
        pages = len(np.unique(self.token_table.astype(np.int64) * (1 << 32) +
                              self.positions.astype(np.int64) // self.page_size))
        return T * (2 * D + 8) + rows * 4 * self.rope_dim + 4 * pages + T * (D + 4)


def rope_table(max_pos: int, rope_dim: int, base: float = 10000.0) -> np.ndarray:
    """cos / sin of the angles p * base^(-2i / R), p < max_pos, i < R / 2, as float32
    [max_pos, R] (cosines first): the caller-side table a RoPE kernel reads."""
    i = np.arange(rope_dim // 2, dtype=np.float64)
    inv = base ** (-2.0 * i / rope_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even) and return the bits."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def key_prologue(seed: int = SEED_BASE + 6, reqs=((0, 16384), (4000, 4096), (100000, 7)),
                 dim: int = 128, rope_dim: int = 64, page_size: int = 64,
                 max_pos: int = 131072) -> KeyBatch:
    """Tokens of several requests in one call: request j contributes n_j tokens at
    positions start_j, ..., start_j + n_j - 1 (a prefill chunk, or a few decode
    tokens). Key channels are N(0,1) times a per-channel spread (exp of N(0, 0.5)) plus
    a per-channel offset N(0, 0.5), rounded to bfloat16; LayerNorm weight 1 + N(0, 0.1),
    bias N(0, 0.1), eps 1e-6; RoPE base 10000. Each request's pages are drawn from one
    shuffled pool of physical pages; the cache has exactly the pool's slots."""
    rng = _rng(seed)
    spread = np.exp(rng.normal(0.0, 0.5, dim))
    offset = rng.normal(0.0, 0.5, dim)
    pos, t2t = [], []
    for j, (start, n) in enumerate(reqs):
        pos.extend(range(start, start + n))
        t2t.extend([j] * n)
    T = len(pos)
    x = (rng.standard_normal((T, dim)) * spread + offset).astype(np.float32)
    ends = np.array([s + n for s, n in reqs], dtype=np.int64)
    table_ld = int(-(-int(ends.max()) // page_size))
    need = [int(-(-e // page_size)) for e in ends]
    pool = _shuffled_pages(rng, sum(need))
    tab = np.full((len(reqs), table_ld), -1, np.int32)
    at = 0
    for j, m in enumerate(need):
        tab[j, :m] = pool[at:at + m]
        at += m
    return KeyBatch("key_prologue", _to_bf16_bits(x),
                    (1.0 + rng.normal(0.0, 0.1, dim)).astype(np.float32),
                    rng.normal(0.0, 0.1, dim).astype(np.float32), 1e-6,
                    np.array(pos, np.int32), rope_table(max_pos, rope_dim), rope_dim,
                    np.array(t2t, np.int32), tab, page_size, int(sum(need)) * page_size)


# ---------------------------------------------------------------- top-K resolver
@dataclasses.dataclass
class ResolverBatch:
    """Requests with a mixed-residency block table, a hot buffer each, their history in
    host memory, and a sequence of per-step top-K selections."""

    name: str
    block_table: np.ndarray   # int32 [R, table_ld]: block id (resident) or -1 (host only)
    page_size: int
    lens: np.ndarray          # int32 [R]: context length of each request
    hot_rows: np.ndarray      # int32 [R, H]: KV rows of each request's hot slots
    kv_rows: int              # rows of the KV tensor
    row_bytes: int
    host_kv: np.ndarray       # uint8 [sum(lens), row_bytes]: every position's KV row
    host_base: np.ndarray     # int64 [R]: host row of position 0 of each request
    kv_init: np.ndarray       # uint8 [kv_rows, row_bytes]: the KV tensor before step 0
    steps: List[np.ndarray]   # int32 [R, k] per step: selected positions (distinct, -1 pad)

    @property
    def rows(self) -> int:
        return int(self.block_table.shape[0])

    @property
    def hot_size(self) -> int:
        return int(self.hot_rows.shape[1])


def hisparse(seed: int = SEED_BASE + 7, reqs: int = 8, k: int = 2048, page_size: int = 64,
             lens=None, tail: int = 4096, resident_frac: float = 0.1, row_bytes: int = 656,
             n_steps: int = 4, keep: float = 0.85, tail_frac: float = 0.1) -> ResolverBatch:
    """Decode steps of `reqs` requests under KV pressure. Each request keeps its last
    `tail` positions resident plus a `resident_frac` share of older pages; the other
    pages are null placeholders whose rows live in host memory. Each request leases a
    hot buffer of 2k rows (whole blocks from the same pool). Step selections: about
    `keep` of the previous step's positions again (decode attends to much the same
    tokens from step to step), the rest new, `tail_frac` of them in the resident tail;
    -1 padding when a request has fewer than k positions. Row bytes 656: one FP8
    sparse-MLA token row (512 fp8 + 64 bf16 + 16 scale bytes)."""
    rng = _rng(seed)
    if lens is None:
        lens = rng.integers(20000, 60000, size=reqs)
    lens = np.asarray(lens, np.int64)
    R = len(lens)
    H = 2 * k
    n_pages = -(-lens // page_size)
    table_ld = int(n_pages.max())
    tab = np.full((R, table_ld), -1, np.int32)
    blocks = 0
    for j in range(R):
        npg = int(n_pages[j])
        res = np.zeros(npg, bool)
        res[max(0, npg - (-(-tail // page_size))):] = True
        res |= rng.random(npg) < resident_frac
        idx = np.nonzero(res)[0]
        tab[j, idx] = np.arange(blocks, blocks + len(idx), dtype=np.int32)
        blocks += len(idx)
    hot_blocks = -(-H // page_size)  # whole blocks; the first H rows are the slots
    hot_rows = np.zeros((R, H), np.int32)
    for j in range(R):
        base = blocks + j * hot_blocks
        hot_rows[j] = (base * page_size + rng.permutation(H)).astype(np.int32)
    kv_rows = (blocks + R * hot_blocks) * page_size
    # shuffle the physical block ids so resident and hot rows interleave in the pool
    perm = rng.permutation(blocks + R * hot_blocks).astype(np.int64)
    tab = np.where(tab >= 0, perm[np.maximum(tab, 0)], -1).astype(np.int32)
    hot_rows = (perm[hot_rows // page_size] * page_size + hot_rows % page_size).astype(np.int32)
    host_base = np.concatenate([[0], np.cumsum(lens)[:-1]]).astype(np.int64)
    host_kv = rng.integers(0, 256, size=(int(lens.sum()), row_bytes), dtype=np.uint8)
    kv_init = rng.integers(0, 256, size=(kv_rows, row_bytes), dtype=np.uint8)
    steps = []
    prev = [None] * R
    for s in range(n_steps):
        sel = np.full((R, k), -1, np.int32)
        for j in range(R):
            L = int(lens[j])
            m = min(k, L)
            chosen: List[int] = []
            seen = set()
            if prev[j] is not None:
                for p in prev[j]:
                    if len(chosen) >= int(keep * m):
                        break
                    if rng.random() < keep and p not in seen:
                        chosen.append(int(p))
                        seen.add(int(p))
            while len(chosen) < m:
                if rng.random() < tail_frac:
                    p = int(rng.integers(max(0, L - tail), L))
                else:
                    p = int(rng.integers(0, L))
                if p not in seen:
                    chosen.append(p)
                    seen.add(p)
            order = rng.permutation(m)
            sel[j, :m] = np.asarray(chosen, np.int32)[order]
            prev[j] = sel[j, :m].copy()
        steps.append(sel)
    return ResolverBatch("hisparse", tab, page_size, lens.astype(np.int32), hot_rows, kv_rows,
                         row_bytes, host_kv, host_base, kv_init, steps)


def hisparse_mtp(seed: int = SEED_BASE + 10, reqs: int = 4, k: int = 512, q_rows: int = 3,
                 page_size: int = 64, lens=None, tail: int = 1024, resident_frac: float = 0.1,
                 row_bytes: int = 64, n_steps: int = 4, keep: float = 0.85, tail_frac: float = 0.1,
                 draft_new: float = 0.2):
    """Multi-token verify steps: each step has q_rows query rows per request (the
    decoded token and its drafts). Row 0 follows the recipe of `hisparse`; each draft
    row takes row 0's positions and replaces about `draft_new` of them with other
    positions of the context (draft tokens attend to much the same tokens). Hot buffers
    hold (q_rows + 1) * k rows, the pages' (num_speculative_tokens + 2) x top-K."""
    base = hisparse(seed=seed, reqs=reqs, k=k, page_size=page_size, lens=lens, tail=tail,
                    resident_frac=resident_frac, row_bytes=row_bytes, n_steps=n_steps,
                    keep=keep, tail_frac=tail_frac)
    rng = _rng(seed + 1)
    R = base.rows
    H = (q_rows + 1) * k
    # re-lease hot buffers of H rows per request from fresh blocks after the base pool
    hot_blocks = -(-H // page_size)
    first = base.kv_rows // page_size
    hot_rows = np.zeros((R, H), np.int32)
    for j in range(R):
        b0 = first + j * hot_blocks
        hot_rows[j] = (b0 * page_size + rng.permutation(hot_blocks * page_size)[:H]).astype(np.int32)
    kv_rows = (first + R * hot_blocks) * page_size
    kv_init = np.concatenate([base.kv_init, rng.integers(0, 256, size=(kv_rows - base.kv_rows,
                                                                       row_bytes), dtype=np.uint8)])
    steps = []
    for sel0 in base.steps:
        st = np.full((R, q_rows, k), -1, np.int32)
        st[:, 0] = sel0
        for j in range(R):
            L = int(base.lens[j])
            m = int((sel0[j] >= 0).sum())
            for q in range(1, q_rows):
                row = sel0[j, :m].copy()
                seen = set(int(x) for x in row)
                for i in range(m):
                    if rng.random() < draft_new:
                        for _ in range(8):
                            p = int(rng.integers(0, L))
                            if p not in seen:
                                seen.discard(int(row[i]))
                                row[i] = p
                                seen.add(p)
                                break
                st[j, q, :m] = row[rng.permutation(m)]
        steps.append(st)
    return dataclasses.replace(base, name="hisparse_mtp", hot_rows=hot_rows, kv_rows=kv_rows,
                               kv_init=kv_init, steps=steps)


# ---------------------------------------------------------------- indexer MQA logits
@dataclasses.dataclass
class LogitsBatch:
    """Inputs of one call of the indexer score producer (MQA logits over the paged FP8
    key cache) and of the top-k selection that consumes its score rows.

    Query rows come in groups of `group_rows` consecutive rows (the tokens of one
    request: a decode token and its draft tokens, or a prefill chunk); every row of
    group g reads the keys of block-table row group_table[g] (g itself when
    group_table is None), each up to its own valid length."""

    name: str
    q: np.ndarray             # uint8 [rows, H, D]: e4m3 codes of the per-head queries
    w: np.ndarray             # float32 [rows, H]: head-gate weights
    cache: np.ndarray         # uint8 [num_slots, D]: e4m3 codes of the keys
    cache_scale: np.ndarray   # float32 [num_slots]: per-key scales
    lens: np.ndarray          # int32 [rows]: keys each query row scores
    max_len: int
    group_rows: int
    group_table: Optional[np.ndarray]  # int32 [n_groups] or None
    block_table: np.ndarray   # int32 [n_tables, table_ld]
    page_size: int
    k: int = 2048

    @property
    def rows(self) -> int:
        return int(self.q.shape[0])

    @property
    def heads(self) -> int:
        return int(self.q.shape[1])

    @property
    def dim(self) -> int:
        return int(self.q.shape[2])

    @property
    def num_slots(self) -> int:
        return int(self.cache.shape[0])

    def row_to_table(self) -> np.ndarray:
        """Block-table row of every query row (int32 [rows])."""
        g = np.arange(self.rows) // self.group_rows
        t = g if self.group_table is None else self.group_table[g]
        return np.asarray(t, np.int32)

    def flops(self) -> int:
        """Multiply-adds of the query-key products, counted as 2 FLOPs each: every
        head of every row against each of the row's keys."""
        return 2 * int(self.lens.astype(np.int64).clip(0).sum()) * self.heads * self.dim


def e4m3_codes(rng: np.random.Generator, shape, exp_mean: float, exp_sd: float) -> np.ndarray:
    """Random e4m3 bit patterns: a fair sign bit, an exponent field drawn as
    round(N(exp_mean, exp_sd)) clipped to [0, 15], a uniform 3-bit mantissa; the
    NaN pattern (exponent 15, mantissa 7) becomes mantissa 6 (the largest finite)."""
    sign = rng.integers(0, 2, size=shape).astype(np.uint8) << 7
    e = np.clip(np.rint(rng.normal(exp_mean, exp_sd, size=shape)), 0, 15).astype(np.uint8)
    m = rng.integers(0, 8, size=shape).astype(np.uint8)
    m = np.where((e == 15) & (m == 7), np.uint8(6), m)
    return (sign | (e << 3) | m).astype(np.uint8)


def logits_batch(name: str, seed: int, lens, group_rows: int, heads: int = 64, dim: int = 128,
                 page_size: int = 64, n_tables: Optional[int] = None, spare_pages: int = 0,
                 k: int = 2048) -> LogitsBatch:
    """Query rows with the given valid lengths, in groups of `group_rows`. Each group
    gets its own block-table row (a shuffled set of physical pages from one pool;
    group_table is a permutation when n_tables > groups, else None); the cache holds
    the pool's pages plus `spare_pages` unused ones.

    Codes stand in for per-token-scaled FP8 tensors, whose largest element sits near
    448: key exponent fields N(13, 1.5), query fields N(12, 1.5); key scales
    exp(N(-6, 0.3)) (about 1/400, an amax near 1); head gates N(0, 1) / 64."""
    rng = _rng(seed)
    lens = np.asarray(lens, np.int32)
    rows = len(lens)
    n_groups = -(-rows // group_rows)
    glen = [int(lens[g * group_rows:(g + 1) * group_rows].clip(0).max()) for g in range(n_groups)]
    max_len = int(lens.max()) if rows else 0
    table_ld = max(1, -(-max_len // page_size))
    need = [-(-L // page_size) for L in glen]
    pool = _shuffled_pages(rng, sum(need) + spare_pages)
    nt = n_groups if n_tables is None else max(n_tables, n_groups)
    tab = np.full((nt, table_ld), -1, np.int32)
    gt = None
    if nt > n_groups:
        gt = rng.permutation(nt)[:n_groups].astype(np.int32)
    at = 0
    for g, m in enumerate(need):
        tab[g if gt is None else gt[g], :m] = pool[at:at + m]
        at += m
    num_slots = (sum(need) + spare_pages) * page_size
    cache = e4m3_codes(rng, (num_slots, dim), 13.0, 1.5)
    scale = np.exp(rng.normal(-6.0, 0.3, num_slots)).astype(np.float32)
    q = e4m3_codes(rng, (rows, heads, dim), 12.0, 1.5)
    w = (rng.standard_normal((rows, heads)) / 64.0).astype(np.float32)
    return LogitsBatch(name, q, w, cache, scale, lens, max_len, group_rows, gt, tab, page_size, k)


def logits_verify_80k(seed: int = SEED_BASE + 8) -> LogitsBatch:
    """bs=1 MTP target verify at 80K context: 7 query rows (1 + 6 draft tokens) of one
    request, causal lengths 80000..80006, 64 heads of 128 channels, pages of 64."""
    return logits_batch("logits_verify_80k", seed, np.arange(80000, 80007), 7)


def logits_verify_1m(seed: int = SEED_BASE + 9) -> LogitsBatch:
    """The same at 1M context: lengths 1,000,000..1,000,006."""
    return logits_batch("logits_verify_1m", seed, np.arange(1000000, 1000007), 7)
