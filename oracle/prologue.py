"""CPU oracle of the indexer key-path prologue: LayerNorm, RoPE, FP8 (e4m3)
quantization with a per-token scale, and the store into the paged indexer KV cache.

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference arm. The product library never imports it.

Source: "Serving GLM5.2 NVFP4 Agentic Workload with SGLang", section "Indexer
Prologue Fusion" (and its Figure 5): the key side of the DSA indexer prologue runs
LayerNorm, RoPE, FP8 quantization and the paged indexer-KV-cache store, fused into one
kernel, on the key activations that the fused wk projection produced (the projection
itself is a GEMM, outside this step; the fused path has no Hadamard transform).

The pages name the steps but fix none of their parameters. Readings taken here:

* LayerNorm over the D channels of one token, with per-channel weight w and bias b:
  y = (x - mean) / sqrt(var + eps) * w + b, var the biased (population) variance.
* RoPE on channels [0, R) in adjacent pairs (2i, 2i + 1), the rotation of the RoFormer
  paper: (a, b) -> (a cos - b sin, a sin + b cos) with the caller's cos/sin table
  entry [position, i]; channels [R, D) pass unrotated.
* FP8 e4m3 ("fn" encoding: bias 7, 3 mantissa bits, largest finite 448, no infinity)
  with one fp32 scale per token: scale = amax / 448 (1 when amax = 0), code =
  e4m3(y / scale) rounded to nearest, ties to even, saturating at +-448.
* The token at logical position p of request r is stored at the physical slot
  table[r][p / page_size] * page_size + p % page_size, the slot rule of the top-k
  path's page translation; codes go to cache[slot, 0:D], the scale to scale[slot].
* A token whose position lies outside the cos/sin table or the table row, whose
  block-table row does not exist, whose page entry is negative, or whose slot lies
  outside the cache is not stored, and sets a status bit (the same bits as the
  kernel's), checked in that order.

Arithmetic is fp64 up to y / scale; the rounding to e4m3 is exact from that value.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
# status bits
ERR_POSITION = 1    # position < 0 or >= the cos/sin table's rows
ERR_TABLE_WIDTH = 2  # position / page_size >= table_ld
ERR_TABLE_ENTRY = 4  # negative page entry
ERR_SLOT = 8        # slot outside [0, num_slots)
ERR_TABLE_ROW = 16  # token's block-table row outside [0, n_tables)

# Deliberately wrong variants, for the pin-strength test (0 = the oracle).
MUTANTS = {
    1: "RoPE rotation with the sign of sin flipped",
    2: "LayerNorm with the unbiased (n - 1) variance",
    3: "e4m3 rounding toward zero instead of to nearest-even",
    4: "RoPE on the last R channels instead of the first",
    5: "scale = amax / 127 (an int8 range) instead of / 448",
    6: "slot = table[p % ps] * ps + p / ps (page and offset swapped)",
    7: "LayerNorm without the bias",
    8: "e4m3 ties rounded away from zero",
}


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns (uint16) to float64: the upper half of an fp32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def e4m3_value(code: np.ndarray) -> np.ndarray:
    """Value of each e4m3 code (uint8): sign, 4 exponent bits (bias 7), 3 mantissa
    bits; exponent field 0 is subnormal (2^-6 * m / 8); S.1111.111 is NaN."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    v = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    v = np.where((e == 15) & (m == 7), np.nan, v)
    return s * v


def e4m3_encode(r: np.ndarray, mutant: int = 0) -> np.ndarray:
    """Nearest e4m3 code to each real r (float64), ties to even, saturating at +-448.
    NaN maps to 0x7F. Written from the format's definition: the representable
    magnitudes in [2^e, 2^(e+1)) are spaced 2^(e-3) for e in [-6, 8]; below 2^-6 they
    are the multiples of 2^-9."""
    r = np.asarray(r, dtype=np.float64)
    a = np.abs(r)
    with np.errstate(divide="ignore", invalid="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.clip(e, -6, 8)
    step = np.ldexp(1.0, (e - 3).astype(np.int64))
    u = a / step
    if mutant == 3:
        n = np.floor(u)
    elif mutant == 8:
        n = np.floor(u + 0.5)
    else:
        n = np.floor(u)
        frac = u - n
        up = (frac > 0.5) | ((frac == 0.5) & (np.mod(n, 2) == 1))
        n = n + up
    q = np.minimum(n * step, E4M3_MAX)
    # code of the magnitude q (exact on the e4m3 grid by construction)
    qe = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    sub = q < np.ldexp(1.0, -6)
    mant = np.where(sub, np.round(q / np.ldexp(1.0, -9)),
                    np.round((q / np.ldexp(1.0, qe.astype(np.int64)) - 1.0) * 8.0))
    expf = np.where(sub, 0, qe + 7)
    code = (expf.astype(np.int64) << 3) | mant.astype(np.int64)
    code = np.where(q == 0, 0, code)
    sign = np.where(np.signbit(r), 0x80, 0)
    code = (code | sign).astype(np.uint8)
    return np.where(np.isnan(r), np.uint8(0x7F), code).astype(np.uint8)


def layer_norm(x: np.ndarray, w: np.ndarray, b: np.ndarray, eps: float,
               mutant: int = 0) -> np.ndarray:
    """Rows of x normalised over the last axis (fp64), then scaled by w, shifted by b."""
    x = np.asarray(x, dtype=np.float64)
    mu = x.mean(axis=-1, keepdims=True)
    d = x - mu
    n = x.shape[-1]
    var = (d * d).sum(axis=-1, keepdims=True) / (n - 1 if mutant == 2 else n)
    y = d / np.sqrt(var + float(eps)) * np.asarray(w, np.float64)
    if mutant != 7:
        y = y + np.asarray(b, np.float64)
    return y


def rope(y: np.ndarray, cos: np.ndarray, sin: np.ndarray, rope_dim: int,
         mutant: int = 0) -> np.ndarray:
    """Rotates adjacent channel pairs (2i, 2i + 1), i < rope_dim / 2, of each row of y
    by the angle whose cosine and sine are cos[row, i], sin[row, i]."""
    y = np.array(y, dtype=np.float64, copy=True)
    D = y.shape[-1]
    off = D - rope_dim if mutant == 4 else 0
    a = y[:, off:off + rope_dim:2].copy()
    b = y[:, off + 1:off + rope_dim:2].copy()
    c = np.asarray(cos, np.float64)
    s = np.asarray(sin, np.float64)
    if mutant == 1:
        s = -s
    y[:, off:off + rope_dim:2] = a * c - b * s
    y[:, off + 1:off + rope_dim:2] = a * s + b * c
    return y


def quantize(y: np.ndarray, mutant: int = 0):
    """Per-row scale (fp32) and e4m3 codes of y / scale."""
    amax = np.abs(y).max(axis=-1)
    qmax = 127.0 if mutant == 5 else E4M3_MAX
    scale = np.where(amax > 0, amax / qmax, 1.0).astype(np.float32)
    codes = e4m3_encode(y / scale.astype(np.float64)[:, None], mutant=mutant)
    return codes, scale


def slots_of(positions, token_table, block_table, page_size, num_slots, mutant=0):
    """Physical slot of each token (int64) and the status bits of the tokens that are
    not stored (slot -1)."""
    pos = np.asarray(positions, np.int64)
    t2t = np.asarray(token_table, np.int64)
    tab = np.asarray(block_table, np.int64)
    ps = int(page_size)
    out = np.full(pos.shape, -1, np.int64)
    err = 0
    for i, (p, t) in enumerate(zip(pos, t2t)):
        if p < 0:
            err |= ERR_POSITION
            continue
        if t < 0 or t >= tab.shape[0]:
            err |= ERR_TABLE_ROW
            continue
        pg, off = (p % ps, p // ps) if mutant == 6 else (p // ps, p % ps)
        if pg >= tab.shape[1]:
            err |= ERR_TABLE_WIDTH
            continue
        page = int(tab[t, pg])
        if page < 0:
            err |= ERR_TABLE_ENTRY
            continue
        slot = page * ps + off
        if slot >= num_slots:
            err |= ERR_SLOT
            continue
        out[i] = slot
    return out, err


def key_prologue(k_bf16, ln_w, ln_b, eps, positions, cos_sin, rope_dim, token_table,
                 block_table, page_size, cache, scales, mutant=0):
    """The fused key path on every token, written into `cache` (uint8 [num_slots, D])
    and `scales` (float32 [num_slots]) in place; returns (status bits, the pre-
    quantization values y (fp64) of every token, the slots used).

    cos_sin: float32 [max_pos, rope_dim]: cos of the rope_dim / 2 pair angles, then
    their sines."""
    k = bf16_to_f64(k_bf16)
    T, D = k.shape
    pos = np.asarray(positions, np.int64)
    max_pos = cos_sin.shape[0]
    half = rope_dim // 2
    num_slots = cache.shape[0]
    # a position outside the cos/sin table is reported as such and never looked up
    bad_pos = (pos < 0) | (pos >= max_pos)
    slots, err = slots_of(np.where(bad_pos, -1, pos), token_table, block_table, page_size,
                          num_slots, mutant)
    pc = np.clip(pos, 0, max_pos - 1)
    y = layer_norm(k, ln_w, ln_b, eps, mutant)
    y = rope(y, cos_sin[pc, :half], cos_sin[pc, half:rope_dim], rope_dim, mutant)
    codes, sc = quantize(y, mutant)
    ok = slots >= 0
    cache[slots[ok]] = codes[ok]
    scales[slots[ok]] = sc[ok]
    return err, y, slots
