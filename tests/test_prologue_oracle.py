"""Pins of the key-path prologue oracle (oracle/prologue.py) to things other than
itself (no GPU needed):

* hand-worked tokens under tests/golden/ (LayerNorm, RoPE, e4m3 codes, slots, status);
* the e4m3 format: closed-form values of its codes, round trips, ties to even,
  saturation, and a cross-check against torch's float8_e4m3fn conversion;
* LayerNorm against torch.nn.functional.layer_norm (fp64) and closed forms;
* RoPE: the identity angle, a quarter turn, pair norms, and inner products that
  depend only on the difference of the two positions;
* the quantization error bound, the slot rule, and invariants on the workload;
* pin strength: each deliberately wrong oracle variant fails at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

import workloads as W
from oracle import prologue as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prologue_hand_worked.json")


def _bf16_bits(values):
    """Bits of values that bfloat16 holds exactly (the golden inputs)."""
    u = np.asarray(values, np.float32).view(np.uint32)
    assert np.all(u & 0xFFFF == 0), "golden input not exact in bfloat16"
    return (u >> 16).astype(np.uint16)


def _golden_table(spec, rope_dim):
    t = np.tile(np.asarray(spec["default"], np.float32), (spec["rows"], 1))
    for r, v in spec["set"].items():
        t[int(r)] = np.asarray(v, np.float32)
    assert t.shape[1] == rope_dim
    return t


# ---------------------------------------------------------------- pin functions
# Each returns None when the oracle variant passes and a message when it fails.

def pin_golden(mutant=0):
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        D = c["dim"]
        cache = np.full((c["num_slots"], D), 0xAA, np.uint8)
        scales = np.full(c["num_slots"], -7.0, np.float32)
        err, _, _ = P.key_prologue(
            _bf16_bits(c["k"]), np.asarray(c["ln_w"], np.float32), np.asarray(c["ln_b"], np.float32),
            c["eps"], np.asarray(c["positions"], np.int32), _golden_table(c["cos_sin"], c["rope_dim"]),
            c["rope_dim"], np.asarray(c["token_table"], np.int32),
            np.asarray(c["block_table"], np.int32), c["page_size"], cache, scales, mutant=mutant)
        if err != c["expect_status"]:
            return f"{c['name']}: status {err} != {c['expect_status']}"
        for slot, e in c["expect"].items():
            s = int(slot)
            if list(cache[s]) != e["codes"]:
                return f"{c['name']}: codes {list(cache[s])} != {e['codes']}"
            want = eval(e["scale"], {"sqrt": math.sqrt})  # noqa: S307 (a fixed fixture)
            if abs(float(scales[s]) - want) > 1e-6 * want:
                return f"{c['name']}: scale {scales[s]} != {want}"
        touched = {int(x) for x in c["expect"]}
        for s in range(c["num_slots"]):
            if s not in touched and (np.any(cache[s] != 0xAA) or scales[s] != -7.0):
                return f"{c['name']}: slot {s} written"
    return None


def pin_e4m3_format(mutant=0):
    """Closed forms of the e4m3 ("fn") codes, their round trip through the encoder,
    ties to even and saturation."""
    codes = np.arange(256, dtype=np.uint8)
    v = P.e4m3_value(codes)
    exp = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0,
           0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x7E: 448.0, 0x76: 224.0, 0xB8: -1.0, 0xFE: -448.0}
    for c, x in exp.items():
        if v[c] != x:
            return f"value of code {c:#x}: {v[c]} != {x}"
    if not (np.isnan(v[0x7F]) and np.isnan(v[0xFF])):
        return "S.1111.111 must be NaN"
    pos = v[:0x7F]
    if not np.all(np.diff(pos) > 0):
        return "positive codes not increasing"
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    if not np.array_equal(P.e4m3_encode(P.e4m3_value(finite), mutant=mutant), finite):
        return "encode(value(c)) != c"
    ties = {1.0625: 0x38, 1.1875: 0x3A, 3 * 2.0 ** -10: 0x02, 2.0 ** -10: 0x00,
            208.0 + 8.0: 0x76, -1.0625: 0xB8, 1.0625 + 1e-9: 0x39}
    for x, c in ties.items():
        got = int(P.e4m3_encode(np.array([x]), mutant=mutant)[0])
        if got != c:
            return f"encode({x!r}) = {got:#x}, want {c:#x}"
    sat = P.e4m3_encode(np.array([448.0, 449.0, 464.0, 479.9, 1e6, -1e30]), mutant=mutant)
    if list(sat) != [0x7E] * 5 + [0xFE]:
        return f"saturation {list(map(hex, sat))}"
    return None


def pin_e4m3_vs_torch(mutant=0):
    """The encoder against torch's float32 -> float8_e4m3fn conversion (round to
    nearest even) on every midpoint between neighbouring codes, their float32
    neighbours and random values inside the finite range."""
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    v = P.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (v[:-1] + v[1:]) / 2
    mids32 = mids.astype(np.float32)
    near = np.concatenate([np.nextafter(mids32, np.float32(0)), mids32,
                           np.nextafter(mids32, np.float32(1e9))])
    rng = np.random.default_rng(5)
    rnd = (rng.standard_normal(20000) * np.exp(rng.uniform(-12, 6, 20000))).astype(np.float32)
    x = np.concatenate([near, -near, rnd, v.astype(np.float32), -v.astype(np.float32)])
    x = x[np.abs(x) <= 448.0]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = P.e4m3_encode(x.astype(np.float64), mutant=mutant)
    # +0 / -0 both denote zero
    same = (got == ref) | ((got & 0x7F) == 0) & ((ref & 0x7F) == 0)
    if not np.all(same):
        i = int(np.argmin(same))
        return f"encode({x[i]!r}) = {got[i]:#x}, torch {ref[i]:#x}"
    return None


def pin_layer_norm(mutant=0):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 128)) * 3 + 1
    w = rng.standard_normal(128)
    b = rng.standard_normal(128)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (128,), torch.from_numpy(w),
                                         torch.from_numpy(b), eps=1e-6).numpy()
    y = P.layer_norm(x, w, b, 1e-6, mutant=mutant)
    if np.max(np.abs(y - ref)) > 1e-9:
        return f"layer_norm differs from torch by {np.max(np.abs(y - ref))}"
    # closed forms: a constant row gives the bias; +-a alternating gives +-1 (eps 0)
    yc = P.layer_norm(np.full((1, 8), 5.0), np.ones(8) * 2, np.arange(8.0), 1e-6, mutant=mutant)
    if not np.allclose(yc, np.arange(8.0), atol=0, rtol=0):
        return "constant row must give the bias"
    ya = P.layer_norm(np.array([[3.0, -3.0] * 4]), np.ones(8), np.zeros(8), 0.0, mutant=mutant)
    if not np.allclose(ya, [[1.0, -1.0] * 4], rtol=0, atol=1e-15):
        return f"alternating row: {ya}"
    return None


def pin_rope(mutant=0):
    rng = np.random.default_rng(9)
    D, R, T = 128, 64, 32
    y = rng.standard_normal((T, D))
    # identity angle
    out = P.rope(y, np.ones((T, R // 2)), np.zeros((T, R // 2)), R, mutant=mutant)
    if not np.array_equal(out, y):
        return "cos 1, sin 0 must be the identity"
    # quarter turn: (a, b) -> (-b, a) on the first R channels, the rest unchanged
    out = P.rope(y, np.zeros((T, R // 2)), np.ones((T, R // 2)), R, mutant=mutant)
    want = y.copy()
    want[:, 0:R:2] = -y[:, 1:R:2]
    want[:, 1:R:2] = y[:, 0:R:2]
    if not np.allclose(out, want, rtol=0, atol=0):
        return "quarter turn"
    # angles p * theta_i: pair norms kept; <q(p1), k(p2)> depends on p1 - p2 only
    theta = 10000.0 ** (-2.0 * np.arange(R // 2) / R)
    def at(v, p):
        a = p * theta
        return P.rope(v[None, :], np.cos(a)[None, :], np.sin(a)[None, :], R, mutant=mutant)[0]
    q, k = y[0], y[1]
    n0 = q[0:R:2] ** 2 + q[1:R:2] ** 2
    q5 = at(q, 5.0)
    if not np.allclose(q5[0:R:2] ** 2 + q5[1:R:2] ** 2, n0, rtol=1e-12, atol=0):
        return "pair norms"
    d1 = at(q, 17.0) @ at(k, 4.0)
    d2 = at(q, 1013.0) @ at(k, 1000.0)
    if abs(d1 - d2) > 1e-9 * (1 + abs(d1)):
        return f"relative position: {d1} != {d2}"
    return None


def pin_quantization_bound(mutant=0):
    """Each dequantized value lies within half an e4m3 step of y (at y's binade, or
    2^-10 * scale below the normal range), and the amax channel codes +-448."""
    rng = np.random.default_rng(11)
    y = rng.standard_normal((200, 128)) * np.exp(rng.uniform(-3, 3, (200, 1)))
    codes, scale = P.quantize(y, mutant=mutant)
    r = y / scale.astype(np.float64)[:, None]
    deq = P.e4m3_value(codes)
    a = np.abs(r)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -6)))
    half = np.ldexp(1.0, (e - 4).astype(np.int64))
    if np.any(np.abs(deq - r) > half * (1 + 1e-12)):
        return "error above half a step"
    top = np.argmax(np.abs(y), axis=1)
    if not np.all(np.abs(deq[np.arange(200), top]) == 448.0):
        return "amax channel must code +-448"
    return None


def pin_slots(mutant=0):
    tab = np.array([[4, 0, 2], [1, 3, 5]], np.int32)
    pos = np.array([0, 5, 11, 3, 7], np.int64)
    t2t = np.array([0, 0, 0, 1, 1], np.int64)
    slots, err = P.slots_of(pos, t2t, tab, 4, 24, mutant=mutant)
    want = [4 * 4 + 0, 0 * 4 + 1, 2 * 4 + 3, 1 * 4 + 3, 3 * 4 + 3]
    if err != 0 or list(slots) != want:
        return f"slots {list(slots)} != {want} (err {err})"
    return None


def pin_workload(mutant=0):
    """On the seeded workload every token is stored, at distinct slots given by the
    slot rule; nothing else is written; dequantized codes approximate y."""
    b = W.key_prologue(reqs=((0, 300), (4000, 70), (100000, 3)))
    cache = np.full((b.num_slots, b.dim), 0xAA, np.uint8)
    scales = np.full(b.num_slots, -7.0, np.float32)
    err, y, slots = P.key_prologue(b.k_bf16, b.ln_w, b.ln_b, b.eps, b.positions, b.cos_sin,
                                   b.rope_dim, b.token_table, b.block_table, b.page_size,
                                   cache, scales, mutant=mutant)
    if err != 0:
        return f"status {err}"
    tab = b.block_table.astype(np.int64)
    p = b.positions.astype(np.int64)
    want = tab[b.token_table, p // b.page_size] * b.page_size + p % b.page_size
    if not np.array_equal(slots, want) or len(np.unique(slots)) != b.tokens:
        return "slots"
    written = np.zeros(b.num_slots, bool)
    written[slots] = True
    if np.any(scales[~written] != -7.0) or np.any(cache[~written] != 0xAA):
        return "a slot outside the tokens' was written"
    deq = P.e4m3_value(cache[slots]) * scales[slots].astype(np.float64)[:, None]
    rel = np.abs(deq - y) / (np.abs(y).max(axis=1, keepdims=True))
    if rel.max() > 1.0 / 16 + 1e-6:
        return f"dequantized error {rel.max()}"
    return None


PINS = [pin_golden, pin_e4m3_format, pin_e4m3_vs_torch, pin_layer_norm, pin_rope,
        pin_quantization_bound, pin_slots, pin_workload]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    msg = pin()
    assert msg is None, msg


@pytest.mark.parametrize("mutant", sorted(P.MUTANTS), ids=lambda m: P.MUTANTS[m])
def test_pin_strength(mutant):
    """Each deliberately wrong variant of the oracle fails at least one pin."""
    failures = []
    for p in PINS:
        try:
            if p(mutant=mutant) is not None:
                failures.append(p.__name__)
        except Exception as ex:  # a crash also counts as caught
            failures.append(f"{p.__name__}: {ex!r}")
    assert failures, f"mutant {mutant} ({P.MUTANTS[mutant]}) passed every pin"
