"""Pins of the sparse MLA decode-attention oracle, none of which goes through the oracle's own arithmetic: an
arbitrary-precision brute force on tiny inputs, closed forms (one row, identical rows, zero query, two rows),
invariances (selection order, padding), and planted mistakes that the pins must catch."""
import math
import os
import types

import numpy as np
import pytest

from oracle import mla_attention as mla

ORACLE_SRC = os.path.join(os.path.dirname(mla.__file__), "mla_attention.py")


def _bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns by round-to-nearest-even of the float32 value (input-side only)."""
    f = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    return ((f + 0x7FFF + ((f >> 16) & 1)) >> 16).astype(np.uint16)


def _mp_decode(q, rows, valid, scale, d_v):
    """Softmax attention in 40-digit arithmetic, one head and one row at a time."""
    import mpmath

    mpmath.mp.dps = 40
    out = np.zeros((q.shape[0], d_v))
    lse = np.zeros(q.shape[0])
    idx = [i for i in range(rows.shape[0]) if valid[i]]
    for h in range(q.shape[0]):
        s = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[h, d]) * mpmath.mpf(rows[i, d]) for d in range(q.shape[1]))
             for i in idx]
        z = mpmath.fsum(mpmath.exp(x) for x in s)
        lse[h] = float(mpmath.log(z))
        for d in range(d_v):
            out[h, d] = float(mpmath.fsum(mpmath.exp(s[j]) * mpmath.mpf(rows[i, d]) for j, i in enumerate(idx)) / z)
    return out, lse


def pin_mpmath_brute_force(m, seed=7, cases=25):
    pytest.importorskip("mpmath")
    rng = np.random.default_rng(seed)
    for c in range(cases):
        h, dqk, n = int(rng.integers(1, 4)), int(rng.integers(2, 9)), int(rng.integers(1, 8))
        d_v = int(rng.integers(1, dqk + 1))
        q = rng.normal(size=(h, dqk)) * rng.uniform(0.2, 3.0)
        rows = rng.normal(size=(n, dqk)) * rng.uniform(0.2, 3.0)
        valid = rng.random(n) < 0.8
        valid[rng.integers(0, n)] = True
        scale = float(rng.uniform(0.05, 2.0))
        out, lse = m.decode_one(q, rows, valid, scale, d_v)
        ref_out, ref_lse = _mp_decode(q, rows, valid, scale, d_v)
        assert np.allclose(out, ref_out, rtol=1e-11, atol=1e-12), c
        assert np.allclose(lse, ref_lse, rtol=1e-12, atol=1e-12), c


def pin_closed_forms(m, seed=8):
    rng = np.random.default_rng(seed)
    h, dqk, d_v = 4, 12, 7
    q = rng.normal(size=(h, dqk))
    r = rng.normal(size=(1, dqk))
    # one valid row among padding: out is that row's value part, lse its score
    rows = np.concatenate([rng.normal(size=(2, dqk)), r, rng.normal(size=(3, dqk))])
    valid = np.array([False, False, True, False, False, False])
    out, lse = m.decode_one(q, rows, valid, 0.3, d_v)
    assert np.array_equal(out, np.repeat(r[:, :d_v], h, axis=0))
    assert np.allclose(lse, 0.3 * (q @ r[0]), rtol=0, atol=1e-14)
    # n identical rows: the same value, lse + log n
    rows = np.repeat(r, 5, axis=0)
    out, lse = m.decode_one(q, rows, np.ones(5, bool), 0.3, d_v)
    assert np.allclose(out, np.repeat(r[:, :d_v], h, axis=0), rtol=0, atol=1e-14)
    assert np.allclose(lse, 0.3 * (q @ r[0]) + math.log(5), rtol=0, atol=1e-13)
    # zero query: the plain mean of the value parts, lse = log n
    rows = rng.normal(size=(6, dqk))
    out, lse = m.decode_one(np.zeros((h, dqk)), rows, np.ones(6, bool), 0.3, d_v)
    assert np.allclose(out, np.repeat(rows[:, :d_v].mean(axis=0, keepdims=True), h, axis=0), rtol=0, atol=1e-14)
    assert np.allclose(lse, math.log(6), rtol=0, atol=1e-14)
    # two rows: weights are the logistic function of the score difference
    rows = rng.normal(size=(2, dqk))
    out, lse = m.decode_one(q, rows, np.ones(2, bool), 0.7, d_v)
    s = 0.7 * (q @ rows.T)
    w = 1.0 / (1.0 + np.exp(s[:, 1] - s[:, 0]))
    assert np.allclose(out, w[:, None] * rows[0, :d_v] + (1 - w[:, None]) * rows[1, :d_v], rtol=0, atol=1e-13)
    # nothing valid: zero output, lse -inf
    out, lse = m.decode_one(q, rows, np.zeros(2, bool), 0.7, d_v)
    assert not out.any() and np.all(np.isneginf(lse))


def pin_invariances(m, seed=9):
    rng = np.random.default_rng(seed)
    h, dqk, n = 3, 10, 9
    q = rng.normal(size=(h, dqk))
    rows = rng.normal(size=(n, dqk))
    valid = rng.random(n) < 0.7
    valid[0] = True
    out, lse = m.decode_one(q, rows, valid, 0.5, 6)
    perm = rng.permutation(n)
    out_p, lse_p = m.decode_one(q, rows[perm], valid[perm], 0.5, 6)
    assert np.allclose(out, out_p, rtol=0, atol=1e-14) and np.allclose(lse, lse_p, rtol=0, atol=1e-14)
    out_c, lse_c = m.decode_one(q, rows[valid], np.ones(int(valid.sum()), bool), 0.5, 6)
    assert np.allclose(out, out_c, rtol=0, atol=1e-14) and np.allclose(lse, lse_c, rtol=0, atol=1e-14)
    # large scores: no overflow, the largest-score row dominates
    big = np.zeros((1, dqk))
    big[0, 0] = 1.0
    rows2 = np.zeros((3, dqk))
    rows2[:, 0] = [1000.0, 990.0, 0.0]
    rows2[:, 1] = [1.0, 2.0, 3.0]
    out, lse = m.decode_one(big, rows2, np.ones(3, bool), 1.0, 2)
    assert abs(out[0, 1] - (1.0 + 2.0 * math.exp(-10)) / (1 + math.exp(-10) + math.exp(-1000))) < 1e-12
    assert abs(lse[0] - (1000.0 + math.log1p(math.exp(-10)))) < 1e-9


def pin_bf16_decoding(m):
    # bf16 bit patterns of exactly representable values decode exactly, batch helper agrees with decode_one
    vals = np.array([0.0, 1.0, -2.0, 0.5, 3.140625, -1e-3, 65280.0])
    bits = _bf16(vals)
    dec = m.bf16_bits_to_f64(bits)
    assert dec[0] == 0.0 and dec[1] == 1.0 and dec[2] == -2.0 and dec[3] == 0.5 and dec[4] == 3.140625
    assert dec[6] == 65280.0 and abs(dec[5] + 1e-3) < 1e-5
    rng = np.random.default_rng(10)
    qb = _bf16(rng.normal(size=(2, 3, 8)))
    rb = _bf16(rng.normal(size=(2, 5, 8)))
    valid = rng.random((2, 5)) < 0.8
    valid[:, 0] = True
    out, lse = m.decode_batch(qb, rb, valid, 0.4, 6)
    for b in range(2):
        o, l = m.decode_one(m.bf16_bits_to_f64(qb[b]), m.bf16_bits_to_f64(rb[b]), valid[b], 0.4, 6)
        assert np.array_equal(out[b], o) and np.array_equal(lse[b], l)


PINS = [pin_mpmath_brute_force, pin_closed_forms, pin_invariances, pin_bf16_decoding]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_attention_oracle_pin(pin):
    pin(mla)


# (name, original text, replacement): mistakes a careful reader could make in the oracle
MUTANTS = [
    ("softmax_over_heads", "m = s.max(axis=1, keepdims=True)", "m = s.max(axis=0, keepdims=True)"),
    ("scale_after_exp", "s = (q @ r.T) * sm_scale", "s = (q @ r.T)"),
    ("value_is_rope_part", "out = (p @ r[:, :d_v]) / l[:, None]", "out = (p @ r[:, -d_v:]) / l[:, None]"),
    ("padding_kept", "r = rows[np.asarray(valid, dtype=bool)]", "r = rows"),
    ("lse_without_max", "lse = m[:, 0] + np.log(l)", "lse = np.log(l)"),
    ("unnormalised", "out = (p @ r[:, :d_v]) / l[:, None]", "out = (p @ r[:, :d_v])"),
    ("bf16_low_half", "return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)",
     "return (b.astype(np.uint32) << 15).view(np.float32).astype(np.float64)"),
]


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_attention_pins_catch_planted_mistake(name, old, new):
    pytest.importorskip("mpmath")
    src = open(ORACLE_SRC).read()
    assert src.count(old) == 1, name
    mod = types.ModuleType(f"mla_mutant_{name}")
    exec(compile(src.replace(old, new), f"<{name}>", "exec"), mod.__dict__)
    caught = []
    for pin in PINS:
        try:
            pin(mod)
        except (AssertionError, FloatingPointError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
