"""CPU ORACLE for the sparse MLA decode attention that consumes the resolver's slot list -- TEST INFRASTRUCTURE
ONLY (the tests, the smoke check and the CPU-baseline leg of the benchmark may call it; the library never does).

What it computes. The resolver exists so that a sparse-attention kernel can read the selected KV rows from the
GPU hot buffer instead of the full history, with model outputs unchanged ("HiSparse" paper, Abstract; the
"Hybrid HiSparse" knowledge card builds on Sparse MLA). For one request and one layer of a multi-head latent
attention decode step in its absorbed form, each selected row holds D = 576 values: the 512-dimensional
compressed latent followed by the 64-dimensional rotary key. Every query head h has a D-dimensional query q[h]
(latent-absorbed part and rotary part). With the selected rows r_0 .. r_{n-1} (padding entries excluded):

    s[h][i]  = sm_scale * sum_d q[h][d] * r_i[d]
    lse[h]   = log sum_i exp(s[h][i])
    out[h]   = sum_i exp(s[h][i] - lse[h]) * r_i[0 : d_v]          (d_v = 512: the latent is also the value)

With no valid row, out is zero and lse is -inf. Everything is evaluated in float64 from the bf16 inputs, with the
maximum subtracted before exponentiation; numpy matrix products and sums are the only library steps.
"""
from __future__ import annotations

import numpy as np

D_QK = 576
D_V = 512


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16, any shape) to float64: the upper half of the float32 with those bits."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_one(q: np.ndarray, rows: np.ndarray, valid: np.ndarray, sm_scale: float, d_v: int = D_V):
    """One request: q float64 [H][D]; rows float64 [n][D] in selection order; valid bool [n].
    Returns (out float64 [H][d_v], lse float64 [H])."""
    h = q.shape[0]
    r = rows[np.asarray(valid, dtype=bool)]
    if r.shape[0] == 0:
        return np.zeros((h, d_v)), np.full(h, -np.inf)
    s = (q @ r.T) * sm_scale
    m = s.max(axis=1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(axis=1)
    out = (p @ r[:, :d_v]) / l[:, None]
    lse = m[:, 0] + np.log(l)
    return out, lse


def decode_batch(q_bits: np.ndarray, rows_bits: np.ndarray, valid: np.ndarray, sm_scale: float, d_v: int = D_V):
    """A batch: q_bits uint16 [B][H][D]; rows_bits uint16 [B][n][D] (the rows each request's selection names, in
    selection order; content of invalid entries is ignored); valid bool [B][n]. Returns (out [B][H][d_v],
    lse [B][H]) in float64."""
    bsz = q_bits.shape[0]
    outs, lses = [], []
    for b in range(bsz):
        o, l = decode_one(bf16_bits_to_f64(q_bits[b]), bf16_bits_to_f64(rows_bits[b]), valid[b], sm_scale, d_v)
        outs.append(o)
        lses.append(l)
    return np.stack(outs), np.stack(lses)
