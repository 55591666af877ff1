"""CPU oracle for chunked linear attention with a decay -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
import this module.  The library never imports it and it never imports the
library: the two share no code.  Plain numpy in float64; every input is
promoted exactly before any arithmetic.

What it computes ("From 1% to 94% of cuBLAS, one kernel at a time", section
"What FLA builds on top of this"): a causal linear-attention layer with a
decay is a recurrence over the tokens t = 0 .. T-1 of each head with a state
matrix S of size K x V:

    S_t = exp(g_t) * S_{t-1} + k_t^T v_t        (S_{-1} = h0, zero by default)
    o_t = scale * q_t S_t

q_t, k_t are rows of K values, v_t and o_t rows of V values, g_t <= 0 the
token's log-decay (no decay: g = 0).  The pages leave the decay's form open
("a decay"); the plainest reading taken here is one scalar per token and
head, in log space.  Vector-valued gates (GLA proper) and the delta rule's
triangular solve are variants outside this reading.

The chunked form the pages describe (same section): cut the sequence into
chunks of BT tokens; h_c, the state before chunk c, passes between chunks,
and inside a chunk everything is a small causally masked dense attention.
With G_t the running sum of g over the chunk up to and including t:

    o_t     = scale * ( exp(G_t) q_t h_c + sum_{s <= t in the chunk} exp(G_t - G_s) (q_t . k_s) v_s )
    h_{c+1} = exp(G_last) h_c + sum_{s in the chunk} exp(G_last - G_s) k_s^T v_s

recurrent() is the definition written out token by token; chunked() takes
the chunked form's steps in that order; tests/test_la_oracle.py pins both
(the masked matrix form, the decayed parallel form, special cases, exact
integer inputs, and planted mistakes).

Shapes: q, k (BH, T, K); v (BH, T, V); g (BH, T) or None; h0 (BH, K, V) or
None; BH = batch x heads, each head independent.
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def recurrent(q, k, v, g=None, scale=1.0, h0=None):
    """The recurrence, one token at a time: returns (o (BH, T, V), S after
    the last token (BH, K, V))."""
    q, k, v, g, h0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(h0)
    BH, T, K = q.shape
    V = v.shape[2]
    S = np.zeros((BH, K, V)) if h0 is None else h0.copy()
    o = np.empty((BH, T, V))
    for t in range(T):
        if g is not None:
            S = S * np.exp(g[:, t])[:, None, None]
        S = S + k[:, t, :, None] * v[:, t, None, :]
        o[:, t] = float(scale) * np.einsum("bk,bkv->bv", q[:, t], S)
    return o, S


def chunked(q, k, v, g=None, scale=1.0, h0=None, BT=64):
    """The chunked form: returns (o (BH, T, V), h (BH, NT, K, V) -- the state
    before each chunk, NT = ceil(T / BT) -- and the state after the last
    chunk (BH, K, V)).  The last chunk may be shorter than BT."""
    q, k, v, g, h0 = _f64(q), _f64(k), _f64(v), _f64(g), _f64(h0)
    BH, T, K = q.shape
    V = v.shape[2]
    NT = -(-T // BT)
    h = np.empty((BH, NT, K, V))
    o = np.empty((BH, T, V))
    state = np.zeros((BH, K, V)) if h0 is None else h0.copy()
    for c in range(NT):
        t0, t1 = c * BT, min(T, (c + 1) * BT)
        n = t1 - t0
        h[:, c] = state
        qc, kc, vc = q[:, t0:t1], k[:, t0:t1], v[:, t0:t1]
        G = np.zeros((BH, n)) if g is None else np.cumsum(g[:, t0:t1], axis=1)
        # inside the chunk: causally masked, decayed attention
        A = np.einsum("btk,bsk->bts", qc, kc)
        causal = np.tril(np.ones((n, n), dtype=bool))
        decay = np.exp(G[:, :, None] - G[:, None, :])
        A = np.where(causal[None], A * decay, 0.0)
        intra = np.einsum("bts,bsv->btv", A, vc)
        # from the chunks before: the decayed state
        inter = np.exp(G)[:, :, None] * np.einsum("btk,bkv->btv", qc, state)
        o[:, t0:t1] = float(scale) * (inter + intra)
        # the state passed on
        w = np.exp(G[:, -1:] - G)
        state = (np.exp(G[:, -1])[:, None, None] * state
                 + np.einsum("bsk,bsv->bkv", kc * w[:, :, None], vc))
    return o, h, state


def magnitudes(q, k, v, g=None, scale=1.0, h0=None, BT=64):
    """Denominators of the accuracy metric: the chunked form on absolute
    values (every decay factor is positive), i.e. for each output and each
    chunk state the sum of the absolute values of the products it adds up.
    Returns (D_o (BH, T, V), D_h (BH, NT, K, V), D_state (BH, K, V))."""
    a = lambda x: None if x is None else np.abs(_f64(x))
    return chunked(a(q), a(k), a(v), g, abs(float(scale)), a(h0), BT)


def max_rel_err(x, ref, D) -> float:
    """max |x - ref| / (D + 1e-30); NaN in x where ref is finite counts as
    infinite."""
    x = np.asarray(x, dtype=np.float64)
    diff = np.abs(x - ref)
    diff = np.where(np.isnan(diff) & ~np.isnan(ref), np.inf, diff)
    if diff.size == 0:
        return 0.0
    return float(np.nanmax(diff / (D + 1e-30)))
