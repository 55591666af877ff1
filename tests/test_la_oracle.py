"""Pins of the linear-attention oracle (oracle/linattn.py) to what the pages
and the mathematics fix, independently of the oracle's own loops:

  - the masked matrix form: without decay the recurrence sums, for every
    token t, (q_t . k_s) v_s over s <= t -- i.e. tril(Q K^T) V, written here
    as numpy matrix products;
  - the decayed parallel form: with G the running sum of g over the whole
    sequence, o = ((Q K^T) * tril(exp(G_t - G_s))) V + exp(G_t) Q h0;
  - the chunked form equals the recurrence for any chunk length, ragged
    last chunks, an initial state, and each chunk's starting state equals
    the recurrence's state after the token before the chunk;
  - closed forms: one token; decay so strong that nothing is remembered;
  - exactness: small integer inputs without decay give the exact integer
    result (int64 matrix products);
  - the magnitudes bound the outputs.
Mutation tests plant mistakes in copies of the oracle's source and check that
these pins reject every one.
"""
import os
import types

import numpy as np
import pytest

from oracle import linattn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def inputs(BH=3, T=37, K=8, V=8, seed=0, decay=True, h0=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((BH, T, K)).astype(np.float32)
    k = rng.standard_normal((BH, T, K)).astype(np.float32)
    v = rng.standard_normal((BH, T, V)).astype(np.float32)
    g = (-rng.uniform(0.0, 0.5, size=(BH, T))).astype(np.float32) if decay else None
    s0 = rng.standard_normal((BH, K, V)).astype(np.float32) if h0 else None
    return q, k, v, g, s0


def close(a, b, rtol=1e-11, atol=1e-11):
    return np.allclose(a, b, rtol=rtol, atol=atol)


# ------------------------------------------------------------ the pin checks

def pin_masked_matrix_form(la):
    q, k, v, _, s0 = inputs(decay=False)
    o, _ = la.recurrent(q, k, v, None, 0.5, s0)
    Q, Kx, Vx, H = (x.astype(np.float64) for x in (q, k, v, s0))
    want = 0.5 * (np.tril(Q @ Kx.transpose(0, 2, 1)) @ Vx + Q @ H)
    assert close(o, want)


def pin_decayed_parallel_form(la):
    q, k, v, g, s0 = inputs(seed=1)
    o, S = la.recurrent(q, k, v, g, 0.25, s0)
    Q, Kx, Vx, H = (x.astype(np.float64) for x in (q, k, v, s0))
    G = np.cumsum(g.astype(np.float64), axis=1)
    T = q.shape[1]
    M = np.where(np.tril(np.ones((T, T), dtype=bool))[None],
                 np.exp(G[:, :, None] - G[:, None, :]), 0.0)
    want = 0.25 * ((Q @ Kx.transpose(0, 2, 1) * M) @ Vx + np.exp(G)[:, :, None] * (Q @ H))
    assert close(o, want)
    # final state: exp(G_T) h0 + sum_s exp(G_T - G_s) k_s^T v_s
    w = np.exp(G[:, -1:] - G)
    S_want = np.exp(G[:, -1])[:, None, None] * H + np.einsum("bsk,bsv->bkv", Kx * w[:, :, None], Vx)
    assert close(S, S_want)


def pin_chunked_equals_recurrent(la):
    for (T, BT, decay, h0) in [(1, 64, True, True), (63, 64, True, False), (64, 64, False, True),
                               (65, 64, True, True), (200, 16, True, True), (37, 5, False, False),
                               (20, 1, True, True)]:
        q, k, v, g, s0 = inputs(T=T, seed=T + BT, decay=decay, h0=h0)
        o_r, S_r = la.recurrent(q, k, v, g, 0.7, s0)
        o_c, h, S_c = la.chunked(q, k, v, g, 0.7, s0, BT)
        assert close(o_c, o_r), (T, BT)
        assert close(S_c, S_r), (T, BT)
        assert h.shape[1] == -(-T // BT)
        for c in range(h.shape[1]):
            if c == 0:
                want = np.zeros_like(S_r) if s0 is None else s0.astype(np.float64)
            else:
                gp = None if g is None else g[:, :c * BT]
                _, want = la.recurrent(q[:, :c * BT], k[:, :c * BT], v[:, :c * BT], gp, 0.7, s0)
            assert close(h[:, c], want), (T, BT, c)


def pin_closed_forms(la):
    # one token: o = scale (exp(g) q h0 + (q . k) v)
    q, k, v, g, s0 = inputs(T=1, seed=5)
    o, _ = la.recurrent(q, k, v, g, 2.0, s0)
    Q, Kx, Vx, H = (x.astype(np.float64)[:, 0] if x.ndim == 3 and x.shape[1] == 1 else
                    x.astype(np.float64) for x in (q, k, v, s0))
    e = np.exp(g.astype(np.float64)[:, 0])
    want = 2.0 * (e[:, None] * np.einsum("bk,bkv->bv", Q, H)
                  + np.einsum("bk,bk->b", Q, Kx)[:, None] * Vx)
    assert close(o[:, 0], want)
    # a decay that forgets everything: o_t = scale (q_t . k_t) v_t
    q, k, v, _, s0 = inputs(T=30, seed=6)
    g = np.full(q.shape[:2], -1.0e4, dtype=np.float32)
    for o in (la.recurrent(q, k, v, g, 1.5, s0)[0], la.chunked(q, k, v, g, 1.5, s0, 8)[0]):
        want = 1.5 * np.einsum("btk,btk->bt", q.astype(np.float64),
                               k.astype(np.float64))[:, :, None] * v.astype(np.float64)
        assert close(o, want)


def pin_exact_integers(la):
    rng = np.random.default_rng(9)
    BH, T, K, V = 2, 50, 6, 7
    q = rng.integers(-3, 4, size=(BH, T, K))
    k = rng.integers(-3, 4, size=(BH, T, K))
    v = rng.integers(-3, 4, size=(BH, T, V))
    s0 = rng.integers(-3, 4, size=(BH, K, V))
    want = np.tril(q @ k.transpose(0, 2, 1)) @ v + q @ s0  # int64, exact
    o_r, _ = la.recurrent(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                          None, 1.0, s0.astype(np.float32))
    o_c, _, _ = la.chunked(q.astype(np.float32), k.astype(np.float32), v.astype(np.float32),
                           None, 1.0, s0.astype(np.float32), 16)
    assert np.array_equal(o_r, want.astype(np.float64))
    assert np.array_equal(o_c, want.astype(np.float64))


def pin_magnitudes(la):
    q, k, v, g, s0 = inputs(T=70, seed=12)
    o, h, S = la.chunked(q, k, v, g, -0.5, s0, 16)
    Do, Dh, DS = la.magnitudes(q, k, v, g, -0.5, s0, 16)
    assert np.all(np.abs(o) <= Do * (1 + 1e-12)) and np.all(np.abs(h) <= Dh * (1 + 1e-12))
    assert np.all(np.abs(S) <= DS * (1 + 1e-12))
    # non-negative inputs and a positive scale: the magnitude is the value
    qa, ka, va, sa = (np.abs(x) for x in (q, k, v, s0))
    assert close(la.magnitudes(qa, ka, va, g, 0.5, sa, 16)[0], la.chunked(qa, ka, va, g, 0.5, sa, 16)[0])


PINS = [pin_masked_matrix_form, pin_decayed_parallel_form, pin_chunked_equals_recurrent,
        pin_closed_forms, pin_exact_integers, pin_magnitudes]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(linattn)


def test_error_metric():
    ref = np.array([1.0, 2.0, np.nan])
    assert linattn.max_rel_err(np.array([1.0, 2.5, np.nan]), ref, np.array([1.0, 1.0, 1.0])) == 0.5
    assert linattn.max_rel_err(np.array([np.nan]), np.array([1.0]), np.array([1.0])) == np.inf


# ----------------------------------------------------------- planted mistakes

MUTATIONS = {
    "future tokens in the chunk's mask": [
        ("causal = np.tril(np.ones((n, n), dtype=bool))", "causal = np.ones((n, n), dtype=bool)")],
    "own token left out of the chunk's mask": [
        ("causal = np.tril(np.ones((n, n), dtype=bool))",
         "causal = np.tril(np.ones((n, n), dtype=bool), -1)")],
    "decay inside the chunk with the wrong sign": [
        ("decay = np.exp(G[:, :, None] - G[:, None, :])",
         "decay = np.exp(G[:, None, :] - G[:, :, None])")],
    "state passed on without its decay": [
        ("state = (np.exp(G[:, -1])[:, None, None] * state", "state = (state")],
    "earlier chunks' term without its decay": [
        ("inter = np.exp(G)[:, :, None] * np.einsum", "inter = np.einsum")],
    "token added before the decay in the recurrence": [
        ("        if g is not None:\n            S = S * np.exp(g[:, t])[:, None, None]\n"
         "        S = S + k[:, t, :, None] * v[:, t, None, :]\n",
         "        S = S + k[:, t, :, None] * v[:, t, None, :]\n        if g is not None:\n"
         "            S = S * np.exp(g[:, t])[:, None, None]\n")],
    "k and v swapped in the state": [
        ("S = S + k[:, t, :, None] * v[:, t, None, :]",
         "S = S + v[:, t, :, None] * k[:, t, None, :]")],
    "scale left off the earlier chunks' term": [
        ("o[:, t0:t1] = float(scale) * (inter + intra)",
         "o[:, t0:t1] = inter + float(scale) * intra")],
    "state update weights with the wrong sign": [
        ("w = np.exp(G[:, -1:] - G)", "w = np.exp(G - G[:, -1:])")],
    "chunk state recorded after the update": [
        ("        h[:, c] = state\n", ""),
        ("vc))\n", "vc))\n        h[:, c] = state\n")],
}


def mutated(edits):
    src = open(os.path.join(ROOT, "oracle", "linattn.py")).read()
    for old, new in edits:
        assert src.count(old) == 1, old
        src = src.replace(old, new)
    mod = types.ModuleType("linattn_mutated")
    exec(compile(src, "linattn_mutated", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_reject_planted_mistake(name):
    mod = mutated(MUTATIONS[name])
    failed = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(mod)
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught: {name}"
