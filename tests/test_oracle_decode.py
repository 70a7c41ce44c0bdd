"""Pins of the oracle's single-token decode step (Eqs. 1-4 with a one-token chunk).

The decode step is checked against two independent formulations of the same
recurrence: the oracle's 64-token chunkwise prefill (a prefill of T + 64 tokens
equals a prefill of T tokens followed by 64 decode steps) and the token-level
brute force of tests/brute.py; plus closed forms for complete forgetting and
for beta = 0.
"""
import numpy as np
import pytest

import gdn_synth
import oracle
from brute import brute_prefill


def token_gates(g):
    """Per-token log2 retention a_t = g_t - g_(t-1) inside each chunk (g_(-1) = 0 at chunk starts)."""
    g = np.asarray(g, dtype=np.float64)
    a = g.copy()
    a[:, 1:] -= g[:, :-1]
    a[:, ::64] = g[:, ::64]
    return a


def decode_tokens(x, t0, t1, S):
    a = token_gates(x.g)
    outs = []
    for t in range(t0, t1):
        r = oracle.decode(x.q[:, t], x.k[:, t], x.v[:, t], x.beta[:, t], a[:, t], S)
        S = r["s"]
        outs.append(r["o"])
    return np.stack(outs, axis=1), S


def rel(a, b):
    return np.linalg.norm(a - b) / np.linalg.norm(b)


@pytest.mark.parametrize("with_h0", [False, True])
def test_decode_continues_the_chunkwise_prefill(with_h0):
    x = gdn_synth.make_inputs(2, 192, 1, 2, d=32, dv=32, dtype="f32", seed=51, mask="ones", with_h0=with_h0)
    h0 = x.h0 if with_h0 else None
    head = oracle.prefill(x.q[:, :128], x.k[:, :128], x.v[:, :128], x.beta[:, :128], x.g[:, :128], h0=h0,
                          solver=oracle.SOLVER_EXACT)
    o_dec, s_dec = decode_tokens(x, 128, 192, head["s_final"])
    full = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, h0=h0, solver=oracle.SOLVER_EXACT)
    assert rel(o_dec, full["o"][:, 128:]) < 1e-12
    assert rel(s_dec, full["s_final"]) < 1e-12


def test_decode_matches_token_brute_force():
    x = gdn_synth.make_inputs(1, 64, 2, 4, d=16, dv=24, dtype="f32", seed=52, mask="ones", with_h0=True)
    o_dec, s_dec = decode_tokens(x, 0, 64, x.h0)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, h0=x.h0)
    assert rel(o_dec, ref["o"]) < 1e-12
    assert rel(s_dec, ref["s_final"]) < 1e-12


def test_decode_closed_forms():
    rng = np.random.default_rng(53)
    B, Nq, Nv, d, dv = 1, 1, 2, 8, 5
    q, k = rng.standard_normal((B, Nq, d)), rng.standard_normal((B, Nq, d))
    v, beta = rng.standard_normal((B, Nv, dv)), rng.uniform(0.1, 0.9, (B, Nv))
    S = rng.standard_normal((B, Nv, d, dv))
    # complete forgetting (2^a = 0): the state becomes the rank-one write beta k v^T
    r = oracle.decode(q, k, v, beta, np.full((B, Nv), -2000.0), S)
    for h in range(Nv):
        np.testing.assert_allclose(r["s"][0, h], beta[0, h] * np.outer(k[0, 0], v[0, h]), rtol=1e-14)
        np.testing.assert_allclose(r["o"][0, h], (q[0, 0] @ k[0, 0]) * beta[0, h] * v[0, h] / np.sqrt(d),
                                   rtol=1e-12)
    # beta = 0: the state only decays and the output reads the decayed state
    a = np.full((B, Nv), -0.75)
    r = oracle.decode(q, k, v, np.zeros((B, Nv)), a, S)
    np.testing.assert_allclose(r["s"], 2 ** -0.75 * S, rtol=1e-14)
    for h in range(Nv):
        np.testing.assert_allclose(r["o"][0, h], 2 ** -0.75 * (q[0, 0] @ S[0, h]) / np.sqrt(d), rtol=1e-12)
    # beta = 1, a = 0, unit k: the value stored along k is replaced exactly by v (delta rule)
    kn = k / np.linalg.norm(k)
    r = oracle.decode(q, kn, v, np.ones((B, Nv)), np.zeros((B, Nv)), S)
    for h in range(Nv):
        np.testing.assert_allclose(kn[0, 0] @ r["s"][0, h], v[0, h], rtol=1e-12, atol=1e-12)
