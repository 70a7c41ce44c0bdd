"""Token-by-token gated delta recurrence in NumPy (fp64): an independent pin of the oracle.

Selected chunk (every chunk on the dense path) -- the plain gated delta rule:
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,   o_t = q_t^T S_t / sqrt(d),
with alpha_t = 2^(g_t - g_{t-1}) and g_{-1} = 0 at each chunk start (g is the
inclusive within-chunk cumulative log2 retention).

Unselected chunk (event-sparse semantics, SparseGDN Secs. 2.6-2.7): the
persistent state only decays, S_t = alpha_t S_{t-1}, while a chunk-local
scratch state X (zero at the chunk start) runs the same delta rule, so the
chunk's tokens still see their own writes.  The second chunk of a two-chunk
group additionally reads the first chunk's final scratch state, decayed
token by token (carry Y); the carry never enters the persistent state.
    o_t = q_t^T (S_t + X_t + Y_t) / sqrt(d).

This restates the recurrence, not the chunkwise algebra, so a slip in the
oracle's chunk formulas (Eqs. 1-8, 17-24) shows up as a mismatch.  Only the
exact (Full64) solver has a token form.
"""
import numpy as np

CHUNK = 64


def brute_prefill(q, k, v, beta, g, mask=None, h0=None):
    q, k, v, beta, g = (np.asarray(a, dtype=np.float64) for a in (q, k, v, beta, g))
    B, T, Nq, d = q.shape
    Nv, dv = v.shape[2], v.shape[3]
    C = (T + CHUNK - 1) // CHUNK
    o = np.zeros((B, T, Nv, dv))
    s_final = np.zeros((B, Nv, d, dv))
    for b in range(B):
        for h in range(Nv):
            p = h // 2
            S = np.zeros((d, dv)) if h0 is None else np.array(h0[b, h], dtype=np.float64)
            X_end = np.zeros((d, dv))
            for c in range(C):
                sel = True if mask is None else bool(mask[b, p, c])
                X = np.zeros((d, dv))
                Y = X_end.copy() if c % 2 == 1 else np.zeros((d, dv))
                g_prev = 0.0
                for t in range(c * CHUNK, min(T, (c + 1) * CHUNK)):
                    alpha = 2.0 ** (g[b, t, h] - g_prev)
                    g_prev = g[b, t, h]
                    kt, vt, qt, bt = k[b, t, p], v[b, t, h], q[b, t, p], beta[b, t, h]
                    if sel:
                        S = alpha * (S - bt * np.outer(kt, kt @ S)) + bt * np.outer(kt, vt)
                    else:
                        S = alpha * S
                        X = alpha * (X - bt * np.outer(kt, kt @ X)) + bt * np.outer(kt, vt)
                    Y = alpha * Y
                    o[b, t, h] = qt @ (S + X + Y) / np.sqrt(d)
                X_end = X
            s_final[b, h] = S
    return {"o": o, "s_final": s_final}
