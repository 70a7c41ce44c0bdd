"""Pins of the CPU oracle against things the pages and the mathematics fix.

None of these compare the oracle with a retyped copy of its own formulas:
  * the token-by-token gated delta recurrence (tests/brute.py) pins the dense
    chunk form and the event-sparse semantics with the exact solver;
  * the block-adjacent solver is pinned by the exactness statement of
    SparseGDN Sec. 2.3 (its seven kept blocks equal those of M^-1) and by
    inputs for which it is exact;
  * Eq. 21 (prefix-gap recovery), Eq. 25 (group minus chunk output) and the
    Sec. 2.7 worked example (skip chunk 4, keep chunk 5) are identities
    between the oracle's own intermediate results;
  * the CSR layout is pinned by a brute enumeration written differently.
"""
import itertools

import numpy as np
import pytest

import gdn_synth
import oracle
from brute import brute_prefill

CH = oracle.CHUNK


def rel_fro(a, b):
    den = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (den if den > 0 else 1.0)


def inputs(T, seed, Nq=1, B=1, mask="ones", with_h0=False, d=128):
    return gdn_synth.make_inputs(B, T, Nq, 2 * Nq, d=d, dv=d, dtype="f32", seed=seed,
                                 mask=mask, with_h0=with_h0)


# ---------------------------------------------------------------- pin (a) ---

@pytest.mark.parametrize("T", [64, 128, 192, 256, 512])
def test_dense_exact_equals_token_recurrence(T):
    x = inputs(T, seed=10 + T)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_EXACT)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g)
    assert rel_fro(r["o"], ref["o"]) < 1e-10
    assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10


def test_dense_exact_with_h0_and_ragged_tail():
    # 100 tokens: one full chunk and a 36-token partial chunk; nonzero initial state
    x = inputs(100, seed=3, with_h0=True)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, h0=x.h0, solver=oracle.SOLVER_EXACT)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, h0=x.h0)
    assert rel_fro(r["o"], ref["o"]) < 1e-10
    assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10


def test_dense_exact_small_d_two_pairs_batch2():
    x = inputs(192, seed=5, Nq=2, B=2, d=32)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_EXACT)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g)
    assert rel_fro(r["o"], ref["o"]) < 1e-10
    assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10


# ------------------------------------------------ sparse semantics, exact ---

@pytest.mark.parametrize("seed", [0, 1])
def test_sparse_all_16_masks_equal_token_rule(seed):
    x = inputs(256, seed=100 + seed, with_h0=(seed == 1))
    for bits in itertools.product([0, 1], repeat=4):
        m = np.array(bits, dtype=np.uint8).reshape(1, 1, 4)
        r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=x.h0, solver=oracle.SOLVER_EXACT)
        ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=x.h0)
        assert rel_fro(r["o"], ref["o"]) < 1e-10, bits
        if np.linalg.norm(ref["s_final"]) > 0:
            assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10, bits
        else:
            assert np.linalg.norm(r["s_final"]) == 0.0


def test_sparse_odd_chunk_count_random_masks():
    # 5 chunks: the last group holds a single chunk (Eq. 22 only)
    x = inputs(320, seed=7, Nq=2, mask="bernoulli")
    rng = np.random.default_rng(1)
    for _ in range(4):
        m = (rng.random((1, 2, 5)) < 0.5).astype(np.uint8)
        r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, solver=oracle.SOLVER_EXACT)
        ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, mask=m)
        assert rel_fro(r["o"], ref["o"]) < 1e-10


@pytest.mark.parametrize("scale", [20.0, 100.0])
def test_strong_decay_sparse_equals_token_rule(scale):
    # the stress gates of the GPU parity test (about -33 and -163 log2 decay per chunk): the oracle's
    # chunkwise form still equals the token recurrence, so it can serve as the reference there
    x = inputs(320, seed=9, Nq=2, mask="bernoulli", with_h0=True)
    g = (np.asarray(x.g, np.float64) * scale).astype(np.float32)
    rng = np.random.default_rng(2)
    m = (rng.random((1, 2, 5)) < 0.5).astype(np.uint8)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, g, mask=m, h0=x.h0, solver=oracle.SOLVER_EXACT)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, g, mask=m, h0=x.h0)
    assert rel_fro(r["o"], ref["o"]) < 1e-10
    assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10


def test_all_ones_mask_is_dense_path():
    x = inputs(320, seed=8)
    for solver in (oracle.SOLVER_EXACT, oracle.SOLVER_BLOCK_ADJ):
        a = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=solver)
        b = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=np.ones((1, 1, 5), np.uint8), solver=solver)
        assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["s_final"], b["s_final"])


# ---------------------------------------------------------------- pin (b) ---

@pytest.mark.parametrize("solver", [oracle.SOLVER_EXACT, oracle.SOLVER_BLOCK_ADJ])
def test_all_ones_group_rule_equals_chunk_rule(solver):
    x = inputs(256, seed=9)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=solver, debug=True)
    assert rel_fro(r["o"], r["o_chunk"]) < 1e-12


# ---------------------------------------------------------------- pin (c) ---

def _kept(ti, si):
    return ti // 16 - si // 16 in (0, 1)


def test_block_adjacent_support_count():
    kept = sum(1 for t in range(64) for s in range(t) if _kept(t, s))
    assert (kept, 64 * 63 // 2) == (1248, 2016)
    assert round(100 * kept / 2016, 1) == 61.9


def test_block_adjacent_kept_blocks_equal_full_inverse():
    x = inputs(256, seed=11)
    ex = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_EXACT, debug=True)["cinv"]
    ba = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_BLOCK_ADJ, debug=True)["cinv"]
    keep = np.array([[_kept(t, s) or t == s for s in range(64)] for t in range(64)])
    lower = np.tril(np.ones((64, 64), bool))
    assert np.max(np.abs(ba[..., keep] - ex[..., keep])) < 1e-12
    assert np.all(ba[..., ~keep] == 0.0)
    # far blocks of the true inverse are not zero for generic inputs: the solver is an approximation
    assert np.max(np.abs(ex[..., lower & ~keep])) > 1e-6
    # the exact solver returns a true inverse: C (I + A) = I where A is read back from C^-1
    Minv = np.linalg.inv(ex[0, 0, 0])
    assert np.allclose(np.triu(Minv), np.eye(64), atol=1e-12)


def _keys_in_subspaces(x, groups):
    """Rewrite keys so that tokens of chunk-position group j live in coordinate block j."""
    k = x.k.copy()
    d = k.shape[-1]
    width = d // len(groups)
    for j, (t0, t1) in enumerate(groups):
        for c in range(x.T // CH):
            seg = k[:, c * CH + t0:c * CH + t1]
            seg[..., :] = 0.0
            sub = np.random.default_rng(j + 7 * c).standard_normal(seg[..., j * width:(j + 1) * width].shape)
            seg[..., j * width:(j + 1) * width] = sub / np.linalg.norm(sub, axis=-1, keepdims=True)
    x.k = k.astype(np.float32)
    return x


@pytest.mark.parametrize("groups", [
    [(0, 32), (32, 64)],                       # far blocks of A_Delta vanish -> M^-1 has no far fill-in
    [(0, 16), (16, 32), (32, 48), (48, 64)],   # A_Delta block-diagonal -> C = M^-1 trivially
])
def test_block_adjacent_exact_on_structured_keys(groups):
    x = _keys_in_subspaces(inputs(256, seed=12), groups)
    m = np.array([[[1, 0, 1, 1]]], np.uint8)
    ba = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, solver=oracle.SOLVER_BLOCK_ADJ)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, mask=m)
    assert rel_fro(ba["o"], ref["o"]) < 1e-10
    assert rel_fro(ba["s_final"], ref["s_final"]) < 1e-10


def test_block_adjacent_differs_on_generic_keys():
    x = inputs(256, seed=13)
    ba = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_BLOCK_ADJ)
    ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g)
    assert rel_fro(ba["o"], ref["o"]) > 1e-8


# ---------------------------------------------------------------- pin (d) ---

@pytest.mark.parametrize("solver", [oracle.SOLVER_EXACT, oracle.SOLVER_BLOCK_ADJ])
def test_decay_only_all_zero_mask(solver):
    x = inputs(320, seed=14, with_h0=True)
    m = np.zeros((1, 1, 5), np.uint8)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=x.h0, solver=solver, debug=True)
    gam = x.g[0, CH - 1::CH, :].astype(np.float64)           # gamma_c for each chunk and head
    PC = gam.sum(axis=0)                                      # P_C per head (Eq. 19)
    expect = (2.0 ** PC)[:, None, None] * x.h0[0]
    assert rel_fro(r["s_final"][0], expect) < 1e-13
    # each skipped chunk only decays the state: S_{c+1} = 2^gamma_c S_c
    for c in range(4):
        for h in range(2):
            assert rel_fro(r["s_in"][0, h, c + 1], 2.0 ** gam[c, h] * r["s_in"][0, h, c]) < 1e-13
    z = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, solver=solver)
    assert np.all(z["s_final"] == 0.0)


def test_prefix_gap_recovery_eq21():
    x = inputs(64 * 12, seed=15, mask="bernoulli")
    m = np.array([[[1, 0, 0, 0, 1, 1, 0, 1, 0, 0, 0, 1]]], np.uint8)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, debug=True)
    gam = x.g[0, CH - 1::CH, :].astype(np.float64)
    P = np.concatenate([np.zeros((1, 2)), np.cumsum(gam, axis=0)])   # P_0 = 0, P_{c+1} = sum_{j<=c} gamma_j
    kept = np.flatnonzero(m[0, 0])
    for c in range(1, 12):
        prev = kept[kept < c]
        if prev.size == 0:
            continue
        e = prev[-1]
        for h in range(2):
            rec = 2.0 ** (P[c, h] - P[e + 1, h]) * r["s_in"][0, h, e + 1]
            assert rel_fro(r["s_in"][0, h, c], rec) < 1e-12


# ------------------------------------------ Eq. 25 and the worked example ---

def _cross_term(x, r, c, h):
    """A_{c+1,c} U'_c / sqrt(d) for value head h (Sec. 2.7)."""
    p = h // 2
    Qn = x.q[0, (c + 1) * CH:(c + 2) * CH, p].astype(np.float64)
    Kc = x.k[0, c * CH:(c + 1) * CH, p].astype(np.float64)
    gn = x.g[0, (c + 1) * CH:(c + 2) * CH, h].astype(np.float64)
    gc = x.g[0, c * CH:(c + 1) * CH, h].astype(np.float64)
    A = (Qn @ Kc.T) * 2.0 ** (gn[:, None] + gc[-1] - gc[None, :])
    return A @ r["u_prime"][0, c * CH:(c + 1) * CH, h] / np.sqrt(x.d)


@pytest.mark.parametrize("solver", [oracle.SOLVER_EXACT, oracle.SOLVER_BLOCK_ADJ])
def test_eq25_group_minus_chunk_output(solver):
    x = inputs(64 * 8, seed=16)
    m = np.array([[[0, 1, 1, 0, 0, 0, 1, 1]]], np.uint8)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, solver=solver, debug=True)
    diff = r["o"] - r["o_chunk"]
    for c in range(8):
        blk = diff[0, c * CH:(c + 1) * CH]
        if c % 2 == 0:
            assert np.max(np.abs(blk)) < 1e-14
            continue
        for h in range(2):
            expect = (1 - m[0, 0, c - 1]) * _cross_term(x, r, c - 1, h)
            assert np.max(np.abs(blk[:, h] - expect)) < 1e-12


def test_worked_example_skip_4_keep_5():
    x = inputs(64 * 8, seed=17)
    m = np.array([[[1, 1, 1, 1, 0, 1, 1, 1]]], np.uint8)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, debug=True)
    for h in range(2):
        gam4 = float(x.g[0, 5 * CH - 1, h])
        S4, S5 = r["s_in"][0, h, 4], r["s_in"][0, h, 5]
        assert rel_fro(S5, 2.0 ** gam4 * S4) < 1e-14                        # S_5 = 2^gamma_4 S_4
        U5, W5 = r["u"][0, 5 * CH:6 * CH, h], r["w"][0, 5 * CH:6 * CH, h]
        assert rel_fro(r["u_prime"][0, 5 * CH:6 * CH, h], U5 - W5 @ S5) < 1e-13  # U'_5 = U_5 - W_5 S_5
        assert np.array_equal(r["u_prime"][0, 4 * CH:5 * CH, h], r["u"][0, 4 * CH:5 * CH, h])  # U'_4 = U_4
        extra = r["o"][0, 5 * CH:6 * CH, h] - r["o_chunk"][0, 5 * CH:6 * CH, h]
        assert rel_fro(extra, _cross_term(x, r, 4, h)) < 1e-12               # O_5 carries A_54 U_4 / sqrt(d)
        assert np.linalg.norm(extra) > 1e-6


# -------------------------------------------------------------- tail score ---

def test_tail16_score():
    x = inputs(256, seed=18)
    r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, debug=True)
    for c in range(4):
        for h in range(2):
            tail = r["u"][0, c * CH + 48:(c + 1) * CH, h]
            assert abs(r["score"][0, h, c] - np.linalg.norm(tail)) < 1e-12 * np.linalg.norm(tail)


# --------------------------------------------------------------------- CSR ---

def csr_by_enumeration(mask):
    B, P, C = mask.shape
    G = (C + 1) // 2
    rows = sorted(range(B * P), key=lambda i: (-int(mask.reshape(B * P, C)[i].sum()), i))
    flat = mask.reshape(B * P, C)
    events = [(i, c) for i in rows for c in range(C) if flat[i, c]]
    row_ptr = [0]
    for i in rows:
        row_ptr.append(row_ptr[-1] + int(flat[i].sum()))
    grp_pred = np.full((B * P, G), -1, np.int32)
    for r in range(G):
        for e, (i, c) in enumerate(events):
            if c < 2 * r and (grp_pred[i, r] < 0 or events[grp_pred[i, r]][1] < c):
                grp_pred[i, r] = e
    refs = sorted(set(int(v) for v in grp_pred.ravel() if v >= 0))
    slot = np.full(len(events), -1, np.int32)
    for n, e in enumerate(refs):
        slot[e] = n
    return (np.array(rows, np.int32), np.array(row_ptr, np.int32),
            np.array([c for _, c in events], np.int32), grp_pred.reshape(B, P, G), slot)


@pytest.mark.parametrize("shape,p", [((1, 1, 4), 0.5), ((2, 3, 7), 0.4), ((3, 4, 9), 0.3),
                                     ((1, 16, 33), 0.29), ((2, 2, 1), 0.5), ((2, 3, 6), 1.0),
                                     ((2, 3, 6), 0.0)])
def test_csr_matches_enumeration(shape, p):
    rng = np.random.default_rng(sum(shape))
    for _ in range(5):
        m = (rng.random(shape) < p).astype(np.uint8)
        r = oracle.events(m)
        rows, row_ptr, ev, pred, slot = csr_by_enumeration(m)
        assert np.array_equal(r["row_pair"], rows)
        assert np.array_equal(r["row_ptr"], row_ptr)
        assert np.array_equal(r["ev_chunk"], ev)
        assert np.array_equal(r["grp_pred"], pred)
        assert np.array_equal(r["snap_slot"], slot)
        assert r["n_events"] == int(m.sum()) == row_ptr[-1]
        assert r["n_snap"] == int((slot >= 0).sum())


def test_csr_all_16_masks_of_4_chunks():
    for bits in itertools.product([0, 1], repeat=4):
        m = np.array(bits, np.uint8).reshape(1, 1, 4)
        r = oracle.events(m)
        rows, row_ptr, ev, pred, slot = csr_by_enumeration(m)
        assert np.array_equal(r["ev_chunk"], ev) and np.array_equal(r["grp_pred"], pred)
        assert np.array_equal(r["snap_slot"], slot)


def test_csr_capacity_overflow_is_reported():
    m = np.ones((1, 2, 4), np.uint8)
    r = oracle.events(m, capacity=7)
    assert r["overflow"] and r["n_events"] == 8


# ------------------------------------------------ partial last chunk (ragged T) ---

@pytest.mark.parametrize("T", [65, 100, 127, 300])
def test_sparse_ragged_tail_equals_token_rule(T):
    # C = ceil(T / 64) chunks, the last one partial; random masks, two pairs, two sequences, h0
    x = gdn_synth.make_inputs(2, T, 2, 4, d=32, dv=32, dtype="f32", seed=T, mask="ones", with_h0=True)
    C = (T + CH - 1) // CH
    rng = np.random.default_rng(T)
    for _ in range(3):
        m = (rng.random((2, 2, C)) < 0.6).astype(np.uint8)
        r = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=x.h0, solver=oracle.SOLVER_EXACT)
        ref = brute_prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=x.h0)
        assert rel_fro(r["o"], ref["o"]) < 1e-10
        assert rel_fro(r["s_final"], ref["s_final"]) < 1e-10


def test_ragged_tail_is_a_prefix_of_the_full_chunk():
    # a partial chunk of n tokens gives the first n outputs of the same chunk with more tokens
    # (causality), and the state after it is that of the n-token prefix
    x = gdn_synth.make_inputs(1, 192, 1, 2, d=32, dv=32, dtype="f32", seed=71, mask="ones")
    full = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_BLOCK_ADJ)
    cut = oracle.prefill(x.q[:, :150], x.k[:, :150], x.v[:, :150], x.beta[:, :150], x.g[:, :150],
                         solver=oracle.SOLVER_BLOCK_ADJ)
    assert rel_fro(cut["o"], full["o"][:, :150]) < 1e-12


# ------------------------------------------------------- Tail-W score windows ---

def test_tail_windows_are_nested_norms():
    # Tail-W = Frobenius norm of the last W rows of U (Eq. 9; W in {8, 16, 32, 64}, Fig. 10):
    # nested windows are monotone, their squares differ by the rows in between, and on a full
    # chunk Tail-64 is the norm of the whole U; a partial chunk shorter than W uses all its rows
    x = gdn_synth.make_inputs(1, 64 * 3 + 20, 1, 2, d=32, dv=32, dtype="f32", seed=81, mask="ones")
    s = {w: oracle.prefill(x.q, x.k, x.v, x.beta, x.g, debug=True, tail=w) for w in (8, 16, 32, 64)}
    u = s[16]["u"]                                           # [B,T,Nv,dv], independent of the window
    for h in range(2):
        for c in range(4):
            n = min(64, 212 - 64 * c)
            rows = u[0, 64 * c:64 * c + n, h]
            sq = {w: s[w]["score"][0, h, c] ** 2 for w in s}
            assert sq[8] <= sq[16] <= sq[32] <= sq[64]
            for w in (16, 32, 64):
                lo, hi = max(0, n - w), max(0, n - w // 2)
                assert abs(sq[w] - sq[w // 2] - np.sum(rows[lo:hi] ** 2)) <= 1e-12 * max(sq[w], 1e-300)
            if n == 64:
                assert abs(sq[64] - np.sum(rows ** 2)) <= 1e-12 * sq[64]
            else:  # 20 rows: every window of 32 or more covers them all
                assert sq[32] == sq[64]
    # the window only changes the score
    assert np.array_equal(s[8]["o"], s[64]["o"]) and np.array_equal(s[8]["s_final"], s[64]["s_final"])
