"""Pins of the oracle's online event selector (SparseGDN Sec. 2.4, Eqs. 10-14).

The pages fix: the candidate budgets (0.08, 0.30, 0.95), anchors (first and
last chunk), nested sets, the tier-count table {1: 11-13, 2: 7-9, 3: 3-5, 4: 0},
the nominal mean retention range 28.44-31.31 % that table implies, and the
preallocation bound E <= 16 k_H.  The other checks use inputs built so that the
tier split or the ranking is known in advance.
"""
import numpy as np
import pytest

import oracle

NP, NV = 16, 32


def rand_inputs(B, C, seed, gamma_lo=-3.2, gamma_hi=-0.064):
    rng = np.random.default_rng(seed)
    s = rng.gamma(2.0, 1.0, size=(B, NV, C)).astype(np.float32)
    g = rng.uniform(gamma_lo, gamma_hi, size=(B, NV, C)).astype(np.float32)
    return s, g


@pytest.mark.parametrize("seed", range(6))
def test_retention_in_pages_nominal_range_and_event_bound(seed):
    C = 4096  # large C: integer rounding of k_l is negligible
    s, g = rand_inputs(2, C, seed)
    r = oracle.select(s, g)
    kL, kM, kH = r["k"]
    for b in range(2):
        counts = r["mask"][b].sum(-1)
        assert set(counts.tolist()) <= {kL, kM, kH}
        E = int(counts.sum())
        assert E <= 16 * kH
        keep = E / (16 * C)
        assert 0.2844 - 1e-3 <= keep <= 0.3131 + 1e-3
        nH = int((r["tier"][b] == 2).sum())
        nM = int((r["tier"][b] == 1).sum())
        assert 1 <= nH <= 4
        assert nM in {1: (11, 12, 13), 2: (7, 8, 9), 3: (3, 4, 5), 4: (0,)}[nH]


def test_nominal_range_endpoints_of_the_tier_table():
    table = {1: (11, 12, 13), 2: (7, 8, 9), 3: (3, 4, 5), 4: (0,)}
    vals = [(nh * 0.95 + nm * 0.30 + (16 - nh - nm) * 0.08) / 16 for nh, row in table.items() for nm in row]
    assert round(100 * min(vals), 2) == 28.44 and round(100 * max(vals), 2) == 31.31


@pytest.mark.parametrize("C", [1, 2, 3, 5, 17, 64, 513])
def test_anchors_and_small_chunk_counts(C):
    s, g = rand_inputs(1, C, 100 + C)
    r = oracle.select(s, g)
    m = r["mask"][0]
    assert np.all(m[:, 0] == 1) and np.all(m[:, C - 1] == 1)  # first and last chunk always kept
    if C <= 2:
        assert np.all(m == 1)
    kL, kM, kH = r["k"]
    assert kL <= kM <= kH <= C and (kL >= 2 or C < 2)


def test_obvious_split_picks_three_high_and_four_mid_pairs():
    C = 512
    s, g = rand_inputs(1, C, 7)
    s[:] = 1.0
    s[0, 0:6] *= 100.0    # pairs 0, 1, 2: far larger gains than every other pair
    s[0, 6:14] *= 10.0    # pairs 3 .. 6: clearly above the rest
    r = oracle.select(s, g)
    assert r["tier"][0].tolist() == [2, 2, 2] + [1] * 4 + [0] * 9


def test_ranking_follows_tail_scores_and_ties_take_lower_chunks():
    C = 100
    s = np.ones((1, NV, C), np.float32)
    g = np.full((1, NV, C), -1.0, np.float32)
    s[0, 0, :] = np.arange(C, dtype=np.float32) + 1.0   # pair 0: score grows with the chunk index
    r = oracle.select(s, g)
    kk = r["k"][r["tier"][0][0]]
    expect = {0, C - 1} | set(range(C - 2, C - 2 - (kk - 2), -1))
    assert set(np.flatnonzero(r["mask"][0, 0]).tolist()) == expect
    kk1 = r["k"][r["tier"][0][1]]                          # pair 1: all scores equal -> lowest indices
    assert set(np.flatnonzero(r["mask"][0, 1]).tolist()) == {0, C - 1} | set(range(1, kk1 - 1))


def test_zero_visibility_pair_is_never_high_tier():
    C = 512
    s, g = rand_inputs(1, C, 9)
    s[0, 0:2] *= 50.0
    eta = np.ones((1, NV), np.float32)
    r1 = oracle.select(s, g, eta)
    assert r1["tier"][0][0] == 2            # large gains -> high tier
    eta[0, 0:2] = 0.0                        # G_h = 0 for both heads of pair 0
    r0 = oracle.select(s, g, eta)
    assert r0["tier"][0][0] != 2
    assert np.array_equal(oracle.select(s, g)["mask"], oracle.select(s, g, np.ones((1, NV), np.float32))["mask"])


# ---- Eq. 11: the memory lifetime r_h, L_h decides these splits (inputs in selector_cases.py) ----

@pytest.mark.parametrize("name", ["window", "sum_from_one", "closed_form"])
def test_memory_lifetime_decides_the_tiers(name):
    from selector_cases import CASES
    s, g, tiers = CASES[name]()
    r = oracle.select(s, g)
    assert r["tier"][0].tolist() == tiers.tolist()
    k = r["k"]
    assert r["mask"][0].sum(-1).tolist() == [k[t] for t in tiers]  # every pair keeps its tier's budget
