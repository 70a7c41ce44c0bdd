"""Selector inputs built so that the tier split depends on the memory lifetime
of SparseGDN Sec. 2.4, Eq. 11: r_h = mean of 2^gamma over the last min(16, C)
chunks, L_h = sum_{j=1}^{C-2} r_h^j.  Every pair gets the same score pattern up
to a per-pair scale, so the upgrade gains (Eq. 12) differ only through the
scale and L_h, and the expected tiers follow from the reading of Eq. 11 alone.

Each builder returns (score [1,32,C] fp32, gamma [1,32,C] fp32, expected tiers
[16] with 2 high, 1 mid, 0 low).
"""
import numpy as np

NP, NV = 16, 32


def window_case():
    """Pairs 0-2 remember long only inside the last-16-chunk window, pairs 3-5
    only before it.  With r_h over the window, pairs 0-2 (L ~ 25) are the high
    tier and pairs 3-5 (L ~ 2e-4) fall below the background (L ~ 1); a mean
    over all chunks would swap them."""
    C = 64
    s = np.ones((1, NV, C), np.float32)
    g = np.full((1, NV, C), -1.0, np.float32)
    g[0, 0:6, :C - 16] = -12.0
    g[0, 0:6, C - 16:] = -0.05
    g[0, 6:12, :C - 16] = -0.05
    g[0, 6:12, C - 16:] = -12.0
    tiers = np.array([2, 2, 2, 0, 0, 0] + [1] * 5 + [0] * 5, np.int32)
    return s, g, tiers


def sum_from_one_case():
    """Pairs 0-2 write 1000x louder but forget at once (r = 2^-20, so
    L = r + r^2 + ... ~ 1e-6); pairs 3-5 remember (r = 2^-0.05, L ~ 25).  The
    sum from j = 1 makes pairs 3-5 the high tier and pairs 0-2 the lowest; a
    sum from j = 0 (or L = 1) would lift the loud pairs to the top."""
    C = 64
    s = np.ones((1, NV, C), np.float32)
    g = np.full((1, NV, C), -1.0, np.float32)
    s[0, 0:6] *= 1000.0
    g[0, 0:6] = -20.0
    g[0, 6:12] = -0.05
    tiers = np.array([0, 0, 0, 2, 2, 2] + [1] * 5 + [0] * 5, np.int32)
    return s, g, tiers


def closed_form_case():
    """Sixteen different constant retentions r_p; each pair's scores are a
    weight w_p divided by the closed form L(r) = r (1 - r^(C-2)) / (1 - r).  If
    L_h is that geometric sum, the gains are proportional to w = (100 x3,
    10 x4, 1 x9) and the tiers are (H x3, M x4, L x9); any other L rescales the
    pairs by factors up to ~400 and scrambles the split."""
    C = 40
    gam = -np.array([0.02, 0.05, 0.1, 0.2, 0.3, 0.5, 0.7, 1.0, 1.3, 1.6, 2.0, 2.4, 2.8, 3.2, 3.6, 4.0])
    w = np.array([100.0] * 3 + [10.0] * 4 + [1.0] * 9)
    r = 2.0 ** gam
    L = r * (1.0 - r ** (C - 2)) / (1.0 - r)
    s = np.empty((1, NV, C), np.float32)
    g = np.empty((1, NV, C), np.float32)
    for p in range(NP):
        s[0, 2 * p:2 * p + 2] = np.float32(w[p] / L[p])
        g[0, 2 * p:2 * p + 2] = np.float32(gam[p])
    tiers = np.array([2] * 3 + [1] * 4 + [0] * 9, np.int32)
    return s, g, tiers


CASES = {"window": window_case, "sum_from_one": sum_from_one_case, "closed_form": closed_form_case}
