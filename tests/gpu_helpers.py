"""Shared helpers of the GPU parity tests: move seeded inputs to the device,
run the CUDA path through the C ABI, compare with the oracle."""
import numpy as np
import torch

import gated_delta_rule_16_gb300 as gdn

# Tolerances on the maximum over (sequence, value head) of the relative
# Frobenius error (O over [T, dv], S over [d, dv]): 2e-2 with bf16 storage and
# fp32 accumulation, 1e-5 for fp32 storage.  When the reference is exactly
# zero, the absolute Frobenius norm must stay below 1e-6.
TOL = {"bf16": 2e-2, "f32": 1e-5}
ABS_ZERO = 1e-6


def dev():
    return torch.device("cuda:0")


def to_dev(x):
    """Inputs on the GPU in their storage dtype."""
    d = dev()
    st = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(d).to(dt)
    out = {"q": f(x.q, st), "k": f(x.k, st), "v": f(x.v, st), "beta": f(x.beta, torch.float32),
           "g": f(x.g, torch.float32), "mask": f(x.mask, torch.uint8)}
    out["h0"] = None if x.h0 is None else f(x.h0, torch.float32)
    return out


def run_gpu(x, solver="block_adj", sparse=True, mask=None, h0=None, score=False, workspace=None):
    t = to_dev(x)
    if mask is not None:
        t["mask"] = torch.from_numpy(np.ascontiguousarray(mask, dtype=np.uint8)).to(dev())
    h0t = t["h0"] if h0 is None else torch.from_numpy(np.ascontiguousarray(h0, np.float32)).to(dev())
    sc = torch.full((x.B, x.Nv, x.C), -1.0, device=dev()) if score else None
    if sparse:
        o, s = gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"], h0=h0t,
                                      solver=solver, score=sc, workspace=workspace)
    else:
        o, s = gdn.gdn_prefill_dense(t["q"], t["k"], t["v"], t["beta"], t["g"], h0=h0t, solver=solver,
                                     score=sc, workspace=workspace)
    torch.cuda.synchronize()
    res = {"o": o.float().cpu().numpy().astype(np.float64), "s_final": s.cpu().numpy().astype(np.float64)}
    if score:
        res["score"] = sc.cpu().numpy().astype(np.float64)
    return res


def max_rel_err(got, want, kind):
    """kind 'o': arrays [B,T,Nv,dv]; kind 's': [B,Nv,d,dv].  Returns (max rel, max abs where ref == 0)."""
    if kind == "o":
        got = np.moveaxis(got, 2, 1)  # [B,Nv,T,dv]
        want = np.moveaxis(want, 2, 1)
    worst_rel, worst_abs = 0.0, 0.0
    for b in range(got.shape[0]):
        for h in range(got.shape[1]):
            den = np.linalg.norm(want[b, h])
            num = np.linalg.norm(got[b, h] - want[b, h])
            if den == 0.0:
                worst_abs = max(worst_abs, num)
            else:
                worst_rel = max(worst_rel, num / den)
    return worst_rel, worst_abs


def max_rel_err_chunks(got, want):
    """O arrays [B,T,Nv,dv]: the largest relative Frobenius error over (sequence, value head,
    64-token chunk), each chunk's error against that chunk's own reference norm (so an error
    confined to one chunk is not diluted by the rest of the sequence).  Chunks whose reference
    is exactly zero are measured by the absolute norm.  Returns (max rel, max abs where zero)."""
    B, T, Nv, dv = want.shape
    C = (T + 63) // 64
    pad = C * 64 - T
    g = np.pad(got, ((0, 0), (0, pad), (0, 0), (0, 0))).reshape(B, C, 64, Nv, dv)
    w = np.pad(want, ((0, 0), (0, pad), (0, 0), (0, 0))).reshape(B, C, 64, Nv, dv)
    num = np.sqrt(((g - w) ** 2).sum(axis=(2, 4)))
    den = np.sqrt((w ** 2).sum(axis=(2, 4)))
    zero = den == 0.0
    rel = np.where(zero, 0.0, num / np.where(zero, 1.0, den))
    return float(rel.max()), float(np.where(zero, num, 0.0).max())


def assert_close(res, ref, dtype, what=""):
    tol = TOL[dtype]
    for key, kind in (("o", "o"), ("s_final", "s")):
        rel, ab = max_rel_err(res[key], ref[key], kind)
        assert rel <= tol, f"{what} {key}: max relative Frobenius error {rel:.3e} > {tol}"
        assert ab <= ABS_ZERO, f"{what} {key}: absolute error {ab:.3e} where the reference is zero"
    # the same bound per 64-token chunk of O
    rel, ab = max_rel_err_chunks(res["o"], ref["o"])
    assert rel <= tol, f"{what} o: max relative Frobenius error of one chunk {rel:.3e} > {tol}"
    assert ab <= ABS_ZERO, f"{what} o: absolute error {ab:.3e} in a chunk where the reference is zero"


def slice_pairs(x, b, pairs):
    """Inputs restricted to sequence b and the given head pairs (pairs are independent)."""
    import copy
    y = copy.copy(x)
    qi = list(pairs)
    vi = [2 * p + j for p in pairs for j in (0, 1)]
    y.q = x.q[b:b + 1][:, :, qi]
    y.k = x.k[b:b + 1][:, :, qi]
    y.v = x.v[b:b + 1][:, :, vi]
    y.beta = x.beta[b:b + 1][:, :, vi]
    y.g = x.g[b:b + 1][:, :, vi]
    y.mask = x.mask[b:b + 1][:, qi]
    y.h0 = None if x.h0 is None else x.h0[b:b + 1][:, vi]
    y.B, y.Nq, y.Nv = 1, len(qi), len(vi)
    return y
