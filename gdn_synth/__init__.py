"""Seeded synthetic inputs for the chunkwise gated-delta prefill core.

This module is shared by the CUDA path's tests/benchmark and by the CPU oracle's
tests. It holds no arithmetic of the method itself: it only draws random
tensors with the shapes and distributions of the SparseGDN workloads and
rounds them to the storage dtype.

Workload recipe (SparseGDN reading notes, Sec. 2.1 problem statement and
Sec. 3.1 setup; these distributions stand in for the RULER timing loads,
which are not available):

* q, k ~ N(0, 1) per element, then L2-normalised per (token, head);
  v ~ N(0, 1).  Drawn in fp32, stored either as fp32 or rounded
  round-to-nearest-even to bf16.
* beta = sigmoid(N(0, 1)) in fp32, one per (token, value head).
* per-token log2 retention a = -U(0.001, 0.05) per value head, and
  g = inclusive cumulative sum of a inside each 64-token chunk (the pages'
  g_{c,h,i}), in fp32.
* event masks over (head pair x chunk):
    - "two_of_four": each pair keeps a seeded random 2 of every 4 chunks
      (the tiny fp32 case);
    - "ones": all chunks kept (dense path);
    - "zeros": no chunk kept;
    - "beta": per pair rho_p ~ Beta(2, 5), rescaled so the mean over the
      sequence's pairs is `retention`, clipped to [2/C, 1]; k_p = round(rho_p C);
      chunks 0 and C-1 are always kept plus k_p - 2 others uniformly without
      replacement.  Each sequence of a batch draws its own mask.

Seeds follow 1000*config + 100*layer + batch_index.  Every draw uses numpy's
PCG64 generator; tensors are drawn in blocks of 2048 tokens, each from its own
SeedSequence child, so the same bits come out on any host and thread count.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

CHUNK = 64


def seed_for(config: int, layer: int = 0, batch_index: int = 0) -> int:
    return 1000 * config + 100 * layer + batch_index


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round-to-nearest-even); returns uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass
class Inputs:
    B: int
    T: int
    Nq: int
    Nv: int
    d: int
    dv: int
    dtype: str                      # "bf16" or "f32": storage type of q, k, v (and o)
    q: np.ndarray                   # float32 [B,T,Nq,d], values exactly representable in `dtype`
    k: np.ndarray                   # float32 [B,T,Nq,d]
    v: np.ndarray                   # float32 [B,T,Nv,dv]
    beta: np.ndarray                # float32 [B,T,Nv]
    g: np.ndarray                   # float32 [B,T,Nv], inclusive within-chunk cumsum of log2 retention
    mask: np.ndarray                # uint8 [B,Nv//2,C]
    h0: np.ndarray | None = None    # float32 [B,Nv,d,dv] or None
    meta: dict = field(default_factory=dict)

    @property
    def C(self) -> int:
        return (self.T + CHUNK - 1) // CHUNK

    @property
    def P(self) -> int:
        return self.Nv // 2

    def storage(self, name: str) -> np.ndarray:
        """q/k/v in their storage representation: uint16 bf16 bits or float32."""
        a = getattr(self, name)
        return f32_to_bf16_bits(a) if self.dtype == "bf16" else a

    def retention(self) -> float:
        return float(self.mask.mean()) if self.mask.size else 0.0


def _l2n(x: np.ndarray) -> np.ndarray:
    n = np.sqrt(np.einsum("...i,...i->...", x, x, dtype=np.float32))[..., None]
    return (x / np.maximum(n, np.float32(1e-30))).astype(np.float32)


def _round(x: np.ndarray, dtype: str) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    return bf16_bits_to_f32(f32_to_bf16_bits(x)) if dtype == "bf16" else x


TOKEN_BLOCK = 2048  # tokens per independently seeded generation block


def _blocks(B: int, T: int):
    return [(b, t0, min(T, t0 + TOKEN_BLOCK)) for b in range(B) for t0 in range(0, T, TOKEN_BLOCK)]


def _fill(seed: int, tag: int, out: np.ndarray, draw) -> None:
    """Fill out[b, t0:t1] block by block; block (b, t0) draws from its own
    SeedSequence child [seed, tag, b, t0 // TOKEN_BLOCK], so the result does
    not depend on thread scheduling or the host."""
    import concurrent.futures as cf

    def work(blk):
        b, t0, t1 = blk
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, b, t0 // TOKEN_BLOCK])))
        out[b, t0:t1] = draw(rng, (t1 - t0,) + out.shape[2:])

    blocks = _blocks(out.shape[0], out.shape[1])
    if len(blocks) <= 1:
        for blk in blocks:
            work(blk)
        return
    with cf.ThreadPoolExecutor(max_workers=min(16, len(blocks))) as ex:
        list(ex.map(work, blocks))


def make_mask(rng: np.random.Generator, B: int, P: int, C: int, kind: str,
              retention: float = 0.29) -> np.ndarray:
    mask = np.zeros((B, P, C), dtype=np.uint8)
    if C == 0:
        return mask
    if kind == "ones":
        mask[:] = 1
    elif kind == "zeros":
        pass
    elif kind == "two_of_four":
        for b in range(B):
            for p in range(P):
                for c0 in range(0, C, 4):
                    n = min(4, C - c0)
                    keep = rng.choice(n, size=min(2, n), replace=False)
                    mask[b, p, c0 + keep] = 1
    elif kind == "bernoulli":
        mask[:] = (rng.random((B, P, C)) < retention).astype(np.uint8)
    elif kind == "beta":
        for b in range(B):
            rho = rng.beta(2.0, 5.0, size=P)
            rho = rho * (retention / rho.mean())
            rho = np.clip(rho, min(1.0, 2.0 / C), 1.0)
            kp = np.clip(np.rint(rho * C).astype(np.int64), min(2, C), C)
            for p in range(P):
                mask[b, p, 0] = 1
                mask[b, p, C - 1] = 1
                inner = np.arange(1, C - 1)
                extra = int(kp[p]) - int(mask[b, p].sum())
                if extra > 0 and inner.size:
                    pick = rng.choice(inner, size=min(extra, inner.size), replace=False)
                    mask[b, p, pick] = 1
    else:
        raise ValueError(f"unknown mask kind {kind!r}")
    return mask


def make_inputs(B: int, T: int, Nq: int, Nv: int, d: int = 128, dv: int = 128,
                dtype: str = "bf16", seed: int = 0, mask: str = "beta",
                retention: float = 0.29, with_h0: bool = False) -> Inputs:
    """Draw one seeded layer of inputs; see the module docstring for the recipe."""
    if Nv != 2 * Nq:
        raise ValueError("value heads come in adjacent pairs per query/key head (Nv == 2*Nq)")
    q = np.empty((B, T, Nq, d), np.float32)
    k = np.empty((B, T, Nq, d), np.float32)
    v = np.empty((B, T, Nv, dv), np.float32)
    beta = np.empty((B, T, Nv), np.float32)
    normal_qk = lambda r, shp: _round(_l2n(r.standard_normal(shp, dtype=np.float32)), dtype)
    _fill(seed, 1, q, normal_qk)
    _fill(seed, 2, k, normal_qk)
    _fill(seed, 3, v, lambda r, shp: _round(r.standard_normal(shp, dtype=np.float32), dtype))
    _fill(seed, 4, beta, lambda r, shp: (1.0 / (1.0 + np.exp(-r.standard_normal(shp, dtype=np.float32)))).astype(np.float32))
    g = make_gates(B, T, Nv, seed)
    C = (T + CHUNK - 1) // CHUNK
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    m = make_mask(rng, B, Nv // 2, C, mask, retention)
    h0 = rng.standard_normal((B, Nv, d, dv), dtype=np.float32) * np.float32(0.1) if with_h0 else None
    return Inputs(B, T, Nq, Nv, d, dv, dtype, q, k, v, beta, g, m, h0,
                  meta={"seed": seed, "mask": mask, "retention_target": retention})


def make_gates(B: int, T: int, Nv: int, seed: int) -> np.ndarray:
    """g [B,T,Nv] fp32: per-token log2 retention -U(0.001, 0.05), summed inside each chunk."""
    a = np.empty((B, T, Nv), np.float32)
    _fill(seed, 5, a, lambda r, shp: -r.uniform(0.001, 0.05, size=shp).astype(np.float32))
    g = np.empty_like(a)
    if T:
        full = (T // CHUNK) * CHUNK
        g[:, :full] = np.cumsum(a[:, :full].reshape(B, T // CHUNK, CHUNK, Nv), axis=2, dtype=np.float32).reshape(B, full, Nv)
        if full < T:
            g[:, full:] = np.cumsum(a[:, full:], axis=1, dtype=np.float32)
    return g


def make_scores(B: int, Nv: int, C: int, seed: int, kind: str = "lognormal") -> np.ndarray:
    """Stand-in Tail-16 write scores [B,Nv,C] fp32 (non-negative, like norms).

    "lognormal": |N(0,1)| times a per-head scale exp(N(0, 0.7)), with a few hot
    chunks (x4) per head; "ties": the same, rounded to 1/4 so many values tie;
    "zero_heads": lognormal with every fourth head all zero.
    """
    rng = np.random.default_rng(np.random.SeedSequence([seed, 7]))
    s = np.abs(rng.standard_normal((B, Nv, C))) * np.exp(0.7 * rng.standard_normal((B, Nv, 1)))
    hot = rng.random((B, Nv, C)) < 0.05
    s = np.where(hot, 4.0 * s, s)
    if kind == "ties":
        s = np.round(4.0 * s) / 4.0
    elif kind == "zero_heads":
        s[:, ::4] = 0.0
    elif kind != "lognormal":
        raise ValueError(f"unknown score kind {kind!r}")
    return s.astype(np.float32)


# The five workloads of the SparseGDN GDN-core study, by what they are.
WORKLOADS = {
    "tiny_fp32_T256": dict(B=1, T=256, Nq=1, Nv=2, dtype="f32", mask="two_of_four", config=0),
    "qwen35_4b_layer_T4096_dense": dict(B=1, T=4096, Nq=16, Nv=32, dtype="bf16", mask="ones", config=1),
    "qwen35_4b_layer_T32768_sparse29": dict(B=1, T=32768, Nq=16, Nv=32, dtype="bf16", mask="beta", config=2),
    "qwen35_4b_24layers_T131072_sparse29": dict(B=1, T=131072, Nq=16, Nv=32, dtype="bf16", mask="beta", config=3),
    "qwen35_4b_layer_B8_T32768_sparse29": dict(B=8, T=32768, Nq=16, Nv=32, dtype="bf16", mask="beta", config=4),
}


def make_workload(name: str, layer: int = 0, batch_index: int = 0, **override) -> Inputs:
    w = dict(WORKLOADS[name])
    w.update(override)
    cfg = w.pop("config")
    return make_inputs(w.pop("B"), w.pop("T"), w.pop("Nq"), w.pop("Nv"),
                       seed=seed_for(cfg, layer, batch_index), **w)


def make_layer_on_device(B: int, T: int, Nq: int, Nv: int, seed: int, device, d: int = 128, dv: int = 128,
                         mask: str = "beta", retention: float = 0.29) -> dict:
    """The same recipe as make_inputs (bf16 storage), drawn on the GPU with a seeded
    torch generator, for workloads too large to draw on the host in a benchmark (the
    24-layer, 128K-token prefill).  The bits differ from make_inputs' for the same
    seed; the distributions are the same.  The mask is drawn on the host with
    make_mask.  Returns device tensors q, k [B,T,Nq,d] bf16; v [B,T,Nv,dv] bf16;
    beta, g [B,T,Nv] fp32; mask [B,Nv/2,C] uint8."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    f32 = torch.float32

    def l2n(x):
        return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)

    q = l2n(torch.randn((B, T, Nq, d), generator=gen, device=device, dtype=f32)).to(torch.bfloat16)
    k = l2n(torch.randn((B, T, Nq, d), generator=gen, device=device, dtype=f32)).to(torch.bfloat16)
    v = torch.randn((B, T, Nv, dv), generator=gen, device=device, dtype=f32).to(torch.bfloat16)
    beta = torch.sigmoid(torch.randn((B, T, Nv), generator=gen, device=device, dtype=f32))
    a = -(0.001 + 0.049 * torch.rand((B, T, Nv), generator=gen, device=device, dtype=f32))
    C = (T + CHUNK - 1) // CHUNK
    pad = C * CHUNK - T
    ap = torch.nn.functional.pad(a, (0, 0, 0, pad)).view(B, C, CHUNK, Nv)
    g = torch.cumsum(ap, dim=2).view(B, C * CHUNK, Nv)[:, :T].contiguous()
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0]))
    m = torch.from_numpy(make_mask(rng, B, Nv // 2, C, mask, retention)).to(device)
    return {"q": q, "k": k, "v": v, "beta": beta, "g": g, "mask": m}
