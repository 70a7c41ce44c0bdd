"""Head-pair sharding of one GDN layer over ranks (tensor parallelism).

Rank r of `world` owns a contiguous block of head pairs [p0, p1) of every
sequence: query/key heads p0..p1-1 and value heads 2 p0 .. 2 p1 - 1, so its
q, k, v, beta, g, mask and o are the head slices a head-sharded projection
produces.  Given a mask, every (sequence, pair) is independent (SparseGDN
Secs. 2.3-2.7 never read another pair's data): each rank runs its block and no
collective is needed.  Online selection (Sec. 2.4) couples a sequence's 16 pairs:
the upgrade gains are normalised by their mean over the pairs and the tier
counts chosen from all of them (Eq. 14).  Each rank then computes its pairs'
Tail-16 scores (first call), the ranks all-gather the scores and the chunk gate
tails gamma (and eta, when given) -- [B, 32, C] fp32 each, 64 KB per sequence
at T = 32K --, every rank runs the same selection on the gathered values and
keeps its own rows of the mask, and each finishes its block (second call).

The orchestration is written against a small backend interface so the same
host logic drives the library (CudaBackend) and, in the tests, a CPU reference.
This module moves and slices tensors only; every step of the method runs in
the backend.
"""
from __future__ import annotations

import torch

CHUNK = 64


def pair_block(rank: int, world: int, P: int) -> tuple[int, int]:
    """[p0, p1) of rank `rank`: contiguous blocks whose sizes differ by at most one."""
    if not 0 <= rank < world:
        raise ValueError("rank out of range")
    base, extra = divmod(P, world)
    p0 = rank * base + min(rank, extra)
    return p0, p0 + base + (1 if rank < extra else 0)


def shard(inputs: dict, rank: int, world: int) -> dict:
    """This rank's head slices of a layer's inputs: q, k [B,T,Nq,d]; v [B,T,Nv,dv];
    beta, g [B,T,Nv]; mask [B,P,C] (optional); eta [B,Nv] (optional); h0 [B,Nv,d,dv]
    (optional).  Returns contiguous tensors."""
    P = inputs["q"].shape[2]
    p0, p1 = pair_block(rank, world, P)
    out = {}
    for name, t in inputs.items():
        if t is None:
            out[name] = None
        elif name in ("q", "k"):
            out[name] = t[:, :, p0:p1].contiguous()
        elif name in ("v", "beta", "g"):
            out[name] = t[:, :, 2 * p0:2 * p1].contiguous()
        elif name == "mask":
            out[name] = t[:, p0:p1].contiguous()
        elif name in ("eta", "h0"):
            out[name] = t[:, 2 * p0:2 * p1].contiguous()
        else:
            raise ValueError(f"unknown input {name!r}")
    return out


def chunk_gamma(g: torch.Tensor) -> torch.Tensor:
    """gamma [B,Nv,C]: g [B,T,Nv] at each chunk's last token (a partial last chunk: token T - 1)."""
    T = g.shape[1]
    C = (T + CHUNK - 1) // CHUNK
    idx = torch.clamp(torch.arange(C, device=g.device) * CHUNK + CHUNK - 1, max=T - 1)
    return g[:, idx, :].transpose(1, 2).contiguous()


def gather_heads(local: torch.Tensor, dim: int, world: int, group=None) -> torch.Tensor:
    """All-gather blocks of `local` along `dim` (block sizes may differ by one between
    ranks: padded to the largest, then cut) and concatenate them in rank order."""
    import torch.distributed as dist
    n = torch.tensor([local.shape[dim]], dtype=torch.int64, device=local.device)
    sizes = [torch.zeros(1, dtype=torch.int64, device=local.device) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(s.item()) for s in sizes]
    m = max(sizes)
    if local.shape[dim] < m:
        pad_shape = list(local.shape)
        pad_shape[dim] = m - local.shape[dim]
        local = torch.cat([local, local.new_zeros(pad_shape)], dim=dim)
    parts = [torch.empty_like(local) for _ in range(world)]
    dist.all_gather(parts, local.contiguous(), group=group)
    return torch.cat([p.narrow(dim, 0, s) for p, s in zip(parts, sizes)], dim=dim)


class CudaBackend:
    """The library on this rank's GPU (bf16 or fp32 storage, block-adjacent solver by default)."""

    def __init__(self, solver: str = "block_adj", stream=None):
        import gated_delta_rule_16_gb300 as gdn
        self.gdn = gdn
        self.solver = solver
        self.stream = stream

    def prefill(self, x: dict, mask: torch.Tensor):
        return self.gdn.gdn_prefill_sparse(x["q"], x["k"], x["v"], x["beta"], x["g"], mask, h0=x.get("h0"),
                                           solver=self.solver, stream=self.stream)

    def scores(self, x: dict):
        B, T, Nv = x["beta"].shape
        C = (T + CHUNK - 1) // CHUNK
        sc = torch.empty((B, Nv, C), dtype=torch.float32, device=x["q"].device)
        ws = self.gdn.Workspace()
        self.gdn.gdn_prefill_ex(x["q"], x["k"], x["v"], x["beta"], x["g"], mode="online", h0=x.get("h0"),
                                solver=self.solver, online_split=1, score=sc, workspace=ws, stream=self.stream)
        return sc, ws

    def select(self, score: torch.Tensor, gamma: torch.Tensor, eta):
        return self.gdn.gdn_select_events_gamma(score, gamma, eta, stream=self.stream)

    def finish(self, x: dict, state, mask: torch.Tensor):
        o, s, _, _ = self.gdn.gdn_prefill_ex(x["q"], x["k"], x["v"], x["beta"], x["g"], mode="online",
                                             mask=mask.contiguous(), h0=x.get("h0"), solver=self.solver,
                                             online_split=2, workspace=state, stream=self.stream)
        return o, s


def prefill_given_mask(backend, x: dict):
    """This rank's block with the given mask rows: (o, s_final) of its pairs; no collective."""
    return backend.prefill(x, x["mask"])


def prefill_online(backend, x: dict, rank: int, world: int, P: int, group=None, comm_device=None):
    """This rank's block with online selection over all ranks' pairs.  Collective: two (three
    with eta) all-gathers of [B, heads, C] tensors over `group`, on `comm_device` (default: where
    the tensors are).  Returns (o, s_final, mask rows, tier rows) of this rank's pairs."""
    p0, p1 = pair_block(rank, world, P)
    score, state = backend.scores(x)
    gamma = chunk_gamma(x["g"])
    dev = score.device
    to_comm = (lambda t: t.to(comm_device)) if comm_device is not None else (lambda t: t)
    score_all = gather_heads(to_comm(score), 1, world, group).to(dev)
    gamma_all = gather_heads(to_comm(gamma), 1, world, group).to(dev)
    eta = x.get("eta")
    eta_all = gather_heads(to_comm(eta), 1, world, group).to(dev) if eta is not None else None
    mask_all, tier_all = backend.select(score_all, gamma_all, eta_all)
    mask = mask_all[:, p0:p1].contiguous()
    o, s = backend.finish(x, state, mask)
    return o, s, mask, tier_all[:, p0:p1]
