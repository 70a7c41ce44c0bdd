"""Head-pair sharding over ranks (gated_delta_rule_16_gb300.sharded), on CPU with gloo.

Two ranks each run the CPU reference on their block of head pairs -- given a
mask with no collective, and with online selection over the gathered scores
and gate tails of both ranks (SparseGDN Sec. 2.4: the tier choice couples the
16 pairs of a sequence, Eq. 14).  The gathered masks, tiers, outputs and final
states must equal the single-process reference bit for bit: every (sequence,
head) unit is computed the same way whichever rank holds it.
"""
import os
import socket

import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gated_delta_rule_16_gb300 import sharded


class OracleBackend:
    """The CPU fp64 reference behind the sharded orchestration's backend interface."""

    def _np(self, t):
        return None if t is None else t.numpy()

    def _run(self, x, mask, debug=False):
        return oracle.prefill(self._np(x["q"]), self._np(x["k"]), self._np(x["v"]), self._np(x["beta"]),
                              self._np(x["g"]), mask=self._np(mask), h0=self._np(x.get("h0")),
                              solver=oracle.SOLVER_BLOCK_ADJ, debug=debug)

    def prefill(self, x, mask):
        r = self._run(x, mask)
        return torch.from_numpy(r["o"]), torch.from_numpy(r["s_final"])

    def scores(self, x):  # Tail-16 scores come from U before the read correction: any mask gives them
        return torch.from_numpy(self._run(x, None, debug=True)["score"]).float(), None

    def select(self, score, gamma, eta):
        r = oracle.select(score.numpy(), gamma.numpy(), self._np(eta))
        return torch.from_numpy(r["mask"]), torch.from_numpy(r["tier"])

    def finish(self, x, state, mask):
        return self.prefill(x, mask)


def layer():
    x = gdn_synth.make_inputs(2, 64 * 9 + 11, 16, 32, dtype="bf16", seed=77, mask="beta", with_h0=True)
    eta = np.abs(np.random.default_rng(77).standard_normal((2, 32))).astype(np.float32)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))
    return x, {"q": t(x.q), "k": t(x.k), "v": t(x.v), "beta": t(x.beta), "g": t(x.g), "mask": t(x.mask),
               "h0": t(x.h0), "eta": t(eta)}


def _worker(rank, world, port, out_dir):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        _, full = layer()
        x = sharded.shard(full, rank, world)
        be = OracleBackend()
        o, s = sharded.prefill_given_mask(be, x)
        res = {"given_o": sharded.gather_heads(o, 2, world), "given_s": sharded.gather_heads(s, 1, world)}
        o, s, m, tier = sharded.prefill_online(be, x, rank, world, 16)
        res.update({"online_o": sharded.gather_heads(o, 2, world), "online_s": sharded.gather_heads(s, 1, world),
                    "online_mask": sharded.gather_heads(m, 1, world), "online_tier": sharded.gather_heads(tier, 1, world)})
        if rank == 0:
            torch.save(res, os.path.join(out_dir, "sharded.pt"))
    finally:
        dist.destroy_process_group()


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_pair_blocks_cover_the_pairs_once():
    for world in (1, 2, 3, 4, 5, 8, 16):
        blocks = [sharded.pair_block(r, world, 16) for r in range(world)]
        assert blocks[0][0] == 0 and blocks[-1][1] == 16
        assert all(a[1] == b[0] for a, b in zip(blocks, blocks[1:]))
        sizes = [p1 - p0 for p0, p1 in blocks]
        assert max(sizes) - min(sizes) <= 1


def test_two_ranks_equal_one_process(tmp_path):
    world = 2
    torch.multiprocessing.spawn(_worker, args=(world, free_port(), str(tmp_path)), nprocs=world, join=True)
    got = torch.load(os.path.join(tmp_path, "sharded.pt"))
    x, full = layer()
    be = OracleBackend()
    ref_o, ref_s = be.prefill(full, full["mask"])
    assert torch.equal(got["given_o"], ref_o) and torch.equal(got["given_s"], ref_s)
    score, _ = be.scores(full)
    mask, tier = be.select(score, sharded.chunk_gamma(full["g"]), full["eta"])
    assert torch.equal(got["online_mask"], mask) and torch.equal(got["online_tier"], tier)
    o, s = be.prefill(full, mask)
    assert torch.equal(got["online_o"], o) and torch.equal(got["online_s"], s)
    # the selection really couples the ranks: selecting each rank's pairs on its own scores
    # (normalising its gains over its 8 pairs only) would give other tiers
    alone = [be.select(score[:, 16 * r:16 * r + 16].repeat(1, 2, 1), sharded.chunk_gamma(full["g"])[:, 16 * r:16 * r + 16]
                       .repeat(1, 2, 1), full["eta"][:, 16 * r:16 * r + 16].repeat(1, 2))[1][:, :8] for r in range(2)]
    assert not torch.equal(torch.cat(alone, dim=1), tier)
