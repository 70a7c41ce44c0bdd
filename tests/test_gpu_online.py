"""Parity of the online event selector (SparseGDN Sec. 2.4, Eqs. 10-14) and of
the prefill that selects its own events, through the C ABI.

The selection is a deterministic function of the Tail-16 scores and the gates,
so the GPU's masks and tiers must equal the oracle's bit for bit on the same
scores.  The prefill that selects online is checked in three parts: its scores
against the oracle's (floating-point tolerance), its mask against the oracle's
selection on the GPU's own scores (bit for bit; near-equal scores may rank
either way, so the oracle's own scores are not the reference for the mask),
and its outputs against the oracle prefill run with that mask.
"""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, assert_close, dev, slice_pairs, to_dev

import gated_delta_rule_16_gb300 as gdn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gated_delta_rule_16_gb300 import build
    build.build()
    gdn.load()


def chunk_gamma(g, C):
    """gamma[b,h,c] = g at the last token of chunk c (of a partial last chunk: token T - 1)."""
    T = g.shape[1]
    idx = np.minimum(np.arange(C) * 64 + 63, T - 1)
    return np.ascontiguousarray(np.moveaxis(g[:, idx, :], 1, 2))


def gpu_select(score, g, eta=None):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev())
    mask, tier = gdn.gdn_select_events_scored(t(score), t(g), None if eta is None else t(eta))
    torch.cuda.synchronize()
    return mask.cpu().numpy(), tier.cpu().numpy()


@pytest.mark.parametrize("B,C,kind", [(1, 1, "lognormal"), (1, 2, "lognormal"), (1, 3, "lognormal"),
                                      (2, 5, "ties"), (1, 15, "lognormal"), (1, 25, "zero_heads"),
                                      (3, 64, "lognormal"), (2, 64, "ties"), (1, 512, "lognormal"),
                                      (4, 512, "zero_heads"), (2, 2048, "lognormal"), (1, 1000, "ties")])
@pytest.mark.parametrize("with_eta", [False, True])
def test_selector_bit_exact(B, C, kind, with_eta):
    seed = 31 * B + C
    score = gdn_synth.make_scores(B, 32, C, seed, kind)
    g = gdn_synth.make_gates(B, 64 * C, 32, seed)
    eta = None
    if with_eta:
        eta = np.abs(np.random.default_rng(seed).standard_normal((B, 32))).astype(np.float32)
        eta[:, 5] = 0.0
    mask, tier = gpu_select(score, g, eta)
    ref = oracle.select(score, chunk_gamma(g, C), eta)
    assert np.array_equal(tier, ref["tier"]), f"tiers {tier} != {ref['tier']}"
    assert np.array_equal(mask, ref["mask"]), f"{np.count_nonzero(mask != ref['mask'])} mask bytes differ"


@pytest.mark.parametrize("name", ["window", "sum_from_one", "closed_form"])
def test_selector_memory_lifetime_cases(name):
    # inputs whose tier split is decided by Eq. 11's memory lifetime (r_h over the last 16 chunks,
    # L_h summed from j = 1): the GPU's tiers and mask equal the expected split and the oracle's
    from selector_cases import CASES
    score, gamma, tiers = CASES[name]()
    C = score.shape[-1]
    g = np.ascontiguousarray(np.repeat(np.moveaxis(gamma, 1, 2), 64, axis=1))  # [1, 64 C, 32]: g = gamma per chunk
    mask, tier = gpu_select(score, g)
    ref = oracle.select(score, chunk_gamma(g, C))
    assert tier[0].tolist() == tiers.tolist()
    assert np.array_equal(tier, ref["tier"]) and np.array_equal(mask, ref["mask"])


def test_selector_all_zero_scores_and_eta():
    score = np.zeros((2, 32, 40), np.float32)
    g = gdn_synth.make_gates(2, 64 * 40, 32, 5)
    eta = np.zeros((2, 32), np.float32)
    for e in (None, eta):
        mask, tier = gpu_select(score, g, e)
        ref = oracle.select(score, chunk_gamma(g, 40), e)
        assert np.array_equal(tier, ref["tier"]) and np.array_equal(mask, ref["mask"])


def test_selector_rejects_other_head_counts():
    score = torch.zeros((1, 4, 8), device=dev())
    g = torch.zeros((1, 512, 4), device=dev())
    with pytest.raises(gdn.GdnError) as ei:
        gdn.gdn_select_events_scored(score, g)
    assert ei.value.status == 6


def run_online(x, solver="block_adj", eta=None):
    t = to_dev(x)
    sc = torch.full((x.B, x.Nv, x.C), -1.0, device=dev())
    et = None if eta is None else torch.from_numpy(eta).to(dev())
    o, s, mask, tier = gdn.gdn_prefill_sparse_online(t["q"], t["k"], t["v"], t["beta"], t["g"], h0=t["h0"],
                                                     eta=et, solver=solver, score=sc)
    torch.cuda.synchronize()
    return {"o": o.float().cpu().numpy().astype(np.float64), "s_final": s.cpu().numpy().astype(np.float64),
            "score": sc.cpu().numpy(), "mask": mask.cpu().numpy(), "tier": tier.cpu().numpy()}


def check_selection(x, res, eta=None):
    ref = oracle.select(res["score"], chunk_gamma(x.g, x.C), eta)
    assert np.array_equal(res["tier"], ref["tier"])
    assert np.array_equal(res["mask"], ref["mask"])


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("solver", ["exact", "block_adj"])
def test_online_prefill_small(dtype, solver):
    # 2 sequences x 16 head pairs x 23 chunks (odd: the last group has one chunk), with h0
    x = gdn_synth.make_inputs(2, 23 * 64, 16, 32, dtype=dtype, seed=41, mask="ones", with_h0=True)
    res = run_online(x, solver)
    ref = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=res["mask"], h0=x.h0,
                         solver={"exact": oracle.SOLVER_EXACT, "block_adj": oracle.SOLVER_BLOCK_ADJ}[solver],
                         debug=True)
    rel = np.abs(res["score"] - ref["score"]) / np.maximum(ref["score"], 1e-30)
    assert rel.max() <= TOL[dtype]
    check_selection(x, res)
    assert_close(res, ref, dtype, f"online {dtype} {solver}")


def test_online_prefill_with_eta():
    x = gdn_synth.make_inputs(1, 40 * 64, 16, 32, dtype="bf16", seed=42, mask="ones")
    eta = np.abs(np.random.default_rng(42).standard_normal((1, 32))).astype(np.float32)
    res = run_online(x, eta=eta)
    check_selection(x, res, eta)
    ref = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=res["mask"], solver=oracle.SOLVER_BLOCK_ADJ)
    assert_close(res, ref, "bf16", "online with eta")


def test_online_layer_T32768_sampled_pairs():
    x = gdn_synth.make_workload("qwen35_4b_layer_T32768_sparse29")
    res = run_online(x)
    check_selection(x, res)
    # the selection keeps the tier budget: retention in [0.08, 0.95], the high tier 1..4 pairs
    ret = res["mask"].mean()
    assert 0.08 <= ret <= 0.95
    assert 1 <= (res["tier"] == 2).sum() <= 4
    for p in (int(np.argmax(res["mask"][0].sum(-1))), int(np.argmin(res["mask"][0].sum(-1)))):
        y = slice_pairs(x, 0, [p])
        ref = oracle.prefill(y.q, y.k, y.v, y.beta, y.g, mask=res["mask"][:, p:p + 1], h0=None,
                             solver=oracle.SOLVER_BLOCK_ADJ)
        got = {"o": res["o"][:, :, 2 * p:2 * p + 2], "s_final": res["s_final"][:, 2 * p:2 * p + 2]}
        assert_close(got, ref, "bf16", f"online T=32768 pair {p}")


@pytest.mark.parametrize("solver", ["exact", "block_adj"])
def test_online_matches_given_mask_path_bitwise(solver):
    # the prefill with the selected mask handed in computes the same thing: W built after the
    # selection from the stored bf16 C-bar blocks equals W built inside the intra step bit for bit
    x = gdn_synth.make_inputs(1, 4096, 16, 32, dtype="bf16", seed=43, mask="ones")
    t = to_dev(x)
    o1, s1, mask, _ = gdn.gdn_prefill_sparse_online(t["q"], t["k"], t["v"], t["beta"], t["g"], solver=solver)
    o2, s2 = gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], mask.clone(), solver=solver)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


def test_online_prefill_ragged_T():
    # 23 full chunks and a 5-token partial chunk
    x = gdn_synth.make_inputs(1, 23 * 64 + 5, 16, 32, dtype="bf16", seed=44, mask="ones")
    res = run_online(x)
    check_selection(x, res)
    ref = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=res["mask"], solver=oracle.SOLVER_BLOCK_ADJ)
    assert_close(res, ref, "bf16", "online ragged T")


@pytest.mark.parametrize("world", [1, 2, 4])
def test_online_selection_split_over_pair_blocks(world):
    # online selection in two calls per rank (gated_delta_rule_16_gb300.sharded with the library as
    # backend), the ranks emulated one after the other on this GPU (no kernel waits for another
    # rank's): gathered scores and gate tails, one selection, each rank's block finished with its
    # mask rows.  Equal, bit for bit, to the one-call online prefill of the whole layer.
    from gated_delta_rule_16_gb300 import sharded
    x = gdn_synth.make_inputs(2, 23 * 64 + 5, 16, 32, dtype="bf16", seed=45, mask="ones", with_h0=True)
    t = to_dev(x)
    eta = torch.from_numpy(np.abs(np.random.default_rng(45).standard_normal((2, 32))).astype(np.float32)).to(dev())
    o_ref, s_ref, m_ref, tier_ref = gdn.gdn_prefill_sparse_online(t["q"], t["k"], t["v"], t["beta"], t["g"],
                                                                  h0=t["h0"], eta=eta)
    full = {"q": t["q"], "k": t["k"], "v": t["v"], "beta": t["beta"], "g": t["g"], "h0": t["h0"], "eta": eta}
    be = sharded.CudaBackend()
    xs = [sharded.shard(full, r, world) for r in range(world)]
    first = [be.scores(xr) for xr in xs]
    score_all = torch.cat([f[0] for f in first], dim=1)
    gamma_all = torch.cat([sharded.chunk_gamma(xr["g"]) for xr in xs], dim=1)
    mask_all, tier_all = be.select(score_all, gamma_all, eta)
    outs = []
    for r, xr in enumerate(xs):
        p0, p1 = sharded.pair_block(r, world, 16)
        outs.append(be.finish(xr, first[r][1], mask_all[:, p0:p1]))
    torch.cuda.synchronize()
    assert torch.equal(mask_all, m_ref) and torch.equal(tier_all, tier_ref)
    assert torch.equal(torch.cat([o for o, _ in outs], dim=2), o_ref)
    assert torch.equal(torch.cat([s for _, s in outs], dim=1), s_ref)
