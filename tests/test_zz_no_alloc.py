"""gdn_prefill_sparse_noalloc: the entry point for callers that cannot allocate.

Callers such as a plugin inside a host runtime that owns all device memory, or
a server that forbids cudaMalloc after start-up, get a prefill whose scratch is
the library's own fixed device array.  These checks call it through the C ABI
and compare it with gdn_prefill_sparse (caller workspace): the two run the same
kernels on the same inputs, so their outputs must agree bit for bit.  Calls
follow each other with different inputs and shapes (one at the 64 MiB limit,
then smaller ones), so a stale scratch from an earlier call would show up, and
the allocation-free status word is read after every call.  This file is
collected last on purpose.
"""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, max_rel_err, to_dev

import gated_delta_rule_16_gb300 as gdn
from gated_delta_rule_16_gb300 import _binding as bnd

pytestmark = pytest.mark.gpu

LIMIT = 64 << 20


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gated_delta_rule_16_gb300 import build
    build.build()
    gdn.load()


def _run_both(x, solver):
    t = to_dev(x)
    ref_o, ref_s = gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"], h0=t["h0"],
                                          solver=solver, workspace=gdn.Workspace())
    o = torch.full_like(ref_o, float("nan"))
    s = torch.full_like(ref_s, float("nan"))
    gdn.gdn_prefill_sparse_noalloc(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"], h0=t["h0"],
                                   solver=solver, o=o, s_final=s)
    assert gdn.gdn_noalloc_status() == 0  # synchronises; nothing latched (no timeout, no capacity overflow)
    return (o, s), (ref_o, ref_s)


def _largest_T(Nq, dtype):
    code = bnd.GDN_BF16 if dtype == "bf16" else bnd.GDN_F32
    fits = lambda T: gdn.gdn_workspace_bytes(bnd.GdnShape(1, T, Nq, 2 * Nq, 128, 128, code), "block_adj", 1) <= LIMIT
    T = 64
    while fits(T + 64):
        T += 64
    return T


@pytest.mark.parametrize("dtype,Nq", [("bf16", 16), ("f32", 2)])
def test_noalloc_equals_workspace_path_over_calls(dtype, Nq):
    T_max = _largest_T(Nq, dtype)
    # at the limit, then smaller shapes (the scratch layout moves with C, R and the snapshot count)
    for call, (B, T, seed) in enumerate(((1, T_max, 41), (1, 1024 + 37, 42), (2, 448, 43))):
        x = gdn_synth.make_inputs(B, T, Nq, 2 * Nq, dtype=dtype, seed=seed, mask="beta", with_h0=(call == 1))
        (o, s), (ref_o, ref_s) = _run_both(x, "block_adj")
        assert torch.equal(o, ref_o), f"call {call} (T={T}): O differs from the workspace path"
        assert torch.equal(s, ref_s), f"call {call} (T={T}): S_final differs from the workspace path"


def test_noalloc_matches_the_oracle():
    x = gdn_synth.make_inputs(1, 512 + 37, 2, 4, dtype="bf16", seed=44, mask="beta", with_h0=True)
    (o, s), _ = _run_both(x, "block_adj")
    ref = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=x.mask, h0=x.h0, solver=oracle.SOLVER_BLOCK_ADJ)
    for got, want, kind in ((o, ref["o"], "o"), (s, ref["s_final"], "s")):
        rel, ab = max_rel_err(got.float().cpu().numpy().astype(np.float64), want, kind)
        assert rel <= TOL["bf16"] and ab <= 1e-6, f"{kind}: {rel:.3e}"


def test_noalloc_rejects_shapes_over_the_limit():
    # needs more than the 64 MiB scratch: rejected on the host, nothing enqueued
    shape = bnd.GdnShape(1, 4096, 16, 32, 128, 128, bnd.GDN_BF16)
    assert gdn.gdn_workspace_bytes(shape, "block_adj", True) > LIMIT
    x = gdn_synth.make_inputs(1, 4096, 16, 32, dtype="bf16", seed=45, mask="beta")
    t = to_dev(x)
    with pytest.raises(bnd.GdnError) as err:
        gdn.gdn_prefill_sparse_noalloc(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"])
    assert err.value.status == 5  # GDN_ERR_WORKSPACE
