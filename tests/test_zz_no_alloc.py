"""gdn_prefill_sparse_noalloc: the entry point for callers that cannot allocate.

Callers such as a plugin inside a host runtime that owns all device memory, or
a server that forbids cudaMalloc after start-up, get a prefill whose scratch is
the library's own fixed device array.  These checks call it through the C ABI
and compare it with gdn_prefill_sparse (caller workspace) on two calls in a
row with different inputs, so a stale scratch from the first call would show
up in the second.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import gdn_synth
from gpu_helpers import TOL, max_rel_err, to_dev

import gated_delta_rule_16_gb300 as gdn
from gated_delta_rule_16_gb300 import _binding as bnd

pytestmark = pytest.mark.gpu


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
    torch.cuda.synchronize()
    return ({"o": o.float().cpu().numpy(), "s_final": s.cpu().numpy()},
            {"o": ref_o.float().cpu().numpy(), "s_final": ref_s.cpu().numpy()})


@pytest.mark.parametrize("dtype,shape", [("bf16", (1, 1024, 16)), ("f32", (2, 448, 2))])
def test_noalloc_matches_workspace_path_two_calls(dtype, shape):
    B, T, Nq = shape
    for call, seed in enumerate((41, 42)):
        x = gdn_synth.make_inputs(B, T, Nq, 2 * Nq, dtype=dtype, seed=seed, mask="beta", with_h0=(call == 1))
        got, want = _run_both(x, "block_adj")
        for key, kind in (("o", "o"), ("s_final", "s")):
            assert np.isfinite(got[key]).all(), f"call {call}: {key} not fully written"
            rel, ab = max_rel_err(got[key].astype(np.float64), want[key].astype(np.float64), kind)
            assert rel <= TOL[dtype] and ab <= 1e-6, f"call {call} {key}: {rel:.3e}"


def test_noalloc_rejects_shapes_over_the_limit():
    # needs more than the 64 MiB scratch: rejected on the host, nothing enqueued
    shape = bnd.GdnShape(1, 4096, 16, 32, 128, 128, bnd.GDN_BF16)
    assert gdn.gdn_workspace_bytes(shape, "block_adj", True) > (64 << 20)
    x = gdn_synth.make_inputs(1, 4096, 16, 32, dtype="bf16", seed=43, mask="beta")
    t = to_dev(x)
    with pytest.raises(bnd.GdnError) as err:
        gdn.gdn_prefill_sparse_noalloc(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"])
    assert err.value.status == 5  # GDN_ERR_WORKSPACE
