"""Parity of the single-token decode step (gdn_decode_step) with the oracle.

One step on random states, both storage dtypes, is compared element-wise with
the oracle's step; then the serving pattern end to end: a GPU prefill of T
tokens followed by 64 GPU decode steps against the oracle's prefill of T + 64
tokens (independent formulations: chunkwise vs one token at a time).
"""
import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, dev, max_rel_err

import gated_delta_rule_16_gb300 as gdn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gated_delta_rule_16_gb300 import build
    build.build()
    gdn.load()


def token_gates(g):
    g = np.asarray(g, dtype=np.float64)
    a = g.copy()
    a[:, 1:] -= g[:, :-1]
    a[:, ::64] = g[:, ::64]
    return a.astype(np.float32)


def to(a, dt):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev()).to(dt)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_step_random_state(dtype):
    x = gdn_synth.make_inputs(3, 64, 2, 4, dtype=dtype, seed=61, mask="ones", with_h0=True)
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    a = token_gates(x.g)
    t = 17
    S = to(x.h0, torch.float32)
    o = gdn.gdn_decode_step(to(x.q[:, t], st), to(x.k[:, t], st), to(x.v[:, t], st), to(x.beta[:, t], torch.float32),
                            to(a[:, t], torch.float32), S)
    torch.cuda.synchronize()
    ref = oracle.decode(x.q[:, t], x.k[:, t], x.v[:, t], x.beta[:, t], a[:, t], x.h0)
    rs, _ = max_rel_err(S.cpu().numpy().astype(np.float64), ref["s"], "s")
    assert rs <= 1e-5
    got_o = o.float().cpu().numpy()
    err = np.linalg.norm(got_o - ref["o"], axis=-1) / np.linalg.norm(ref["o"], axis=-1)
    assert err.max() <= (1e-5 if dtype == "f32" else 8e-3)


def test_prefill_then_decode_matches_longer_prefill():
    # one Qwen3.5-4B-shaped layer: prefill 4096 tokens on the GPU, decode 64 more one at a time
    x = gdn_synth.make_inputs(1, 4160, 16, 32, dtype="bf16", seed=62, mask="ones")
    T0 = 4096
    bf = torch.bfloat16
    q, k, v = to(x.q, bf), to(x.k, bf), to(x.v, bf)
    beta, g = to(x.beta, torch.float32), to(x.g, torch.float32)
    _, S = gdn.gdn_prefill_dense(q[:, :T0].contiguous(), k[:, :T0].contiguous(), v[:, :T0].contiguous(),
                                 beta[:, :T0].contiguous(), g[:, :T0].contiguous(), solver="exact")
    a = to(token_gates(x.g), torch.float32)
    outs = []
    for t in range(T0, T0 + 64):
        outs.append(gdn.gdn_decode_step(q[:, t].contiguous(), k[:, t].contiguous(), v[:, t].contiguous(),
                                        beta[:, t].contiguous(), a[:, t].contiguous(), S).float())
    torch.cuda.synchronize()
    o_dec = torch.stack(outs, dim=1).cpu().numpy().astype(np.float64)  # [1, 64, Nv, dv]
    ref = oracle.prefill(x.q, x.k, x.v, x.beta, x.g, solver=oracle.SOLVER_EXACT)
    ro, _ = max_rel_err(o_dec, ref["o"][:, T0:], "o")
    rs, _ = max_rel_err(S.cpu().numpy().astype(np.float64), ref["s_final"], "s")
    assert ro <= TOL["bf16"] and rs <= TOL["bf16"], (ro, rs)
