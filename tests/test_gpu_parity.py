"""Parity of the CUDA path (through the C ABI) with the CPU fp64 oracle.

Element-by-element comparisons on seeded inputs at sizes the oracle finishes
in seconds (several chunks, groups, pairs, sequences, and an odd chunk count),
plus the full-size sparse layer (T = 32768) and two layers of the 128K-token
prefill on every head pair, and the eight-sequence batch on sampled pairs.
Errors are bounded per (sequence, value head) and per 64-token chunk of O.
CSR event lists are compared bit for bit.
"""
import itertools

import numpy as np
import pytest
import torch

import gdn_synth
import oracle
from gpu_helpers import TOL, assert_close, dev, max_rel_err, run_gpu, slice_pairs, to_dev

import gated_delta_rule_16_gb300 as gdn

pytestmark = pytest.mark.gpu

SOLVER = {"exact": oracle.SOLVER_EXACT, "block_adj": oracle.SOLVER_BLOCK_ADJ}


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from gated_delta_rule_16_gb300 import build
    build.build()
    gdn.load()


def oracle_run(x, solver, sparse=True, mask=None, h0="inputs", debug=False):
    m = (x.mask if mask is None else mask) if sparse else None
    h = x.h0 if isinstance(h0, str) else h0
    return oracle.prefill(x.q, x.k, x.v, x.beta, x.g, mask=m, h0=h, solver=SOLVER[solver], debug=debug)


# ------------------------------------------------------------- tiny fp32 ---

@pytest.mark.parametrize("solver", ["exact", "block_adj"])
@pytest.mark.parametrize("sparse", [True, False])
def test_tiny_fp32(solver, sparse):
    x = gdn_synth.make_workload("tiny_fp32_T256")
    res = run_gpu(x, solver=solver, sparse=sparse)
    assert_close(res, oracle_run(x, solver, sparse), "f32", f"tiny {solver} sparse={sparse}")


@pytest.mark.parametrize("solver", ["exact", "block_adj"])
def test_tiny_fp32_all_16_masks(solver):
    x = gdn_synth.make_workload("tiny_fp32_T256", with_h0=True)
    for bits in itertools.product([0, 1], repeat=4):
        m = np.array(bits, np.uint8).reshape(1, 1, 4)
        for h0 in (None, x.h0):
            res = run_gpu(x, solver=solver, mask=m, h0=h0 if h0 is not None else np.zeros_like(x.h0))
            ref = oracle_run(x, solver, mask=m, h0=h0)
            assert_close(res, ref, "f32", f"mask {bits} h0={h0 is not None}")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ragged_groups_batch_and_h0(dtype):
    # 5 chunks (last group has one chunk), 3 pairs, 2 sequences, random masks and an initial state
    x = gdn_synth.make_inputs(2, 320, 3, 6, dtype=dtype, seed=21, mask="bernoulli", retention=0.5, with_h0=True)
    for solver in ("exact", "block_adj"):
        res = run_gpu(x, solver=solver, score=True)
        ref = oracle_run(x, solver, debug=True)
        assert_close(res, ref, dtype, f"ragged {dtype} {solver}")
        rel = np.abs(res["score"] - ref["score"]) / np.maximum(ref["score"], 1e-30)
        assert rel.max() <= TOL[dtype]


def test_single_chunk_and_empty_sequence():
    x = gdn_synth.make_inputs(1, 64, 2, 4, dtype="f32", seed=22, mask="ones", with_h0=True)
    for sparse in (True, False):
        assert_close(run_gpu(x, sparse=sparse), oracle_run(x, "block_adj", sparse), "f32", "T=64")
    # T = 0: the final state is the initial state
    t = to_dev(x)
    e = lambda *s: torch.empty(*s, device=dev())
    q = e((1, 0, 2, 128)); v = e((1, 0, 4, 128)); bg = e((1, 0, 4))
    o, s = gdn.gdn_prefill_dense(q, q, v, bg, bg, h0=t["h0"])
    torch.cuda.synchronize()
    assert torch.equal(s, t["h0"])
    o, s = gdn.gdn_prefill_dense(q, q, v, bg, bg)
    torch.cuda.synchronize()
    assert torch.count_nonzero(s).item() == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_all_zero_mask_decay_only(dtype):
    x = gdn_synth.make_inputs(1, 512, 2, 4, dtype=dtype, seed=23, mask="zeros", with_h0=True)
    assert_close(run_gpu(x), oracle_run(x, "block_adj"), dtype, "zero mask with h0")
    r = run_gpu(x, h0=np.zeros_like(x.h0))
    assert np.count_nonzero(r["s_final"]) == 0


def test_all_ones_sparse_equals_dense_bitwise():
    x = gdn_synth.make_inputs(1, 512, 2, 4, dtype="bf16", seed=24, mask="ones")
    for solver in ("exact", "block_adj"):
        a = run_gpu(x, solver=solver, sparse=True)
        b = run_gpu(x, solver=solver, sparse=False)
        assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["s_final"], b["s_final"])


@pytest.mark.parametrize("scale", [20.0, 100.0])
def test_strong_decay(scale):
    # Gates scaled so that the decay over a run of chunks passes 2^-64: the tensor-core scan then
    # applies decays to its TMEM state and restarts the state's scale inside runs (scale 20: about
    # every second event chunk; scale 100: every event).  Scale 100 (about -160 log2 decay per chunk)
    # also sends the output's decay mask to its per-element path (a two-chunk range above 200).
    x = gdn_synth.make_inputs(1, 4096, 2, 4, dtype="bf16", seed=73, mask="bernoulli", retention=0.5,
                              with_h0=True)
    x.g = (x.g.astype(np.float64) * scale).astype(np.float32)
    for solver in ("block_adj", "exact"):
        res = run_gpu(x, solver=solver)
        assert_close(res, oracle_run(x, solver), "bf16", f"gates x{scale} {solver}")


# ----------------------------------------------------------------- CSR ---

@pytest.mark.parametrize("shape,p", [((1, 1, 4), 0.5), ((2, 3, 7), 0.4), ((3, 16, 33), 0.29),
                                     ((1, 16, 512), 0.29), ((8, 16, 512), 0.29), ((2, 3, 6), 1.0),
                                     ((2, 3, 6), 0.0), ((1, 16, 2048), 0.1), ((4, 5, 1), 0.5),
                                     ((1, 16, 16384), 0.002), ((2, 16, 10000), 0.05), ((64, 16, 1024), 0.29)])
def test_csr_bit_exact(shape, p):
    # the last case is too large for the word-parallel compaction and takes the row-per-warp kernel
    rng = np.random.default_rng(sum(shape))
    m = (rng.random(shape) < p).astype(np.uint8)
    ev = gdn.gdn_select_events(torch.from_numpy(m).to(dev()))
    assert gdn.gdn_events_status(ev) == 0
    ref = oracle.events(m)
    E = ref["n_events"]
    counts = ev["counts"].cpu().numpy()
    assert counts[0] == E and counts[1] == ref["n_snap"] and counts[2] == 0
    B, P, C = shape
    assert np.array_equal(ev["row_pair"].cpu().numpy()[:B * P], ref["row_pair"])
    assert np.array_equal(ev["row_ptr"].cpu().numpy(), ref["row_ptr"])
    assert np.array_equal(ev["ev_chunk"].cpu().numpy()[:E], ref["ev_chunk"])
    assert np.array_equal(ev["grp_pred"].cpu().numpy()[:B * P * ((C + 1) // 2)], ref["grp_pred"].ravel())
    assert np.array_equal(ev["snap_slot"].cpu().numpy()[:E], ref["snap_slot"])


def test_csr_all_16_masks():
    for bits in itertools.product([0, 1], repeat=4):
        m = np.array(bits, np.uint8).reshape(1, 1, 4)
        ev = gdn.gdn_select_events(torch.from_numpy(m).to(dev()))
        ref = oracle.events(m)
        E = ref["n_events"]
        assert np.array_equal(ev["ev_chunk"].cpu().numpy()[:E], ref["ev_chunk"])
        assert np.array_equal(ev["grp_pred"].cpu().numpy()[:2], ref["grp_pred"].ravel())
        assert np.array_equal(ev["snap_slot"].cpu().numpy()[:E], ref["snap_slot"])


def test_csr_capacity_overflow_latched():
    m = np.ones((1, 2, 8), np.uint8)
    ev = gdn.gdn_select_events(torch.from_numpy(m).to(dev()), capacity=5)
    assert gdn.gdn_events_status(ev) == 9
    assert ev["counts"][0].item() == 16


# ------------------------------------------------------- layer-sized bf16 ---

@pytest.mark.parametrize("solver", ["exact", "block_adj"])
def test_dense_layer_T4096(solver):
    x = gdn_synth.make_workload("qwen35_4b_layer_T4096_dense")
    res = run_gpu(x, solver=solver, sparse=False)
    assert_close(res, oracle_run(x, solver, sparse=False), "bf16", f"T=4096 dense {solver}")


def test_sparse_layer_T32768_all_pairs():
    # the benchmark's layer, every head pair (all 32 value heads) against the oracle
    x = gdn_synth.make_workload("qwen35_4b_layer_T32768_sparse29")
    res = run_gpu(x, solver="block_adj")
    assert_close(res, oracle_run(x, "block_adj"), "bf16", "T=32768 all pairs")


@pytest.mark.parametrize("scan_runs", [False, True])
def test_sparse_layer_T32768_scan_variants_sampled(scan_runs):
    # both event-scan schedules (one pass per row / run maps + chain + fix-up) on the longest and
    # the shortest row
    x = gdn_synth.make_workload("qwen35_4b_layer_T32768_sparse29")
    t = to_dev(x)
    o, s, _, _ = gdn.gdn_prefill_ex(t["q"], t["k"], t["v"], t["beta"], t["g"], mode="sparse", mask=t["mask"],
                                    solver="block_adj", scan_runs=scan_runs)
    torch.cuda.synchronize()
    counts = x.mask[0].sum(-1)
    for p in (int(np.argmax(counts)), int(np.argmin(counts))):
        y = slice_pairs(x, 0, [p])
        got = {"o": o[:, :, 2 * p:2 * p + 2].float().cpu().numpy().astype(np.float64),
               "s_final": s[:, 2 * p:2 * p + 2].cpu().numpy().astype(np.float64)}
        assert_close(got, oracle_run(y, "block_adj"), "bf16", f"scan_runs={scan_runs} pair {p}")


def test_batch8_T32768_sampled_pairs():
    # eight sequences with their own masks; two head pairs of every sequence
    x = gdn_synth.make_workload("qwen35_4b_layer_B8_T32768_sparse29")
    res = run_gpu(x, solver="block_adj")
    for b in range(8):
        pairs = [(3 * b) % 16, (3 * b + 8) % 16]
        y = slice_pairs(x, b, pairs)
        ref = oracle_run(y, "block_adj")
        vi = [2 * p + j for p in pairs for j in (0, 1)]
        got = {"o": res["o"][b:b + 1][:, :, vi], "s_final": res["s_final"][b:b + 1][:, vi]}
        assert_close(got, ref, "bf16", f"B=8 seq {b} pairs {pairs}")


def test_workspace_status_ok_after_prefill():
    x = gdn_synth.make_inputs(1, 256, 1, 2, dtype="bf16", seed=25, mask="two_of_four")
    ws = gdn.Workspace()
    run_gpu(x, workspace=ws)
    assert gdn.gdn_workspace_status(ws) == 0


def test_bounded_wait_times_out_and_context_survives():
    # a barrier nothing arrives at: the wait must give up after its limit and latch the bit
    rc, waited_ms, bits = gdn.gdn_selftest_wait_timeout(50)
    assert rc == 0 and bits & 4 and 50 <= waited_ms < 2000
    # the context is still usable: a prefill right after runs and matches the oracle
    x = gdn_synth.make_workload("tiny_fp32_T256")
    assert_close(run_gpu(x), oracle_run(x, "block_adj"), "f32", "after timeout self-test")


@pytest.mark.parametrize("layer", [0, 23])
def test_long_context_T131072_layer_all_pairs(layer):
    # one layer of the 24-layer, 128K-token prefill: output and final state of every head pair
    x = gdn_synth.make_workload("qwen35_4b_24layers_T131072_sparse29", layer=layer)
    res = run_gpu(x, solver="block_adj")
    assert_close(res, oracle_run(x, "block_adj"), "bf16", f"T=131072 layer {layer}")


def test_long_context_24_layers_every_layer_sampled_pair():
    # the 24-layer, 128K-token prefill as the benchmark runs it (inputs drawn on the GPU, layers
    # back to back on one workspace): every layer's output and final state on one sampled head
    # pair, against the oracle run on that pair's inputs (all 24 pairs as one batch of sequences)
    L, T = 24, 131072
    ws = gdn.Workspace()
    qs, ks, vs, bs, gs, ms, os_, ss = [], [], [], [], [], [], [], []
    for layer in range(L):
        t = gdn_synth.make_layer_on_device(1, T, 16, 32, gdn_synth.seed_for(3, layer), dev())
        o, s = gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"], solver="block_adj",
                                      workspace=ws)
        p = (7 * layer + 3) % 16
        hv = [2 * p, 2 * p + 1]
        f64 = lambda a: a.float().cpu().numpy().astype(np.float64)
        qs.append(f64(t["q"][:, :, p:p + 1])); ks.append(f64(t["k"][:, :, p:p + 1]))
        vs.append(f64(t["v"][:, :, hv])); bs.append(f64(t["beta"][:, :, hv])); gs.append(f64(t["g"][:, :, hv]))
        ms.append(t["mask"][:, p:p + 1].cpu().numpy())
        os_.append(f64(o[:, :, hv])); ss.append(s[:, hv].cpu().numpy().astype(np.float64))
        del t, o, s
    assert gdn.gdn_workspace_status(ws) == 0
    cat = lambda a: np.concatenate(a, axis=0)
    ref = oracle.prefill(cat(qs), cat(ks), cat(vs), cat(bs), cat(gs), mask=cat(ms), solver=oracle.SOLVER_BLOCK_ADJ)
    assert_close({"o": cat(os_), "s_final": cat(ss)}, ref, "bf16", "24 layers x T=131072")


@pytest.mark.parametrize("sparse", [True, False])
@pytest.mark.parametrize("T1", [128, 1024 + 128])
def test_chunked_prefill_resume(sparse, T1):
    # prefill(T1) then prefill(rest, h0 = its S_final) equals prefill(T1 + rest): T1 a multiple of
    # 128, so both halves keep the two-chunk groups of the whole (the pages return S_C for later use)
    x = gdn_synth.make_inputs(2, 2048 + 37, 4, 8, dtype="bf16", seed=30 + T1, mask="beta", with_h0=True)
    whole = run_gpu(x, solver="block_adj", sparse=sparse)
    ref = oracle_run(x, "block_adj", sparse)
    assert_close(whole, ref, "bf16", "whole")
    C1 = T1 // 64
    first, second = slice_tokens(x, 0, T1), slice_tokens(x, T1, x.T)
    first.mask, second.mask = x.mask[:, :, :C1], x.mask[:, :, C1:]
    r1 = run_gpu(first, solver="block_adj", sparse=sparse)
    r2 = run_gpu(second, solver="block_adj", sparse=sparse, h0=r1["s_final"].astype(np.float32))
    joined = {"o": np.concatenate([r1["o"], r2["o"]], axis=1), "s_final": r2["s_final"]}
    assert_close(joined, ref, "bf16", f"resumed at T1={T1}")
    assert_close(joined, whole, "bf16", f"resumed vs whole at T1={T1}")


def slice_tokens(x, t0, t1):
    """Inputs restricted to tokens [t0, t1) of every sequence (h0 kept)."""
    import copy
    y = copy.copy(x)
    y.q, y.k, y.v = x.q[:, t0:t1], x.k[:, t0:t1], x.v[:, t0:t1]
    y.beta, y.g = x.beta[:, t0:t1], x.g[:, t0:t1]
    y.T = t1 - t0
    return y


@pytest.mark.parametrize("dtype,sparse", [("bf16", True), ("bf16", False), ("f32", True)])
def test_host_buffer_prefill_equals_device_path(dtype, sparse):
    # gdn_prefill_host: the same kernels behind host copies, so the same bits
    x = gdn_synth.make_inputs(2, 640, 16, 32, dtype=dtype, seed=26, mask="beta", with_h0=True)
    res = run_gpu(x, sparse=sparse)
    st = torch.bfloat16 if dtype == "bf16" else torch.float32
    h = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dt).pin_memory()
    stream = torch.cuda.Stream()
    o, s = gdn.gdn_prefill_host(h(x.q, st), h(x.k, st), h(x.v, st), h(x.beta, torch.float32),
                                h(x.g, torch.float32), h(x.mask, torch.uint8) if sparse else None,
                                h0=h(x.h0, torch.float32), stream=stream)
    stream.synchronize()
    assert np.array_equal(o.float().numpy().astype(np.float64), res["o"])
    assert np.array_equal(s.numpy().astype(np.float64), res["s_final"])


# ------------------------------------------------- partial last chunk (ragged T) ---

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T", [100, 150, 337])
def test_ragged_T_partial_last_chunk(dtype, T):
    # two sequences (the partial chunk of the first must not touch the second), 3 pairs, h0,
    # random masks; C = ceil(T / 64)
    x = gdn_synth.make_inputs(2, T, 3, 6, dtype=dtype, seed=27 + T, mask="bernoulli", retention=0.6,
                              with_h0=True)
    for solver in ("exact", "block_adj"):
        for sparse in (True, False):
            res = run_gpu(x, solver=solver, sparse=sparse, score=True)
            ref = oracle_run(x, solver, sparse, debug=True)
            assert_close(res, ref, dtype, f"T={T} {dtype} {solver} sparse={sparse}")
            rel = np.abs(res["score"] - ref["score"]) / np.maximum(ref["score"], 1e-30)
            assert rel.max() <= TOL[dtype]


def test_ragged_T_qwen_layer_sampled_pairs():
    # one Qwen3.5-4B-shaped layer with a ragged tail, two sequences, 29% events
    x = gdn_synth.make_inputs(2, 4096 + 37, 16, 32, dtype="bf16", seed=28, mask="beta")
    res = run_gpu(x, solver="block_adj")
    for b, p in ((0, 5), (1, 12)):
        y = slice_pairs(x, b, [p])
        ref = oracle_run(y, "block_adj")
        got = {"o": res["o"][b:b + 1, :, 2 * p:2 * p + 2], "s_final": res["s_final"][b:b + 1, 2 * p:2 * p + 2]}
        assert_close(got, ref, "bf16", f"ragged layer seq {b} pair {p}")


def test_maximum_chunk_count_one_pair():
    # the largest sequence the boundary accepts: C = 16384 chunks (T = 1,048,576), one head pair,
    # 29% events and an initial state: 1024 scan runs per row (the chain's limit), the compaction's
    # largest mask staging; compared with the oracle on every token and the final state
    x = gdn_synth.make_inputs(1, 64 * 16384, 1, 2, dtype="bf16", seed=29, mask="beta", with_h0=True)
    res = run_gpu(x, solver="block_adj")
    ref = oracle_run(x, "block_adj")
    assert_close(res, ref, "bf16", "C=16384")
