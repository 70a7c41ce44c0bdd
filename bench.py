#!/usr/bin/env python3
"""GDN-core prefill throughput on one GB300: tokens/s per layer and % of roofline.

One step = one pass of the whole hot path over one synthetic layer: mask ->
CSR compaction, log-decay prefix, intra-chunk solve, deferred W, event scan and
group output, all in libgdn's CUDA kernels through the C ABI.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline]

Default workload: one Qwen3.5-4B-shaped GDN layer, B=1, T=32768, N_q=16,
N_v=32, d=d_v=128, bf16, event-sparse path at 29% retention (Beta(2,5)
per-pair budgets), block-adjacent solver.  Under torchrun every rank runs its
own independent sequence (weak scaling, no collective on the data path).

--impl reference times the CPU fp64 oracle (the only reference there is)
on a bounded sample of the same workload, on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "GDN-core prefill tokens/s per layer at T=32K, 29% events; % of roofline"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0


# DRAM bytes (read + write) of one launch, measured with ncu (dram__bytes_read.sum +
# dram__bytes_write.sum) on the current version of each kernel and workload (all launches of
# one prefill summed per kernel); an entry must be removed whenever its kernel changes (the
# traffic is then reported as null).
PROFILED_TRAFFIC = {
    ("qwen35_4b_layer_T32768_sparse29", "select"): 0.09e6,
    ("qwen35_4b_layer_T32768_sparse29", "prefix"): 0.14e6,
    ("qwen35_4b_layer_T32768_sparse29", "intra"): 609.1e6,
    ("qwen35_4b_layer_T32768_sparse29", "scan"): 242.0e6,
    ("qwen35_4b_layer_T32768_sparse29", "output"): 837.1e6,
}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen35_4b_layer_T32768_sparse29")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=0,
                    help="steps of the end-to-end (host-buffer) timing; 0: the same as --steps")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' timings")
    ap.add_argument("--shard", choices=["pairs", "sequences"], default="pairs",
                    help="with several ranks: split the layer's head pairs over the ranks (tensor "
                         "parallelism, strong scaling) or give each rank its own sequence (weak scaling)")
    args = ap.parse_args()
    if args.e2e_steps <= 0:
        args.e2e_steps = args.steps
    return args


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def rank_batch_index(rank: int) -> int:
    """Weak scaling: rank r processes its own independent sequence(s), drawn with batch index r."""
    return rank


def reduce_step_ms(ms: float, world: int, device=None) -> float:
    """Max over ranks of the per-step time (the slowest rank sets the job's step time)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, step_ms: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's step time."""
    return tokens_per_rank * world / (step_ms / 1000.0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ accounting ---

def compulsory_share(x, kernel: str) -> float:
    """The part of the step's compulsory bytes each kernel moves (inputs read once,
    outputs written once): intra k, v, beta, g; scan S_final; output q and o;
    compaction the mask."""
    es = 2 if x.dtype == "bf16" else 4
    B, T, Nq, Nv, d, dv = x.B, x.T, x.Nq, x.Nv, x.d, x.dv
    qk, vo, bg = B * T * Nq * d * es, B * T * Nv * dv * es, B * T * Nv * 4
    return {"intra": qk + vo + 2 * bg, "scan": B * Nv * d * dv * 4, "output": qk + vo,
            "select": x.mask.size, "prefix": 0}.get(kernel, 0)


def algorithmic_bytes(x, kernel: str, n_snap: int = 0) -> float:
    """Compulsory bytes of one launch: inputs read once, outputs written once.

    step   : q, k, v, beta, g, mask in; o and s_final out (the whole core).
    output : q, k, U' (the workspace U buffer), g in; o out; plus one entry
             state per (group, value head) read from the fp32 snapshots.
    intra  : k, v, beta, g in; U out, and W of the event chunks out (bf16 storage:
             W is built inside intra; fp32 storage writes compact C-bar blocks instead).
    scan   : per selected (pair-)event, for both value heads: W and U read, U'
             written (dtype), K read once per pair; g in; the post-event fp32
             snapshots that output groups reference written; s_final out.
    """
    es = 2 if x.dtype == "bf16" else 4
    B, T, Nq, Nv, d, dv, C = x.B, x.T, x.Nq, x.Nv, x.d, x.dv, x.C
    G = (C + 1) // 2
    qk = B * T * Nq * d * es
    vo = B * T * Nv * dv * es
    bg = B * T * Nv * 4
    if kernel == "step":
        return 2 * qk + 2 * vo + 2 * bg + B * Nv * d * dv * 4 + x.mask.size
    if kernel == "output":
        return 2 * qk + 2 * vo + bg + B * Nv * G * d * dv * 4
    if kernel == "intra":
        if x.dtype == "bf16":
            return qk + 2 * vo + 2 * bg + int(x.mask.sum()) * 2 * 64 * d * es
        return qk + 2 * vo + 2 * bg + B * Nv * C * 7 * 256 * 4
    if kernel == "scan":
        E = int(x.mask.sum())
        per_event = 64 * d * es + 2 * (2 * 64 * d * es + 2 * 64 * dv * es + 64 * 4)
        return E * per_event + n_snap * 2 * d * dv * 4 + B * Nv * d * dv * 4
    raise ValueError(kernel)


# ------------------------------------------------------------------ clocks ---

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((float(r[3]) for r in rows if r[3].replace(".", "").isdigit()), default=None)}


# -------------------------------------------------------------- the oracle ---

def oracle_sample(x, pairs, t_tokens, nthreads):
    """Time the oracle on head pairs `pairs` of sequence 0 over the first t_tokens tokens."""
    import oracle
    vi = [2 * p + j for p in pairs for j in (0, 1)]
    C = t_tokens // 64
    sl = lambda a, idx: np.ascontiguousarray(a[0:1, :t_tokens][:, :, idx])
    q, k = sl(x.q, pairs), sl(x.k, pairs)
    v, beta, g = sl(x.v, vi), sl(x.beta, vi), sl(x.g, vi)
    mask = np.ascontiguousarray(x.mask[0:1][:, pairs, :C])
    t0 = time.perf_counter()
    oracle.prefill(q, k, v, beta, g, mask=mask, solver=oracle.SOLVER_BLOCK_ADJ, nthreads=nthreads)
    dt = time.perf_counter() - t0
    # tokens of the whole layer this sample stands for: t_tokens x (fraction of the layer's heads)
    return t_tokens * len(pairs) / x.Nq / dt, dt, min(nthreads, 2 * len(pairs))


def cpu_model() -> str:
    """The host CPU's model name (lscpu), or 'unknown'."""
    try:
        outp = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in outp.splitlines():
            if ln.lower().startswith("model name"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return "unknown"


def cpu_baseline(x):
    cores = os.cpu_count() or 1
    npairs = max(1, min(x.Nq, cores))
    pairs = list(range(npairs))
    t_tokens = min(x.T, 16384)
    value, dt, used = oracle_sample(x, pairs, t_tokens, nthreads=min(2 * npairs, cores))
    return {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "cpu_model": cpu_model(),
            "host_cores": cores,
            "sample": f"fp64 C oracle, head pairs 0..{npairs - 1} of {x.Nq}, tokens 0..{t_tokens - 1} of sequence 0 "
                      f"({dt:.1f} s wall, {used} threads); tokens/s scaled to the full layer by the head fraction"}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import gdn_synth
    x = gdn_synth.make_workload(args.workload)
    cores = os.cpu_count() or 1
    npairs = max(1, min(x.Nq, cores // 2, 4))
    t_tokens = min(x.T, 4096)
    times, vals = [], []
    used = 1
    for step in range(args.warmup + args.steps):
        pairs = [(step * npairs + i) % x.Nq for i in range(npairs)]
        v, dt, used = oracle_sample(x, pairs, t_tokens, nthreads=2 * npairs)
        if step >= args.warmup:
            times.append(dt)
            vals.append(v)
    ms = 1000.0 * statistics.mean(times)
    value = t_tokens * npairs / x.Nq / (ms / 1000.0)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, "B": x.B, "T": x.T, "Nq": x.Nq, "Nv": x.Nv, "d": x.d, "dv": x.dv,
                       "retention": round(x.retention(), 4), "solver": "block_adj"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": used, "kind": "oracle", "cpu_model": cpu_model(),
                             "sample": f"each step: {npairs} head pairs (cycling) x tokens 0..{t_tokens - 1} of "
                                       f"sequence 0; tokens/s scaled to the full layer by the head fraction"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ our CUDA path ---

def count_launches(gdn, call, steps):
    """Kernels that `steps` calls launch on their normal schedule (profile mode 2: counted, not timed)."""
    import torch
    gdn.gdn_profile_enable(2)
    for _ in range(steps):
        call()
    torch.cuda.synchronize()
    _, _, n_launch = gdn.gdn_profile_read(with_launches=True)
    gdn.gdn_profile_enable(False)
    return n_launch


def time_plain(call, steps, world, dev, warmup=3):
    """Mean ms of `call()` over `steps` after `warmup` calls (CUDA events on the current stream)."""
    import torch
    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    return reduce_step_ms(e0.elapsed_time(e1) / steps, world, dev)


def other_configs(gdn, gdn_synth, args, world, dev, stream, rank):
    """The other workloads of the study, timed on their own inputs (tokens/s per layer):
    the T=4096 dense layer through gdn_prefill_dense with both solvers, the batch of
    B = 2, 4, 8 sequences at T=32K (29% events), and the 24-layer, 128K-token prefill
    timed end to end (24 independently seeded layers back to back in one stream)."""
    import torch
    out = {}
    st = torch.bfloat16

    def dev_inputs(x):
        f = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(dt)
        return {"q": f(x.q, st), "k": f(x.k, st), "v": f(x.v, st), "beta": f(x.beta, torch.float32),
                "g": f(x.g, torch.float32), "mask": f(x.mask, torch.uint8)}

    x = gdn_synth.make_workload("qwen35_4b_layer_T4096_dense", batch_index=rank_batch_index(rank))
    t = dev_inputs(x)
    ws = gdn.Workspace()
    for solver in ("exact", "block_adj"):
        call = lambda: gdn.gdn_prefill_dense(t["q"], t["k"], t["v"], t["beta"], t["g"], solver=solver, workspace=ws,
                                             stream=stream)
        ms = time_plain(call, args.steps, world, dev)
        out[f"qwen35_4b_layer_T4096_dense_{solver}"] = {
            "ms_per_step": ms, "value": job_throughput(x.B * x.T, world, ms), "unit": UNIT,
            "api": "gdn_prefill_dense", "gpu_launches": count_launches(gdn, call, 1)}
    del t, ws
    for B in (2, 4, 8):
        x = gdn_synth.make_workload("qwen35_4b_layer_B8_T32768_sparse29", B=B, batch_index=rank_batch_index(rank))
        t = dev_inputs(x)
        ws = gdn.Workspace()
        call = lambda: gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"],
                                              solver="block_adj", workspace=ws, stream=stream)
        ms = time_plain(call, max(3, args.steps // 4), world, dev)
        out[f"qwen35_4b_layer_B{B}_T32768_sparse29"] = {
            "ms_per_step": ms, "value": job_throughput(x.B * x.T, world, ms), "unit": UNIT,
            "retention": round(x.retention(), 4), "api": "gdn_prefill_sparse",
            "gpu_launches": count_launches(gdn, call, 1)}
        del t, ws
        torch.cuda.empty_cache()
    # 24 layers x T = 131072: inputs drawn on the GPU (the same recipe, a device generator)
    name, L, T = "qwen35_4b_24layers_T131072_sparse29", 24, 131072
    layers = [gdn_synth.make_layer_on_device(1, T, 16, 32, gdn_synth.seed_for(3, layer, rank_batch_index(rank)), dev)
              for layer in range(L)]
    o = torch.empty((1, T, 32, 128), dtype=st, device=dev)
    finals = torch.empty((L, 1, 32, 128, 128), dtype=torch.float32, device=dev)
    ws = gdn.Workspace()

    def prefill_24():
        for i, t in enumerate(layers):
            gdn.gdn_prefill_sparse(t["q"], t["k"], t["v"], t["beta"], t["g"], t["mask"], solver="block_adj",
                                   o=o, s_final=finals[i], workspace=ws, stream=stream)

    ms = time_plain(prefill_24, 3, world, dev, warmup=1)
    ok = bool(torch.isfinite(finals).all().item()) and gdn.gdn_workspace_status(ws) == 0
    out[name] = {"ms_per_prefill": ms, "value": job_throughput(L * T, world, ms), "unit": "tokens/s per layer",
                 "layers": L, "T": T, "timed": "24 layers back to back in one stream, end to end",
                 "inputs": "seeded, drawn on the GPU (gdn_synth.make_layer_on_device)",
                 "retention": round(float(sum(t["mask"].float().mean().item() for t in layers) / L), 4),
                 "s_final_finite_and_status_ok": ok, "gpu_launches": count_launches(gdn, prefill_24, 1)}
    del layers, o, finals, ws
    torch.cuda.empty_cache()
    return out


def timed_variant(gdn, call, x, steps, world, dev, stream):
    """Time `call()` (one prefill) over `steps` after 3 warm-ups: ms per step, tokens/s, stages, kernels."""
    import torch
    for _ in range(3):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    gdn.gdn_profile_enable(True)  # stage breakdown on a second pass (stage events serialise the kernels)
    for _ in range(steps):
        call()
    torch.cuda.synchronize()
    stage_ms, nrec, _ = gdn.gdn_profile_read(with_launches=True)
    gdn.gdn_profile_enable(False)
    n_launch = count_launches(gdn, call, steps)
    ms = reduce_step_ms(e0.elapsed_time(e1) / steps, world, dev)
    return {"ms_per_step": ms, "value": job_throughput(x.B * x.T, world, ms), "unit": UNIT, "gpu_launches": n_launch,
            "stages_ms": {k: round(v / max(nrec, 1), 4) for k, v in stage_ms.items()}}


def online_variant(gdn, d_in, x, ws, stream, steps, world, dev):
    """The same step with the events chosen on the GPU from the Tail-16 scores
    (SparseGDN Sec. 2.4) instead of the given mask: time, stages and retention."""
    if x.Nv != 32:
        return None
    last = []

    def step():
        last[:] = [gdn.gdn_prefill_sparse_online(d_in["q"], d_in["k"], d_in["v"], d_in["beta"], d_in["g"],
                                                 solver="block_adj", workspace=ws, stream=stream)]

    r = timed_variant(gdn, step, x, steps, world, dev, stream)
    out = last[0]
    r["retention"] = round(float(out[2].float().mean().item()), 4)
    r["tiers_low_mid_high"] = [int((out[3] == t).sum().item()) for t in range(3)]
    return r


def run_ours(args):
    import torch
    import torch.distributed as dist

    import gated_delta_rule_16_gb300 as gdn
    import gdn_synth

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    pair_shard = world > 1 and args.shard == "pairs"
    x = gdn_synth.make_workload(args.workload, batch_index=0 if pair_shard else rank_batch_index(rank))
    tok = x.B * x.T  # tokens of this rank's layer (with pair sharding: the layer all ranks share)
    if pair_shard:  # this rank's block of head pairs (gated_delta_rule_16_gb300.sharded.pair_block)
        from gated_delta_rule_16_gb300.sharded import pair_block
        p0, p1 = pair_block(rank, world, x.Nq)
        x.q, x.k = x.q[:, :, p0:p1], x.k[:, :, p0:p1]
        x.v, x.beta, x.g = x.v[:, :, 2 * p0:2 * p1], x.beta[:, :, 2 * p0:2 * p1], x.g[:, :, 2 * p0:2 * p1]
        x.mask = x.mask[:, p0:p1]
        x.Nq, x.Nv = p1 - p0, 2 * (p1 - p0)
    st = torch.bfloat16 if x.dtype == "bf16" else torch.float32
    c = np.ascontiguousarray
    host = {
        "q": torch.from_numpy(c(x.q)).to(st).pin_memory(), "k": torch.from_numpy(c(x.k)).to(st).pin_memory(),
        "v": torch.from_numpy(c(x.v)).to(st).pin_memory(), "beta": torch.from_numpy(c(x.beta)).pin_memory(),
        "g": torch.from_numpy(c(x.g)).pin_memory(), "mask": torch.from_numpy(c(x.mask)).pin_memory(),
    }
    d_in = {n: t.to(dev) for n, t in host.items()}
    o = torch.empty((x.B, x.T, x.Nv, x.dv), dtype=st, device=dev)
    s_final = torch.empty((x.B, x.Nv, x.d, x.dv), dtype=torch.float32, device=dev)
    ws = gdn.Workspace()
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.gdn_prefill_sparse(d_in["q"], d_in["k"], d_in["v"], d_in["beta"], d_in["g"], d_in["mask"],
                               solver="block_adj", o=o, s_final=s_final, workspace=ws, stream=stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    if gdn.gdn_workspace_status(ws) != 0:
        raise RuntimeError("device-side capacity overflow in the warm-up")
    # the library's device counters at workspace offset 0: E, snapshots written, status
    n_events, n_snap = (int(v) for v in ws.buf[:8].view(torch.int32).cpu().tolist())

    clocks = ClockSampler(local).start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    # stage breakdown and kernel count: the same steps again with the library's stage events
    # (which serialise the kernels, so they are not part of the timed loop above)
    gdn.gdn_profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    stage_ms, nrec, _ = gdn.gdn_profile_read(with_launches=True)
    gdn.gdn_profile_enable(False)
    n_launch = count_launches(gdn, step, args.steps)
    ms = reduce_step_ms(ev0.elapsed_time(ev1) / args.steps, world, dev)
    # with pair sharding the ranks share one layer: its tokens over the slowest rank's time
    ranks_tokens = 1 if pair_shard else world
    value = job_throughput(tok, ranks_tokens, ms)

    # end to end through the C ABI with host buffers (gdn_prefill_host): each step copies its
    # inputs from pinned host memory, runs the prefill and copies O and S_final back.  Serial:
    # one stream.  Pipelined (the e2e value): two workspaces on two streams, so one step's
    # copies overlap the other step's kernels; every step still does all of its own copies.
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = o.numel() * o.element_size() + s_final.numel() * s_final.element_size()
    streams = [stream, torch.cuda.Stream(dev)]
    wss = [gdn.Workspace(), gdn.Workspace()]
    h_out = [(torch.empty(o.shape, dtype=st).pin_memory(), torch.empty(s_final.shape, dtype=torch.float32).pin_memory())
             for _ in range(2)]

    def e2e_step(j):
        gdn.gdn_prefill_host(host["q"], host["k"], host["v"], host["beta"], host["g"], host["mask"],
                             solver="block_adj", o=h_out[j][0], s_final=h_out[j][1], workspace=wss[j],
                             device=dev, stream=streams[j])

    def time_e2e(pipelined):
        for i in range(2):
            e2e_step(i % 2 if pipelined else 0)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(streams[0])
        streams[1].wait_event(e0)
        for i in range(args.e2e_steps):
            e2e_step(i % 2 if pipelined else 0)
        streams[0].wait_stream(streams[1])
        e1.record(streams[0])
        torch.cuda.synchronize()
        return reduce_step_ms(e0.elapsed_time(e1) / args.e2e_steps, world, dev)

    e2e_serial_ms = time_e2e(False)
    e2e_ms = time_e2e(True)
    # the host copy of O must equal the device-path result of the same inputs
    if not torch.equal(h_out[(args.e2e_steps - 1) % 2][0], o.cpu()):
        raise RuntimeError("host-buffer prefill disagrees with the device-buffer prefill")

    online = online_variant(gdn, d_in, x, ws, stream, args.steps, world, dev)
    # the pages' ablation axes on the same inputs (gdn_prefill_ex): W deferred to its own kernel
    # (bit-identical result), the exact Full64 solver with the same mask, the run-map event scan
    def ex_call(**kw):
        return lambda: gdn.gdn_prefill_ex(d_in["q"], d_in["k"], d_in["v"], d_in["beta"], d_in["g"], mode="sparse",
                                          mask=d_in["mask"], o=o, s_final=s_final, workspace=ws, stream=stream, **kw)
    w_deferred = timed_variant(gdn, ex_call(solver="block_adj", w_deferred=True), x, args.steps, world, dev, stream)
    exact = timed_variant(gdn, ex_call(solver="exact"), x, args.steps, world, dev, stream)
    scan_runs = timed_variant(gdn, ex_call(solver="block_adj", scan_runs=True), x, args.steps, world, dev, stream)
    # the pages' reference paths (Table 6), bit-identical results: the masked full scan, and the
    # dense group entry states read by group instead of compact snapshots through the group map
    scan_full = timed_variant(gdn, ex_call(solver="block_adj", scan_full=True), x, args.steps, world, dev, stream)
    expanded = timed_variant(gdn, ex_call(solver="block_adj", states_expanded=True), x, args.steps, world, dev,
                             stream)
    # the library's own dense path on the same layer (every chunk an event, gdn_prefill_dense)
    dense = timed_variant(gdn, lambda: gdn.gdn_prefill_dense(
        d_in["q"], d_in["k"], d_in["v"], d_in["beta"], d_in["g"], solver="block_adj", o=o, s_final=s_final,
        workspace=ws, stream=stream), x, args.steps, world, dev, stream)
    variants = {"online_selection": online, "w_deferred": w_deferred, "solver_exact": exact, "scan_runs": scan_runs,
                "scan_full_masked": scan_full, "states_expanded_unmapped_o": expanded, "dense_same_layer": dense}
    del o, s_final
    ws = None
    torch.cuda.empty_cache()
    configs = {} if args.no_configs or world > 1 else other_configs(gdn, gdn_synth, args, world, dev, stream, rank)

    peak, peak_kind = peaks()
    per_stage = {k: v / max(nrec, 1) for k, v in stage_ms.items()}
    step_bytes = algorithmic_bytes(x, "step")
    step_gbs = step_bytes / (ms / 1000.0) / 1e9
    traffic = {k: PROFILED_TRAFFIC.get((args.workload, k)) for k in ("select", "prefix", "intra", "scan", "output")}
    step_traffic = sum(traffic.values()) if all(v is not None for v in traffic.values()) else None
    kernels = {}
    for k in ("select", "prefix", "intra", "scan", "output"):
        share = compulsory_share(x, k)
        t = per_stage.get(k, 0.0)
        kernels[k] = {"ms_one_stream": round(t, 4), "compulsory_bytes": share,
                      "frac_of_peak": (share / (t / 1000.0) / 1e9 / peak) if t > 0 and share else None,
                      "dram_bytes": traffic[k],
                      "dram_over_compulsory": (traffic[k] / share) if traffic[k] and share else None}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if pair_shard else "weak",
        "vs_baseline": None, "dtype": x.dtype, "data": "synthetic",
        "config": {"workload": args.workload, "B": x.B, "T": x.T, "Nq": x.Nq, "Nv": x.Nv, "d": x.d, "dv": x.dv,
                   "retention": round(x.retention(), 4), "events": n_events, "snapshots": n_snap,
                   "solver": "block_adj",
                   "l2": "inputs larger than L2 (%.0f MB compulsory bytes per step), no flush" % (step_bytes / 1e6),
                   "parallelism": (f"head pairs split over {world} GPUs (tensor parallel, no collective with a "
                                   f"given mask)" if pair_shard else
                                   "one independent sequence per GPU" if world > 1 else "single GPU")},
        "clocks": clk,
        "e2e": {"value": job_throughput(tok, ranks_tokens, e2e_ms), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "api": "gdn_prefill_host (C ABI, host buffers)",
                "pipelining": "2 streams x 2 workspaces", "serial_ms_per_step": e2e_serial_ms,
                "steps": args.e2e_steps},
        "gpu_launches": n_launch,
        "roofline": {"bound": "hbm", "kernel": "step (the whole hot path: compaction, prefix, intra, scan, output)",
                     "achieved": step_gbs, "peak": peak, "unit": "GB/s", "frac": step_gbs / peak,
                     "traffic": step_traffic, "peak_source": peak_kind,
                     "note": f"achieved = the step's compulsory bytes ({step_bytes / 1e6:.1f} MB: q, k, v, beta, g, "
                             f"mask read once; o, S_final written once) / ms_per_step; frac of {peak_kind} HBM copy "
                             f"bandwidth; traffic = ncu DRAM bytes of one prefill summed over its kernels",
                     "kernels": kernels},
        "stages_ms_one_stream": {k: round(v, 4) for k, v in per_stage.items()},
        "variants": variants,
        "configs": configs,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(x)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
