#!/usr/bin/env python
"""Benchmark of one-layer attention-matching compaction on GB300.

Workload: one GQA layer with 8 KV heads x 4 query heads per group,
T = 8192 cached positions, n_q = 4*T = 32768 context-prefill reference
queries per KV head, d = 128, t = 256 keys kept (32x), bf16 Q/K/V with the
synthetic "peaked" recipe (outlier key channels, queries drawn near keys).
A step compacts one layer: all five steps (full statistics, key scores,
top-t selection, NNLS biases, OLS values) on inputs already in HBM.
Successive steps cycle through four distinct layers (400 MB of inputs, more
than the 129 MB L2), so no step finds its inputs in L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl lc|reference]

Prints one JSON line.  `value` is ms per compacted layer over the whole job;
`roofline` is the dominant kernel's algorithmic throughput against the
measured peak; `e2e` is the same metric through the host-buffer entry point
with the host<->device copies inside the timed region; `cpu_baseline` is the
float64 oracle timed on this machine's host cores on a bounded sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ms per layer compaction (8 KV heads, T=8192, t=256); QK^T TFLOP/s vs peak"
WORKLOAD = "cfg3"
N_LAYERS = 4


def rank_layer_ids(rank: int, n_layers: int = N_LAYERS):
    """Layer indices (generator seeds) a rank compacts: ranks own disjoint
    layers, so per-GPU work is fixed as the job grows (weak scaling)."""
    return [rank * n_layers + l for l in range(n_layers)]


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The largest value of x over all ranks: a step of the job takes as long
    as its slowest rank."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(ms_step_max: float, world: int) -> float:
    """ms per compacted layer over the whole job: each of the `world` ranks
    compacts one layer per step."""
    return ms_step_max / world


def args_():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="lc", choices=["lc", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--fast-steps", type=int, default=100,
                    help="steps of the two-pass / redistribution path (0: skip)")
    ap.add_argument("--fast-n-sub", type=int, default=256)
    ap.add_argument("--fast-k", type=int, default=4)
    ap.add_argument("--sweep-layers", type=int, default=36,
                    help="layers of the full-model sweep timed through the pipelined "
                         "multi-layer call (0: skip)")
    ap.add_argument("--sweep-steps", type=int, default=3)
    ap.add_argument("--long-steps", type=int, default=2,
                    help="timed compactions of one long-context layer (T = 131072, "
                         "t = 1024); 0 skips it (drawing its inputs takes about a minute)")
    ap.add_argument("--select-steps", type=int, default=20,
                    help="timed top-t selections of 8 x 2^select-log2t scores (0: skip)")
    ap.add_argument("--select-log2t", type=int, default=24,
                    help="log2 of the scores per head in the select sweep")
    ap.add_argument("--quality-queries", type=int, default=4096,
                    help="held-out queries per head for the quality comparison (0: skip)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=20.0,
                    help="seconds of oracle work for the cpu_baseline sample")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            m = json.load(f)
        return {"hbm_gbs": m["hbm_gbs"], "bf16_tflops": m["bf16_tflops"],
                "bf16_tflops_sustained": m.get("bf16_tflops_sustained", m["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def workload():
    import synth
    return synth.workload(WORKLOAD)


def flops(w):
    """Algorithmic flops of one layer (per launch of each kernel)."""
    H, nq, T, d, t = w.H, w.n_q, w.T, w.d, w.t
    return {
        "attn_stats": 4.0 * nq * T * d * H,        # S = Q K^T and O = P V
        "key_scores": 2.0 * nq * T * d * H,        # S recomputed
        "gram_mass": H * (2.0 * nq * t * d + 2.0 * nq * t * t),
        "gram_out": H * (2.0 * nq * t * d + 2.0 * nq * t * t + 2.0 * nq * t * d),
        "layer": H * (6.0 * nq * T * d + 6.0 * nq * t * d + 4.0 * nq * t * t),
    }


# ------------------------------------------------------------------ clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.f = None

    def start(self):
        try:
            self.f = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = max(mx, float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ oracle
def oracle_sample(budget_s: float):
    """Time the float64 oracle on one KV head of the workload with a subset of
    the reference queries sized to about `budget_s` seconds, and scale to ms
    per layer by the ratio of work (linear in the number of queries) times the
    number of heads."""
    import numpy as np

    import oracle
    import synth
    w = workload()
    d = synth.make(w, heads=[0])
    Q, K, V = d["Q"][0], d["K"][0], d["V"][0]
    s = w.softmax_scale

    def run(nq):
        q = Q[:nq].astype(np.float64)
        t0 = time.perf_counter()
        oracle.compact_head(q, K, V, w.t, s)
        return time.perf_counter() - t0

    probe_n = 1024
    tp = run(probe_n)
    n = int(min(w.n_q, max(probe_n, probe_n * budget_s / max(tp, 1e-3))))
    n = max(probe_n, n // 1024 * 1024)
    t_s = run(n)
    ms_layer = t_s * 1e3 * (w.n_q / n) * w.H
    return ms_layer, n, t_s


def reference_arm(a):
    """The float64 oracle as it stands, on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = workload()
    total_budget = 120.0
    per_step = max(0.5, min(10.0, total_budget / max(1, a.steps + a.warmup)))
    times = []
    n_used = None
    for i in range(a.warmup + a.steps):
        ms, n, _ = oracle_sample(per_step)
        n_used = n
        if i >= a.warmup:
            times.append(ms)
    value = statistics.mean(times)
    cores = os.cpu_count()
    sample = (f"extrapolated: 1 of {w.H} KV heads of one {WORKLOAD} layer, {n_used} of "
              f"{w.n_q} reference queries per step, timed and scaled to a full layer by "
              f"query count x heads")
    line = {
        "metric": METRIC, "value": value, "unit": "ms", "impl": "reference",
        "n_gpus": a.gpus, "steps": a.steps, "warmup": a.warmup, "ms_per_step": value,
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(w, a.gpus),
        "cpu_baseline": {"value": value, "unit": "ms", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "ms", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_dict(w, n):
    return {"workload": f"{WORKLOAD}: one GQA layer, {w.H} KV heads x {w.G} query heads, "
                        f"T={w.T}, n_q={w.n_q} per KV head, d={w.d}, t={w.t}, bf16, "
                        f"peaked synthetic Q/K/V",
            "H": w.H, "G": w.G, "T": w.T, "n_q": w.n_q, "d": w.d, "t": w.t,
            "parallelism": f"independent layers, {n} GPU(s)",
            "l2": f"steps cycle over {N_LAYERS} distinct layers ({N_LAYERS * 100} MB of inputs > 129 MB L2)"}


def traffic_for(kernel: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel
    source has not changed since it was taken."""
    p = os.path.join(ROOT, "profiles", f"{kernel}_{WORKLOAD}.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "kv_cache_compaction_gb300", "csrc", rec.get("source", ""))
    if not os.path.exists(src):
        return None
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    return rec.get("dram_bytes_per_launch") if h == rec.get("source_sha256") else None


# ------------------------------------------------------------------ main arm
def main():
    a = args_()
    if a.impl == "reference":
        reference_arm(a)
        return
    import numpy as np
    import torch

    import synth
    from kv_cache_compaction_gb300 import build as lcbuild
    lcbuild.build()
    import kv_cache_compaction_gb300 as lc

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = workload()
    fl = flops(w)

    def up(arr):
        bits = synth.bf16_bits(arr).view(np.int16)
        return torch.from_numpy(np.ascontiguousarray(bits)).view(torch.bfloat16)

    layers_host = []
    layers = []
    for l in range(N_LAYERS):
        d = synth.make(w.layer(rank_layer_ids(rank)[l]))
        if l == 0:
            K0 = d["K"]
        hq, hk, hv = up(d["Q"]), up(d["K"]), up(d["V"])
        layers_host.append((hq, hk, hv))
        layers.append((hq.to(dev), hk.to(dev), hv.to(dev)))
    comp = lc.Compactor(local)
    H, t, dd = w.H, w.t, w.d
    out = (torch.empty((H, t), dtype=torch.int32, device=dev),
           torch.empty((H, t), dtype=torch.float32, device=dev),
           torch.empty((H, t), dtype=torch.float32, device=dev),
           torch.empty((H, t, dd), dtype=torch.float32, device=dev))

    def step(i):
        Q, K, V = layers[i % N_LAYERS]
        comp.compact_layer(Q, K, V, t, out=out)

    for i in range(a.warmup):
        step(i)
    torch.cuda.synchronize()
    rep = comp.report(H)
    if rep.device_error_bits:
        raise RuntimeError(f"device error bits {rep.device_error_bits}")

    stream = torch.cuda.current_stream(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(local)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clk.start()
    time.sleep(0.3)  # let the sampler start before the timed work
    # the headline: K steps with the library's per-kernel events off
    t_wall = time.perf_counter()
    ev0.record(stream)
    for i in range(a.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    wall_s = time.perf_counter() - t_wall
    if dist:
        dist.barrier()
    ms_total = ev0.elapsed_time(ev1)
    ms_step = max_over_ranks(ms_total / a.steps, dist, dev)
    value = job_value(ms_step, world)
    # a second timed region of the same K steps with per-kernel CUDA events
    # recorded on the launching streams: the per-kernel times and the roofline
    comp.profile_read()
    comp.profile(True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for i in range(a.steps):
        step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_step_profiled = ev0.elapsed_time(ev1) / a.steps
    clocks = clk.stop()
    comp.profile(False)
    kern = comp.profile_read()

    # per-kernel breakdown (per step) and the dominant kernel's roofline
    pk = peaks()
    per_kernel = {k: {"ms_per_step": v[0] / a.steps, "launches_per_step": v[1] / a.steps}
                  for k, v in kern.items()}
    launches = int(sum(v[1] for v in kern.values()))
    dom = max(kern, key=lambda k: kern[k][0])
    dom_ms = kern[dom][0] / max(kern[dom][1], 1)
    if dom in ("attn_stats", "key_scores", "gram_mass", "gram_out"):
        # a launch lasts under a millisecond, inside 2 ms steps: the burst
        # peak applies; the sustained one is given beside it
        ach = fl[dom] / (dom_ms * 1e-3) / 1e12
        roof = {"kernel": dom, "bound": "tensor", "achieved": ach,
                "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "traffic": traffic_for(dom),
                "peak_kind": f"bf16 dense burst ({pk['source']})",
                "frac_of_sustained": ach / pk["bf16_tflops_sustained"],
                "sustained_peak": pk["bf16_tflops_sustained"],
                "algorithmic_flops_per_launch": fl[dom], "avg_launch_ms": dom_ms}
    else:
        roof = {"kernel": dom, "bound": "alu", "achieved": None, "peak": None, "unit": None,
                "frac": None, "traffic": None, "avg_launch_ms": dom_ms}
    qkt = {}
    for k, f in (("attn_stats", fl["attn_stats"]), ("key_scores", fl["key_scores"])):
        if k in kern:
            ms = kern[k][0] / max(kern[k][1], 1)
            tf = f / (ms * 1e-3) / 1e12
            qkt[k] = {"tflops": tf, "frac_of_burst": tf / pk["bf16_tflops"],
                      "frac_of_sustained": tf / pk["bf16_tflops_sustained"], "ms": ms,
                      "traffic": traffic_for(k)}
    # the two small memory-side kernels against HBM: the top-t select reads
    # the scores u and writes idx; the key gather reads and writes t rows of K
    hbm_bytes = {"select_topt": H * w.T * 4 + H * t * 4, "gather_keys": 2 * H * t * dd * 2}
    hbm = {}
    for k, nb in hbm_bytes.items():
        if k in kern:
            ms = kern[k][0] / max(kern[k][1], 1)
            gbs = nb / (ms * 1e-3) / 1e9
            hbm[k] = {"bytes": nb, "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"]}

    # the top-t select on long score arrays (the sampled-threshold path of
    # lc_select_topt): 8 heads x 2^24 fp32 scores by default, t = 1024, two
    # arrays used in turn (2 x 537 MB) so that no call finds its scores in L2
    if a.select_steps > 0:
        Hs, Ts, ts = 8, 1 << a.select_log2t, 1024
        gen = torch.Generator(device=dev)
        gen.manual_seed(11)
        us = [-20.0 * torch.rand((Hs, Ts), generator=gen, device=dev) for _ in range(2)]
        for i in range(3):
            comp.select_topt(us[i % 2], ts)
        torch.cuda.synchronize()
        q0 = torch.cuda.Event(enable_timing=True)
        q1 = torch.cuda.Event(enable_timing=True)
        q0.record(stream)
        for i in range(a.select_steps):
            comp.select_topt(us[i % 2], ts)
        q1.record(stream)
        torch.cuda.synchronize()
        ms_sel = q0.elapsed_time(q1) / a.select_steps
        comp.profile_read()
        comp.profile(True)
        for i in range(a.select_steps):
            comp.select_topt(us[i % 2], ts)
        torch.cuda.synchronize()
        comp.profile(False)
        sk = comp.profile_read()
        stage_ms = {k: v[0] / max(v[1], 1) for k, v in sk.items()}
        nb = Hs * Ts * 4 + Hs * ts * 4
        filt = None
        if "select_filter" in stage_ms:
            fb = Hs * Ts * 4
            fg = fb / (stage_ms["select_filter"] * 1e-3) / 1e9
            filt = {"bytes": fb, "ms": stage_ms["select_filter"], "gbs": fg,
                    "frac_of_hbm": fg / pk["hbm_gbs"]}
        hbm.setdefault("select_topt", {})["large_n_sweep"] = {
            "workload": f"{Hs} heads x {Ts} fp32 scores (uniform in [-20, 0]), t = {ts}, "
                        "two arrays in turn (> L2)",
            "bytes": nb, "ms": ms_sel, "gbs": nb / (ms_sel * 1e-3) / 1e9,
            "frac_of_hbm": nb / (ms_sel * 1e-3) / 1e9 / pk["hbm_gbs"],
            "steps": a.select_steps, "stage_ms": stage_ms, "filter_kernel": filt}
        del us

    # end to end through the host-buffer entry point
    e2e = None
    if a.e2e_steps > 0:
        pinned = [tuple(x.pin_memory() for x in L) for L in layers_host]
        hout = (torch.empty((H, t), dtype=torch.int32).pin_memory(),
                torch.empty((H, t)).pin_memory(), torch.empty((H, t)).pin_memory(),
                torch.empty((H, t, dd)).pin_memory())
        for i in range(2):
            Q, K, V = pinned[i % N_LAYERS]
            comp.compact_layer_host(Q, K, V, t, hout)
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(a.e2e_steps):
            Q, K, V = pinned[i % N_LAYERS]
            comp.compact_layer_host(Q, K, V, t, hout)
        e1.record(stream)
        torch.cuda.synchronize()
        ms_e2e = max_over_ranks(e0.elapsed_time(e1) / a.e2e_steps, dist, dev)
        h2d = sum(x.numel() * x.element_size() for x in pinned[0])
        d2h = sum(x.numel() * x.element_size() for x in hout)
        # this machine's pinned host -> device copy rate for the same tensors,
        # copies alone: the floor under the upload that e2e overlaps with step 1
        dst = [torch.empty_like(x, device=dev) for x in pinned[0]]
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        for i in range(4):
            for d_, s_ in zip(dst, pinned[i % N_LAYERS]):
                d_.copy_(s_, non_blocking=True)
        c1.record(stream)
        torch.cuda.synchronize()
        ms_copy = c0.elapsed_time(c1) / 4
        del dst
        e2e = {"value": job_value(ms_e2e, world), "unit": "ms", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "h2d_copy_ms": ms_copy,
               "h2d_copy_gbs": h2d / (ms_copy * 1e-3) / 1e9}

    # the fast path (two-pass selection, redistributed beta, direct values)
    # on the same layers, 256-query subsets drawn per layer
    fast = None
    if a.fast_steps > 0:
        qsels = [torch.from_numpy(np.stack([
            np.random.default_rng(1000 + rank * N_LAYERS + l + 7919 * h).choice(
                w.n_q, a.fast_n_sub, replace=False) for h in range(H)]).astype(np.int32)).to(dev)
            for l in range(N_LAYERS)]
        fout = (out[0], out[2], out[3])

        def fstep(i):
            Q, K, V = layers[i % N_LAYERS]
            comp.compact_layer_fast(Q, K, V, qsels[i % N_LAYERS], t, a.fast_k, out=fout)

        for i in range(max(a.warmup, 3)):
            fstep(i)
        torch.cuda.synchronize()
        f0 = torch.cuda.Event(enable_timing=True)
        f1 = torch.cuda.Event(enable_timing=True)
        f0.record(stream)
        for i in range(a.fast_steps):
            fstep(i)
        f1.record(stream)
        torch.cuda.synchronize()
        ms_fast = f0.elapsed_time(f1) / a.fast_steps
        comp.profile_read()
        comp.profile(True)
        for i in range(20):
            fstep(i)
        torch.cuda.synchronize()
        comp.profile(False)
        fk = comp.profile_read()
        if comp.report(H).device_error_bits:
            raise RuntimeError("device error in the fast path")
        fast = {"ms_per_layer": ms_fast, "n_sub": a.fast_n_sub, "k": a.fast_k,
                "steps": a.fast_steps, "vs_full_path": ms_step / ms_fast,
                "launches_per_step": sum(v[1] for v in fk.values()) / 20,
                "per_kernel_ms": {k: v[0] / 20 for k, v in fk.items()}}

    # the full-model sweep (36 layers of the benchmark shape) through the
    # pipelined multi-layer call; the layers cycle over the drawn ones
    sweep = None
    if a.sweep_layers > 0:
        L = a.sweep_layers
        SQ = torch.empty((L,) + tuple(layers[0][0].shape), dtype=torch.bfloat16, device=dev)
        SK = torch.empty((L,) + tuple(layers[0][1].shape), dtype=torch.bfloat16, device=dev)
        SV = torch.empty((L,) + tuple(layers[0][2].shape), dtype=torch.bfloat16, device=dev)
        for l in range(L):
            SQ[l].copy_(layers[l % N_LAYERS][0])
            SK[l].copy_(layers[l % N_LAYERS][1])
            SV[l].copy_(layers[l % N_LAYERS][2])
        sout = (torch.empty((L, H, t), dtype=torch.int32, device=dev),
                torch.empty((L, H, t), dtype=torch.float32, device=dev),
                torch.empty((L, H, t), dtype=torch.float32, device=dev),
                torch.empty((L, H, t, dd), dtype=torch.float32, device=dev))
        comp.compact_layers(SQ, SK, SV, t, out=sout)
        torch.cuda.synchronize()
        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(a.sweep_steps):
            comp.compact_layers(SQ, SK, SV, t, out=sout)
        s1.record(stream)
        torch.cuda.synchronize()
        rep = comp.report(L * H)
        if rep.device_error_bits:
            raise RuntimeError("device error in the layer sweep")
        ms_sweep = s0.elapsed_time(s1) / a.sweep_steps
        sweep = {"workload": f"cfg4: {L} layers of the benchmark shape, one pipelined call; "
                             f"the {L} layers' inputs reuse {N_LAYERS} drawn layers in turn",
                 "layers": L, "ms": ms_sweep, "ms_per_layer": ms_sweep / L,
                 "serial_ms_per_layer": ms_step, "speedup_vs_serial": ms_step * L / ms_sweep,
                 "steps": a.sweep_steps}
        del SQ, SK, SV, sout

    # one long-context layer (T = 131072 keys, 524288 reference queries per KV
    # head, t = 1024): heads 0-1 of the seeded draw, repeated to the layer's 8
    # heads (same shapes and kernels; drawing all 8 takes minutes)
    long_ctx = None
    if a.long_steps > 0 and rank == 0:
        w5 = synth.workload("cfg5")
        d5 = synth.make(w5, heads=[0, 1])
        rep_h = (w5.H + 1) // 2
        Q5, K5, V5 = (up(np.concatenate([d5[k]] * rep_h)[: w5.H]).to(dev) for k in ("Q", "K", "V"))
        del d5
        comp.compact_layer(Q5, K5, V5, w5.t)
        torch.cuda.synchronize()
        comp.profile(True)
        l0 = torch.cuda.Event(enable_timing=True)
        l1 = torch.cuda.Event(enable_timing=True)
        l0.record(stream)
        for _ in range(a.long_steps):
            comp.compact_layer(Q5, K5, V5, w5.t)
        l1.record(stream)
        torch.cuda.synchronize()
        comp.profile(False)
        k5 = comp.profile_read()
        rep = comp.report(w5.H)
        if rep.device_error_bits:
            raise RuntimeError("device error in the long-context layer")
        f5 = flops(w5)
        pk5 = {k: v[0] / a.long_steps for k, v in k5.items()}
        dom5 = max(k5, key=lambda k: k5[k][0])
        ms5 = k5[dom5][0] / max(k5[dom5][1], 1)
        roof5 = None
        if dom5 in f5:
            # launches of ~0.2 s inside a step of ~0.4 s: the sustained peak applies
            ach5 = f5[dom5] / (ms5 * 1e-3) / 1e12
            roof5 = {"kernel": dom5, "bound": "tensor", "achieved": ach5,
                     "peak": pk["bf16_tflops_sustained"], "unit": "TFLOP/s",
                     "frac": ach5 / pk["bf16_tflops_sustained"], "traffic": None,
                     "peak_kind": f"bf16 dense sustained ({pk['source']})",
                     "frac_of_burst": ach5 / pk["bf16_tflops"],
                     "algorithmic_flops_per_launch": f5[dom5], "avg_launch_ms": ms5}
        long_ctx = {
            "workload": "cfg5: one layer, 8 KV heads x 4 query heads, T=131072, n_q=524288 "
                        "per KV head, d=128, t=1024, bf16, 64 needles per head (heads 0-1 of "
                        "the draw repeated to 8)",
            "ms_per_layer": l0.elapsed_time(l1) / a.long_steps, "steps": a.long_steps,
            "attn_stats_tflops": f5["attn_stats"] / (pk5["attn_stats"] * 1e-3) / 1e12,
            "key_scores_tflops": f5["key_scores"] / (pk5["key_scores"] * 1e-3) / 1e12,
            "layer_tflops": f5["layer"] / (l0.elapsed_time(l1) / a.long_steps * 1e-3) / 1e12,
            "nnls_iters": rep.nnls_iters, "per_kernel_ms": pk5, "roofline": roof5}
        del Q5, K5, V5

    # quality of three compactions of the first layer on held-out queries
    # drawn from the same recipe: attention matching (NNLS beta, OLS values),
    # the fast path (two-pass keys, redistributed beta, direct values) and
    # the baseline variant (RMS keys, bounded beta, OLS values)
    quality = None
    if a.quality_queries > 0:
        Qh = up(synth.heldout_queries(w, K0, a.quality_queries, 9001)).to(dev)
        Q, K, V = layers[0]
        qsel0 = torch.from_numpy(np.stack([
            np.random.default_rng(2000 + h).choice(w.n_q, a.fast_n_sub, replace=False)
            for h in range(H)]).astype(np.int32)).to(dev)

        def errs(idx, beta, Cv):
            me, oe = comp.heldout_errors(Qh, K, V, idx, beta, Cv)
            return {"mass_err": float(me.mean()), "out_err": float(oe.mean())}

        i1, _, b1, c1 = comp.compact_layer(Q, K, V, t)
        i2, b2, c2 = comp.compact_layer_fast(Q, K, V, qsel0, t, a.fast_k)
        i3, _, b3, c3 = comp.compact_layer_baseline(Q, K, V, t)
        quality = {"heldout_queries_per_head": a.quality_queries,
                   "definition": "per head mean |log Z_cmp - log Z_full| and mean "
                                 "||A_cmp - A_full||_2 over held-out queries, averaged over heads",
                   "attention_matching": errs(i1, b1, c1),
                   "fast_path": errs(i2, b2, c2),
                   "baseline_variant": errs(i3, b3, c3)}
        torch.cuda.synchronize()
        if comp.report(H).device_error_bits:
            raise RuntimeError("device error in the quality comparison")

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        ms_l, n, t_s = oracle_sample(a.cpu_budget)
        cpu = {"value": ms_l, "unit": "ms", "cores": os.cpu_count(), "kind": "oracle",
               "sample": f"extrapolated: 1 of {w.H} KV heads of one {WORKLOAD} layer with "
                         f"{n} of {w.n_q} reference queries ({t_s:.1f} s of CPU work), scaled "
                         f"to a full layer by query count x heads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "ms", "n_gpus": world, "steps": a.steps,
            "warmup": a.warmup, "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_dict(w, world), "roofline": roof, "qkt": qkt, "hbm": hbm,
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
            "per_kernel": per_kernel, "ms_per_step_profiled": ms_step_profiled,
            "timing": "value: K steps with the library's per-kernel events off; roofline, "
                      "qkt, hbm and per_kernel: a second timed region of the same K steps "
                      "with per-kernel CUDA events on the launching streams",
            "fast_path": fast, "sweep": sweep, "long_context": long_ctx, "quality": quality,
            "layer_tflops": fl["layer"] / (ms_step * 1e-3) / 1e12, "wall_s_timed": wall_s,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
