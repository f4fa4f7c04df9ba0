"""Benchmark of the MC-Sparse hot path on one GB300 (or N independent replicas).

Workload: the 720p kernel-benchmark layer (B=1, H=40, N=75,600 tokens on a
21x45x80 grid, d=128, bf16, C=128 -> 591 groups, density 0.2 -> K=15,120),
synthetic inputs from the seeded generator, generated on the device.

One step = one anchor period of the meta-cache schedule (anchor every 10 steps):
  anchor: PDDP grouping, dense attention + LSE, pass-2 column sums + exact top-K,
          anchor sparse attention + residual store;
  9 reuse steps: token-gather sparse attention of the current Q/K/V + residual.
Every kernel is timed with CUDA events on the launching stream. The headline
value is the sparse attention layer time (ms/layer, lower is better) of the
reuse kernel; the roofline object covers that kernel (kept FLOPs / time against
the measured sustained bf16 peak). After the timed steps (outside the timed
region) the 118,800-token schedule (24 heads, 50 steps, densities 0.15 and 0.25)
runs once to report the total time including anchors and the anchor overhead as
equivalent extra density (`anchor_overhead`; `--no-schedule` skips it), and the
65,536-token density/tile sweep (d and C in {64, 128}, densities 0.05-1.0) reports
the sparse kernel against the dense kernel per point (`sweep`; `--no-sweep`).
`matched_density` compares, on the same layer at its density, the captured
attention mass and the sparse output's relative error (||R|| / ||O_dense||) of
the group-shared selection with the PDDP groups against contiguous tile groups
(`--no-matched` skips it).
It also times the reuse step with the meta-cache kept in pinned host memory
through the cache ring (three layers' entries, the next one prefetched while
the current one computes; `cache_ring`; `--no-ring` skips it), and the reuse
kernel on uniform random sorted key sets of the same size (`stress_random_idx`;
`--no-stress` skips it).
`--impl reference` times the float64 CPU oracle instead, on a bounded sample of
groups, extrapolated to ms/layer.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-attn ms/layer & TFLOP/s (frac of bf16 roofline) at density 0.15-0.25"
UNIT = "ms/layer"
REUSE_PER_STEP = 9
# DRAM bytes (read + write) of one reuse-kernel launch on the 40-head layer: an
# 8-head ncu capture of the same kernel (dram__bytes_read.sum 1.0906 GB +
# dram__bytes_write.sum 0.1489 GB per 8-head launch) scaled by heads (traffic
# grows in proportion). Set to None when the kernel changes.
SPARSE_TRAFFIC_BYTES_H40 = (1.0906e9 + 0.1489e9) * 40 / 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("mcs", "reference"), default="mcs")
    ap.add_argument("--workload", default="kernel-bench-720p")
    ap.add_argument("--density", default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-schedule", action="store_true", help="skip the 118,800-token schedule (anchor overhead)")
    ap.add_argument("--no-sweep", action="store_true", help="skip the 65,536-token density/tile sweep")
    ap.add_argument("--no-ring", action="store_true", help="skip the host-resident meta-cache (cache ring) timing")
    ap.add_argument("--no-stress", action="store_true",
                    help="skip the reuse kernel on uniform random key sets (stress variant of the selected ones)")
    ap.add_argument("--no-matched", action="store_true", help="skip the PDDP-vs-contiguous group mass comparison")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the tiny fp32 layer and the 480p-shaped layer (1 anchor + reuse steps each)")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end leg (profiler launch lists of the timed steps only)")
    ap.add_argument("--heads", type=int, default=None, help="override H (smaller case for profiler captures)")
    ap.add_argument("--group-size", type=int, choices=(64, 128), default=None,
                    help="override C (the 64-query form of the sparse kernel, for profiler captures)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="oracle sample budget (CPU seconds)")
    ap.add_argument("--ref-seconds", type=float, default=60.0,
                    help="--impl reference: total oracle budget over the warm-up and timed steps (CPU seconds)")
    ap.add_argument("--e2e-chunks", type=int, default=40, help="head chunks of the host-buffer reuse step (one head each by default)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(vals, device=None):
    """Element-wise maximum of a list of floats over all ranks of the default
    process group (NCCL on GPUs, gloo on CPUs); the values unchanged without one."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in vals]
    t = torch.tensor([float(v) for v in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], bf16=j["bf16_tflops"], bf16_sus=j["bf16_tflops_sustained"],
                    sm_max_mhz=float(j.get("sm_max_mhz", 2070.0)), src="measured")
    except Exception:
        return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, sm_max_mhz=2070.0, src="fallback")


class Clocks:
    """nvidia-smi sampler running during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def flops_sparse(wl, K):
    return 4.0 * wl.B * wl.H * wl.N * K * wl.d


def flops_dense(wl):
    return 4.0 * wl.B * wl.H * wl.N * wl.N * wl.d


# ---------------------------------------------------------------- CPU oracle sample
def oracle_sample(wl, K, budget_s, seed=0):
    """Time the float64 oracle's reuse-step sparse attention (+ residual) on
    random query groups of one head until `budget_s` seconds have been spent
    (at least 2 groups); returns (seconds, groups, threads)."""
    import numpy as np
    import torch
    from oracle import mcs_oracle as orc
    from sparse_attention_diffusion_gb300 import synth

    one = wl.with_(B=1, H=1, grid=wl.grid)
    layer = synth.make_layer(one, device="cpu", seed=seed)
    q, k, v = (t[0, 0].float().numpy().astype(np.float64) for t in layer.cast())
    rng = np.random.default_rng(seed)
    resid = rng.standard_normal((wl.C, wl.d))
    n_groups = 0
    t0 = time.perf_counter()
    while n_groups < 2 or time.perf_counter() - t0 < budget_s:
        rows = rng.choice(wl.N, wl.C, replace=False)
        idx = np.sort(rng.choice(wl.N, K, replace=False))
        o = orc.sparse_attention(q[rows], k, v, idx) + resid
        n_groups += 1
    dt = time.perf_counter() - t0
    threads = torch.get_num_threads()
    try:
        from threadpoolctl import threadpool_info
        threads = max(int(i.get("num_threads", 1)) for i in threadpool_info()) or threads
    except Exception:
        threads = os.cpu_count() or threads
    return dt, n_groups, threads


def oracle_anchor_sample(wl, K, n_groups=8, seed=0):
    """Time the float64 oracle's anchor step on one head of the layer: the full
    PDDP grouping, then for `n_groups` seeded groups of it the dense rows and
    their LSE, the group scores, the top-K, the sparse rows and the residual, and
    the reuse step (sparse rows + residual) of the same groups. Returns seconds
    for the grouping of one head, per anchor group and per reuse group, and the
    threads used; the caller extrapolates to the layer."""
    import numpy as np
    import torch
    from oracle import mcs_oracle as orc
    from sparse_attention_diffusion_gb300 import synth

    one = wl.with_(B=1, H=1)
    layer = synth.make_layer(one, device="cpu", seed=seed)
    q, k, v = (t[0, 0].float().numpy().astype(np.float64) for t in layer.cast())
    N, C = wl.N, wl.C
    x = np.zeros((wl.N_pad, wl.d))
    x[:N] = q
    t0 = time.perf_counter()
    perm, _ = orc.pddp_groups(x, N, C, 20)
    t_pddp = time.perf_counter() - t0
    rng = np.random.default_rng(seed)
    groups = rng.choice(wl.G, min(n_groups, wl.G), replace=False)
    t_anchor = t_reuse = 0.0
    for g in groups:
        mem = perm[g * C:(g + 1) * C]
        mem = mem[mem < N]
        t1 = time.perf_counter()
        o_d, lse = orc.dense_attention(q[mem], k, v)
        S = orc.group_scores(q[mem], lse, k)
        idx = orc.topk_ascending(S, K)
        r = o_d - orc.sparse_attention(q[mem], k, v, idx)
        t2 = time.perf_counter()
        _ = orc.sparse_attention(q[mem], k, v, idx) + r
        t3 = time.perf_counter()
        t_anchor += t2 - t1
        t_reuse += t3 - t2
    threads = torch.get_num_threads()
    try:
        from threadpoolctl import threadpool_info
        threads = max(int(i.get("num_threads", 1)) for i in threadpool_info()) or threads
    except Exception:
        threads = os.cpu_count() or threads
    return dict(pddp_s=t_pddp, anchor_group_s=t_anchor / len(groups), reuse_group_s=t_reuse / len(groups),
                groups=len(groups), threads=threads)


def oracle_layer_ms(wl, smp):
    """Per-layer extrapolation of an oracle_anchor_sample: anchor and reuse ms."""
    BH = wl.B * wl.H
    return dict(anchor=(smp["pddp_s"] * BH + smp["anchor_group_s"] * BH * wl.G) * 1e3,
                reuse=smp["reuse_group_s"] * BH * wl.G * 1e3)


def run_reference(args, wl, K):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    per = []
    budget = max(0.5, args.ref_seconds / max(1, args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        dt, g, thr = oracle_sample(wl, K, budget, seed=i)
        if i >= args.warmup:
            per.append(dt / g)
    groups_layer = wl.B * wl.H * wl.G
    val = statistics.mean(per) * groups_layer * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": val, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "C": wl.C,
                   "density": float(wl.density), "K": K},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": thr, "kind": "oracle",
                         "sample": f"each step: random query groups of one head for ~{budget:.0f} s of float64 numpy "
                                   f"reuse-step sparse attention, extrapolated to {groups_layer} groups"},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU arm
RING_LAYERS = 3


def cache_ring_timing(desc, K, q, k, v, cache, stream):
    """Reuse steps whose meta-cache lives in pinned host memory: RING_LAYERS
    entries (copies of this layer's anchor cache, written out through the ring
    as an anchor step would), then passes over the layers where each layer's
    entry is already resident from the previous layer's prefetch and the next
    one is copied in during its kernel. Returns ms per layer of the second
    pass (device events on the compute stream)."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs
    ring = mcs.CacheRing(desc, K, RING_LAYERS, q.dtype)
    o = torch.empty_like(q)
    try:
        for l in range(RING_LAYERS):
            c = ring.acquire(l, fill=False, prefetch_next=False, stream=stream)
            for key in ("perm", "idx", "residual"):
                c[key].copy_(cache[key])
            ring.release(l, store=True, stream=stream)
        per_pass = []
        for _ in range(2):
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for l in range(RING_LAYERS):
                c = ring.acquire(l, fill=True, prefetch_next=True, stream=stream)
                mcs.mcs_sparse_attn_gather(desc, q, k, v, c["perm"], c["idx"], K, c["residual"], o, stream)
                ring.release(l, stream=stream)
            b.record(stream)
            torch.cuda.synchronize()
            per_pass.append(a.elapsed_time(b) / RING_LAYERS)
        mcs.mcs_check_status()
        return {"ms_per_layer": per_pass[-1], "first_pass_ms_per_layer": per_pass[0],
                "entry_bytes": ring.entry, "layers": RING_LAYERS,
                "note": "perm+idx+residual per layer in pinned host memory, two device slots; second pass over the layers timed"}
    finally:
        ring.close()


def stress_random_indices(desc, K, q, k, v, cache, stream, peak, wl, reps=5, warm=3, seed=1234):
    """The reuse kernel on the same layer with uniform random key sets instead of
    the anchor's selection: per (head, group) K distinct keys drawn uniformly
    (seeded), sorted ascending. The gathers then follow no locality of the
    selected keys; the arithmetic is unchanged."""
    import torch
    from sparse_attention_diffusion_gb300 import mcs

    idx = torch.empty_like(cache["idx"])
    rows = idx.numel() // K
    flat = idx.view(rows, K)
    gen = torch.Generator(device=q.device)
    gen.manual_seed(seed)
    for r0 in range(0, rows, 1024):
        r1 = min(rows, r0 + 1024)
        u = torch.rand((r1 - r0, wl.N), generator=gen, device=q.device)
        flat[r0:r1] = torch.sort(torch.topk(u, K, dim=1, sorted=False).indices.to(torch.int32), dim=1).values
        del u
    o = torch.empty_like(q)
    f = lambda: mcs.mcs_sparse_attn_gather(desc, q, k, v, cache["perm"], idx, K, cache["residual"], o)
    for _ in range(warm):
        f()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        f()
        b.record(stream)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    mcs.mcs_check_status()
    ms = statistics.median(ts)
    tf = flops_sparse(wl, K) / (ms * 1e-3) / 1e12
    del idx, o
    return {"what": "reuse kernel, uniform random sorted key sets (seeded), same layer and K",
            "ms": ms, "tflops": tf, "frac": tf / peak, "calls_ms": [round(x, 3) for x in ts], "stat": f"median of {reps}"}


def matched_density(desc, K, q, k, v, o_dense, cache, ws):
    """Group-shared selection on the benchmark layer with the PDDP groups (the
    anchor's cache) and with contiguous tile groups (identity perm): mean captured
    mass over groups and the anchor sparse output's relative error."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs

    def rel_err(R):
        return float(torch.linalg.vector_norm(R.float()) / torch.linalg.vector_norm(o_dense.float()))

    out = {"mass_group_pddp": float(cache["mass"].float().mean()), "rel_err_group_pddp": rel_err(cache["residual"])}
    G, N_pad = mcs.geometry(desc)
    perm = torch.arange(N_pad, dtype=torch.int32, device=q.device).expand_as(cache["perm"]).contiguous()
    idx, mass = torch.empty_like(cache["idx"]), torch.empty_like(cache["mass"])
    R = torch.empty_like(cache["residual"])
    mcs.mcs_anchor_select(desc, q, k, perm, None, K, idx, mass, ws)
    mcs.mcs_anchor_residual(desc, q, k, v, perm, idx, K, o_dense, R)
    mcs.mcs_check_status()
    out.update(mass_group_contiguous=float(mass.float().mean()), rel_err_group_contiguous=rel_err(R),
               note="mean over groups of the captured fraction of dense attention mass; error of the sparse "
                    "output before the residual")
    del perm, idx, mass, R
    torch.cuda.empty_cache()
    return out


def schedule_overhead(dev, peak_tflops, warm_iters=4):
    """The full meta-cache schedule on the 118,800-token layer (24 heads, 50 steps:
    5 dense warm-up steps, an anchor every 10 steps, reuse steps otherwise, drift
    0.05) at densities 0.15 and 0.25: total time including anchors and the anchor
    cost as equivalent extra density (post-warm-up time over 45 dense steps).
    Each density runs twice: grouping every anchor from the fixed start, and the
    amortised ("fast PDDP") grouping that starts each node from the previous
    anchor's direction with `warm_iters` iterations (`fast_pddp`: its grouping
    time, overhead, and the anchors' mean captured attention mass beside the
    cold run's)."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs, schedule, synth

    out = {"workload": synth.SCHEDULE_HY.name, "steps": 50, "warmup": 5, "period": 10}
    for rho in ("0.15", "0.25"):
        wl = synth.SCHEDULE_HY.with_(density=rho)
        res = {}
        for mode in ("cold", "warm"):
            layer = synth.make_layer(wl, device=dev)
            q0, _, _ = layer.cast()
            desc = mcs.desc_for(q0, wl.C)
            ml = schedule.MetaCacheLayer(desc, wl.K, q0.dtype, dev, warm_iters=warm_iters if mode == "warm" else None)
            del q0
            recs = schedule.run(ml, schedule.Schedule(steps=50, warmup=5, period=10), layer.cast,
                                lambda: layer.drift_step())
            mcs.mcs_check_status()
            res[mode] = (recs, ml.masses)
            del ml, layer
            torch.cuda.empty_cache()
        recs = res["cold"][0]
        t_dense = statistics.median(r.ms for r in recs[1:5])  # the first dense step pays one-off costs
        rho_eq, extra = schedule.anchor_overhead(recs, t_dense, float(wl.density), 5)
        kinds = {k: [r.ms for r in recs if r.kind == k] for k in ("dense", "anchor", "reuse")}
        n_post = len(recs) - 5
        n_anchor, n_reuse = len(kinds["anchor"]), len(kinds["reuse"])
        t_reuse = statistics.mean(kinds["reuse"])
        reuse_tf = flops_sparse(wl, wl.K) / (t_reuse * 1e-3) / 1e12
        wrecs, wmass = res["warm"]
        w_rho_eq, w_extra = schedule.anchor_overhead(wrecs, t_dense, float(wl.density), 5)
        w_anchor = [r for r in wrecs if r.kind == "anchor"]
        out[rho] = {"K": wl.K, "total_ms": sum(r.ms for r in recs), "post_warmup_ms": sum(r.ms for r in recs[5:]),
                    "dense_step_ms": t_dense, "anchor_step_ms": statistics.mean(kinds["anchor"]),
                    "anchor_stages_ms": {n: statistics.mean(r.stages[n] for r in recs if r.kind == "anchor")
                                         for n in ("pddp", "dense", "select", "anchor_residual")},
                    "reuse_step_ms": t_reuse, "reuse_tflops": reuse_tf, "reuse_frac": reuse_tf / peak_tflops,
                    "rho_eq": rho_eq, "anchor_overhead_points": 100.0 * extra,
                    # what an anchor that only ran dense attention would cost, with reuse at 1/rho of dense
                    "floor_points_dense_anchor_ideal_reuse": 100.0 * n_anchor * (1.0 - float(rho)) / n_post,
                    # the same with the measured reuse steps
                    "floor_points_dense_anchor_measured_reuse":
                        100.0 * ((n_anchor * t_dense + n_reuse * t_reuse) / (n_post * t_dense) - float(rho)),
                    "vs_all_dense": 50 * t_dense / sum(r.ms for r in recs),
                    "anchor_mass_mean": statistics.mean(res["cold"][1]),
                    "fast_pddp": {"warm_iters": warm_iters, "total_ms": sum(r.ms for r in wrecs),
                                  "anchor_overhead_points": 100.0 * w_extra,
                                  "pddp_ms_first_anchor": w_anchor[0].stages["pddp"],
                                  "pddp_ms_warm_anchors": statistics.mean(r.stages["pddp"] for r in w_anchor[1:]),
                                  "anchor_mass_mean": statistics.mean(wmass)}}
    return out


def sweep_table(dev, peak_tflops, peak_texp=None):
    """The density/tile sweep layer (16 heads, N = 65,536, bf16) for d and C in
    {64, 128}: groups and dense attention once per (d, C), then for every density
    the anchor selection and the reuse-step sparse kernel, timed with CUDA events
    (median of 5 launches) against the dense kernel (median of 3)."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs, synth

    stream = torch.cuda.current_stream()

    def timed(fn, n):
        ts = []
        for _ in range(n):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    rows = []
    for d, C in ((128, 128), (128, 64), (64, 128), (64, 64)):
        wl0 = synth.SWEEP.with_(d=d, C=C)
        layer = synth.make_layer(wl0, device=dev)
        q, k, v = layer.cast()
        del layer
        desc = mcs.desc_for(q, C)
        o_dense = torch.empty_like(q)
        lse = torch.empty((wl0.B, wl0.H, wl0.N), dtype=torch.float32, device=dev)
        o = torch.empty_like(q)
        cache = mcs.alloc_cache(desc, wl0.N, q.dtype, device=dev)
        ws = mcs.workspace(desc, wl0.N, device=dev)
        mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
        t_dense = timed(lambda: mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse), 3)
        for rho in ("0.05", "0.1", "0.15", "0.2", "0.3", "0.5", "1.0"):
            K = synth.SWEEP.with_(d=d, C=C, density=rho).K
            idx = cache["idx"].view(-1)[: wl0.B * wl0.H * wl0.G * K].view(wl0.B, wl0.H, wl0.G, K)
            mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, idx, cache["mass"], ws)
            mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], idx, K, o_dense, cache["residual"])
            t = timed(lambda: mcs.mcs_sparse_attn_gather(desc, q, k, v, cache["perm"], idx, K, cache["residual"], o), 5)
            tf = 4.0 * wl0.B * wl0.H * wl0.N * K * d / (t * 1e-3) / 1e12
            texp = wl0.B * wl0.H * wl0.N * K / (t * 1e-3) / 1e12   # kept (real query, key) exponentials
            rows.append({"d": d, "C": C, "density": float(rho), "K": K, "sparse_ms": t, "tflops": tf,
                         "frac": tf / peak_tflops, "exp_frac": (texp / peak_texp) if peak_texp else None,
                         "dense_ms": t_dense, "speedup_vs_dense": t_dense / t, "ideal_speedup": 1.0 / float(rho)})
        mcs.mcs_check_status()
        del q, k, v, o_dense, lse, o, cache, ws
        torch.cuda.empty_cache()
    table = {}
    for r in rows:
        t = table.setdefault(f"d{r['d']}-c{r['C']}", {"density": [], "K": [], "sparse_ms": [], "tflops": [],
                                                       "frac": [], "exp_frac": [], "speedup_vs_dense": [],
                                                       "dense_ms": r["dense_ms"]})
        for key in ("density", "K"):
            t[key].append(r[key])
        for key in ("sparse_ms", "tflops", "frac", "exp_frac", "speedup_vs_dense"):
            t[key].append(_r(r[key]))
    return {"workload": synth.SWEEP.name, "B": 1, "H": synth.SWEEP.H, "N": synth.SWEEP.N,
            "peak_kind": "measured sustained bf16",
            "exp_frac_of": "kept exponentials (B*H*N*K per launch) per second over the measured ex2 peak",
            "by_shape": table}


def exp_peak(dev, sm_max_mhz):
    """Peak exponential rate (T exp/s): the library's ex2 diagnostic measures
    exponentials per SM clock (one CTA per SM), scaled by the SM count and the
    maximum SM clock."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs

    per_clk = mcs.ex2_per_clock_per_sm()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    return {"ex2_per_clk_sm": per_clk, "sms": sms, "sm_mhz": sm_max_mhz,
            "peak_texp_s": per_clk * sms * sm_max_mhz * 1e6 / 1e12,
            "how": "mcs_selftest_ex2_rate: 1,024 threads x 8 chains of ex2.approx.ftz.f32 per CTA, one CTA per SM, "
                   "median over SMs of exponentials / clock64 cycles"}


def fp32_alu_peak_tflops(sm_max_mhz):
    """FP32 FMA peak of the CUDA cores: SMs x 128 fp32 lanes x 2 FLOP x max SM clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * sm_max_mhz * 1e6 / 1e12


def config_measure(wl, dev, pk, n_reuse, cpu=True, reps=3, warm=2):
    """One anchor step and `n_reuse` drifted reuse steps of a layer, repeated
    (warm untimed + reps timed): per-stage ms (CUDA events, median), the reuse
    kernel's kept TFLOP/s and roofline fraction, its speedup over the dense
    kernel, and the float64 oracle on the host cores (the whole layer when it has
    one head of at most 4,096 tokens, else one head's grouping and 8 sampled
    groups, extrapolated)."""
    import torch

    from sparse_attention_diffusion_gb300 import mcs, schedule, synth

    layer = synth.make_layer(wl, device=dev)
    steps = [layer.cast()]
    for _ in range(n_reuse):
        layer.drift_step()
        steps.append(layer.cast())
    del layer
    q, k, v = steps[0]
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    ml = schedule.MetaCacheLayer(desc, K, q.dtype, dev)
    stream = torch.cuda.current_stream()
    ev = {n: [] for n in ("pddp", "dense", "select", "anchor_residual", "sparse")}

    def timer(name, fn, keep=True):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        if keep:
            ev[name].append((a, b))

    for rep in range(warm + reps):
        keep = rep >= warm
        ml.anchor(q, k, v, lambda n, fn: timer(n, fn, keep))
        for (q2, k2, v2) in steps[1:]:
            timer("sparse", lambda: ml.reuse(q2, k2, v2), keep)
    torch.cuda.synchronize()
    mcs.mcs_check_status()
    ms = {n: statistics.median(a.elapsed_time(b) for a, b in v) for n, v in ev.items()}
    bf16 = wl.dtype == "bf16"
    peak = pk["bf16_sus"] if bf16 else fp32_alu_peak_tflops(pk.get("sm_max_mhz", 2070.0))
    tf = flops_sparse(wl, K) / (ms["sparse"] * 1e-3) / 1e12
    out = {"workload": wl.name, "H": wl.H, "N": wl.N, "d": wl.d, "C": wl.C, "dtype": wl.dtype, "K": K,
           "steps": f"1 anchor + {n_reuse} reuse", "stages_ms": ms,
           "anchor_ms": sum(ms[n] for n in ("pddp", "dense", "select", "anchor_residual")),
           "sparse_tflops": tf, "frac": tf / peak,
           "peak": {"value": peak, "kind": f"{pk['src']} sustained bf16" if bf16 else
                    "fp32 FMA lanes x 2 x max SM clock (derived)"},
           "dense_tflops": flops_dense(wl) / (ms["dense"] * 1e-3) / 1e12,
           "speedup_vs_dense": ms["dense"] / ms["sparse"], "ideal_speedup": 1.0 / float(wl.density)}
    del ml, steps, q, k, v
    torch.cuda.empty_cache()
    if cpu:
        out["cpu_baseline"] = oracle_config(wl, K)
    return out


def oracle_config(wl, K):
    """The float64 oracle on the host cores for a config line: the whole layer
    (anchor_head + reuse_head) for one head of <= 4,096 tokens, else one head's
    grouping plus 8 sampled groups extrapolated to the layer."""
    import numpy as np
    import torch
    from oracle import mcs_oracle as orc
    from sparse_attention_diffusion_gb300 import synth

    if wl.B * wl.H == 1 and wl.N <= 4096:
        layer = synth.make_layer(wl, device="cpu")
        q, k, v = (t[0, 0].float().numpy().astype(np.float64) for t in layer.cast())
        t0 = time.perf_counter()
        ref = orc.anchor_head(q, k, v, wl.C, K)
        t1 = time.perf_counter()
        orc.reuse_head(q, k, v, ref["perm"], ref["idx"], ref["residual"], wl.C)
        t2 = time.perf_counter()
        return {"anchor_ms": (t1 - t0) * 1e3, "reuse_ms": (t2 - t1) * 1e3, "cores": torch.get_num_threads(),
                "kind": "oracle", "sample": "whole layer (one head), float64 numpy"}
    smp = oracle_anchor_sample(wl, K)
    ext = oracle_layer_ms(wl, smp)
    return {"anchor_ms": ext["anchor"], "reuse_ms": ext["reuse"], "cores": smp["threads"], "kind": "oracle",
            "sample": f"one head: full grouping ({smp['pddp_s']:.1f} s) + {smp['groups']} sampled groups "
                      f"(dense rows, LSE, scores, top-K, sparse, residual; reuse), float64 numpy, "
                      f"extrapolated to {wl.B * wl.H} heads x {wl.G} groups"}


def _r(x, n=4):
    """Round to n significant digits (compact summary)."""
    if x is None or not isinstance(x, (int, float)) or x == 0 or not math.isfinite(x):
        return x
    return round(x, -int(math.floor(math.log10(abs(x)))) + n - 1)


def run_mcs(args, wl, K):
    import torch
    import torch.distributed as dist

    from sparse_attention_diffusion_gb300 import mcs, synth

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", init_method="env://", rank=rank, world_size=world)
    mcs.load(build_if_missing=True)
    dev = torch.device("cuda", local)

    layer = synth.make_layer(wl, device=dev, seed=wl.seed + rank)
    q, k, v = layer.cast()
    layer.drift_step()
    q2, k2, v2 = layer.cast()
    del layer
    desc = mcs.desc_for(q, wl.C)
    G, N_pad = mcs.geometry(desc)
    cache = mcs.alloc_cache(desc, K, q.dtype, device=dev)
    ws = mcs.workspace(desc, K, device=dev)
    o_dense = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device=dev)
    o = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    stages = ("pddp", "dense", "select", "anchor_residual", "sparse")
    ev = {s: [] for s in stages}

    def timed(name, fn, record):
        if record:
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev[name].append((a, b))
        else:
            fn()

    def step(record):
        timed("pddp", lambda: mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws), record)
        timed("dense", lambda: mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse), record)
        timed("select", lambda: mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"],
                                                      cache["mass"], ws), record)
        timed("anchor_residual", lambda: mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], cache["idx"], K,
                                                                 o_dense, cache["residual"]), record)
        for _ in range(REUSE_PER_STEP):
            timed("sparse", lambda: mcs.mcs_sparse_attn_gather(desc, q2, k2, v2, cache["perm"], cache["idx"], K,
                                                               cache["residual"], o), record)

    for _ in range(args.warmup):
        step(False)
    mcs.mcs_check_status()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    n0 = mcs.mcs_launch_count()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with Clocks(local) as clk:
        t_start.record(stream)
        for _ in range(args.steps):
            step(True)
        t_end.record(stream)
        torch.cuda.synchronize()
    launches = mcs.mcs_launch_count() - n0
    mcs.mcs_check_status()
    total_ms = t_start.elapsed_time(t_end)
    stage_ms = {s: [a.elapsed_time(b) for a, b in ev[s]] for s in stages}
    sparse_ms = statistics.mean(stage_ms["sparse"])
    total_ms, sparse_ms = max_over_ranks([total_ms, sparse_ms], dev)

    e2e_ms, e2e_calls = None, []
    if not args.no_e2e:
        # end to end through the C ABI from pinned host buffers: one call copies q, k, v in,
        # runs the reuse step and copies o out, pipelined over head chunks
        hq, hk, hv = (x.cpu().pin_memory() for x in (q2, k2, v2))
        ho = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        hws = mcs.host_gather_workspace(desc, args.e2e_chunks)
        mcs.mcs_sparse_attn_gather_host(desc, hq, hk, hv, cache["perm"], cache["idx"], K, cache["residual"], ho, hws,
                                        args.e2e_chunks, stream)
        # per-call device times; the median rejects a call slowed by other traffic on the host link
        e2e_calls = []
        for _ in range(5):
            torch.cuda.synchronize()
            ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ea.record(stream)
            mcs.mcs_sparse_attn_gather_host(desc, hq, hk, hv, cache["perm"], cache["idx"], K, cache["residual"], ho, hws,
                                            args.e2e_chunks, stream)
            eb.record(stream)
            torch.cuda.synchronize()
            e2e_calls.append(ea.elapsed_time(eb))
        mcs.mcs_check_status()
        e2e_ms = statistics.median(e2e_calls)
        del hws
    if e2e_ms is not None:
        e2e_ms = max_over_ranks([e2e_ms], dev)[0]
    if world > 1:
        dist.barrier()

    if rank == 0:
        pk = peaks()
        fl = flops_sparse(wl, K)
        achieved = fl / (sparse_ms * 1e-3) / 1e12
        dense_ms = statistics.mean(stage_ms["dense"])
        clocks = clk.summary()
        line = {
            "metric": METRIC,
            "value": sparse_ms / world,
            "unit": UNIT,
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps,
            "higher_is_better": False,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "bf16",
            "data": "synthetic (seeded smooth-field + noise generator, generated on the device)",
            "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "N": wl.N, "grid": list(wl.grid), "d": wl.d,
                       "C": wl.C, "G": G, "density": float(wl.density), "K": K,
                       "step": f"1 anchor (pddp, dense+lse, select, anchor residual) + {REUSE_PER_STEP} reuse",
                       "l2": "inputs larger than L2 (q/k/v 774 MB each; 40 heads cycled per kernel)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "tflops": achieved,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_sus"], "unit": "TFLOP/s",
                         "frac": achieved / pk["bf16_sus"],
                         "traffic": (SPARSE_TRAFFIC_BYTES_H40 * wl.H / 40
                                     if (SPARSE_TRAFFIC_BYTES_H40 is not None and wl.name == "kernel-bench-720p"
                                         and wl.d == 128 and wl.C == 128 and K == 15120) else None),
                         "kernel": f"attn_sparse_cs_kernel<{wl.d}, add-residual, "
                                   + ("64-query groups>" if wl.C <= 64 else "128-query groups>"),
                         "peak_kind": f"{pk['src']} sustained bf16",
                         "algorithmic": "4*B*H*N*K*d kept FLOPs per launch"},
            "stages_ms": {s: statistics.mean(v) for s, v in stage_ms.items()},
            "dense_ms": dense_ms,
            "speedup_vs_dense": dense_ms / sparse_ms,
            "ideal_speedup": 1.0 / float(wl.density),
            "fraction_of_ideal": dense_ms / sparse_ms * float(wl.density),
            "dense_tflops": flops_dense(wl) / (dense_ms * 1e-3) / 1e12,
            "gpu_launches": launches,
            "e2e": None if e2e_ms is None else {
                    "value": e2e_ms / world, "unit": UNIT, "h2d_bytes_per_step": 3 * q2.numel() * q2.element_size(),
                    "d2h_bytes_per_step": o.numel() * o.element_size(),
                    "api": f"mcs_sparse_attn_gather_host, pinned host q/k/v/o, {args.e2e_chunks} head chunks",
                    "calls_ms": [round(x, 3) for x in e2e_calls], "stat": "median of 5 calls"},
            "clocks": clocks,
        }
        if world == 1 and not args.no_matched:
            line["matched_density"] = matched_density(desc, K, q, k, v, o_dense, cache, ws)
        if world == 1 and not args.no_stress:
            line["stress_random_idx"] = stress_random_indices(desc, K, q2, k2, v2, cache, stream, pk["bf16_sus"], wl)
        if world == 1 and not args.no_ring:
            ring = cache_ring_timing(desc, K, q2, k2, v2, cache, stream)
            ring["resident_ms_per_layer"] = sparse_ms
            line["cache_ring"] = ring
        if world == 1 and not args.no_schedule:
            line["anchor_overhead"] = schedule_overhead(dev, pk["bf16_sus"])
        ep = exp_peak(dev, pk["sm_max_mhz"])
        texp = wl.B * wl.H * wl.N * K / (sparse_ms * 1e-3) / 1e12
        line["exp_unit"] = dict(ep, sparse_texp_s=texp, sparse_exp_frac=texp / ep["peak_texp_s"])
        if world == 1 and not args.no_sweep:
            line["sweep"] = sweep_table(dev, pk["bf16_sus"], ep["peak_texp_s"])
        if world == 1 and not args.no_configs:
            line["configs"] = {c.name: config_measure(c, dev, pk, n, cpu=not args.no_cpu_baseline)
                               for c, n in ((synth.TINY, 1), (synth.WAN13_480P, 4))}
        if world == 1 and not args.no_cpu_baseline:
            dt, g, thr = oracle_sample(wl, K, args.cpu_seconds)
            val = dt / g * wl.B * wl.H * wl.G * 1e3
            line["cpu_baseline"] = {"value": val, "unit": UNIT, "cores": thr, "kind": "oracle",
                                    "sample": f"{g} random query groups of one head, reuse-step sparse attention "
                                              f"in float64 numpy ({dt:.1f} s), extrapolated to "
                                              f"{wl.B * wl.H * wl.G} groups"}
            smp = oracle_anchor_sample(wl, K)
            ext = oracle_layer_ms(wl, smp)
            line["cpu_baseline"]["anchor"] = {
                "value": ext["anchor"], "unit": "ms/layer", "cores": smp["threads"],
                "sample": f"one head: full grouping ({smp['pddp_s']:.1f} s) + {smp['groups']} sampled groups "
                          f"(dense rows, LSE, scores, top-K, sparse, residual), float64 numpy, extrapolated to "
                          f"{wl.B * wl.H} heads x {wl.G} groups"}
        line["per_config"] = summary(line, wl)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def summary(line, wl):
    """Compact per-config digest, printed last in the JSON line: ms per stage,
    the reuse kernel's kept TFLOP/s and roofline fraction, its speedup over the
    dense kernel, and the oracle's time on the host cores."""
    out = {}
    for name, c in (line.get("configs") or {}).items():
        cb = c.get("cpu_baseline") or {}
        out[name] = {"stages_ms": {k: _r(v) for k, v in c["stages_ms"].items()}, "sparse_tflops": _r(c["sparse_tflops"]),
                     "frac": _r(c["frac"], 3), "speedup": _r(c["speedup_vs_dense"], 3),
                     "cpu_ms": {"anchor": _r(cb.get("anchor_ms")), "reuse": _r(cb.get("reuse_ms"))}}
    cb = line.get("cpu_baseline") or {}
    out[wl.name] = {"stages_ms": {k: _r(v) for k, v in line["stages_ms"].items()}, "sparse_tflops": _r(line["tflops"]),
                    "frac": _r(line["roofline"]["frac"], 3), "speedup": _r(line["speedup_vs_dense"], 3),
                    "cpu_ms": {"anchor": _r((cb.get("anchor") or {}).get("value")), "reuse": _r(cb.get("value"))}}
    st = line.get("stress_random_idx")
    if st:
        out[wl.name]["random_idx"] = {"ms": _r(st["ms"]), "frac": _r(st["frac"], 3)}
    ao = line.get("anchor_overhead")
    if ao:
        out[ao["workload"]] = {rho: {"total_ms": _r(v["total_ms"]), "overhead_pts": _r(v["anchor_overhead_points"], 3),
                                     "floor_pts": _r(v["floor_points_dense_anchor_ideal_reuse"], 3),
                                     "reuse_tflops": _r(v["reuse_tflops"]), "frac": _r(v["reuse_frac"], 3),
                                     "vs_dense": _r(v["vs_all_dense"], 3),
                                     "pddp_ms": _r(v["anchor_stages_ms"]["pddp"], 3),
                                     "mass": _r(v["anchor_mass_mean"], 4),
                                     "fast_pddp": {"overhead_pts": _r(v["fast_pddp"]["anchor_overhead_points"], 3),
                                                   "pddp_ms": _r(v["fast_pddp"]["pddp_ms_warm_anchors"], 3),
                                                   "mass": _r(v["fast_pddp"]["anchor_mass_mean"], 4)}}
                               for rho, v in ao.items() if isinstance(v, dict) and "total_ms" in v}
    sw = line.get("sweep")
    if sw:
        out[sw["workload"]] = {shape: {"frac": t["frac"], "exp_frac": t.get("exp_frac"),
                                       "speedup": [_r(x, 3) for x in t["speedup_vs_dense"]]}
                               for shape, t in sw["by_shape"].items()}
    return out


def main():
    args = parse()
    from sparse_attention_diffusion_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.density:
        wl = wl.with_(density=args.density)
    if args.heads:
        wl = wl.with_(H=args.heads)
    if args.group_size:
        wl = wl.with_(C=args.group_size)
    K = wl.K
    if args.impl == "reference":
        run_reference(args, wl, K)
    else:
        run_mcs(args, wl, K)


if __name__ == "__main__":
    main()
