"""Meta-cache denoising schedule over the C ABI [MC-Sparse summary: grouping and
exact selection run only on anchor steps; later steps reuse the query groups, the
KV indices and the output residual; groups, indices and residual refresh together].

A schedule of `steps` denoising steps for one attention layer:
  * the first `warmup` steps run dense attention;
  * step `warmup + i*period` is an anchor: PDDP grouping, dense attention + LSE,
    pass-2 column sums + exact top-K, anchor sparse attention + residual store;
    the anchor's output is the dense output;
  * every other step is a reuse step: sparse attention of the current Q/K/V over
    the cached groups and indices, plus the cached residual.
The warm-up length and anchor period are not on the pages; the 118,800-token
schedule workload uses 5 warm-up steps and an anchor every 10 steps.

Inputs drift between steps through a caller-supplied callback (the generator's
variance-preserving drift), which runs outside the per-step kernel timing.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import mcs


@dataclass
class StepRecord:
    kind: str          # "dense" | "anchor" | "reuse"
    ms: float
    stages: dict = field(default_factory=dict)


@dataclass
class Schedule:
    steps: int = 50
    warmup: int = 5
    period: int = 10

    def kind(self, t: int) -> str:
        if t < self.warmup:
            return "dense"
        return "anchor" if (t - self.warmup) % self.period == 0 else "reuse"


class MetaCacheLayer:
    """One attention layer with its caller-owned meta-cache buffers.

    warm_iters: None groups every anchor from the fixed start (desc.pddp_iters
    power iterations); an integer keeps the grouping's per-node directions
    between anchors, so that every anchor after the first starts each node from
    the previous anchor's direction and runs warm_iters iterations ("fast PDDP",
    the amortised grouping). `masses` collects each anchor's mean captured
    attention mass (untimed), the quality measure of the grouping."""

    def __init__(self, desc: mcs.mcs_desc, K: int, dtype, device, warm_iters=None):
        self.desc, self.K = desc, K
        self.cache = mcs.alloc_cache(desc, K, dtype, device=device)
        self.ws = mcs.workspace(desc, K, device=device)
        shape = (desc.B, desc.H, desc.N, desc.d)
        self.o_dense = torch.empty(shape, dtype=dtype, device=device)
        self.lse = torch.empty((desc.B, desc.H, desc.N), dtype=torch.float32, device=device)
        self.out = torch.empty(shape, dtype=dtype, device=device)
        self.warm_iters = warm_iters
        self.masses = []
        self._anchors = 0
        if warm_iters is not None:
            self.dirs = mcs.pddp_dirs(desc, device=device)
            self.desc_warm = mcs.make_desc(desc.B, desc.H, desc.N, desc.d, desc.C, dtype, desc.scale, warm_iters)

    def group(self, q):
        c = self.cache
        if self.warm_iters is None:
            mcs.mcs_group_pddp(self.desc, q, c["perm"], c["group_of"], self.ws)
        elif self._anchors == 0:
            mcs.mcs_group_pddp_warm(self.desc, q, None, self.dirs, c["perm"], c["group_of"], self.ws)
        else:
            mcs.mcs_group_pddp_warm(self.desc_warm, q, self.dirs, self.dirs, c["perm"], c["group_of"], self.ws)
        self._anchors += 1

    def dense(self, q, k, v):
        mcs.mcs_dense_attn(self.desc, q, k, v, self.o_dense, self.lse)
        return self.o_dense

    def anchor(self, q, k, v, timer=None):
        c = self.cache
        t = timer or (lambda name, fn: fn())
        t("pddp", lambda: self.group(q))
        t("dense", lambda: mcs.mcs_dense_attn(self.desc, q, k, v, self.o_dense, self.lse))
        t("select", lambda: mcs.mcs_anchor_select(self.desc, q, k, c["perm"], self.lse, self.K, c["idx"], c["mass"],
                                                  self.ws))
        t("anchor_residual", lambda: mcs.mcs_anchor_residual(self.desc, q, k, v, c["perm"], c["idx"], self.K,
                                                             self.o_dense, c["residual"]))
        return self.o_dense

    def after_step(self, kind, q):
        """Untimed work after a step: the anchor's mean captured mass."""
        if kind == "anchor":
            self.masses.append(float(self.cache["mass"].float().mean()))

    def reuse(self, q, k, v):
        c = self.cache
        mcs.mcs_sparse_attn_gather(self.desc, q, k, v, c["perm"], c["idx"], self.K, c["residual"], self.out)
        return self.out


def run(layer: MetaCacheLayer, sched: Schedule, inputs, advance, on_output=None):
    """Run the schedule. `inputs()` returns the current (q, k, v); `advance()`
    drifts them to the next step. Returns the per-step records (CUDA-event ms)."""
    stream = torch.cuda.current_stream()
    recs = []
    for t in range(sched.steps):
        q, k, v = inputs()
        kind = sched.kind(t)
        stages = {}
        ev = []

        def timer(name, fn):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ev.append((name, a, b))

        a0, b0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        if kind == "dense":
            out = layer.dense(q, k, v)
        elif kind == "anchor":
            out = layer.anchor(q, k, v, timer)
        else:
            out = layer.reuse(q, k, v)
        b0.record(stream)
        if hasattr(layer, "after_step"):
            layer.after_step(kind, q)
        if on_output is not None:
            on_output(t, kind, out)
        recs.append((kind, a0, b0, ev))
        advance()
    torch.cuda.synchronize()
    out = []
    for kind, a0, b0, ev in recs:
        out.append(StepRecord(kind, a0.elapsed_time(b0), {n: a.elapsed_time(b) for n, a, b in ev}))
    return out


def anchor_overhead(records, t_dense_ms: float, density: float, warmup: int):
    """Anchor cost spread over the trajectory, as extra density points: the
    post-warm-up time divided by what dense attention would have cost on those
    steps gives an equivalent density; the overhead is that minus the density."""
    post = [r for r in records[warmup:]]
    t_post = sum(r.ms for r in post)
    rho_eq = t_post / (len(post) * t_dense_ms)
    return rho_eq, rho_eq - density
