"""The meta-cache schedule end to end (dense warm-up, anchors, reuse steps with
drifting inputs) on the tiny fp32 layer, step by step against the oracle's own
schedule (its own groups, indices and residuals): every step within 1e-5."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, schedule, synth
from tests import parity

pytestmark = pytest.mark.gpu


def test_schedule_tiny_f32():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.TINY
    layer = synth.make_layer(wl)
    sched = schedule.Schedule(steps=8, warmup=2, period=3)     # anchors at steps 2 and 5
    state = {}

    def inputs():
        state["qkv"] = tuple(t.cuda() for t in layer.cast())
        return state["qkv"]

    outs, kinds, qkvs = [], [], []

    def on_output(t, kind, out):
        outs.append(out.clone())
        kinds.append(kind)
        qkvs.append(tuple(x.clone() for x in state["qkv"]))

    desc = mcs.desc_for(layer.q0, wl.C)
    desc.dtype = mcs.MCS_F32
    ml = schedule.MetaCacheLayer(desc, wl.K, torch.float32, "cuda")
    recs = schedule.run(ml, sched, inputs, lambda: layer.drift_step(), on_output)
    mcs.mcs_check_status()
    assert [r.kind for r in recs] == ["dense", "dense", "anchor", "reuse", "reuse", "anchor", "reuse", "reuse"]
    assert all(r.ms > 0 for r in recs)
    cache = None
    for t, (kind, out, qkv) in enumerate(zip(kinds, outs, qkvs)):
        q, k, v = (parity.f64(x[0, 0]) for x in qkv)
        if kind == "dense":
            want, _ = orc.dense_attention(q, k, v)
        elif kind == "anchor":
            cache = orc.anchor_head(q, k, v, wl.C, wl.K)
            want = cache["o_dense"]
        else:
            want = orc.reuse_head(q, k, v, cache["perm"], cache["idx"], cache["residual"], wl.C)
        parity.assert_close(parity.f64(out[0, 0]), want, "f32", f"step {t} ({kind})")
    rho_eq, extra = schedule.anchor_overhead(recs, np.mean([r.ms for r in recs[:2]]), float(wl.density), 2)
    assert rho_eq > 0
