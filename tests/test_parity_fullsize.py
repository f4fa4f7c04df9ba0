"""Full-size layers in the launch configuration the benchmark uses: the 720p
kernel-benchmark layer (B=1, H=40, N=75,600 on a 21x45x80 grid, d=128, bf16,
C=128, K=15,120), the Wan2.1-1.3B-shaped 480p layer (H=12, N=32,768, K=6,554),
the 118,800-token schedule layer (H=24, 929 groups with 112 pad rows,
K=17,820) and the density sweep's layer (H=16, N=65,536, K=13,108) with
64-query groups at d = 128 and d = 64. The whole path runs on the GPU (grouping, dense attention + LSE,
pass-2 selection, anchor residual, one drifted reuse step), and sampled heads,
groups and rows are checked one by one against the float64 oracle fed the very
tensors the GPU received (the oracle cannot run a whole layer in a test)."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

GROUPS_PER_HEAD = 2        # sampled groups per head (selection, residual, reuse)
ROWS_PER_HEAD = 64         # sampled query rows per head (dense output and LSE)
LAYERS = {
    "kernel-bench-720p": synth.KBENCH_720P,
    "wan2.1-1.3b-480p": synth.WAN13_480P,
    "schedule-118800": synth.SCHEDULE_HY,
    # the density sweep's 65,536-token layer with 64-query groups (each query on two
    # lanes of the sparse kernel), at both head dims, density 0.2
    "sweep-65536-d128-c64": synth.SWEEP.with_(C=64),
    "sweep-65536-d64-c64": synth.SWEEP.with_(d=64, C=64),
}


@pytest.fixture(scope="module", params=list(LAYERS))
def run(request):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = LAYERS[request.param]
    heads = (0, wl.H // 2 - 3, wl.H - 1)   # first, middle, last
    layer = synth.make_layer(wl, device="cuda")
    q, k, v = layer.cast()
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    o_dense = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], cache["idx"], K, o_dense, cache["residual"])
    layer.drift_step()
    q2, k2, v2 = layer.cast()
    o_reuse = torch.empty_like(q2)
    mcs.mcs_sparse_attn_gather(desc, q2, k2, v2, cache["perm"], cache["idx"], K, cache["residual"], o_reuse)
    mcs.mcs_check_status()
    torch.cuda.synchronize()
    host = lambda t, h: parity.f64(t[0, h])
    out = dict(wl=wl, K=K, heads={})
    rng = np.random.default_rng(20261202)
    for h in heads:
        groups = rng.choice(wl.G, GROUPS_PER_HEAD, replace=False)
        if wl.N_pad > wl.N:
            groups[-1] = wl.G - 1          # the group that holds the pad rows
        out["heads"][h] = dict(
            q=host(q, h), k=host(k, h), v=host(v, h), q2=host(q2, h), k2=host(k2, h), v2=host(v2, h),
            o_dense=host(o_dense, h), lse=lse[0, h].double().cpu().numpy(), o_reuse=host(o_reuse, h),
            residual=host(cache["residual"], h), perm=cache["perm"][0, h].cpu().numpy(),
            group_of=cache["group_of"][0, h].cpu().numpy(), idx=cache["idx"][0, h].cpu().numpy(),
            mass=cache["mass"][0, h].cpu().numpy(),
            rows=rng.choice(wl.N, ROWS_PER_HEAD, replace=False), groups=groups)
    del q, k, v, q2, k2, v2, o_dense, lse, o_reuse, cache, ws, layer
    torch.cuda.empty_cache()
    return out


def test_groups_fullsize(run):
    """Each sampled head's grouping against the oracle's, split by split: the
    fraction of identical groups, and for every split where the GPU's left child
    differs, the oracle's own key gap there (fp32 accumulation on bf16 inputs may
    only differ from the float64 oracle where that gap is small)."""
    wl = run["wl"]
    report = []
    for h, d in run["heads"].items():
        parity.assert_valid_partition(d["perm"], wl.N, wl.C)
        gid = np.empty(wl.N, dtype=np.int64)
        for g in range(wl.G):
            gid[parity.group_members(d["perm"], g, wl.C, wl.N)] = g
        assert np.array_equal(d["group_of"], gid), f"head {h}: group_of disagrees with perm"
        x = np.zeros((wl.N_pad, wl.d))
        x[:wl.N] = d["q"]
        agree, _, bad = parity.pddp_split_report(d["perm"], x, wl.N, wl.C)
        report.append((h, agree, bad))
    for h, agree, bad in report:
        gaps = ", ".join(f"node(g0={b['g0']}, n={b['n']}): gap {b['gap']:.2e} sd, {b['moved']} moved" for b in bad)
        print(f"{wl.name} head {h}: group agreement {agree:.4f}; {len(bad)} disagreeing splits [{gaps}]")
    for h, agree, bad in report:
        assert agree >= parity.PDDP_AGREE_FLOOR_FULLSIZE, f"head {h}: agreement {agree:.4f}"
        for b in bad:
            assert b["gap"] <= parity.PDDP_GAP_MAX, f"head {h}: disagreeing split with oracle gap {b['gap']:.3g} sd"


def test_dense_rows_fullsize(run):
    for h, d in run["heads"].items():
        rows = d["rows"]
        o_ref, lse_ref = orc.dense_attention(d["q"][rows], d["k"], d["v"])
        parity.assert_close(d["o_dense"][rows], o_ref, "bf16", f"dense rows head {h}")
        assert np.abs(d["lse"][rows] - lse_ref).max() < 1e-3, f"head {h}: lse"


def test_selection_residual_reuse_fullsize(run):
    wl, K = run["wl"], run["K"]
    for h, d in run["heads"].items():
        for g in d["groups"]:
            mem = parity.group_members(d["perm"], g, wl.C, wl.N)
            # pass 2 on this group with the oracle's own pass-1 lse of its queries
            _, lse_g = orc.dense_attention(d["q"][mem], d["k"], np.zeros((wl.N, 1)))
            S = orc.group_scores(d["q"][mem], lse_g, d["k"])
            parity.check_selection(d["idx"][g], S, K, mem.size, f"head {h} group {g}")
            assert abs(d["mass"][g] - orc.captured_mass(S, d["idx"][g], mem.size)) < 1e-4
            # residual of the anchor step (the GPU's own dense output, as the path uses it)
            r_ref = d["o_dense"][mem] - orc.sparse_attention(d["q"][mem], d["k"], d["v"], d["idx"][g])
            parity.assert_close(d["residual"][mem], r_ref, "bf16", f"residual head {h} group {g}")
            # reuse step on the drifted inputs over the cached group, indices and residual
            want = orc.sparse_attention(d["q2"][mem], d["k2"], d["v2"], d["idx"][g]) + d["residual"][mem]
            parity.assert_close(d["o_reuse"][mem], want, "bf16", f"reuse head {h} group {g}")


@pytest.mark.parametrize("d,C", [(128, 128), (64, 64)])
def test_sweep_layer_k_equals_n(d, C):
    """The 65,536-token sweep layer at density 1.0 (K = N): the anchor's sparse
    output reproduces dense attention, so the residual is zero, and a reuse step
    on the unchanged inputs reproduces the dense output [residual paragraph]."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.SWEEP.with_(d=d, C=C, density="1.0")
    layer = synth.make_layer(wl, device="cuda")
    q, k, v = layer.cast()
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    assert K == wl.N
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    o_dense = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], cache["idx"], K, o_dense, cache["residual"])
    o_reuse = torch.empty_like(q)
    mcs.mcs_sparse_attn_gather(desc, q, k, v, cache["perm"], cache["idx"], K, cache["residual"], o_reuse)
    mcs.mcs_check_status()
    want_idx = torch.arange(wl.N, dtype=torch.int32, device="cuda")
    assert torch.equal(cache["idx"], want_idx.expand_as(cache["idx"])), "K = N must select every key"
    assert torch.allclose(cache["mass"], torch.ones_like(cache["mass"]), atol=1e-4), "K = N keeps all the mass"
    R = cache["residual"].float()
    err = (o_reuse.float() - o_dense.float()).abs()
    assert float(R.abs().max()) <= 2e-2 and float(R.pow(2).mean().sqrt()) <= 5e-3, "residual not ~0"
    assert float(err.max()) <= 2e-2 and float(err.pow(2).mean().sqrt()) <= 5e-3, "reuse != dense"
