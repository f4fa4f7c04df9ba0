"""bf16 layers small enough for the oracle, spanning several tiles with ragged
tails (N not a multiple of 128, K not a multiple of 128, pad queries, K = N),
both head dims and both group sizes, and a layer of one group per head. Every
stage of the CUDA path is checked against the float64 oracle run on the very
tensors the GPU received."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    "n600-d128-c128-k120": synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.2", seed=3),
    "n600-d128-c128-k300": synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.5", seed=4),
    "n600-d64-c64-k200": synth.Workload("t", 1, 2, (2, 12, 25), 64, "bf16", 64, "0.3334", seed=5),
    "n600-d128-c64-k90": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 64, "0.15", seed=6),
    "n600-d64-c128-k150": synth.Workload("t", 1, 1, (3, 10, 20), 64, "bf16", 128, "0.25", seed=7),
    "n1024-d128-c128-k205": synth.Workload("t", 2, 1, (2, 16, 32), 128, "bf16", 128, "0.2", seed=8),
    "n600-d128-c128-kN": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 128, "1.0", seed=9),
    # d = 64 with 16 key tiles per group: the deeper key/value rings wrap twice
    "n4096-d64-c128-k2048": synth.Workload("t", 1, 1, (4, 32, 32), 64, "bf16", 128, "0.5", seed=11),
    "n4000-d64-c64-k1500": synth.Workload("t", 1, 1, (4, 25, 40), 64, "bf16", 64, "0.375", seed=12),
    # one group per head (G = 1, 28 pad rows): no split at all, a key list shorter than one tile
    "n100-d128-c128-k30": synth.Workload("t", 1, 2, (1, 10, 10), 128, "bf16", 128, "0.3", seed=10),
    # d = 64, G = 2 (28 pad rows), one key tile per group: the odd-tile chain has nothing to issue
    "n100-d64-c64-k30": synth.Workload("t", 1, 2, (1, 10, 10), 64, "bf16", 64, "0.3", seed=13),
    # C = 64 splits each row's keys over two lanes (keys 0-63 / 64-127 of every tile):
    # exactly one half's worth of keys (the second lane sees none), one key past it,
    # and a second tile holding a single key
    "n600-d128-c64-k64": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 64, "0.1066", seed=14),
    "n600-d64-c64-k65": synth.Workload("t", 1, 2, (3, 10, 20), 64, "bf16", 64, "0.1075", seed=15),
    "n600-d128-c64-k129": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 64, "0.2149", seed=16),
    # C = 128 splits every tile's keys over two softmax warpgroups (keys 0-63 / 64-127):
    # exactly the first half (the second warpgroup never sees a key), one key past it,
    # and a last tile whose second half is empty
    "n600-d128-c128-k64": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 128, "0.1066", seed=17),
    "n600-d128-c128-k65": synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.1075", seed=18),
    "n600-d64-c128-k129": synth.Workload("t", 1, 1, (3, 10, 20), 64, "bf16", 128, "0.2149", seed=19),
    # one selected key per group: the sparse output is that key's value row, and all
    # but one softmax thread of a row see no key
    "n600-d128-c128-k1": synth.Workload("t", 1, 1, (3, 10, 20), 128, "bf16", 128, "0.001", seed=20),
    "n600-d64-c64-k1": synth.Workload("t", 1, 1, (3, 10, 20), 64, "bf16", 64, "0.001", seed=21),
}


def _run(wl):
    layer = synth.make_layer(wl)
    q, k, v = (t.cuda() for t in layer.cast())
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
    q2, k2, v2 = (t.cuda() for t in layer.cast())
    o_reuse = torch.empty_like(q2)
    mcs.mcs_sparse_attn_gather(desc, q2, k2, v2, cache["perm"], cache["idx"], K, cache["residual"], o_reuse)
    idx_nolse = torch.empty_like(cache["idx"])
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], None, K, idx_nolse, None, ws)
    mcs.mcs_check_status()
    return dict(wl=wl, K=K, q=q, k=k, v=v, q2=q2, k2=k2, v2=v2, o_dense=o_dense, lse=lse, cache=cache,
                o_reuse=o_reuse, idx_nolse=idx_nolse)


@pytest.fixture(scope="module", params=list(CASES))
def run(request):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    return _run(CASES[request.param])


def _heads(run):
    wl = run["wl"]
    for b in range(wl.B):
        for h in range(wl.H):
            yield b, h


def test_dense(run):
    for b, h in _heads(run):
        q, k, v = (parity.f64(run[n][b, h]) for n in ("q", "k", "v"))
        o_ref, lse_ref = orc.dense_attention(q, k, v)
        parity.assert_close(parity.f64(run["o_dense"][b, h]), o_ref, "bf16", f"dense o head {b},{h}")
        assert np.abs(parity.f64(run["lse"][b, h]) - lse_ref).max() < 1e-3


def test_groups(run):
    wl = run["wl"]
    for b, h in _heads(run):
        x = np.zeros((wl.N_pad, wl.d))
        x[:wl.N] = parity.f64(run["q"][b, h])
        perm = run["cache"]["perm"][b, h].cpu().numpy()
        parity.assert_valid_partition(perm, wl.N, wl.C)
        group_of = run["cache"]["group_of"][b, h].cpu().numpy()
        for g in range(wl.G):
            mem = parity.group_members(perm, g, wl.C, wl.N)
            assert np.all(group_of[mem] == g)
        agree, _, bad = parity.pddp_split_report(perm, x, wl.N, wl.C)
        gaps = ", ".join(f"g0={s['g0']} n={s['n']} gap {s['gap']:.2e} sd moved {s['moved']}" for s in bad)
        print(f"PDDP group agreement head {b},{h}: {agree:.3f} [{gaps}]")
        assert agree >= parity.PDDP_AGREE_FLOOR_SMALL, f"head {b},{h}: agreement {agree:.3f}"
        for s in bad:
            assert s["gap"] <= parity.PDDP_GAP_MAX, f"head {b},{h}: disagreeing split with oracle gap {s['gap']:.3g} sd"


def test_selection(run):
    wl, K = run["wl"], run["K"]
    exact = total = 0
    for b, h in _heads(run):
        q, k = parity.f64(run["q"][b, h]), parity.f64(run["k"][b, h])
        _, lse_ref = orc.dense_attention(q, k, np.zeros((wl.N, 1)))
        perm = run["cache"]["perm"][b, h].cpu().numpy()
        idx = run["cache"]["idx"][b, h].cpu().numpy()
        mass = run["cache"]["mass"][b, h].cpu().numpy()
        for g in range(wl.G):
            mem = parity.group_members(perm, g, wl.C, wl.N)
            S = orc.group_scores(q[mem], lse_ref[mem], k)
            exact += parity.check_selection(idx[g], S, K, mem.size, f"head {b},{h} group {g}")
            total += 1
            assert abs(mass[g] - orc.captured_mass(S, idx[g], mem.size)) < 1e-4
    print(f"index sets identical to the oracle: {exact}/{total}")
    assert torch.equal(run["idx_nolse"], run["cache"]["idx"])


def test_residual_and_reuse(run):
    wl = run["wl"]
    for b, h in _heads(run):
        perm = run["cache"]["perm"][b, h].cpu().numpy()
        idx = run["cache"]["idx"][b, h].cpu().numpy()
        q, k, v = (parity.f64(run[n][b, h]) for n in ("q", "k", "v"))
        o_d = parity.f64(run["o_dense"][b, h])
        R_ref = np.empty_like(o_d)
        for g in range(wl.G):
            mem = parity.group_members(perm, g, wl.C, wl.N)
            R_ref[mem] = o_d[mem] - orc.sparse_attention(q[mem], k, v, idx[g])
        R = parity.f64(run["cache"]["residual"][b, h])
        parity.assert_close(R, R_ref, "bf16", f"residual head {b},{h}")
        if run["K"] == wl.N:
            assert np.abs(R).max() < 2e-2
        q2, k2, v2 = (parity.f64(run[n][b, h]) for n in ("q2", "k2", "v2"))
        want = orc.reuse_head(q2, k2, v2, perm, idx, R, wl.C)
        parity.assert_close(parity.f64(run["o_reuse"][b, h]), want, "bf16", f"reuse head {b},{h}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_residual_store_apply_exact(dtype):
    mcs.load(build_if_missing=True)
    g = torch.Generator().manual_seed(0)
    shape = (1, 3, 333, 64)
    a, b = (torch.randn(shape, generator=g).to(dtype) for _ in range(2))
    desc = mcs.make_desc(1, 3, 333, 64, 64, dtype)
    ad, bd = a.cuda(), b.cuda()
    r, o = torch.empty_like(ad), torch.empty_like(ad)
    mcs.mcs_residual_store(desc, ad, bd, r)
    mcs.mcs_residual_apply(desc, bd, r, o)
    mcs.mcs_check_status()
    # one rounding of the exact fp64 result (differences of bf16 values are exact in fp32)
    want_r = (a.double() - b.double()).to(dtype)
    want_o = (b.double() + want_r.double()).to(dtype)
    assert torch.equal(r.cpu(), want_r)
    assert torch.equal(o.cpu(), want_o)
