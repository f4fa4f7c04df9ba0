"""Warm-started PDDP grouping ("fast PDDP": every tree node's power iteration
starts from a stored direction, e.g. the previous anchor's) against the float64
oracle given the same start directions [grouping paragraph; the kernel-benchmark
paragraph's amortised grouping cost].

* fp32 inputs with pads and odd nodes: seeded random start directions and a few
  iterations, bit-exact perm and group_of;
* an anchor chain: a cold grouping writes its directions, the inputs drift, a
  warm grouping with 4 iterations starts from them; the oracle runs the same
  chain on its own directions;
* the stored directions used as they are (0 iterations), in place (the input and
  output tables are one buffer);
* bf16 at d = 128 (tensor-core moments) and d = 64, split by split against the
  oracle."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

F32 = {
    "n700-d64-c128": synth.Workload("t", 1, 2, (1, 20, 35), 64, "f32", 128, "0.2", seed=71),
    "n1100-d128-c64": synth.Workload("t", 1, 1, (1, 22, 50), 128, "f32", 64, "0.2", seed=72),
}
BF16 = {
    "n1024-d128-c128": synth.Workload("t", 1, 2, (2, 16, 32), 128, "bf16", 128, "0.2", seed=73),
    "n600-d64-c64": synth.Workload("t", 1, 2, (2, 12, 25), 64, "bf16", 64, "0.2", seed=74),
}


def _padded(q_head, wl):
    x = np.zeros((wl.N_pad, wl.d))
    x[:wl.N] = parity.f64(q_head)
    return x


def _random_dirs(desc, seed):
    """Seeded random unit start directions, one row per tree node (test input)."""
    S = mcs.pddp_dirs(desc, device="cpu").shape[2]
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((desc.B, desc.H, S, desc.d)).astype(np.float32)
    v /= np.linalg.norm(v, axis=-1, keepdims=True)
    return torch.from_numpy(v)


def _group(desc, q, iters, dirs_in, dirs_out, wl):
    d2 = mcs.make_desc(desc.B, desc.H, desc.N, desc.d, desc.C, q.dtype, 0.0, iters)
    perm = torch.empty((wl.B, wl.H, wl.N_pad), dtype=torch.int32, device="cuda")
    group_of = torch.empty((wl.B, wl.H, wl.N), dtype=torch.int32, device="cuda")
    ws = mcs.workspace(d2, 1)
    mcs.mcs_group_pddp_warm(d2, q, dirs_in, dirs_out, perm, group_of, ws)
    mcs.mcs_check_status()
    return perm, group_of


@pytest.fixture(autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)


@pytest.mark.parametrize("name", list(F32))
def test_random_start_directions_bit_exact(name):
    wl = F32[name]
    q = synth.make_layer(wl).cast()[0].cuda()
    desc = mcs.desc_for(q, wl.C)
    dirs = _random_dirs(desc, 7)
    perm, group_of = _group(desc, q, 3, dirs.cuda(), None, wl)
    for h in range(wl.H):
        perm_ref, group_ref = orc.pddp_groups(_padded(q[0, h], wl), wl.N, wl.C, 3,
                                              v_init=dirs[0, h].double().numpy())
        assert np.array_equal(perm[0, h].cpu().numpy(), perm_ref), f"head {h}"
        assert np.array_equal(group_of[0, h].cpu().numpy(), group_ref), f"head {h}"


@pytest.mark.parametrize("name", list(F32))
def test_anchor_chain_cold_then_warm(name):
    wl = F32[name]
    layer = synth.make_layer(wl)
    q0 = layer.cast()[0].cuda()
    for _ in range(10):          # ten denoising steps between two anchors
        layer.drift_step()
    q1 = layer.cast()[0].cuda()
    desc = mcs.desc_for(q0, wl.C)
    dirs = mcs.pddp_dirs(desc)
    _group(desc, q0, 20, None, dirs, wl)
    perm, _ = _group(desc, q1, 4, dirs, dirs, wl)            # warm, in place
    for h in range(wl.H):
        S = dirs.shape[2]
        v = np.full((S, wl.d), np.nan)
        orc.pddp_groups(_padded(q0[0, h], wl), wl.N, wl.C, 20, v_out=v)
        v32 = np.where(np.isnan(v), 0.0, v).astype(np.float32).astype(np.float64)   # the table is fp32
        perm_ref, _ = orc.pddp_groups(_padded(q1[0, h], wl), wl.N, wl.C, 4, v_init=v32)
        assert np.array_equal(perm[0, h].cpu().numpy(), perm_ref), f"head {h}"


def test_stored_directions_used_as_they_are():
    wl = F32["n700-d64-c128"]
    q = synth.make_layer(wl).cast()[0].cuda()
    desc = mcs.desc_for(q, wl.C)
    for h in range(wl.H):
        x = _padded(q[0, h], wl)
        S = mcs.pddp_dirs(desc, device="cpu").shape[2]
        v = np.zeros((S, wl.d))
        perm_cold, _ = orc.pddp_groups(x, wl.N, wl.C, 20, v_out=v)
        dirs = torch.zeros((1, wl.H, S, wl.d), dtype=torch.float32)
        dirs[0, h] = torch.from_numpy(v.astype(np.float32))
        perm, _ = _group(desc, q, 0, dirs.cuda(), None, wl)
        perm_ref, _ = orc.pddp_groups(x, wl.N, wl.C, 0, v_init=dirs[0, h].double().numpy())
        assert np.array_equal(perm[0, h].cpu().numpy(), perm_ref)
        assert np.array_equal(perm_ref, perm_cold)   # a converged direction reproduces the cold groups


@pytest.mark.parametrize("name", list(BF16))
def test_bf16_random_start_directions(name):
    wl = BF16[name]
    q = synth.make_layer(wl).cast()[0].cuda()
    desc = mcs.desc_for(q, wl.C)
    dirs = _random_dirs(desc, 9)
    perm, _ = _group(desc, q, 4, dirs.cuda(), None, wl)
    for h in range(wl.H):
        trace_dirs = dirs[0, h].double().numpy()
        p = perm[0, h].cpu().numpy()
        parity.assert_valid_partition(p, wl.N, wl.C)
        perm_ref, _ = orc.pddp_groups(_padded(q[0, h], wl), wl.N, wl.C, 4, v_init=trace_dirs)
        agree = parity.pddp_agreement(p, perm_ref, wl.C)
        print(f"{name} head {h}: warm-start group agreement {agree:.3f}")
        assert agree >= parity.PDDP_AGREE_FLOOR_SMALL
