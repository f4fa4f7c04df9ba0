"""mcs_anchor_select_noalloc: anchor selection for callers that cannot allocate
device memory (the score rows live in a fixed array inside the library instead
of a caller workspace). Its results must equal mcs_anchor_select's on the same
inputs, on two calls in a row (the second call reuses the array the first one
left behind). Kept in a file pytest collects last."""
import ctypes

import pytest
import torch

from sparse_attention_diffusion_gb300 import mcs, synth

pytestmark = pytest.mark.gpu

CASES = [
    synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.2", seed=21),
    synth.Workload("t", 1, 1, (2, 12, 25), 64, "bf16", 64, "0.3", seed=22),
    synth.TINY,
]


@pytest.mark.parametrize("wl", CASES, ids=["bf16-d128-c128", "bf16-d64-c64", "f32-tiny"])
def test_matches_workspace_entry_point_twice(wl):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    layer = synth.make_layer(wl)
    q, k, v = (t.cuda() for t in layer.cast())
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, None, lse)
    idx_ref = torch.empty_like(cache["idx"])
    mass_ref = torch.empty_like(cache["mass"])
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, idx_ref, mass_ref, ws)
    for _ in range(2):
        idx = torch.full_like(cache["idx"], -7)
        mass = torch.full_like(cache["mass"], -1.0)
        mcs.mcs_anchor_select_noalloc(desc, q, k, cache["perm"], lse, K, idx, mass)
        mcs.mcs_check_status()
        assert torch.equal(idx, idx_ref)
        assert torch.allclose(mass, mass_ref, rtol=0, atol=1e-5)


def _select_both_ways(desc, q, k, K, twice=True):
    ws = mcs.workspace(desc, K)
    G, N_pad = mcs.geometry(desc)
    perm = torch.empty((desc.B, desc.H, N_pad), dtype=torch.int32, device="cuda")
    group_of = torch.empty((desc.B, desc.H, desc.N), dtype=torch.int32, device="cuda")
    lse = torch.empty((desc.B, desc.H, desc.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, perm, group_of, ws)
    mcs.mcs_dense_attn(desc, q, k, k, None, lse)
    idx_ref = torch.empty((desc.B, desc.H, G, K), dtype=torch.int32, device="cuda")
    mass_ref = torch.empty((desc.B, desc.H, G), dtype=torch.float32, device="cuda")
    mcs.mcs_anchor_select(desc, q, k, perm, lse, K, idx_ref, mass_ref, ws)
    del ws
    for _ in range(2 if twice else 1):
        idx = torch.full_like(idx_ref, -7)
        mass = torch.full_like(mass_ref, -1.0)
        mcs.mcs_anchor_select_noalloc(desc, q, k, perm, lse, K, idx, mass)
        mcs.mcs_check_status()
        assert torch.equal(idx, idx_ref)
        assert torch.allclose(mass, mass_ref, rtol=0, atol=1e-5)


def test_group_rows_spanning_several_fills_of_the_array():
    """One 720p-shaped head (N = 75,600, 591 groups): the array holds 221 score
    rows, so the call runs three launches whose boundaries (rows 221 and 442) fall
    inside two-group pairs of the pass-2 kernel."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.KBENCH_720P.with_(H=1, seed=23)
    q, k, _ = synth.make_layer(wl, device="cuda").cast()
    desc = mcs.desc_for(q, wl.C)
    assert (64 << 20) // (wl.N * 4) == 221 and wl.G == 591
    _select_both_ways(desc, q, k, wl.K)


def test_many_short_heads_keep_launch_grids_small():
    """fp32, N = 100 (one score row is 400 bytes): 80,000 group rows would fit in
    the array at once, more than one launch grid dimension takes, so rows go 4,096
    per launch as in the workspace entry point."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    g = torch.Generator(device="cuda").manual_seed(24)
    H, N, d = 40_000, 100, 64
    q = torch.randn((1, H, N, d), generator=g, device="cuda")
    k = torch.randn((1, H, N, d), generator=g, device="cuda")
    desc = mcs.make_desc(1, H, N, d, 64, torch.float32)
    _select_both_ways(desc, q, k, 30, twice=False)


def test_rejects_rows_beyond_the_fixed_scratch():
    lib = mcs.load(build_if_missing=True)
    d = mcs.make_desc(1, 1, 20_000_000, 128, 128, torch.bfloat16)   # one score row > 64 MiB
    fake = ctypes.c_void_p(4096)
    assert lib.mcs_anchor_select_noalloc(ctypes.byref(d), fake, fake, fake, fake, 10, fake, None, None) == 2
    d = mcs.make_desc(1, 1, 600, 128, 128, torch.bfloat16)
    assert lib.mcs_anchor_select_noalloc(ctypes.byref(d), fake, fake, fake, None, 10, fake, None, None) == 1  # lse required
