"""Pass-2 column sums with two groups per CTA (d = 128, C = 128): a launch covers
4,096 group rows, so with 5 groups per head the pair (4095, 4096) of head 819 is
split between two launches and each launch masks the half it does not own; odd
G also leaves a single group in every head's last pair. The groups around the
launch boundary, and each head's last group there, are checked against the
float64 oracle (selection rule and captured mass)."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu


def test_pairs_across_the_launch_boundary():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.Workload("t", 1, 1000, (3, 10, 20), 128, "bf16", 128, "0.2", seed=51)   # G = 5, 5,000 rows
    q, k, v = synth.make_layer(wl, device="cuda").cast()
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, torch.empty_like(q), lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_check_status()
    assert wl.G == 5 and wl.H * wl.G > 4096
    rows = list(range(4090, 4102)) + [4 * wl.G + 4]          # around row 4,096, and head 4's last group
    for row in rows:
        h, g = divmod(row, wl.G)
        qh, kh = parity.f64(q[0, h]), parity.f64(k[0, h])
        perm = cache["perm"][0, h].cpu().numpy()
        mem = parity.group_members(perm, g, wl.C, wl.N)
        _, lse_g = orc.dense_attention(qh[mem], kh, np.zeros((wl.N, 1)))
        S = orc.group_scores(qh[mem], lse_g, kh)
        idx = cache["idx"][0, h, g].cpu().numpy()
        parity.check_selection(idx, S, K, mem.size, f"row {row} (head {h} group {g})")
        assert abs(float(cache["mass"][0, h, g]) - orc.captured_mass(S, idx, mem.size)) < 1e-4
