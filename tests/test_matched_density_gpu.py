"""The GPU selection measured the way the matched-density analysis measures it:
per-group captured mass with the method's PDDP groups and with contiguous tile
groups (identity perm), and the relative error of the anchor's sparse output
(||R|| / ||O_dense||), against the float64 analysis oracle on the very inputs
the GPU received."""
import numpy as np
import pytest
import torch

from oracle import matched_density as md
from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

WL = synth.Workload("t", 1, 2, (4, 32, 32), 128, "bf16", 128, "0.2", seed=31)


def _gpu(perm_kind):
    q, k, v = (t.cuda() for t in synth.make_layer(WL).cast())
    desc = mcs.desc_for(q, WL.C)
    K = WL.K
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    if perm_kind == "pddp":
        mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    else:
        cache["perm"].copy_(torch.arange(WL.N_pad, dtype=torch.int32, device="cuda").expand_as(cache["perm"]))
    o_dense = torch.empty_like(q)
    lse = torch.empty((WL.B, WL.H, WL.N), dtype=torch.float32, device="cuda")
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], cache["idx"], K, o_dense, cache["residual"])
    mcs.mcs_check_status()
    return q, k, v, o_dense, cache


@pytest.mark.parametrize("perm_kind", ["pddp", "contiguous"])
def test_group_mass_and_sparse_error_match_analysis(perm_kind):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    q, k, v, o_dense, cache = _gpu(perm_kind)
    for h in range(WL.H):
        qh, kh, vh = (parity.f64(t[0, h]) for t in (q, k, v))
        P = md.probabilities(qh, kh)
        perm = cache["perm"][0, h].cpu().numpy()
        groups = [parity.group_members(perm, g, WL.C, WL.N) for g in range(WL.G)]
        sets = md.group_shared_sets(P, groups, WL.K)
        gpu_mass = cache["mass"][0, h].cpu().numpy()
        for g, mem in enumerate(groups):
            S = P[mem].sum(axis=0)
            want = orc.captured_mass(S, sets[mem[0]], mem.size)
            assert abs(gpu_mass[g] - want) < 1e-5, f"{perm_kind} head {h} group {g}: mass"
        _, err = md.evaluate(P, vh, sets)
        R, Od = parity.f64(cache["residual"][0, h]), parity.f64(o_dense[0, h])
        gpu_err = np.linalg.norm(R) / np.linalg.norm(Od)
        assert gpu_err == pytest.approx(err, rel=2e-2), f"{perm_kind} head {h}: sparse output error"
