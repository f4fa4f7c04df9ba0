"""PDDP grouping on fp32 inputs with pad rows and odd tree nodes, bit-exact
against the float64 oracle (perm and group_of). N is not a multiple of C, so the
last group holds pads, and G is not a power of two, so some nodes hold an odd
number of groups and split floor(n/2) : ceil(n/2) [grouping paragraph: groups of
exactly C by principal-direction projection and median split]."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    # G = 6 (nodes of 3 groups), 68 pads
    "n700-d64-c128": synth.Workload("t", 1, 2, (1, 20, 35), 64, "f32", 128, "0.2", seed=41),
    # G = 18 (nodes of 9 and 5 groups), 52 pads
    "n1100-d128-c64": synth.Workload("t", 1, 1, (1, 22, 50), 128, "f32", 64, "0.2", seed=42),
    # G = 6, 51 pads, C = 64
    "n333-d64-c64": synth.Workload("t", 1, 1, (1, 9, 37), 64, "f32", 64, "0.2", seed=43),
    # G = 5 (nodes of 5, 3 and 2 groups), one pad
    "n639-d128-c128": synth.Workload("t", 1, 1, (1, 9, 71), 128, "f32", 128, "0.2", seed=44),
}


@pytest.mark.parametrize("name", list(CASES))
def test_groups_bit_exact_with_pads_and_odd_nodes(name):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = CASES[name]
    assert wl.N_pad > wl.N and wl.G & (wl.G - 1) != 0
    q = synth.make_layer(wl).cast()[0].cuda()
    desc = mcs.desc_for(q, wl.C)
    cache = mcs.alloc_cache(desc, wl.K, q.dtype)
    ws = mcs.workspace(desc, wl.K)
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_check_status()
    for h in range(wl.H):
        x = np.zeros((wl.N_pad, wl.d))
        x[:wl.N] = parity.f64(q[0, h])
        perm_ref, group_ref = orc.pddp_groups(x, wl.N, wl.C, 20)
        perm = cache["perm"][0, h].cpu().numpy()
        assert np.array_equal(perm, perm_ref), f"head {h}: perm differs from the oracle"
        assert np.array_equal(cache["group_of"][0, h].cpu().numpy(), group_ref), f"head {h}: group_of differs"


def test_groups_bit_exact_many_heads():
    """A layer with many heads: heads x ceil(G / 8) >= 256, so the fp64 moments use
    chunks of up to 8 groups (small layers use one group per chunk). G = 18 with
    pads as above; three heads checked against the oracle, every head's
    partition checked for validity."""
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.Workload("t", 1, 86, (1, 22, 50), 64, "f32", 64, "0.2", seed=45)
    assert wl.H * ((wl.G + 7) // 8) >= 256 and wl.N_pad > wl.N
    q = synth.make_layer(wl).cast()[0].cuda()
    desc = mcs.desc_for(q, wl.C)
    cache = mcs.alloc_cache(desc, wl.K, q.dtype)
    ws = mcs.workspace(desc, wl.K)
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_check_status()
    perm_all = cache["perm"][0].cpu().numpy()
    for h in range(wl.H):
        parity.assert_valid_partition(perm_all[h], wl.N, wl.C)
    for h in (0, wl.H // 2, wl.H - 1):
        x = np.zeros((wl.N_pad, wl.d))
        x[:wl.N] = parity.f64(q[0, h])
        perm_ref, group_ref = orc.pddp_groups(x, wl.N, wl.C, 20)
        assert np.array_equal(perm_all[h], perm_ref), f"head {h}: perm differs from the oracle"
        assert np.array_equal(cache["group_of"][0, h].cpu().numpy(), group_ref), f"head {h}: group_of differs"
