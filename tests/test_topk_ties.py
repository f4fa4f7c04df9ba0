"""Exact ties in the top-K kernel. All-equal scores (zero queries: every key
gets the same summed weight) over a 16,384-token row must keep the K lowest
ids; duplicated keys make exact ties at the K-th score inside ordinary rows,
where the lower id must win."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu


def _select(q, k, C, K):
    desc = mcs.desc_for(q, C)
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    G, N_pad = mcs.geometry(desc)
    cache["perm"].copy_(torch.arange(N_pad, dtype=torch.int32, device="cuda").expand_as(cache["perm"]))
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], None, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_check_status()
    return cache


def test_all_equal_scores_keep_the_lowest_ids():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.Workload("t", 1, 1, (4, 64, 64), 64, "bf16", 64, "0.1", seed=41)
    _, k, _ = (t.cuda() for t in synth.make_layer(wl).cast())
    q = torch.zeros_like(k)
    K = 1000
    cache = _select(q, k, wl.C, K)
    want = torch.arange(K, dtype=torch.int32, device="cuda")
    assert torch.equal(cache["idx"][0, 0], want.expand(wl.G, K)), "ties must keep the lowest ids"
    assert torch.allclose(cache["mass"], torch.full_like(cache["mass"], K / wl.N), rtol=1e-4)


def test_duplicated_keys_tie_to_the_lower_id():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.Workload("t", 1, 1, (2, 16, 32), 128, "bf16", 128, "0.25", seed=43)
    q, k, _ = (t.cuda() for t in synth.make_layer(wl).cast())
    k = k.clone()
    k[0, 0, 1::2] = k[0, 0, 0::2]          # key 2i+1 repeats key 2i: every score appears twice
    K = wl.K | 1                            # odd K: the K-th score's twin is the first key left out
    cache = _select(q, k, wl.C, K)
    qh, kh = parity.f64(q[0, 0]), parity.f64(k[0, 0])
    _, lse = orc.dense_attention(qh, kh, np.zeros((wl.N, 1)))
    for g in range(wl.G):
        mem = np.arange(g * wl.C, min((g + 1) * wl.C, wl.N))
        S = orc.group_scores(qh[mem], lse[mem], kh)
        idx = cache["idx"][0, 0, g].cpu().numpy()
        parity.check_selection(idx, S, K, mem.size, f"group {g}")
        pairs = set(idx.tolist())
        # ties go to the lower id: a kept odd key always has its even twin kept
        assert all((j - 1) in pairs for j in idx if j % 2 == 1), f"group {g}: odd twin kept without its even twin"
