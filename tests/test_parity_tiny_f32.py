"""Tiny anchor + reuse layer in fp32 (1 head, 1024 tokens on a 4x16x16 grid,
d=64, C=64, K=256): every stage of the CUDA path against the float64 oracle on
the same inputs. Groups must be bit-exact; outputs within 1e-5."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def run():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = synth.TINY
    layer = synth.make_layer(wl)
    q, k, v = (t.cuda() for t in layer.cast())
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    G, N_pad = mcs.geometry(desc)
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    o_dense = torch.empty_like(q)
    lse = torch.empty((1, 1, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    mcs.mcs_anchor_residual(desc, q, k, v, cache["perm"], cache["idx"], K, o_dense, cache["residual"])
    mcs.mcs_check_status()
    # reuse step on drifted inputs
    layer.drift_step()
    q2, k2, v2 = (t.cuda() for t in layer.cast())
    o_reuse = torch.empty_like(q2)
    mcs.mcs_sparse_attn_gather(desc, q2, k2, v2, cache["perm"], cache["idx"], K, cache["residual"], o_reuse)
    mcs.mcs_check_status()
    return dict(wl=wl, q=q, k=k, v=v, q2=q2, k2=k2, v2=v2, o_dense=o_dense, lse=lse, cache=cache,
                o_reuse=o_reuse, K=K, G=G)


def test_groups_bit_exact(run):
    wl = run["wl"]
    x = np.zeros((wl.N_pad, wl.d))
    x[:wl.N] = parity.f64(run["q"][0, 0])
    perm_ref, group_ref = orc.pddp_groups(x, wl.N, wl.C, 20)
    perm = run["cache"]["perm"][0, 0].cpu().numpy()
    assert np.array_equal(perm, perm_ref)
    assert np.array_equal(run["cache"]["group_of"][0, 0].cpu().numpy(), group_ref)


def test_dense_and_lse(run):
    o_ref, lse_ref = orc.dense_attention(parity.f64(run["q"][0, 0]), parity.f64(run["k"][0, 0]),
                                         parity.f64(run["v"][0, 0]))
    parity.assert_close(parity.f64(run["o_dense"][0, 0]), o_ref, "f32", "dense o")
    parity.assert_close(parity.f64(run["lse"][0, 0]), lse_ref, "f32", "lse")


def test_selection(run):
    wl, K = run["wl"], run["K"]
    q, k = parity.f64(run["q"][0, 0]), parity.f64(run["k"][0, 0])
    _, lse_ref = orc.dense_attention(q, k, np.zeros((wl.N, 1)))
    perm = run["cache"]["perm"][0, 0].cpu().numpy()
    idx = run["cache"]["idx"][0, 0].cpu().numpy()
    mass = run["cache"]["mass"][0, 0].cpu().numpy()
    for g in range(run["G"]):
        mem = parity.group_members(perm, g, wl.C, wl.N)
        S = orc.group_scores(q[mem], lse_ref[mem], k)
        parity.check_selection(idx[g], S, K, mem.size, f"group {g}")
        assert abs(mass[g] - orc.captured_mass(S, idx[g], mem.size)) < 1e-5


def test_anchor_residual_and_reuse(run):
    wl, K = run["wl"], run["K"]
    perm = run["cache"]["perm"][0, 0].cpu().numpy()
    idx = run["cache"]["idx"][0, 0].cpu().numpy()
    q, k, v = (parity.f64(run[n][0, 0]) for n in ("q", "k", "v"))
    o_d = parity.f64(run["o_dense"][0, 0])
    R_ref = np.empty_like(o_d)
    for g in range(run["G"]):
        mem = parity.group_members(perm, g, wl.C, wl.N)
        R_ref[mem] = o_d[mem] - orc.sparse_attention(q[mem], k, v, idx[g])
    R = parity.f64(run["cache"]["residual"][0, 0])
    parity.assert_close(R, R_ref, "f32", "residual")
    q2, k2, v2 = (parity.f64(run[n][0, 0]) for n in ("q2", "k2", "v2"))
    want = orc.reuse_head(q2, k2, v2, perm, idx, R, wl.C)
    parity.assert_close(parity.f64(run["o_reuse"][0, 0]), want, "f32", "reuse output")


def test_end_to_end_against_oracle_anchor(run):
    """Whole anchor + reuse chain of the oracle (its own groups and indices)."""
    wl, K = run["wl"], run["K"]
    q, k, v = (parity.f64(run[n][0, 0]) for n in ("q", "k", "v"))
    ref = orc.anchor_head(q, k, v, wl.C, K)
    q2, k2, v2 = (parity.f64(run[n][0, 0]) for n in ("q2", "k2", "v2"))
    want = orc.reuse_head(q2, k2, v2, ref["perm"], ref["idx"], ref["residual"], wl.C)
    parity.assert_close(parity.f64(run["o_reuse"][0, 0]), want, "f32", "end-to-end reuse output")
