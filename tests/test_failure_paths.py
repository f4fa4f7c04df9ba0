"""Device-side failure detection, exercised without faulting the GPU.

* Out-of-range indices: ids outside [0, N) planted (on the host) in a copy of a
  layer's key index lists, and a query slot outside [0, N_pad) planted in a copy
  of perm. Every kernel that forms an address from such an id checks it first,
  skips the access and raises a sticky flag: mcs_check_status() must report
  MCS_ERR_DEVICE_BOUNDS once, and the groups that were left alone must come out
  bit for bit as in a clean run.
* Bounded waits: a diagnostic kernel waits on a barrier nothing arrives at with
  a 1 ms limit; it must give up, report MCS_ERR_DEVICE_TIMEOUT once, and leave
  the context usable for the next real call."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    "bf16-d128-c128": synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.2", seed=61),
    "bf16-d64-c64": synth.Workload("t", 1, 1, (2, 12, 25), 64, "bf16", 64, "0.3", seed=62),
    "f32-d64-c64": synth.Workload("t", 1, 1, (4, 16, 16), 64, "f32", 64, "0.25", seed=63),
}


def _expect_status(code):
    with pytest.raises(mcs.McsError) as e:
        mcs.mcs_check_status()
    assert e.value.code == code
    mcs.mcs_check_status()          # the flag was cleared by the first report


@pytest.fixture(scope="module", params=list(CASES))
def layer(request):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = CASES[request.param]
    q, k, v = (t.cuda() for t in synth.make_layer(wl).cast())
    desc = mcs.desc_for(q, wl.C)
    K = wl.K
    cache = mcs.alloc_cache(desc, K, q.dtype)
    ws = mcs.workspace(desc, K)
    o_dense = torch.empty_like(q)
    lse = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, cache["perm"], cache["group_of"], ws)
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, cache["perm"], lse, K, cache["idx"], cache["mass"], ws)
    o = torch.zeros_like(q)
    mcs.mcs_sparse_attn_gather(desc, q, k, v, cache["perm"], cache["idx"], K, None, o)
    mcs.mcs_check_status()
    return dict(wl=wl, desc=desc, K=K, q=q, k=k, v=v, lse=lse, ws=ws, cache=cache, o=o)


def _tokens(perm_row, groups, C, N):
    return np.concatenate([parity.group_members(perm_row, g, C, N) for g in groups])


def test_out_of_range_key_ids_are_flagged_and_skipped(layer):
    wl, desc, K, cache = layer["wl"], layer["desc"], layer["K"], layer["cache"]
    idx = cache["idx"].clone()
    bad = {0: [(0, wl.N), (K - 1, 2**31 - 1)], wl.G - 1: [(K // 2, -1)]}   # (slot, id) per group of head 0
    for g, plants in bad.items():
        for slot, val in plants:
            idx[0, 0, g, slot] = val
    o = torch.zeros_like(layer["q"])
    mcs.mcs_sparse_attn_gather(desc, layer["q"], layer["k"], layer["v"], cache["perm"], idx, K, None, o)
    _expect_status(5)
    perm0 = cache["perm"][0, 0].cpu().numpy()
    keep = _tokens(perm0, [g for g in range(wl.G) if g not in bad], wl.C, wl.N)
    assert torch.equal(o[0, 0, keep], layer["o"][0, 0, keep]), "groups without bad ids changed"
    assert torch.equal(o[:, 1:], layer["o"][:, 1:]), "other heads changed"
    # the anchor residual pass reads the same lists
    r = torch.empty_like(o)
    mcs.mcs_anchor_residual(desc, layer["q"], layer["k"], layer["v"], cache["perm"], idx, K, o, r)
    _expect_status(5)


def test_out_of_range_query_slot_is_flagged_and_skipped(layer):
    wl, desc, K, cache = layer["wl"], layer["desc"], layer["K"], layer["cache"]
    perm = cache["perm"].clone()
    g_bad = 1 if wl.G > 1 else 0
    victim = int(perm[0, 0, g_bad * wl.C + 3])
    perm[0, 0, g_bad * wl.C + 3] = wl.N_pad + 9
    o = torch.zeros_like(layer["q"])
    mcs.mcs_sparse_attn_gather(desc, layer["q"], layer["k"], layer["v"], perm, cache["idx"], K, None, o)
    _expect_status(5)
    assert not bool(o[0, 0, victim].any()), "the row of a bad slot must not be written"
    others = np.setdiff1d(np.arange(wl.N), [victim])
    assert torch.equal(o[0, 0, others], layer["o"][0, 0, others]), "rows of valid slots changed"
    # selection: the bad slot is left out of its group's column sums, other groups unchanged
    idx = torch.empty_like(cache["idx"])
    mcs.mcs_anchor_select(desc, layer["q"], layer["k"], perm, layer["lse"], K, idx, None, layer["ws"])
    _expect_status(5)
    same = [g for g in range(wl.G) if g != g_bad]
    assert torch.equal(idx[0, 0, same], cache["idx"][0, 0, same])
    assert torch.equal(idx[:, 1:], cache["idx"][:, 1:])


def test_bounded_wait_times_out_and_context_survives():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    mcs.mcs_check_status()
    elapsed = torch.zeros(1, dtype=torch.int64, device="cuda")
    limit = 1_000_000                                       # 1 ms
    mcs.mcs_selftest_wait_timeout(limit, elapsed)
    _expect_status(6)
    ns = int(elapsed.item())
    assert limit <= ns < 500 * limit, f"wait gave up after {ns} ns"
    # the context is usable: a real call right after gives oracle-close results
    wl = synth.Workload("t", 1, 1, (2, 8, 16), 64, "f32", 64, "0.25", seed=64)
    q, k, v = (t.cuda() for t in synth.make_layer(wl).cast())
    desc = mcs.desc_for(q, wl.C)
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, wl.N), dtype=torch.float32, device="cuda")
    mcs.mcs_dense_attn(desc, q, k, v, o, lse)
    mcs.mcs_check_status()
    o_ref, _ = orc.dense_attention(parity.f64(q[0, 0]), parity.f64(k[0, 0]), parity.f64(v[0, 0]))
    parity.assert_close(parity.f64(o[0, 0]), o_ref, "f32", "dense after a timed-out wait")
