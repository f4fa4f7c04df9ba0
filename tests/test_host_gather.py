"""The host-buffer reuse step (q, k, v copied in and the output copied out in
head chunks, overlapped with the kernel) returns exactly what the device-buffer
reuse step returns, for any chunking, with and without a residual; the
device-buffer step itself is held to the float64 oracle by the other parity
tests."""
import pytest
import torch

from sparse_attention_diffusion_gb300 import mcs, synth

pytestmark = pytest.mark.gpu

CASES = {
    "bf16-b2h3-n600-d128": synth.Workload("t", 2, 3, (3, 10, 20), 128, "bf16", 128, "0.2", seed=11),
    "bf16-b1h5-n600-d64-c64": synth.Workload("t", 1, 5, (2, 12, 25), 64, "bf16", 64, "0.3334", seed=12),
    "f32-b1h3-n1024-d64": synth.Workload("t", 1, 3, (4, 16, 16), 64, "f32", 64, "0.25", seed=13),
}


@pytest.fixture(scope="module", params=list(CASES))
def prepared(request):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = CASES[request.param]
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
    q2, k2, v2 = layer.cast()
    mcs.mcs_check_status()
    return dict(wl=wl, desc=desc, K=K, cache=cache, host=[t.contiguous().pin_memory() for t in (q2, k2, v2)])


@pytest.mark.parametrize("chunks", [1, 2, 4, 1000])
@pytest.mark.parametrize("with_residual", [True, False])
def test_host_gather_matches_device_gather(prepared, chunks, with_residual):
    desc, K, cache = prepared["desc"], prepared["K"], prepared["cache"]
    hq, hk, hv = prepared["host"]
    res = cache["residual"] if with_residual else None
    dq, dk, dv = (t.cuda() for t in (hq, hk, hv))
    want = torch.empty_like(dq)
    mcs.mcs_sparse_attn_gather(desc, dq, dk, dv, cache["perm"], cache["idx"], K, res, want)
    ho = torch.full(hq.shape, float("nan"), dtype=hq.dtype).pin_memory()
    ws = mcs.host_gather_workspace(desc, chunks)
    mcs.mcs_sparse_attn_gather_host(desc, hq, hk, hv, cache["perm"], cache["idx"], K, res, ho, ws, chunks)
    torch.cuda.current_stream().synchronize()
    mcs.mcs_check_status()
    assert torch.equal(ho, want.cpu()), "host-buffer reuse step differs from the device-buffer one"


def test_host_gather_from_pageable_memory(prepared):
    """Pageable host buffers are correct too (the copies then serialise)."""
    desc, K, cache = prepared["desc"], prepared["K"], prepared["cache"]
    hq, hk, hv = (t.clone() for t in prepared["host"])          # plain (pageable) host copies
    assert not hq.is_pinned()
    dq, dk, dv = (t.cuda() for t in (hq, hk, hv))
    want = torch.empty_like(dq)
    mcs.mcs_sparse_attn_gather(desc, dq, dk, dv, cache["perm"], cache["idx"], K, cache["residual"], want)
    ho = torch.empty(hq.shape, dtype=hq.dtype)
    ws = mcs.host_gather_workspace(desc, 2)
    mcs.mcs_sparse_attn_gather_host(desc, hq, hk, hv, cache["perm"], cache["idx"], K, cache["residual"], ho, ws, 2)
    torch.cuda.current_stream().synchronize()
    mcs.mcs_check_status()
    assert torch.equal(ho, want.cpu())


def test_host_gather_repeated_calls_on_one_stream(prepared):
    """Back-to-back calls reuse one workspace: each call's copy-in waits for the
    previous call's kernels and copy-out through the caller's stream."""
    desc, K, cache = prepared["desc"], prepared["K"], prepared["cache"]
    hq, hk, hv = prepared["host"]
    ws = mcs.host_gather_workspace(desc, 2)
    outs = [torch.empty(hq.shape, dtype=hq.dtype).pin_memory() for _ in range(3)]
    for o in outs:
        mcs.mcs_sparse_attn_gather_host(desc, hq, hk, hv, cache["perm"], cache["idx"], K, cache["residual"], o, ws, 2)
    torch.cuda.current_stream().synchronize()
    mcs.mcs_check_status()
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
