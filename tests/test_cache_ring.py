"""The meta-cache ring: anchor entries written into a device slot and copied out
to host memory, then brought back (with the next layer prefetched) for reuse
steps, give bit for bit the reuse outputs of caches that never left the
device, and those outputs match the float64 oracle's reuse step run on the
entry the ring brought back; acquire/release out of order is refused."""
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    "bf16-d128-c128": [synth.Workload("t", 1, 2, (3, 10, 20), 128, "bf16", 128, "0.2", seed=21 + l) for l in range(3)],
    "f32-d64-c64": [synth.Workload("t", 1, 2, (4, 16, 16), 64, "f32", 64, "0.25", seed=31 + l) for l in range(3)],
}


def _anchor(desc, K, q, k, v, perm, idx, residual):
    wl_ws = mcs.workspace(desc, K)
    group_of = torch.empty((desc.B, desc.H, desc.N), dtype=torch.int32, device="cuda")
    o_dense = torch.empty_like(q)
    lse = torch.empty((desc.B, desc.H, desc.N), dtype=torch.float32, device="cuda")
    mcs.mcs_group_pddp(desc, q, perm, group_of, wl_ws)
    mcs.mcs_dense_attn(desc, q, k, v, o_dense, lse)
    mcs.mcs_anchor_select(desc, q, k, perm, lse, K, idx, None, wl_ws)
    mcs.mcs_anchor_residual(desc, q, k, v, perm, idx, K, o_dense, residual)


@pytest.fixture(scope="module", params=list(CASES))
def layers(request):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    out = []
    for wl in CASES[request.param]:
        layer = synth.make_layer(wl)
        q, k, v = (t.cuda() for t in layer.cast())
        layer.drift_step()
        q2, k2, v2 = (t.cuda() for t in layer.cast())
        desc = mcs.desc_for(q, wl.C)
        K = wl.K
        cache = mcs.alloc_cache(desc, K, q.dtype)
        _anchor(desc, K, q, k, v, cache["perm"], cache["idx"], cache["residual"])
        want = torch.empty_like(q2)
        mcs.mcs_sparse_attn_gather(desc, q2, k2, v2, cache["perm"], cache["idx"], K, cache["residual"], want)
        out.append(dict(desc=desc, K=K, qkv=(q, k, v), qkv2=(q2, k2, v2), want=want, dtype=q.dtype))
    mcs.mcs_check_status()
    return out


def test_ring_round_trip_matches_resident_caches(layers):
    desc, K = layers[0]["desc"], layers[0]["K"]
    ring = mcs.CacheRing(desc, K, len(layers), layers[0]["dtype"])
    try:
        for l, L in enumerate(layers):               # anchor step: fresh entries, stored to host
            c = ring.acquire(l, fill=False, prefetch_next=False)
            _anchor(desc, K, *L["qkv"], c["perm"], c["idx"], c["residual"])
            ring.release(l, store=True)
        for rnd in range(2):                          # reuse steps: entries from host, next layer prefetched
            outs, entries = [], []
            for l, L in enumerate(layers):
                c = ring.acquire(l, fill=True, prefetch_next=True)
                o = torch.empty_like(L["want"])
                mcs.mcs_sparse_attn_gather(desc, *L["qkv2"], c["perm"], c["idx"], K, c["residual"], o)
                if rnd == 0:   # the entry as the kernel read it (copied before the slot is released)
                    entries.append({n: c[n].cpu() for n in ("perm", "idx", "residual")})
                ring.release(l)
                outs.append(o)
            torch.cuda.synchronize()
            mcs.mcs_check_status()
            for l, (o, L) in enumerate(zip(outs, layers)):
                assert torch.equal(o, L["want"]), f"pass {rnd} layer {l}: ring cache differs from resident cache"
            # the reuse step against the float64 oracle, fed the entry the ring brought back
            for l, (o, L, e) in enumerate(zip(outs, layers, entries)):
                for h in range(desc.H):
                    q2, k2, v2 = (parity.f64(t[0, h]) for t in L["qkv2"])
                    want = orc.reuse_head(q2, k2, v2, e["perm"][0, h].numpy(), e["idx"][0, h].numpy(),
                                          parity.f64(e["residual"][0, h]), desc.C)
                    parity.assert_close(parity.f64(o[0, h]), want, "bf16" if L["dtype"] == torch.bfloat16 else "f32",
                                        f"layer {l} head {h}: ring reuse output vs oracle")
    finally:
        ring.close()


def test_ring_refuses_out_of_order_calls(layers):
    desc, K = layers[0]["desc"], layers[0]["K"]
    with mcs.CacheRing(desc, K, 3, layers[0]["dtype"]) as ring:
        ring.acquire(0, fill=False, prefetch_next=False)
        with pytest.raises(mcs.McsError):
            ring.acquire(0, fill=False)               # acquired twice
        ring.acquire(1, fill=False, prefetch_next=False)
        with pytest.raises(mcs.McsError):
            ring.acquire(2, fill=False)               # both slots in use
        with pytest.raises(mcs.McsError):
            ring.release(2)                           # never acquired
        ring.release(0)
        ring.release(1)
        ring.acquire(2, fill=False, prefetch_next=False)
        ring.release(2)
        torch.cuda.synchronize()
