"""The sparse kernels' lazy rescaling under keys whose logits grow tile by tile.

The softmax keeps a running reference maximum per query row and only moves it
(rescaling the output accumulator and the partial sums) when a later key tile's
maximum exceeds it by more than a factor 2^8. With ordinary inputs that seldom
happens after the first tile; here the key rows of tile t are scaled by
(1 + 0.6 t), so nearly every row moves its reference several times, in tiles
of both parities. The reuse-step output (sparse attention over the selected
keys, plus the residual) and the anchor residual are checked against the
float64 oracle on the very tensors the GPU received."""
import numpy as np
import pytest
import torch

from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import mcs, synth
from tests import parity

pytestmark = pytest.mark.gpu

CASES = {
    "d128-kN": synth.Workload("t", 1, 2, (2, 16, 32), 128, "bf16", 128, "1.0", seed=81),
    "d128-k0.5": synth.Workload("t", 1, 1, (2, 16, 32), 128, "bf16", 128, "0.5", seed=82),
    "d64-c64-k0.75": synth.Workload("t", 1, 1, (2, 16, 32), 64, "bf16", 64, "0.75", seed=83),
    "d64-c128-n4096": synth.Workload("t", 1, 1, (4, 32, 32), 64, "bf16", 128, "0.5", seed=84),
    "d128-c64-k0.5": synth.Workload("t", 1, 1, (2, 16, 32), 128, "bf16", 64, "0.5", seed=85),
}


def _growing_keys(k):
    N = k.shape[2]
    f = 1.0 + 0.6 * (torch.arange(N, dtype=torch.float32) // 128)
    return (k.float() * f[None, None, :, None].to(k.device)).to(k.dtype)


@pytest.mark.parametrize("name", list(CASES))
def test_rescaling_against_the_oracle(name):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    mcs.load(build_if_missing=True)
    wl = CASES[name]
    q, k, v = (t.cuda() for t in synth.make_layer(wl).cast())
    k = _growing_keys(k)
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
    o = torch.empty_like(q)
    mcs.mcs_sparse_attn_gather(desc, q, k, v, cache["perm"], cache["idx"], K, cache["residual"], o)
    mcs.mcs_check_status()
    for h in range(wl.H):
        qh, kh, vh = (parity.f64(t[0, h]) for t in (q, k, v))
        o_ref, _ = orc.dense_attention(qh, kh, vh)
        parity.assert_close(parity.f64(o_dense[0, h]), o_ref, "bf16", f"dense head {h}")
        perm = cache["perm"][0, h].cpu().numpy()
        idx = cache["idx"][0, h].cpu().numpy()
        o_d = parity.f64(o_dense[0, h])
        R = parity.f64(cache["residual"][0, h])
        R_ref = np.empty_like(o_d)
        for g in range(wl.G):
            mem = parity.group_members(perm, g, wl.C, wl.N)
            R_ref[mem] = o_d[mem] - orc.sparse_attention(qh[mem], kh, vh, idx[g])
        parity.assert_close(R, R_ref, "bf16", f"anchor residual head {h}")
        want = orc.reuse_head(qh, kh, vh, perm, idx, R, wl.C)
        parity.assert_close(parity.f64(o[0, h]), want, "bf16", f"reuse output head {h}")
