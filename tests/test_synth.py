"""The seeded generator: shapes, K rounding, determinism and the logit-std recipe. CPU only."""
import math

import numpy as np
import pytest
import torch

from sparse_attention_diffusion_gb300 import synth


def test_workload_sizes():
    w = synth.WORKLOADS
    assert (w["tiny-anchor-reuse"].N, w["tiny-anchor-reuse"].G, w["tiny-anchor-reuse"].K) == (1024, 16, 256)
    assert (w["wan2.1-1.3b-480p"].N, w["wan2.1-1.3b-480p"].K) == (32768, 6554)
    kb = w["kernel-bench-720p"]
    assert (kb.N, kb.N_pad, kb.G, kb.K) == (75600, 75648, 591, 15120)
    sc = w["schedule-118800"]
    assert (sc.N, sc.N_pad, sc.G, sc.K, sc.with_(density="0.25").K) == (118800, 118912, 929, 17820, 29700)
    sw = w["sweep-65536"]
    ks = [sw.with_(density=r).K for r in ("0.05", "0.1", "0.15", "0.2", "0.3", "0.5", "1.0")]
    assert ks == [3277, 6554, 9831, 13108, 19661, 32768, 65536]


def test_generator_is_deterministic_and_standardised():
    wl = synth.TINY
    a, b = synth.make_layer(wl), synth.make_layer(wl)
    for x, y in ((a.q0, b.q0), (a.k0, b.k0), (a.v0, b.v0)):
        assert torch.equal(x, y)
        assert abs(float(x.mean())) < 1e-5 and abs(float(x.std()) - 1.0) < 1e-4
    q, k, v = a.cast()
    assert q.dtype == torch.float32 and q.shape == (1, 1, 1024, 64)


def test_logit_std_is_about_three():
    wl = synth.TINY
    L = synth.make_layer(wl)
    q, k, _ = L.cast()
    s = (q[0, 0] @ k[0, 0].T) / math.sqrt(wl.d)
    assert 2.5 < float(s.std()) < 3.5


def test_drift_is_variance_preserving():
    L = synth.make_layer(synth.TINY)
    before = L.q0.clone()
    L.drift_step(0.1)
    c = float(torch.nn.functional.cosine_similarity(before.flatten(), L.q0.flatten(), dim=0))
    assert abs(c - math.sqrt(1 - 0.01)) < 0.01
    assert abs(float(L.q0.std()) - 1.0) < 0.02


def test_bf16_cast_is_round_to_nearest_even():
    x = torch.tensor([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8], dtype=torch.float32)
    got = synth.round_bf16(x).float()
    assert got.tolist() == [1.0, 1.0 + 2 ** -6, -1.0]
