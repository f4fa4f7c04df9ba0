"""Seeded synthetic Q/K/V layers shaped like the DiT attention inputs the MC-Sparse
pages measure on (video latents on a (t, y, x) token grid).

This module only makes inputs. It holds none of the attention, grouping or
selection arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe (per head h, per tensor q/k/v):
  * token n = (t*Y + y)*X + x, normalised position p = (t/T, y/Y, x/X);
  * per head, 32 random Fourier features shared by q, k, v:
        omega_m ~ N(0, 2^2 I_3),  b_m ~ U[0, 2*pi),
        f_m(p) = sqrt(2/32) * cos(2*pi*omega_m . p + b_m);
  * per tensor, x = F A^T + 0.3 * N(0,1) with A ~ N(0,1)^{d x 32};
  * standardise each (head, tensor) to zero mean and unit element std;
  * scale q and k by alpha, alpha^2 chosen so that the std of q.k/sqrt(d)
    over 4096 seeded (i, j) pairs is 3.0 (logits with std about 3);
  * drift between denoising steps: x <- sqrt(1 - delta^2) x + delta * xi on
    the standardised tensors, xi ~ N(0,1), then alpha is applied again;
  * cast once to the workload dtype (bf16 by round-to-nearest-even).

Draw order per head: omega, b, then (A, noise) for q, k, v, then the 4096
(i, j) pairs; drift noise is drawn per step, per head, for q, k, v in turn.
Generation runs in torch on the device given (CPU for small cases, CUDA for
full-size layers); the values are a function of (seed, device type, torch
build) and every consumer receives the same tensors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from fractions import Fraction

import torch

N_FEATURES = 32
OMEGA_STD = 2.0
NOISE_STD = 0.3
LOGIT_STD = 3.0
ALPHA_PAIRS = 4096


@dataclass(frozen=True)
class Workload:
    """One attention layer: B x H heads of N tokens on a (T, Y, X) grid."""
    name: str
    B: int
    H: int
    grid: tuple
    d: int
    dtype: str            # "f32" or "bf16"
    C: int                # query-group size (tile width)
    density: str          # decimal string, e.g. "0.2"; K = ceil(density * N)
    seed: int = 0
    drift: float = 0.1

    @property
    def N(self) -> int:
        t, y, x = self.grid
        return t * y * x

    @property
    def G(self) -> int:
        return -(-self.N // self.C)

    @property
    def N_pad(self) -> int:
        return self.G * self.C

    @property
    def K(self) -> int:
        # exact rational arithmetic: 0.2 * 75600 must give 15120, not 15121
        return int(math.ceil(Fraction(self.density) * self.N))

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


# The five layers the hot path is measured and checked on.
TINY = Workload("tiny-anchor-reuse", 1, 1, (4, 16, 16), 64, "f32", 64, "0.25", seed=0, drift=0.1)
WAN13_480P = Workload("wan2.1-1.3b-480p", 1, 12, (16, 32, 64), 128, "bf16", 128, "0.2", seed=0, drift=0.1)
KBENCH_720P = Workload("kernel-bench-720p", 1, 40, (21, 45, 80), 128, "bf16", 128, "0.2", seed=0, drift=0.1)
SCHEDULE_HY = Workload("schedule-118800", 1, 24, (33, 45, 80), 128, "bf16", 128, "0.15", seed=0, drift=0.05)
SWEEP = Workload("sweep-65536", 1, 16, (16, 64, 64), 128, "bf16", 128, "0.2", seed=1, drift=0.1)
WORKLOADS = {w.name: w for w in (TINY, WAN13_480P, KBENCH_720P, SCHEDULE_HY, SWEEP)}


def positions(grid, device="cpu") -> torch.Tensor:
    """[N, 3] normalised (t/T, y/Y, x/X) positions in token order."""
    T, Y, X = grid
    t = torch.arange(T, device=device, dtype=torch.float32) / T
    y = torch.arange(Y, device=device, dtype=torch.float32) / Y
    x = torch.arange(X, device=device, dtype=torch.float32) / X
    tt, yy, xx = torch.meshgrid(t, y, x, indexing="ij")
    return torch.stack([tt.reshape(-1), yy.reshape(-1), xx.reshape(-1)], dim=1)


def round_bf16(x: torch.Tensor) -> torch.Tensor:
    """Round-to-nearest-even to bf16 (torch's float->bf16 cast is RNE)."""
    return x.to(torch.bfloat16)


@dataclass
class Layer:
    """Standardised pre-scale tensors (fp32) plus the fixed per-head alpha."""
    wl: Workload
    q0: torch.Tensor      # [B, H, N, d] fp32, standardised
    k0: torch.Tensor
    v0: torch.Tensor
    alpha: torch.Tensor   # [B, H] fp32
    gen: torch.Generator = field(repr=False)

    def cast(self):
        """(q, k, v) in the workload dtype, contiguous [B, H, N, d]."""
        a = self.alpha[:, :, None, None]
        dt = self.wl.torch_dtype
        return ((self.q0 * a).to(dt).contiguous(),
                (self.k0 * a).to(dt).contiguous(),
                self.v0.to(dt).contiguous())

    def drift_step(self, delta: float | None = None):
        """Advance one denoising step: variance-preserving drift of q0, k0, v0 in place."""
        delta = self.wl.drift if delta is None else delta
        c = math.sqrt(1.0 - delta * delta)
        B, H, N, d = self.q0.shape
        for b in range(B):
            for h in range(H):
                for t in (self.q0, self.k0, self.v0):
                    xi = torch.randn((N, d), generator=self.gen, device=t.device, dtype=torch.float32)
                    t[b, h].mul_(c).add_(xi, alpha=delta)


def make_layer(wl: Workload, device="cpu", seed: int | None = None) -> Layer:
    """Generate one layer's standardised q/k/v and alpha, following the module recipe."""
    seed = wl.seed if seed is None else seed
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    N, d = wl.N, wl.d
    p = positions(wl.grid, device)
    out = [torch.empty((wl.B, wl.H, N, d), device=device, dtype=torch.float32) for _ in range(3)]
    alpha = torch.empty((wl.B, wl.H), dtype=torch.float32)
    for b in range(wl.B):
        for h in range(wl.H):
            omega = torch.randn((N_FEATURES, 3), generator=g, device=device) * OMEGA_STD
            phase = torch.rand((N_FEATURES,), generator=g, device=device) * (2 * math.pi)
            F = math.sqrt(2.0 / N_FEATURES) * torch.cos(2 * math.pi * (p @ omega.T) + phase)
            for t in out:
                A = torch.randn((d, N_FEATURES), generator=g, device=device)
                x = F @ A.T + NOISE_STD * torch.randn((N, d), generator=g, device=device)
                x = (x - x.mean()) / x.std()
                t[b, h] = x
            ii = torch.randint(0, N, (ALPHA_PAIRS,), generator=g, device=device)
            jj = torch.randint(0, N, (ALPHA_PAIRS,), generator=g, device=device)
            s = (out[0][b, h][ii] * out[1][b, h][jj]).sum(-1) / math.sqrt(d)
            alpha[b, h] = math.sqrt(LOGIT_STD / float(s.std()))
    return Layer(wl, out[0], out[1], out[2], alpha.to(device), g)
