"""Thin ctypes binding of libmcs (the C ABI in include/mcs.h).

Functions carry the C names and only marshal arguments: torch tensors become
device pointers, the current torch CUDA stream becomes the stream argument, and
a non-OK status raises McsError. Every step of the path runs in libmcs's CUDA
kernels; there is no fallback. Loading fails loudly when libmcs.so is missing.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

from . import build as _build

MCS_OK = 0
STATUS_NAMES = {0: "MCS_OK", 1: "MCS_ERR_INVALID_ARG", 2: "MCS_ERR_UNSUPPORTED", 3: "MCS_ERR_WORKSPACE",
                4: "MCS_ERR_CUDA", 5: "MCS_ERR_DEVICE_BOUNDS", 6: "MCS_ERR_DEVICE_TIMEOUT"}
MCS_F32, MCS_BF16 = 0, 1

EXPORTS = ("mcs_workspace_size", "mcs_group_pddp", "mcs_dense_attn", "mcs_anchor_select",
           "mcs_sparse_attn_gather", "mcs_anchor_residual", "mcs_residual_store", "mcs_residual_apply",
           "mcs_check_status", "mcs_status_string", "mcs_launch_count", "mcs_selftest_tc_mma",
           "mcs_selftest_tma_gather", "mcs_anchor_select_noalloc", "mcs_sparse_attn_gather_host",
           "mcs_sparse_attn_gather_host_workspace_size", "mcs_cache_entry_bytes", "mcs_cache_ring_create",
           "mcs_cache_ring_acquire", "mcs_cache_ring_release", "mcs_cache_ring_destroy",
           "mcs_selftest_wait_timeout", "mcs_pddp_dirs_size", "mcs_group_pddp_warm", "mcs_selftest_ex2_rate")


class McsError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(code, code)} ({_status_string(code)})")


class mcs_desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("N", ctypes.c_int), ("d", ctypes.c_int),
                ("C", ctypes.c_int), ("dtype", ctypes.c_int), ("scale", ctypes.c_float),
                ("pddp_iters", ctypes.c_int)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """Load libmcs.so (optionally building it first) and declare the signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_build.LIB):
        if not build_if_missing:
            raise RuntimeError(f"libmcs.so not built at {_build.LIB}: run sparse_attention_diffusion_gb300.build.build()")
        _build.build()
    L = ctypes.CDLL(_build.LIB)
    P, I, Z, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p
    D = ctypes.POINTER(mcs_desc)
    sig = {
        "mcs_workspace_size": (Z, [D, I]),
        "mcs_group_pddp": (I, [D, P, P, P, P, Z, S]),
        "mcs_pddp_dirs_size": (Z, [D]),
        "mcs_group_pddp_warm": (I, [D, P, P, P, P, P, P, Z, S]),
        "mcs_dense_attn": (I, [D, P, P, P, P, P, S]),
        "mcs_anchor_select": (I, [D, P, P, P, P, I, P, P, P, Z, S]),
        "mcs_sparse_attn_gather": (I, [D, P, P, P, P, P, I, P, P, S]),
        "mcs_anchor_residual": (I, [D, P, P, P, P, P, I, P, P, S]),
        "mcs_residual_store": (I, [D, P, P, P, S]),
        "mcs_residual_apply": (I, [D, P, P, P, S]),
        "mcs_check_status": (I, [S]),
        "mcs_status_string": (ctypes.c_char_p, [I]),
        "mcs_launch_count": (ctypes.c_uint64, []),
        "mcs_selftest_tc_mma": (I, [P, P, P, I, ctypes.c_uint32, ctypes.c_uint32, S]),
        "mcs_selftest_tma_gather": (I, [P, I, P, P, S]),
        "mcs_selftest_wait_timeout": (I, [ctypes.c_uint64, P, S]),
        "mcs_selftest_ex2_rate": (I, [I, I, P, S]),
        "mcs_anchor_select_noalloc": (I, [D, P, P, P, P, I, P, P, S]),
        "mcs_sparse_attn_gather_host": (I, [D, P, P, P, P, P, I, P, P, P, Z, I, S]),
        "mcs_sparse_attn_gather_host_workspace_size": (Z, [D, I]),
        "mcs_cache_entry_bytes": (Z, [D, I]),
        "mcs_cache_ring_create": (I, [D, I, I, P, P, ctypes.POINTER(ctypes.c_void_p)]),
        "mcs_cache_ring_acquire": (I, [P, I, I, I, S, ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                                       ctypes.POINTER(ctypes.c_void_p)]),
        "mcs_cache_ring_release": (I, [P, I, I, S]),
        "mcs_cache_ring_destroy": (I, [P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype, fn.argtypes = res, args
    _lib = L
    return L


def _status_string(code) -> str:
    try:
        return load().mcs_status_string(code).decode()
    except Exception:
        return "?"


def _check(fn, code):
    if code != MCS_OK:
        raise McsError(fn, code)


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("libmcs takes device tensors")
    if not t.is_contiguous():
        raise ValueError("libmcs takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def make_desc(B, H, N, d, C, dtype, scale=0.0, pddp_iters=20) -> mcs_desc:
    dt = MCS_BF16 if dtype in (torch.bfloat16, "bf16", MCS_BF16) else MCS_F32
    return mcs_desc(B, H, N, d, C, dt, float(scale), int(pddp_iters))


def desc_for(x: torch.Tensor, C: int, pddp_iters: int = 20) -> mcs_desc:
    B, H, N, d = x.shape
    return make_desc(B, H, N, d, C, x.dtype, 0.0, pddp_iters)


def geometry(desc: mcs_desc):
    G = -(-desc.N // desc.C)
    return G, G * desc.C


def mcs_workspace_size(desc: mcs_desc, K: int = 1) -> int:
    return int(load().mcs_workspace_size(ctypes.byref(desc), int(K)))


def workspace(desc: mcs_desc, K: int = 1, device="cuda") -> torch.Tensor:
    n = mcs_workspace_size(desc, K)
    if n == 0:
        raise McsError("mcs_workspace_size", 2)
    return torch.empty(n, dtype=torch.uint8, device=device)


def _io_dtype(desc):
    return torch.bfloat16 if desc.dtype == MCS_BF16 else torch.float32


def _expect(desc, K=None, **tensors):
    """Host check of tensors against the descriptor before their pointers cross
    the ABI (the library trusts the descriptor's sizes): x-like tensors are
    [B,H,N,d] in the I/O dtype, perm [B,H,N_pad] int32, group_of [B,H,N] int32,
    lse [B,H,N] fp32, idx [B,H,G,K] int32, mass [B,H,G] fp32. None is allowed."""
    G, N_pad = geometry(desc)
    B, H, N, d = desc.B, desc.H, desc.N, desc.d
    want = {"x": ((B, H, N, d), _io_dtype(desc)), "perm": ((B, H, N_pad), torch.int32),
            "group_of": ((B, H, N), torch.int32), "lse": ((B, H, N), torch.float32),
            "idx": ((B, H, G, K), torch.int32), "mass": ((B, H, G), torch.float32)}
    for name, t in tensors.items():
        if t is None:
            continue
        kind = name if name in want else "x"
        shape, dtype = want[kind]
        if tuple(t.shape) != tuple(shape) or t.dtype != dtype:
            raise ValueError(f"{name}: expected {tuple(shape)} {dtype}, got {tuple(t.shape)} {t.dtype}")


def mcs_group_pddp(desc, q, perm, group_of, ws, stream=None):
    _expect(desc, q=q, perm=perm, group_of=group_of)
    _check("mcs_group_pddp", load().mcs_group_pddp(ctypes.byref(desc), _ptr(q), _ptr(perm), _ptr(group_of), _ptr(ws),
                                                   ws.numel(), _stream(stream)))


def pddp_dirs(desc, device="cuda") -> torch.Tensor:
    """A zeroed PDDP direction table [B, H, S, d] fp32 (S = 2^ceil(log2 G) - 1)."""
    n = int(load().mcs_pddp_dirs_size(ctypes.byref(desc)))
    S = n // (4 * desc.B * desc.H * desc.d)
    return torch.zeros((desc.B, desc.H, S, desc.d), dtype=torch.float32, device=device)


def mcs_group_pddp_warm(desc, q, dirs_in, dirs_out, perm, group_of, ws, stream=None):
    """PDDP grouping whose power iterations start from stored directions (dirs_in,
    or None for the fixed start); final directions go to dirs_out (or None)."""
    _expect(desc, q=q, perm=perm, group_of=group_of)
    n = int(load().mcs_pddp_dirs_size(ctypes.byref(desc)))
    for name, t in (("dirs_in", dirs_in), ("dirs_out", dirs_out)):
        if t is not None and (t.dtype != torch.float32 or t.numel() * 4 != n):
            raise ValueError(f"{name}: expected {n // 4} fp32 elements, got {t.numel()} {t.dtype}")
    _check("mcs_group_pddp_warm", load().mcs_group_pddp_warm(ctypes.byref(desc), _ptr(q), _ptr(dirs_in), _ptr(dirs_out),
                                                             _ptr(perm), _ptr(group_of), _ptr(ws), ws.numel(),
                                                             _stream(stream)))


def mcs_dense_attn(desc, q, k, v, o, lse, stream=None):
    _expect(desc, q=q, k=k, v=v, o=o, lse=lse)
    _check("mcs_dense_attn", load().mcs_dense_attn(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                                   _stream(stream)))


def mcs_anchor_select(desc, q, k, perm, lse, K, idx, mass, ws, stream=None):
    _expect(desc, int(K), q=q, k=k, perm=perm, lse=lse, idx=idx, mass=mass)
    _check("mcs_anchor_select", load().mcs_anchor_select(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(perm), _ptr(lse),
                                                         int(K), _ptr(idx), _ptr(mass), _ptr(ws), ws.numel(),
                                                         _stream(stream)))


def mcs_anchor_select_noalloc(desc, q, k, perm, lse, K, idx, mass, stream=None):
    """mcs_anchor_select without a workspace (scores kept in the library's fixed device array)."""
    _expect(desc, int(K), q=q, k=k, perm=perm, lse=lse, idx=idx, mass=mass)
    _check("mcs_anchor_select_noalloc", load().mcs_anchor_select_noalloc(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(perm),
                                                                         _ptr(lse), int(K), _ptr(idx), _ptr(mass),
                                                                         _stream(stream)))


def mcs_sparse_attn_gather(desc, q, k, v, perm, idx, K, residual, o, stream=None):
    _expect(desc, int(K), q=q, k=k, v=v, perm=perm, idx=idx, residual=residual, o=o)
    _check("mcs_sparse_attn_gather", load().mcs_sparse_attn_gather(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v),
                                                                   _ptr(perm), _ptr(idx), int(K), _ptr(residual),
                                                                   _ptr(o), _stream(stream)))


def _host_ptr(t):
    if t.is_cuda:
        raise ValueError("expected a host tensor")
    if not t.is_contiguous():
        raise ValueError("libmcs takes contiguous tensors")
    return ctypes.c_void_p(t.data_ptr())


def host_gather_workspace(desc, head_chunks, device="cuda") -> torch.Tensor:
    n = load().mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(desc), int(head_chunks))
    if n == 0:
        raise McsError("mcs_sparse_attn_gather_host_workspace_size", 1)
    return torch.empty(n, dtype=torch.uint8, device=device)


def mcs_sparse_attn_gather_host(desc, q_host, k_host, v_host, perm, idx, K, residual, o_host, ws, head_chunks,
                                stream=None):
    """Reuse-step sparse attention from host q/k/v (pinned for overlap) to a host output."""
    _expect(desc, int(K), q=q_host, k=k_host, v=v_host, perm=perm, idx=idx, residual=residual, o=o_host)
    _check("mcs_sparse_attn_gather_host", load().mcs_sparse_attn_gather_host(
        ctypes.byref(desc), _host_ptr(q_host), _host_ptr(k_host), _host_ptr(v_host), _ptr(perm), _ptr(idx), int(K),
        _ptr(residual), _host_ptr(o_host), _ptr(ws), ws.numel() * ws.element_size(), int(head_chunks),
        _stream(stream)))


class CacheRing:
    """The per-layer meta-cache {perm, idx, residual} of n_layers layers in pinned
    host memory with two device slots (mcs_cache_ring_*). acquire() returns
    device tensors viewing the layer's slot; they stay valid until release()."""

    def __init__(self, desc, K, n_layers, dtype, device="cuda"):
        lib = load()
        self.desc, self.K, self.n_layers, self.dtype = desc, int(K), int(n_layers), dtype
        self.entry = lib.mcs_cache_entry_bytes(ctypes.byref(desc), self.K)
        if self.entry == 0:
            raise McsError("mcs_cache_entry_bytes", 1)
        self.host = torch.empty(self.n_layers * self.entry + 256, dtype=torch.uint8, pin_memory=True)
        self.dev = torch.empty(2 * self.entry + 256, dtype=torch.uint8, device=device)
        h = ctypes.c_void_p((self.host.data_ptr() + 255) & ~255)
        d = ctypes.c_void_p((self.dev.data_ptr() + 255) & ~255)
        self._h0, self._d0 = h.value, d.value
        self._ring = ctypes.c_void_p()
        _check("mcs_cache_ring_create", lib.mcs_cache_ring_create(ctypes.byref(desc), self.K, self.n_layers, h, d,
                                                                  ctypes.byref(self._ring)))
        G, N_pad = geometry(desc)
        self._shapes = ((desc.B, desc.H, N_pad), (desc.B, desc.H, G, self.K), (desc.B, desc.H, desc.N, desc.d))

    def _view(self, addr, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        off = addr - self.dev.data_ptr()
        return self.dev[off:off + nbytes].view(dtype).view(shape)

    def acquire(self, layer, fill=True, prefetch_next=True, stream=None):
        """fill: make the layer's host entry resident (False: the caller overwrites the slot)."""
        p, i, r = ctypes.c_void_p(), ctypes.c_void_p(), ctypes.c_void_p()
        _check("mcs_cache_ring_acquire", load().mcs_cache_ring_acquire(
            self._ring, int(layer), int(bool(fill)), int(bool(prefetch_next)), _stream(stream), ctypes.byref(p),
            ctypes.byref(i), ctypes.byref(r)))
        sp, si, sr = self._shapes
        return {"perm": self._view(p.value, sp, torch.int32), "idx": self._view(i.value, si, torch.int32),
                "residual": self._view(r.value, sr, self.dtype)}

    def release(self, layer, store=False, stream=None):
        _check("mcs_cache_ring_release", load().mcs_cache_ring_release(self._ring, int(layer), int(bool(store)),
                                                                         _stream(stream)))

    def close(self):
        """Wait for the ring's copies and free it (the buffers stay with this object)."""
        if self._ring:
            _check("mcs_cache_ring_destroy", load().mcs_cache_ring_destroy(self._ring))
            self._ring = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def mcs_anchor_residual(desc, q, k, v, perm, idx, K, o_dense, r, stream=None):
    _expect(desc, int(K), q=q, k=k, v=v, perm=perm, idx=idx, o_dense=o_dense, r=r)
    _check("mcs_anchor_residual", load().mcs_anchor_residual(ctypes.byref(desc), _ptr(q), _ptr(k), _ptr(v), _ptr(perm),
                                                             _ptr(idx), int(K), _ptr(o_dense), _ptr(r),
                                                             _stream(stream)))


def mcs_residual_store(desc, o_dense, o_sparse, r, stream=None):
    _expect(desc, o_dense=o_dense, o_sparse=o_sparse, r=r)
    _check("mcs_residual_store", load().mcs_residual_store(ctypes.byref(desc), _ptr(o_dense), _ptr(o_sparse), _ptr(r),
                                                           _stream(stream)))


def mcs_residual_apply(desc, o_sparse, r, o, stream=None):
    _expect(desc, o_sparse=o_sparse, r=r, o=o)
    _check("mcs_residual_apply", load().mcs_residual_apply(ctypes.byref(desc), _ptr(o_sparse), _ptr(r), _ptr(o),
                                                           _stream(stream)))


def mcs_check_status(stream=None):
    _check("mcs_check_status", load().mcs_check_status(_stream(stream)))


def mcs_launch_count() -> int:
    return int(load().mcs_launch_count())


def mcs_selftest_tc_mma(a, b, d, mode, mn_lbo=16384, mn_sbo=1024, stream=None):
    _check("mcs_selftest_tc_mma", load().mcs_selftest_tc_mma(_ptr(a), _ptr(b), _ptr(d), int(mode), int(mn_lbo),
                                                             int(mn_sbo), _stream(stream)))


def mcs_selftest_wait_timeout(limit_ns, elapsed=None, stream=None):
    """Launch the bounded-wait diagnostic (a wait that must time out after limit_ns).
    elapsed: optional int64 device tensor of one element receiving the wait in ns."""
    _check("mcs_selftest_wait_timeout", load().mcs_selftest_wait_timeout(int(limit_ns), _ptr(elapsed),
                                                                         _stream(stream)))


def mcs_selftest_ex2_rate(iters, out, stream=None):
    """Launch the exponential-rate diagnostic: out is an int64 device tensor [nblocks, 2]
    receiving each CTA's duration in SM clock cycles and its exponential count."""
    _check("mcs_selftest_ex2_rate", load().mcs_selftest_ex2_rate(int(iters), int(out.shape[0]), _ptr(out),
                                                                 _stream(stream)))


def ex2_per_clock_per_sm(iters=1 << 14):
    """Exponentials (ex2.approx.ftz.f32) per SM clock cycle, median over one CTA per SM."""
    import torch
    n = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    out = torch.zeros((n, 2), dtype=torch.int64, device="cuda")
    mcs_selftest_ex2_rate(iters, out)
    mcs_check_status()
    cyc, cnt = out[:, 0].double().cpu(), out[:, 1].double().cpu()
    return float((cnt / cyc).median())


def mcs_selftest_tma_gather(src, rows, out, stream=None):
    _check("mcs_selftest_tma_gather", load().mcs_selftest_tma_gather(_ptr(src), int(src.shape[0]), _ptr(rows), _ptr(out),
                                                                     _stream(stream)))


# ---------------------------------------------------------------- convenience: buffers for one layer
def alloc_cache(desc: mcs_desc, K: int, dtype, device="cuda"):
    """Caller-owned meta-cache buffers {perm, group_of, idx, mass, residual} for one layer."""
    G, N_pad = geometry(desc)
    BH = desc.B * desc.H
    return dict(
        perm=torch.empty((desc.B, desc.H, N_pad), dtype=torch.int32, device=device),
        group_of=torch.empty((desc.B, desc.H, desc.N), dtype=torch.int32, device=device),
        idx=torch.empty((desc.B, desc.H, G, K), dtype=torch.int32, device=device),
        mass=torch.empty((desc.B, desc.H, G), dtype=torch.float32, device=device),
        residual=torch.empty((desc.B, desc.H, desc.N, desc.d), dtype=dtype, device=device),
    )


def density_K(density, N) -> int:
    from fractions import Fraction
    return int(math.ceil(Fraction(str(density)) * N))
