"""The C-ABI library loads, exports every entry point include/mcs.h declares, and
rejects bad arguments on the host before any launch. CPU only: nothing here
touches a GPU (validation returns before the first CUDA call)."""
import ctypes
import os
import re

import pytest

from sparse_attention_diffusion_gb300 import mcs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return mcs.load(build_if_missing=True)


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mcs.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mcs_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(mcs.EXPORTS)


def test_status_strings(lib):
    for code in range(7):
        s = lib.mcs_status_string(code)
        assert s and s.decode() != "unknown status"
    assert lib.mcs_status_string(99).decode() == "unknown status"


def _desc(**kw):
    base = dict(B=1, H=2, N=600, d=128, C=128, dtype=mcs.MCS_BF16, scale=0.0, pddp_iters=20)
    base.update(kw)
    return mcs.mcs_desc(*[base[k] for k in ("B", "H", "N", "d", "C", "dtype", "scale", "pddp_iters")])


def test_workspace_size_host_only(lib):
    d = _desc()
    n = lib.mcs_workspace_size(ctypes.byref(d), 120)
    assert n > 2 * 600 * 4
    assert lib.mcs_workspace_size(ctypes.byref(_desc(d=96)), 1) == 0
    assert lib.mcs_workspace_size(None, 1) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), 2), (dict(C=32), 2), (dict(dtype=7), 2), (dict(N=0), 1), (dict(B=0), 1),
    (dict(scale=float("nan")), 1), (dict(H=70000), 2),
])
def test_bad_descriptors_rejected(lib, kw, code):
    d = _desc(**kw)
    fake = ctypes.c_void_p(256)
    assert lib.mcs_dense_attn(ctypes.byref(d), fake, fake, fake, fake, None, None) == code


def test_bad_pointers_and_sizes_rejected(lib):
    d = _desc()
    a = ctypes.c_void_p(4096)
    mis = ctypes.c_void_p(4096 + 8)
    assert lib.mcs_dense_attn(ctypes.byref(d), None, a, a, a, None, None) == 1
    assert lib.mcs_dense_attn(ctypes.byref(d), a, a, a, None, None, None) == 1         # no output at all
    assert lib.mcs_dense_attn(ctypes.byref(d), mis, a, a, a, None, None) == 1
    assert lib.mcs_sparse_attn_gather(ctypes.byref(d), a, a, a, a, a, 0, None, a, None) == 1     # K < 1
    assert lib.mcs_sparse_attn_gather(ctypes.byref(d), a, a, a, a, a, 601, None, a, None) == 1   # K > N
    assert lib.mcs_anchor_select(ctypes.byref(d), a, a, a, None, 10, a, None, None, 0, None) == 3  # no workspace
    need = lib.mcs_workspace_size(ctypes.byref(d), 10)
    assert lib.mcs_anchor_select(ctypes.byref(d), a, a, a, None, 10, a, None, a, need - 1, None) == 3
    assert lib.mcs_group_pddp(ctypes.byref(d), a, a, a, a, 16, None) == 3
    assert lib.mcs_residual_store(ctypes.byref(d), a, a, None, None) == 1
    assert lib.mcs_residual_apply(ctypes.byref(d), a, mis, a, None) == 1
    assert lib.mcs_anchor_residual(ctypes.byref(d), a, a, a, a, a, 10, None, a, None) == 1
    assert lib.mcs_selftest_tc_mma(a, a, a, 5, 0, 0, None) == 1
    assert lib.mcs_selftest_ex2_rate(0, 1, a, None) == 1                # iters < 1
    assert lib.mcs_selftest_ex2_rate(16, 0, a, None) == 1               # no CTA
    assert lib.mcs_selftest_ex2_rate(16, 1, None, None) == 1            # no output
    assert lib.mcs_selftest_ex2_rate(16, 1, ctypes.c_void_p(4096 + 4), None) == 1   # misaligned output


def test_launch_counter_is_monotone(lib):
    c0 = lib.mcs_launch_count()
    d = _desc(d=96)
    lib.mcs_dense_attn(ctypes.byref(d), None, None, None, None, None, None)
    assert lib.mcs_launch_count() == c0          # a rejected call launches nothing


def test_host_gather_validation(lib):
    d = _desc()                                   # B=1, H=2, N=600, d=128, bf16
    one = lib.mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(d), 1)
    assert one == 2 * 4 * (((2 * 600 * 128 * 2) + 255) // 256 * 256)    # two slots of q, k, v, o
    two = lib.mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(d), 2)
    assert two == 2 * 4 * (((600 * 128 * 2) + 255) // 256 * 256)
    assert lib.mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(d), 9) == two   # at most one chunk per head
    assert lib.mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(d), 0) == 0
    assert lib.mcs_sparse_attn_gather_host_workspace_size(ctypes.byref(_desc(d=96)), 1) == 0
    a = ctypes.c_void_p(4096)
    g = lib.mcs_sparse_attn_gather_host
    assert g(ctypes.byref(d), None, a, a, a, a, 10, None, a, a, one, 1, None) == 1       # no q
    assert g(ctypes.byref(d), a, a, a, a, a, 10, None, None, a, one, 1, None) == 1       # no output
    assert g(ctypes.byref(d), a, a, a, a, a, 0, None, a, a, one, 1, None) == 1           # K < 1
    assert g(ctypes.byref(d), a, a, a, a, a, 10, None, a, a, one, 0, None) == 1          # no chunks
    assert g(ctypes.byref(d), a, a, a, a, a, 10, None, a, a, one - 1, 1, None) == 3      # small workspace
    assert g(ctypes.byref(d), a, a, a, a, a, 10, None, a, None, one, 1, None) == 3       # no workspace
    assert g(ctypes.byref(d), a, a, a, a, a, 10, None, a, ctypes.c_void_p(4104), one, 1, None) == 3


def test_cache_ring_validation(lib):
    d = _desc()                                   # B=1, H=2, N=600 (N_pad 640, G 5), d=128, bf16
    n = lib.mcs_cache_entry_bytes(ctypes.byref(d), 120)
    a256 = lambda x: (x + 255) // 256 * 256
    assert n == a256(2 * 640 * 4) + a256(2 * 5 * 120 * 4) + a256(2 * 600 * 128 * 2)
    assert lib.mcs_cache_entry_bytes(ctypes.byref(d), 0) == 0
    assert lib.mcs_cache_entry_bytes(ctypes.byref(d), 601) == 0
    ring = ctypes.c_void_p()
    a = ctypes.c_void_p(4096)
    c = lib.mcs_cache_ring_create
    assert c(ctypes.byref(d), 120, 0, a, a, ctypes.byref(ring)) == 1                     # no layers
    assert c(ctypes.byref(d), 120, 3, None, a, ctypes.byref(ring)) == 1                  # no host entries
    assert c(ctypes.byref(d), 120, 3, a, ctypes.c_void_p(4096 + 16), ctypes.byref(ring)) == 1  # slots not 256-aligned
    assert c(ctypes.byref(d), 120, 3, a, a, None) == 1
    assert c(ctypes.byref(_desc(d=96)), 120, 3, a, a, ctypes.byref(ring)) == 2
    p = ctypes.c_void_p()
    assert lib.mcs_cache_ring_acquire(None, 0, 1, 1, None, ctypes.byref(p), ctypes.byref(p), ctypes.byref(p)) == 1
    assert lib.mcs_cache_ring_release(None, 0, 0, None) == 1
    assert lib.mcs_cache_ring_destroy(None) == 1


def test_binding_checks_shapes_against_the_descriptor():
    import torch

    d = _desc()                                   # B=1, H=2, N=600 (N_pad 640, G 5), d=128, bf16
    ok = dict(q=torch.empty(1, 2, 600, 128, dtype=torch.bfloat16), perm=torch.empty(1, 2, 640, dtype=torch.int32),
              idx=torch.empty(1, 2, 5, 120, dtype=torch.int32), lse=torch.empty(1, 2, 600))
    mcs._expect(d, 120, **ok)
    for name, bad in [("q", torch.empty(1, 2, 600, 64, dtype=torch.bfloat16)),
                      ("q", torch.empty(1, 2, 600, 128, dtype=torch.float32)),
                      ("perm", torch.empty(1, 2, 600, dtype=torch.int32)),
                      ("idx", torch.empty(1, 2, 5, 121, dtype=torch.int32)),
                      ("lse", torch.empty(1, 2, 600, dtype=torch.float64))]:
        with pytest.raises(ValueError):
            mcs._expect(d, 120, **dict(ok, **{name: bad}))
    mcs._expect(d, 120, lse=None, mass=None)      # optional outputs may be absent
