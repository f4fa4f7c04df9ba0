"""CPU oracle for the MC-Sparse hot path (test infrastructure only).

Plain, slow, float64 numpy restatement of what the method computes, written from
the method's description on the page "MC-Sparse: Deconstructing and Closing the
Dense-Sparse Attention Gap in Diffusion Transformers" (summary of arXiv
2610.06801). Paragraphs cited below by their subject:
  [grouping]  the paragraph on index gathering and PDDP (project onto the
              principal direction, split at the median, repeat; groups of exactly C);
  [selection] the paragraph on the anchor step's two-pass top-K by summed
              attention weight (Q, K, V come from the current step);
  [residual]  the paragraph on the stored dense-minus-sparse output and its
              reuse (groups, indices and residual refresh together).

Only tests, the package smoke check and the benchmark's CPU-baseline leg use
this module. It shares no code with the CUDA path and imports nothing from it.
Every function works on one head: arrays are [N, d] float64 (inputs widened
exactly from fp32 or bf16).

Readings where the page is silent (each is listed with its pin in the design notes):
  * grouping is per head, over the real tokens plus zero pad rows appended at
    ids >= N so that N_pad = G*C; pads take key +inf in every split and are
    excluded from means, covariance products and scores;
  * the principal direction is the top eigenvector of the node's centred
    covariance, computed by exactly `iters` power iterations from 1/sqrt(d)*ones
    with no convergence test;
  * "split at the median" is a rank split: the lower floor(n/2)*C members (by
    projection, then token index) go left, which is the median for even n;
  * group ids are the depth-first leaf order; members are listed ascending;
  * the summed attention weight of key j for group g is the sum over g's real
    queries of the dense softmax probability exp(s_ij - lse_i);
  * top-K ties go to the lower index; indices are emitted ascending;
  * sparse attention renormalises over the kept keys;
  * K = ceil(density * N); scale = 1/sqrt(d).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = [
    "principal_direction", "pddp_node_slot", "pddp_groups", "dense_attention", "group_scores",
    "topk_ascending", "sparse_attention", "captured_mass", "anchor_head",
    "reuse_head", "default_scale",
]


def default_scale(d: int) -> float:
    return 1.0 / math.sqrt(d)


# ---------------------------------------------------------------- [grouping]
def principal_direction(xc: np.ndarray, iters: int, v0: np.ndarray | None = None) -> np.ndarray:
    """Power iteration on the centred rows xc [n, d]: w = xc^T (xc v), v <- w/|w|.

    Exactly `iters` steps from v0 (default 1/sqrt(d) * ones); a zero w leaves v
    unchanged.
    """
    d = xc.shape[1]
    v = np.full(d, 1.0 / math.sqrt(d)) if v0 is None else np.asarray(v0, dtype=np.float64).copy()
    for _ in range(iters):
        w = xc.T @ (xc @ v)
        nrm = math.sqrt(float(w @ w))
        if nrm > 0.0:
            v = w / nrm
    return v


def pddp_node_slot(level: int, k: int) -> int:
    """Slot of tree node k of `level` in a per-head direction table: nodes are
    numbered level by level (root 0; the children of node k are 2k and 2k+1 of
    the next level), so node (level, k) sits at 2^level - 1 + k."""
    return (1 << level) - 1 + k


def pddp_groups(x: np.ndarray, n_real: int, C: int, iters: int = 20, trace: list | None = None,
                v_init: np.ndarray | None = None, v_out: np.ndarray | None = None):
    """PDDP grouping of one head's queries into G = ceil(N/C) groups of exactly C.

    x is [N_pad, d] (rows >= n_real are pads and are ignored). Recursive
    principal-direction split at the rank floor(n/2)*C [grouping].
    Returns (perm [N_pad] int64: token ids group by group, ascending within a
    group; group_of [n_real] int64).
    trace: if a list is given, one record per split node is appended (a report
    only; it changes nothing): g0 (first group id of the node), n (groups),
    left (sorted member ids sent left) and gap (the key gap at the rank split,
    key[n_left*C] - key[n_left*C - 1] among the sorted keys, divided by the
    standard deviation of the node's real keys; inf when the split is at a pad).
    v_init / v_out: optional direction tables [2^L - 1, d] (L = ceil(log2 G))
    indexed by pddp_node_slot. With v_init the power iteration of each split
    node starts from its row instead of 1/sqrt(d)*ones (the warm start of an
    amortised grouping: the previous anchor's directions, so that fewer
    iterations are needed); v_out receives every split node's final direction.
    """
    N_pad = x.shape[0]
    assert N_pad % C == 0 and N_pad - n_real < C and n_real > 0
    groups = []

    def split(members: np.ndarray, n: int, level: int, k: int):
        if n == 1:
            groups.append(np.sort(members))
            return
        real = members[members < n_real]
        mu = x[real].mean(axis=0)
        slot = pddp_node_slot(level, k)
        v = principal_direction(x[real] - mu, iters, None if v_init is None else v_init[slot])
        if v_out is not None:
            v_out[slot] = v
        proj = (x[members] - mu) @ v
        key = np.where(members < n_real, proj, np.inf)
        order = np.lexsort((members, key))          # by key, then token index
        n_left = n // 2
        left = np.sort(members[order[: n_left * C]])
        right = np.sort(members[order[n_left * C:]])
        if trace is not None:
            ks = key[order]
            sd = float(np.std(proj[members < n_real]))
            gap = float(ks[n_left * C] - ks[n_left * C - 1])
            trace.append(dict(g0=len(groups), n=n, left=left,
                              gap=gap / sd if np.isfinite(gap) and sd > 0 else math.inf))
        split(left, n_left, level + 1, 2 * k)
        split(right, n - n_left, level + 1, 2 * k + 1)

    split(np.arange(N_pad), N_pad // C, 0, 0)
    perm = np.concatenate(groups)
    group_of = np.empty(n_real, dtype=np.int64)
    for g, mem in enumerate(groups):
        real = mem[mem < n_real]
        group_of[real] = g
    return perm.astype(np.int64), group_of


# ---------------------------------------------------------------- dense attention
def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float | None = None,
                    row_block: int = 512):
    """Softmax attention of every query row over every key row, with the row log-sum-exp.

    o_i = sum_j exp(s_ij - lse_i) v_j, s_ij = scale q_i.k_j, lse_i = log sum_j exp(s_ij).
    Rows are independent; they are processed `row_block` at a time to bound memory.
    """
    scale = default_scale(q.shape[1]) if scale is None else scale
    o = np.empty((q.shape[0], v.shape[1]))
    lse = np.empty(q.shape[0])
    for r0 in range(0, q.shape[0], row_block):
        s = scale * (q[r0:r0 + row_block] @ k.T)
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        l = e.sum(axis=1, keepdims=True)
        lse[r0:r0 + row_block] = (m + np.log(l))[:, 0]
        o[r0:r0 + row_block] = (e / l) @ v
    return o, lse


# ---------------------------------------------------------------- [selection]
def group_scores(q_real: np.ndarray, lse_real: np.ndarray, k: np.ndarray,
                 scale: float | None = None) -> np.ndarray:
    """Summed dense attention weight of every key over one group's real queries.

    S[j] = sum_i exp(scale q_i.k_j - lse_i): pass 1 gives lse, this is pass 2.
    """
    scale = default_scale(k.shape[1]) if scale is None else scale
    s = scale * (q_real @ k.T)
    return np.exp(s - lse_real[:, None]).sum(axis=0)


def topk_ascending(S: np.ndarray, K: int) -> np.ndarray:
    """Indices of the K largest scores, ties to the lower index, returned ascending."""
    order = np.lexsort((np.arange(S.shape[0]), -S))
    return np.sort(order[:K])


def captured_mass(S: np.ndarray, idx: np.ndarray, n_real_in_group: int) -> float:
    """Fraction of the group's total attention weight kept by the index set."""
    return float(S[idx].sum()) / n_real_in_group


# ---------------------------------------------------------------- sparse attention
def sparse_attention(q_rows: np.ndarray, k: np.ndarray, v: np.ndarray, idx: np.ndarray,
                     scale: float | None = None) -> np.ndarray:
    """Attention of the given query rows over the gathered keys k[idx], v[idx] only,
    with the softmax renormalised over the kept keys [grouping: keys gathered by index]."""
    scale = default_scale(k.shape[1]) if scale is None else scale
    s = scale * (q_rows @ k[idx].T)
    m = s.max(axis=1, keepdims=True)
    e = np.exp(s - m)
    return (e / e.sum(axis=1, keepdims=True)) @ v[idx]


# ---------------------------------------------------------------- [residual] + schedule
def anchor_head(q, k, v, C: int, K: int, iters: int = 20, scale: float | None = None):
    """One head's anchor step: groups, dense output + lse, per-group top-K, sparse
    output and the residual R = O_dense - O_sparse (token order, real rows)."""
    N, d = q.shape
    G = -(-N // C)
    xq = np.zeros((G * C, d))
    xq[:N] = q
    perm, group_of = pddp_groups(xq, N, C, iters)
    o_dense, lse = dense_attention(q, k, v, scale)
    idx = np.empty((G, K), dtype=np.int64)
    mass = np.empty(G)
    o_sparse = np.empty_like(o_dense)
    for g in range(G):
        mem = perm[g * C:(g + 1) * C]
        real = mem[mem < N]
        S = group_scores(q[real], lse[real], k, scale)
        idx[g] = topk_ascending(S, K)
        mass[g] = captured_mass(S, idx[g], real.size)
        o_sparse[real] = sparse_attention(q[real], k, v, idx[g], scale)
    return dict(perm=perm, group_of=group_of, o_dense=o_dense, lse=lse, idx=idx,
                mass=mass, o_sparse=o_sparse, residual=o_dense - o_sparse)


def reuse_head(q, k, v, perm, idx, residual, C: int, scale: float | None = None):
    """One head's reuse step: fresh sparse attention of the current q, k, v over the
    cached groups and indices, plus the cached residual [residual]."""
    N = q.shape[0]
    out = np.empty((N, v.shape[1]))
    for g in range(idx.shape[0]):
        mem = perm[g * C:(g + 1) * C]
        real = mem[mem < N]
        out[real] = sparse_attention(q[real], k, v, idx[g], scale) + residual[real]
    return out
