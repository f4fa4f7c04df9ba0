"""Matched-density analysis of one head (test infrastructure only; CPU, float64).

Written from the page "MC-Sparse: Deconstructing and Closing the Dense-Sparse
Attention Gap in Diffusion Transformers" (summary of arXiv 2610.06801), the
paragraphs on block-sparse practice and on matched-density oracles [oracles]:
block-sparse attention cuts queries and keys into tile blocks, scores them with
mean-pooled vectors and keeps or drops blocks whole; oracles that keep as much
true attention mass as a budget allows gain fidelity from whole blocks, to one
shared key set per query group, to a private set per query; the gap to the
mean-pooled baseline splits into structural binding, selection error and the
discarded tail.

Readings (the page gives no formulas):
  * P is the dense softmax of one head, P_ij = exp(s_ij - lse_i);
  * a selection gives every query i a key set I_i; its captured mass is
    sum_{j in I_i} P_ij, averaged over the queries; its output is attention
    renormalised over I_i (the sparse output, no residual), and its output error
    is ||O_sel - O_dense||_F / ||O_dense||_F;
  * the budget is K = ceil(rho N) keys per query; block selections keep
    nb = K // Bk whole key blocks of Bk tokens (K a multiple of Bk matches the
    budget exactly);
  * per-query oracle: I_i = the K largest P_ij of row i;
  * group-shared oracle: the queries of a group share the K keys with the
    largest column sums of P over the group (ties to the lower index); with the
    method's PDDP groups this is the anchor step's selection, with contiguous
    blocks of C queries it is the same rule on the tile grid;
  * block oracle: contiguous query blocks of C, key blocks of Bk; each query block
    keeps the nb key blocks of largest true mass;
  * mean-pooled block-sparse: the same grid, key blocks ranked by the pooled logit
    scale * mean(q over the query block) . mean(k over the key block);
  * decomposition of the mass the mean-pooled baseline loses, 1 - m_pool =
      discarded tail   1 - m_query          (what even a private top-K drops)
    + structural binding m_query - m_block  (whole blocks, shared by a query block)
    + selection error  m_block - m_pool     (pooled scores instead of true mass);
    binding is further split at m_group (contiguous groups, token-level keys):
    key-block binding m_group - m_block and query binding m_query - m_group.
"""
from __future__ import annotations

import math

import numpy as np

from oracle.mcs_oracle import default_scale, pddp_groups, topk_ascending


def probabilities(q: np.ndarray, k: np.ndarray, scale: float | None = None) -> np.ndarray:
    """Dense softmax probabilities P [N, N] of one head (rows sum to 1)."""
    scale = default_scale(q.shape[1]) if scale is None else scale
    s = scale * (q @ k.T)
    e = np.exp(s - s.max(axis=1, keepdims=True))
    return e / e.sum(axis=1, keepdims=True)


def evaluate(P: np.ndarray, v: np.ndarray, sets) -> tuple[float, float]:
    """Mean captured mass and relative output error of per-query key sets
    (`sets[i]` is the index array of query i)."""
    o_dense = P @ v
    mass = np.empty(P.shape[0])
    o = np.empty_like(o_dense)
    for i, I in enumerate(sets):
        w = P[i, I]
        mass[i] = w.sum()
        o[i] = (w / mass[i]) @ v[I]
    err = float(np.linalg.norm(o - o_dense) / np.linalg.norm(o_dense))
    return float(mass.mean()), err


def per_query_sets(P: np.ndarray, K: int):
    return [topk_ascending(P[i], K) for i in range(P.shape[0])]


def group_shared_sets(P: np.ndarray, groups, K: int):
    """`groups`: list of query-index arrays; every member gets its group's set."""
    sets = [None] * P.shape[0]
    for mem in groups:
        I = topk_ascending(P[mem].sum(axis=0), K)
        for i in mem:
            sets[i] = I
    return sets


def contiguous_groups(N: int, C: int):
    return [np.arange(b, min(b + C, N)) for b in range(0, N, C)]


def pddp_group_list(q: np.ndarray, C: int, iters: int = 20):
    """The method's query groups (real members only), from the PDDP oracle."""
    N, d = q.shape
    G = -(-N // C)
    x = np.zeros((G * C, d))
    x[:N] = q
    perm, _ = pddp_groups(x, N, C, iters)
    return [m[m < N] for m in (perm[g * C:(g + 1) * C] for g in range(G))]


def _block_union(kblocks, Bk: int, N: int) -> np.ndarray:
    return np.sort(np.concatenate([np.arange(b * Bk, min((b + 1) * Bk, N)) for b in kblocks]))


def block_oracle_sets(P: np.ndarray, C: int, Bk: int, nb: int):
    N = P.shape[0]
    nkb = -(-N // Bk)
    sets = [None] * N
    for mem in contiguous_groups(N, C):
        col = P[mem].sum(axis=0)
        bm = np.array([col[b * Bk:(b + 1) * Bk].sum() for b in range(nkb)])
        I = _block_union(topk_ascending(bm, nb), Bk, N)
        for i in mem:
            sets[i] = I
    return sets


def mean_pooled_block_sets(q: np.ndarray, k: np.ndarray, C: int, Bk: int, nb: int, scale: float | None = None):
    scale = default_scale(q.shape[1]) if scale is None else scale
    N = q.shape[0]
    nkb = -(-N // Bk)
    kbar = np.stack([k[b * Bk:(b + 1) * Bk].mean(axis=0) for b in range(nkb)])
    sets = [None] * N
    for mem in contiguous_groups(N, C):
        score = scale * (kbar @ q[mem].mean(axis=0))
        I = _block_union(topk_ascending(score, nb), Bk, N)
        for i in mem:
            sets[i] = I
    return sets


def analyse(q, k, v, C: int, Bk: int, rho: float, iters: int = 20, scale: float | None = None) -> dict:
    """Captured mass and output error of every selection at density rho, plus the
    mass decomposition of the mean-pooled baseline's gap."""
    N = q.shape[0]
    K = math.ceil(rho * N)
    nb = max(1, K // Bk)
    P = probabilities(q, k, scale)
    res = {"N": N, "K": K, "nb": nb}
    sel = {
        "per_query": per_query_sets(P, K),
        "group_pddp": group_shared_sets(P, pddp_group_list(q, C, iters), K),
        "group_contiguous": group_shared_sets(P, contiguous_groups(N, C), K),
        "block_oracle": block_oracle_sets(P, C, Bk, nb),
        "mean_pooled": mean_pooled_block_sets(q, k, C, Bk, nb, scale),
    }
    for name, sets in sel.items():
        res[name] = evaluate(P, v, sets)
    m = {name: res[name][0] for name in sel}
    res["decomposition"] = {
        "tail": 1.0 - m["per_query"],
        "binding": m["per_query"] - m["block_oracle"],
        "binding_keys": m["group_contiguous"] - m["block_oracle"],
        "binding_queries": m["per_query"] - m["group_contiguous"],
        "selection": m["block_oracle"] - m["mean_pooled"],
        "gap": 1.0 - m["mean_pooled"],
    }
    return res


def report(heads=2, grid=(4, 32, 32), d=128, C=128, Bk=128, rhos=(0.1, 0.15, 0.2, 0.25, 0.3), seed=0) -> str:
    """Markdown table of the analysis on the synthetic generator's heads."""
    from sparse_attention_diffusion_gb300 import synth

    wl = synth.Workload("matched-density", 1, heads, tuple(grid), d, "f32", C, "0.2", seed=seed)
    layer = synth.make_layer(wl)
    q, k, v = (np.asarray(t.double().numpy()) for t in layer.cast())
    names = ("per_query", "group_pddp", "group_contiguous", "block_oracle", "mean_pooled")
    lines = [f"Synthetic heads: {heads} x N = {wl.N} ({grid[0]}x{grid[1]}x{grid[2]}), d = {d}, C = {C}, "
             f"key blocks Bk = {Bk}; mass / relative output error, averaged over heads.", "",
             "| rho | K | " + " | ".join(names) + " | tail | binding (keys + queries) | selection |",
             "|---|---|" + "---|" * (len(names) + 3)]
    for rho in rhos:
        rs = [analyse(q[0, h], k[0, h], v[0, h], C, Bk, rho) for h in range(heads)]
        cell = lambda n: f"{np.mean([r[n][0] for r in rs]):.4f} / {np.mean([r[n][1] for r in rs]):.4f}"
        dec = lambda n: float(np.mean([r["decomposition"][n] for r in rs]))
        lines.append(f"| {rho} | {rs[0]['K']} | " + " | ".join(cell(n) for n in names) +
                     f" | {dec('tail'):.4f} | {dec('binding'):.4f} ({dec('binding_keys'):.4f} + "
                     f"{dec('binding_queries'):.4f}) | {dec('selection'):.4f} |")
    return "\n".join(lines)


if __name__ == "__main__":
    print(report())
