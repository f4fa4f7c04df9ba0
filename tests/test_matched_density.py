"""Pins of the matched-density analysis oracle (CPU): the mass ordering the
oracles' definitions force, the full-budget and degenerate cases where two
selections coincide, brute force over subsets on a tiny head, the pooled scorer
on block-constant inputs, and the renormalised output against the oracle's own
sparse attention."""
import itertools

import numpy as np
import pytest

from oracle import matched_density as md
from oracle import mcs_oracle as orc
from sparse_attention_diffusion_gb300 import synth


def _head(grid=(4, 16, 16), d=64, seed=3):
    wl = synth.Workload("t", 1, 1, grid, d, "f32", 64, "0.25", seed=seed)
    q, k, v = (t.double().numpy()[0, 0] for t in synth.make_layer(wl).cast())
    return q, k, v


def test_masses_ordered_at_matched_budget():
    q, k, v = _head()
    r = md.analyse(q, k, v, C=64, Bk=64, rho=0.25)       # K = 256 = 4 whole key blocks
    assert r["K"] == 256 and r["nb"] == 4
    m = {n: r[n][0] for n in ("per_query", "group_pddp", "group_contiguous", "block_oracle", "mean_pooled")}
    assert m["per_query"] >= m["group_pddp"] - 1e-12
    assert m["per_query"] >= m["group_contiguous"] >= m["block_oracle"] >= m["mean_pooled"] > 0
    dec = r["decomposition"]
    assert abs(dec["tail"] + dec["binding"] + dec["selection"] - dec["gap"]) < 1e-12
    assert abs(dec["binding_keys"] + dec["binding_queries"] - dec["binding"]) < 1e-12


def test_full_budget_keeps_everything():
    q, k, v = _head(grid=(2, 8, 16))
    r = md.analyse(q, k, v, C=64, Bk=64, rho=1.0)
    for n in ("per_query", "group_pddp", "group_contiguous", "block_oracle", "mean_pooled"):
        mass, err = r[n]
        assert abs(mass - 1.0) < 1e-12 and err < 1e-12, n


def test_unit_key_blocks_equal_group_selection():
    q, k, v = _head(grid=(2, 8, 16))
    P = md.probabilities(q, k)
    K = 64
    a = md.block_oracle_sets(P, C=64, Bk=1, nb=K)
    b = md.group_shared_sets(P, md.contiguous_groups(P.shape[0], 64), K)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_singleton_groups_equal_per_query():
    q, k, v = _head(grid=(2, 8, 16))
    P = md.probabilities(q, k)
    a = md.group_shared_sets(P, md.contiguous_groups(P.shape[0], 1), 40)
    b = md.per_query_sets(P, 40)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_brute_force_tiny_head():
    rng = np.random.default_rng(5)
    N, d, K, C, Bk = 8, 4, 3, 4, 2
    q, k = rng.normal(size=(N, d)) * 2, rng.normal(size=(N, d)) * 2
    P = md.probabilities(q, k)
    best_row = [max(P[i, list(s)].sum() for s in itertools.combinations(range(N), K)) for i in range(N)]
    assert np.allclose([P[i, I].sum() for i, I in enumerate(md.per_query_sets(P, K))], best_row, atol=1e-15)
    groups = md.contiguous_groups(N, C)
    sets = md.group_shared_sets(P, groups, K)
    for mem in groups:
        best = max(P[np.ix_(mem, list(s))].sum() for s in itertools.combinations(range(N), K))
        assert abs(P[np.ix_(mem, sets[mem[0]])].sum() - best) < 1e-15
    bsets = md.block_oracle_sets(P, C, Bk, 1)
    for mem in groups:
        best = max(P[np.ix_(mem, list(range(b * Bk, (b + 1) * Bk)))].sum() for b in range(N // Bk))
        assert abs(P[np.ix_(mem, bsets[mem[0]])].sum() - best) < 1e-15


def test_pooled_scores_exact_on_block_constant_inputs():
    """Identical rows inside every query block and every key block: the pooled
    logit is the true logit, so the pooled ranking is the block oracle's."""
    rng = np.random.default_rng(7)
    N, d, C, Bk = 64, 8, 16, 8
    q = np.repeat(rng.normal(size=(N // C, d)), C, axis=0)
    k = np.repeat(rng.normal(size=(N // Bk, d)) * 1.5, Bk, axis=0)
    P = md.probabilities(q, k)
    a = md.mean_pooled_block_sets(q, k, C, Bk, 3)
    b = md.block_oracle_sets(P, C, Bk, 3)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))


def test_renormalised_output_matches_sparse_attention():
    q, k, v = _head(grid=(2, 8, 16))
    P = md.probabilities(q, k)
    groups = md.contiguous_groups(P.shape[0], 64)
    sets = md.group_shared_sets(P, groups, 50)
    o = np.concatenate([orc.sparse_attention(q[m], k, v, sets[m[0]]) for m in groups])
    o_dense, _ = orc.dense_attention(q, k, v)
    want_err = np.linalg.norm(o - o_dense) / np.linalg.norm(o_dense)
    _, err = md.evaluate(P, v, sets)
    assert err == pytest.approx(want_err, rel=1e-10)
