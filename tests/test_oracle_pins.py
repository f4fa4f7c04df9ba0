"""Pins of the CPU oracle to facts it does not compute itself: closed forms,
invariants of the method, reductions to library routines it does not call,
brute force on tiny inputs and hand-worked cases. CPU only."""
import itertools
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import mcs_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _sdpa(q, k, v, scale=None):
    """torch scaled_dot_product_attention in float64 on CPU (library routine)."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a))[None, None] for a in (q, k, v))
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)[0, 0].numpy()


# ---------------------------------------------------------------- PDDP grouping
@pytest.mark.parametrize("N,C,d", [(1000, 64, 16), (1024, 64, 64), (700, 128, 8), (129, 64, 3)])
def test_pddp_groups_are_an_exact_partition(N, C, d):
    x = _rng(N).standard_normal((N, d))
    G = -(-N // C)
    xp = np.zeros((G * C, d))
    xp[:N] = x
    perm, group_of = orc.pddp_groups(xp, N, C, iters=20)
    assert perm.shape == (G * C,)
    assert np.array_equal(np.sort(perm), np.arange(G * C))        # a permutation of 0..N_pad-1
    for g in range(G):
        mem = perm[g * C:(g + 1) * C]
        assert mem.size == C and np.all(np.diff(mem) > 0)        # exactly C, ascending
        assert np.all(group_of[mem[mem < N]] == g)
    assert np.all(perm[:(G - 1) * C] < N)                           # pads only in the last group
    assert np.all(perm[(G - 1) * C:][C - (G * C - N):] >= N)


@pytest.mark.parametrize("N,C", [(64, 8), (96, 8), (200, 16), (77, 4)])
def test_pddp_d1_is_sort_and_chunk(N, C):
    """d = 1: the principal direction is +1, so PDDP reduces to sorting by
    (value, index) and cutting into consecutive chunks of C (depth-first order)."""
    x = np.round(_rng(N + C).standard_normal(N) * 3) / 2          # many exact duplicates
    G = -(-N // C)
    xp = np.zeros((G * C, 1))
    xp[:N, 0] = x
    perm, _ = orc.pddp_groups(xp, N, C, iters=20)
    order = list(np.lexsort((np.arange(N), x))) + list(range(N, G * C))
    expect = np.concatenate([np.sort(order[g * C:(g + 1) * C]) for g in range(G)])
    assert np.array_equal(perm, expect)


def test_principal_direction_matches_eigh():
    rng = _rng(7)
    d = 24
    basis, _ = np.linalg.qr(rng.standard_normal((d, d)))
    x = rng.standard_normal((4000, d)) * np.r_[4.0, np.linspace(2.0, 0.5, d - 1)] @ basis.T   # eigengap ratio 1/4
    xc = x - x.mean(axis=0)
    v = orc.principal_direction(xc, iters=60)
    w, U = np.linalg.eigh(xc.T @ xc)
    assert abs(abs(v @ U[:, -1]) - 1.0) < 1e-10
    assert abs(np.linalg.norm(v) - 1.0) < 1e-12


def test_principal_direction_collinear():
    rng = _rng(3)
    u = rng.standard_normal(10)
    u /= np.linalg.norm(u)
    t = rng.standard_normal(50)
    v = orc.principal_direction(np.outer(t - t.mean(), u), iters=3)
    assert abs(abs(v @ u) - 1.0) < 1e-12


def test_principal_direction_fixed_start_and_zero():
    d = 5
    v = orc.principal_direction(np.zeros((7, d)), iters=20)         # w = 0: v stays at the start
    assert np.allclose(v, np.full(d, 1 / math.sqrt(d)))
    v0 = orc.principal_direction(np.eye(d)[:1] * 2.0 - 0.0, iters=0)
    assert np.allclose(v0, np.full(d, 1 / math.sqrt(d)))


def test_pddp_recovers_planted_clusters_far_from_origin():
    """Four tight clusters at the corners of a 10 x 3 rectangle, shifted far along a
    third axis. Centred PCA splits the long side, then the short sides, so the groups
    are the clusters. An uncentred direction would point along the shift and fail."""
    rng = _rng(11)
    C, d = 32, 8
    corners = [(0, 0), (10, 0), (0, 3), (10, 3)]
    pts, labels = [], []
    for c, (a, b) in enumerate(corners):
        base = np.zeros(d)
        base[0], base[1], base[2] = a, b, 50.0
        pts.append(base + 0.05 * rng.standard_normal((C, d)))
        labels += [c] * C
    x = np.concatenate(pts)
    shuffle = rng.permutation(x.shape[0])
    x, labels = x[shuffle], np.array(labels)[shuffle]
    perm, group_of = orc.pddp_groups(x, x.shape[0], C, iters=20)
    got = {frozenset(perm[g * C:(g + 1) * C].tolist()) for g in range(4)}
    want = {frozenset(np.nonzero(labels == c)[0].tolist()) for c in range(4)}
    assert got == want


def test_pddp_line_clusters_in_order():
    """Eight clusters along a line: the depth-first leaf order walks the line."""
    rng = _rng(5)
    C, d = 16, 6
    direction = rng.standard_normal(d)
    direction /= np.linalg.norm(direction)
    x = np.concatenate([c * 5.0 * direction + 0.01 * rng.standard_normal((C, d)) for c in range(8)])
    perm, _ = orc.pddp_groups(x, 8 * C, C, iters=20)
    firsts = [perm[g * C] // C for g in range(8)]
    assert firsts == list(range(8)) or firsts == list(range(7, -1, -1))
    for g in range(8):
        assert len(set((perm[g * C:(g + 1) * C] // C).tolist())) == 1


def _golden_kv(name):
    """Parse a `key | values` golden file; lines under `points` are `id | x | y`."""
    kv, pts = {}, []
    in_points = False
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            if line.strip() == "points":
                in_points = True
                continue
            parts = [t.strip() for t in line.split("|")]
            if in_points and len(parts) == 3 and parts[0].lstrip("-").isdigit():
                pts.append((int(parts[0]), float(parts[1]), float(parts[2])))
                continue
            in_points = False
            kv[parts[0]] = parts[1]
    return kv, pts


def test_pddp_hand_worked_odd_split():
    """G = 3: the root sends floor(3/2) = 1 group left, and the right node's own
    principal direction (not the root's) cuts the remaining points. Hand-worked in
    tests/golden/pddp_odd_split.txt; a ceil(n/2) split gives different groups."""
    kv, pts = _golden_kv("pddp_odd_split.txt")
    C = int(kv["C"])
    x = np.zeros((len(pts), 2))
    for i, a, b in pts:
        x[i] = (a, b)
    perm, group_of = orc.pddp_groups(x, len(pts), C, iters=20)
    assert perm.tolist() == [int(t) for t in kv["perm"].split()]
    assert group_of.tolist() == [int(t) for t in kv["group_of"].split()]


def test_pddp_hand_worked_warm_start():
    """Stored start directions per tree node (level-by-level slots) with 0 power
    iterations: the right node is then cut along x instead of its own principal
    direction. Hand-worked in tests/golden/pddp_odd_split.txt."""
    kv, pts = _golden_kv("pddp_odd_split.txt")
    C = int(kv["C"])
    x = np.zeros((len(pts), 2))
    for i, a, b in pts:
        x[i] = (a, b)
    dirs = np.array([[float(t) for t in row.split()] for row in kv["warm_dirs"].split(";")])
    perm, _ = orc.pddp_groups(x, len(pts), C, iters=int(kv["warm_iters"]), v_init=dirs)
    assert perm.tolist() == [int(t) for t in kv["warm_perm"].split()]


@pytest.mark.parametrize("N,C,d", [(1000, 64, 16), (700, 128, 8)])
def test_pddp_warm_start_from_own_directions_reproduces_groups(N, C, d):
    """Directions written by one grouping, fed back as start vectors with zero
    iterations, give back the same groups (every node reads its own slot); the
    default start equals a table of 1/sqrt(d) rows."""
    x = _rng(N + d).standard_normal((N, d)) * np.linspace(3, 1, d)
    G = -(-N // C)
    xp = np.zeros((G * C, d))
    xp[:N] = x
    L = int(math.ceil(math.log2(G))) if G > 1 else 0
    dirs = np.full(((1 << L) - 1, d), np.nan)
    perm, _ = orc.pddp_groups(xp, N, C, iters=20, v_out=dirs)
    perm0, _ = orc.pddp_groups(xp, N, C, iters=0, v_init=dirs)
    assert np.array_equal(perm0, perm)
    ones = np.full(((1 << L) - 1, d), 1 / math.sqrt(d))
    perm1, _ = orc.pddp_groups(xp, N, C, iters=7, v_init=ones)
    assert np.array_equal(perm1, orc.pddp_groups(xp, N, C, iters=7)[0])


def test_principal_direction_warm_start_converges_to_eigh():
    rng = _rng(17)
    d = 12
    basis, _ = np.linalg.qr(rng.standard_normal((d, d)))
    x = rng.standard_normal((3000, d)) * np.r_[3.0, np.linspace(1.5, 0.5, d - 1)] @ basis.T
    xc = x - x.mean(axis=0)
    v0 = rng.standard_normal(d)
    v = orc.principal_direction(xc, iters=60, v0=v0 / np.linalg.norm(v0))
    U = np.linalg.eigh(xc.T @ xc)[1]
    assert abs(abs(v @ U[:, -1]) - 1.0) < 1e-10


def test_pddp_hand_worked_pads_excluded():
    """Pads (zero rows at ids >= N) enter neither the node mean nor its covariance:
    with them, the x axis would win and a different real token would share the pad
    group. Hand-worked in tests/golden/pddp_pads.txt."""
    kv, _ = _golden_kv("pddp_pads.txt")
    N, C = int(kv["N"]), int(kv["C"])
    i = np.arange(N)
    y = (37 * i % 65) - 32.0
    x = np.zeros((2 * C, 2))
    x[:N, 0] = 100.0 + 0.001 * (352.0 - y * y)
    x[:N, 1] = y
    perm, group_of = orc.pddp_groups(x, N, C, iters=20)
    want1 = [int(t) for t in kv["group1"].split()]
    assert perm[C:].tolist() == want1
    assert perm[:C].tolist() == [t for t in range(N) if t not in want1]
    assert np.all(group_of[want1[:1]] == 1) and int((group_of == 0).sum()) == N - 1


# ---------------------------------------------------------------- dense attention
@pytest.mark.parametrize("N,Nk,d", [(37, 53, 16), (300, 300, 64), (5, 1, 8)])
def test_dense_matches_sdpa_and_logsumexp(N, Nk, d):
    rng = _rng(N * Nk)
    q, k, v = rng.standard_normal((N, d)) * 2, rng.standard_normal((Nk, d)) * 2, rng.standard_normal((Nk, d))
    o, lse = orc.dense_attention(q, k, v, row_block=16)
    assert np.allclose(o, _sdpa(q, k, v), rtol=0, atol=1e-12)
    ref_lse = scipy.special.logsumexp((q @ k.T) / math.sqrt(d), axis=1)
    assert np.allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_dense_rows_sum_to_one():
    rng = _rng(1)
    q, k = rng.standard_normal((50, 8)) * 3, rng.standard_normal((70, 8)) * 3
    ones = np.ones((70, 1))
    o, _ = orc.dense_attention(q, k, ones)
    assert np.allclose(o, 1.0, atol=1e-14)


# ---------------------------------------------------------------- selection
def test_group_scores_sum_to_group_size_and_match_softmax_rows():
    rng = _rng(2)
    d = 16
    q, k = rng.standard_normal((40, d)) * 2, rng.standard_normal((90, d)) * 2
    _, lse = orc.dense_attention(q, k, np.zeros((90, 1)))
    S = orc.group_scores(q[:13], lse[:13], k)
    assert abs(S.sum() - 13) < 1e-12
    P = torch.softmax(torch.from_numpy(q[:13] @ k.T / math.sqrt(d)), dim=1).numpy()
    assert np.allclose(S, P.sum(axis=0), atol=1e-13)


def _golden_topk():
    cases = []
    with open(os.path.join(GOLDEN, "topk_ties.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            K, scores, want = (s.strip() for s in line.split("|"))
            cases.append((int(K), np.array([float(t) for t in scores.split()]),
                          np.array([int(t) for t in want.split()])))
    return cases


@pytest.mark.parametrize("K,S,want", _golden_topk())
def test_topk_hand_worked_ties(K, S, want):
    assert np.array_equal(orc.topk_ascending(S, K), want)


@pytest.mark.parametrize("seed", range(12))
def test_topk_brute_force_max_mass(seed):
    """Among all K-subsets, the oracle's set has the largest sum; among equal
    sums it is the lexicographically smallest ascending index tuple (ties to the
    lower index). Scores are multiples of 1/8 so subset sums are exact."""
    rng = _rng(100 + seed)
    N = int(rng.integers(4, 13))
    K = int(rng.integers(1, min(6, N) + 1))
    S = rng.integers(0, 6, N) / 8.0
    best = None
    for sub in itertools.combinations(range(N), K):
        key = (-S[list(sub)].sum(), sub)
        best = key if best is None or key < best else best
    assert tuple(orc.topk_ascending(S, K)) == best[1]


@pytest.mark.parametrize("seed", range(6))
def test_anchor_selection_is_max_summed_weight_subset(seed):
    """End to end on a tiny head: each group's index set maximises the group's
    summed softmax weight (computed here with torch.softmax) over all K-subsets."""
    rng = _rng(200 + seed)
    N, d, C, K = 12, 4, 4, 3
    q, k, v = (rng.standard_normal((N, d)) * 1.5 for _ in range(3))
    res = orc.anchor_head(q, k, v, C, K, iters=20)
    P = torch.softmax(torch.from_numpy(q @ k.T / math.sqrt(d)), dim=1).numpy()
    for g in range(N // C):
        mem = res["perm"][g * C:(g + 1) * C]
        w = P[mem].sum(axis=0)
        best = max(itertools.combinations(range(N), K), key=lambda s: w[list(s)].sum())
        assert tuple(res["idx"][g]) == best
        assert abs(res["mass"][g] - w[list(best)].sum() / C) < 1e-12


# ---------------------------------------------------------------- sparse + residual
def test_sparse_is_sdpa_on_gathered_keys():
    rng = _rng(4)
    q, k, v = rng.standard_normal((9, 32)) * 2, rng.standard_normal((80, 32)) * 2, rng.standard_normal((80, 32))
    idx = np.sort(rng.choice(80, 23, replace=False))
    assert np.allclose(orc.sparse_attention(q, k, v, idx), _sdpa(q, k[idx], v[idx]), atol=1e-12)


def _head(seed, N, d):
    rng = _rng(seed)
    return (rng.standard_normal((N, d)) * 1.7, rng.standard_normal((N, d)) * 1.7, rng.standard_normal((N, d)))


@pytest.mark.parametrize("N,C", [(256, 64), (200, 64)])
def test_full_density_sparse_equals_dense_and_residual_is_zero(N, C):
    q, k, v = _head(N, N, 16)
    res = orc.anchor_head(q, k, v, C, N)
    assert np.allclose(res["o_sparse"], res["o_dense"], atol=1e-13)
    assert np.abs(res["residual"]).max() < 1e-13
    assert np.allclose(res["mass"], 1.0, atol=1e-12)


def test_anchor_plus_residual_reproduces_dense():
    q, k, v = _head(9, 300, 16)
    res = orc.anchor_head(q, k, v, 64, 60)
    assert np.abs(res["residual"]).max() > 1e-3                       # a real residual
    recon = res["o_sparse"] + res["residual"]
    ulp = np.spacing(np.abs(res["o_dense"]).max())
    assert np.abs(recon - res["o_dense"]).max() <= 2 * ulp


def test_reuse_with_zero_drift_reproduces_anchor_dense():
    q, k, v = _head(10, 300, 16)
    res = orc.anchor_head(q, k, v, 64, 45)
    out = orc.reuse_head(q, k, v, res["perm"], res["idx"], res["residual"], 64)
    assert np.allclose(out, res["o_dense"], atol=1e-13)


# ---------------------------------------------------------------- pages' printed ratios
def test_pages_ratios_are_consistent():
    with open(os.path.join(GOLDEN, "pages_ratios.txt")) as f:
        rows = [l.split("|") for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 3
    for name, num, den, ratio, tol, _src in rows:
        assert abs(float(num) / float(den) - float(ratio)) <= float(tol), name
