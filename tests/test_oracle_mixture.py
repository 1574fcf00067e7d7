"""Pins for the oracle's latent-mixture trees (no GPU).

DBlast's dependent block proposal is a mixture over a latent branch z,
q_dep(x_1..b) = sum_z q(z) prod_i q_i(x_i | z) (third page, "Methodologie" 1);
the tree is grown best-first on the induced prefix score
rho(x_1..d) = sum_z pi_z prod_{k<=d} q_k^z(x_k) with Bastion's controller.
The pins tie it to the pinned single-branch tree oracle (one branch, identical
branches), to brute force over all prefix-closed trees, to a closed form at
depth 1, and to invariants of the construction.
"""
import itertools
import math

import numpy as np
import pytest

import oracle
import synth


def _branch_topk(B, Z, b, V, K, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=(B, Z, b, V)) * scale).astype(np.float32)
    tk = oracle.topk_marginals(x.reshape(B * Z * b, V), K)
    return (tk.logit.reshape(B, Z, b, K), tk.tok.reshape(B, Z, b, K), tk.lse.reshape(B, Z, b))


def _flat(n_max):
    return np.full((1, n_max + 1), 5.0, np.float32)


def _common(B):
    return np.zeros(B, np.int32), np.full(B, 7, np.int32), np.full(B, 18.0, np.float32)


@pytest.mark.parametrize("cost", ["flat", "workload"])
def test_one_branch_is_the_tree_oracle(cost):
    B, b, V, K, n_max = 3, 6, 400, 8, 40
    lg, tk, ls = _branch_topk(B, 1, b, V, K, 1)
    roots, ctx, lar = _common(B)
    c = _flat(n_max) if cost == "flat" else synth.cost_table(synth.workload(2, n_max=n_max))
    m = oracle.build_tree_mixture(lg, tk, ls, np.ones((B, 1)), n_max, roots, ctx, c, lar)
    t = oracle.build_tree(lg[:, 0], tk[:, 0], ls[:, 0], n_max, roots, ctx, c, lar)
    assert np.array_equal(m.n_nodes, t.n_nodes)
    for r in range(B):
        n = t.n_nodes[r]
        for f in ("parent", "depth", "pos_id", "token"):
            assert np.array_equal(getattr(m, f)[r, :n], getattr(t, f)[r, :n]), f
        assert np.array_equal(m.log_rho[r, :n], t.log_rho[r, :n])
        assert np.array_equal(m.anc_mask[r, :n], t.anc_mask[r, :n])


def test_identical_branches_are_one_branch():
    """A mixture of Z copies of one proposal is that proposal."""
    B, Z, b, V, K, n_max = 2, 3, 5, 300, 6, 30
    lg, tk, ls = _branch_topk(B, 1, b, V, K, 2)
    roots, ctx, lar = _common(B)
    rep = lambda a: np.repeat(a, Z, axis=1)
    pi = np.tile([0.2, 0.3, 0.5], (B, 1))
    m = oracle.build_tree_mixture(rep(lg), rep(tk), rep(ls), pi, n_max, roots, ctx, _flat(n_max), lar)
    t = oracle.build_tree(lg[:, 0], tk[:, 0], ls[:, 0], n_max, roots, ctx, _flat(n_max), lar)
    assert np.array_equal(m.n_nodes, t.n_nodes)
    for r in range(B):
        n = t.n_nodes[r]
        assert np.array_equal(m.parent[r, :n], t.parent[r, :n])
        assert np.array_equal(m.token[r, :n], t.token[r, :n])
        assert np.allclose(m.log_rho[r, :n], t.log_rho[r, :n], rtol=0, atol=1e-12)


def _rho_of_path(path, lg, tk, ls, pi):
    """Mixture probability of a token path from the definition."""
    total = 0.0
    for z in range(len(pi)):
        p = pi[z]
        for k, t in enumerate(path):
            hit = np.flatnonzero(tk[z, k] == t)
            p *= math.exp(float(lg[z, k, hit[0]]) - ls[z, k]) if hit.size else 0.0
        total += p
    return total


def test_best_first_maximises_the_score_sum_brute_force():
    """Every prefix-closed tree of N nodes drawn from the candidate universe
    has a score sum at most best-first's A_hat(T_N), for every N."""
    Z, b, K, n_max = 2, 2, 2, 7
    rng = np.random.default_rng(3)
    V = 6
    x = rng.normal(size=(1, Z, b, V)).astype(np.float32) * 1.5
    tkr = oracle.topk_marginals(x.reshape(Z * b, V), K)
    lg, tk, ls = tkr.logit.reshape(1, Z, b, K), tkr.tok.reshape(1, Z, b, K), tkr.lse.reshape(1, Z, b)
    pi = np.array([[0.35, 0.65]])
    roots, ctx, lar = _common(1)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar)
    # the candidate universe: paths whose tokens come from the union of the branches' lists
    level = [sorted(set(tk[0, :, k].ravel().tolist())) for k in range(b)]
    paths = [(t,) for t in level[0]] + [(t, u) for t in level[0] for u in level[1]]
    rho = {p: _rho_of_path(p, lg[0], tk[0], ls[0], pi[0]) for p in paths}
    n_tree = int(m.n_nodes[0])
    for N in range(1, n_tree + 1):
        best = 0.0
        for sub in itertools.combinations(paths, N - 1):
            s = set(sub)
            if all(len(p) == 1 or p[:1] in s for p in sub):
                best = max(best, 1.0 + sum(rho[p] for p in sub))
        assert m.a_hat[0, N - 1] == pytest.approx(best, rel=1e-12), N


def test_depth_one_closed_form_with_disjoint_branches():
    """Branches whose position-1 lists share no token: a depth-1 node's score
    is pi_z q_1^z(x) of the one branch that lists x."""
    B, Z, b, V, K, n_max = 1, 2, 3, 100, 5, 12
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 4)
    tk[0, 1, 0] = np.arange(K) + 1000   # branch 1's position-1 tokens: none in branch 0's list
    pi = np.array([[0.4, 0.6]])
    roots, ctx, lar = _common(B)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar)
    n = int(m.n_nodes[0])
    seen = 0
    for i in range(1, n):
        if m.depth[0, i] != 1:
            continue
        t = m.token[0, i]
        z = 0 if t < 1000 else 1
        j = int(np.flatnonzero(tk[0, z, 0] == t)[0])
        assert m.log_rho[0, i] == pytest.approx(math.log(pi[0, z]) + float(lg[0, z, 0, j]) - ls[0, z, 0],
                                                abs=1e-13)
        seen += 1
    assert seen >= 2


def test_invariants_and_branch_relabelling():
    B, Z, b, V, K, n_max = 2, 3, 6, 500, 10, 64
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 5)
    rng = np.random.default_rng(6)
    pi = rng.dirichlet(np.ones(Z), size=B)
    roots, ctx, lar = _common(B)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar)
    for r in range(B):
        n = int(m.n_nodes[r])
        assert n == n_max                                   # a flat cost fills the budget
        par = m.parent[r, :n]
        assert np.all(par[1:] < np.arange(1, n))            # prefix closure, pop order
        assert np.all(m.log_rho[r, 1:n] <= m.log_rho[r, par[1:]] + 1e-15)   # rho(child) <= rho(parent)
        assert np.all(np.diff(m.log_rho[r, 1:n]) <= 1e-15)  # non-increasing pops: A_hat concave
        assert np.all(m.depth[r, 1:n] == m.depth[r, par[1:]] + 1)
    perm = [2, 0, 1]
    m2 = oracle.build_tree_mixture(lg[:, perm], tk[:, perm], ls[:, perm], pi[:, perm], n_max, roots,
                                   ctx, _flat(n_max), lar)
    assert np.array_equal(m.parent, m2.parent) and np.array_equal(m.token, m2.token)
    assert np.allclose(m.log_rho, m2.log_rho, rtol=0, atol=1e-12)


def _tie_case():
    """Z = 2, pi = (1/2, 1/2), b = 2, K = 2, logits log p with lse = 0:
    position 1: branch 0 {10: 1/2, 11: 1/4}, branch 1 {10: 1/2, 12: 1/4};
    position 2: branch 0 {20: 1/2, 21: 1/2}, branch 1 {20: 1/2, 22: 1/4}.
    rho: (10) 1/2, (10,20) 1/4, then (11), (12) and (10,21) all 1/8: a tie
    across depths 1 and 2 and across branches."""
    tk = np.array([[[[10, 11], [20, 21]], [[10, 12], [20, 22]]]], np.int32)
    p = np.array([[[[0.5, 0.25], [0.5, 0.5]], [[0.5, 0.25], [0.5, 0.25]]]])
    lg = np.log(p).astype(np.float32)
    ls = np.zeros((1, 2, 2))
    pi = np.array([[0.5, 0.5]])
    return lg, tk, ls, pi


def test_tie_across_depths_is_flagged_and_follows_the_guide():
    lg, tk, ls, pi = _tie_case()
    n_max = 6
    roots, ctx, lar = _common(1)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar)
    # own order: the tie goes to the lower depth, then to the lower token
    assert m.token[0, :6].tolist() == [0, 10, 20, 11, 12, 21]
    assert m.parent[0, :6].tolist() == [-1, 0, 1, 0, 0, 1]
    assert np.allclose(np.exp(m.log_rho[0, :6]), [1, 0.5, 0.25, 0.125, 0.125, 0.125], rtol=1e-12)
    assert m.flagged_pops >= 2 and m.guided == 0
    # a guide that takes the depth-2 node first is followed at the flagged pop
    guide = (np.array([6], np.int32), np.array([[-1, 0, 1, 1, 0, 0]], np.int32),
             np.array([[0, 10, 20, 21, 11, 12]], np.int32))
    g = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar, guide=guide)
    assert g.guided == 1
    assert g.parent[0].tolist() == guide[1][0].tolist() and g.token[0].tolist() == guide[2][0].tolist()
    assert g.a_hat[0, 5] == pytest.approx(m.a_hat[0, 5], rel=1e-12)


def test_guide_outside_the_band_is_ignored():
    lg, tk, ls, pi = _tie_case()
    n_max = 6
    roots, ctx, lar = _common(1)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar)
    # at the flagged pop the guide names (11, 20), rho 1/16: not a near tie
    guide = (np.array([6], np.int32), np.array([[-1, 0, 1, 3, 0, 0]], np.int32),
             np.array([[0, 10, 20, 20, 11, 12]], np.int32))
    g = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, _flat(n_max), lar, guide=guide)
    assert g.guided == 0
    assert np.array_equal(g.parent, m.parent) and np.array_equal(g.token, m.token)


def test_stop_at_the_boundary_is_flagged_and_follows_the_guide():
    """After the root (A_hat = 1) the best candidate has rho = 1/2; with
    C(1) = 2 and C(2) = 3 the stop test rho C(1) < A_hat (C(2) - C(1)) is an
    equality: either tree is correct."""
    lg, tk, ls, pi = _tie_case()
    n_max = 4
    roots, ctx, lar = _common(1)
    c = np.array([[0.0, 2.0, 3.0, 3.0, 3.0]], np.float32)
    m = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert m.flagged_stops >= 1
    stop = (np.array([1], np.int32), np.full((1, n_max), -1, np.int32), np.zeros((1, n_max), np.int32))
    g = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, c, lar, guide=stop)
    assert int(g.n_nodes[0]) == 1
    go = (np.array([4], np.int32), np.array([[-1, 0, 1, 0]], np.int32),
          np.array([[0, 10, 20, 11]], np.int32))
    g2 = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, c, lar, guide=go)
    assert int(g2.n_nodes[0]) == 4       # C flat after N = 2: nothing else stops it
    assert g2.token[0, :4].tolist() == [0, 10, 20, 11]
    assert g.guided + g2.guided == 1     # the oracle's own decision matches one of the two


def test_no_flags_on_random_logits_without_ties():
    """Random fp32 logits: near ties within 1e-5 are rare; identical branch
    copies tie only within one parent with identical logits, never flagged."""
    B, Z, b, V, K, n_max = 2, 3, 5, 300, 6, 30
    lg, tk, ls = _branch_topk(B, 1, b, V, K, 2)
    rep = lambda a: np.repeat(a, Z, axis=1)
    pi = np.tile([0.2, 0.3, 0.5], (B, 1))
    roots, ctx, lar = _common(B)
    m = oracle.build_tree_mixture(rep(lg), rep(tk), rep(ls), pi, n_max, roots, ctx, _flat(n_max), lar)
    t = oracle.build_tree(lg[:, 0], tk[:, 0], ls[:, 0], n_max, roots, ctx, _flat(n_max), lar)
    assert m.flagged_pops == t.flagged_pops == 0
