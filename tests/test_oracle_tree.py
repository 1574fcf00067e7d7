"""Pins for the oracle's best-first tree and online controller (no GPU).

Bastion (gist.science/nl/paper/2605.29727), Methodologie:
  §1 rho(i) = prod_k q_k(x_ik);  §2 A_hat(T) = sum rho, best-first is optimal for
  A_hat under a fixed budget and A_hat(T_N) is concave in N;  §3 stop when
  S(N) = A_hat(T_N) L_AR / C(N) starts to decrease.
Each pin below reaches the expected value by a different computation than the
oracle's (enumeration, closed form, dynamic programming, pruned search,
library routines).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
import synth
from treecheck import check_tree, rank_paths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def ranked_q(rows):
    """Library path: softmax (scipy) and rank order (numpy lexsort) of fp64 rows."""
    rows = np.asarray(rows, np.float64)
    q = softmax(rows, axis=-1)
    logq = rows - logsumexp(rows, axis=-1, keepdims=True)
    order = np.stack([np.lexsort((np.arange(rows.shape[1]), -r)) for r in rows])
    return (np.take_along_axis(q, order, -1), np.take_along_axis(logq, order, -1), order)


def run_oracle(x, K, n_max, cost_row=None, l_ar=20.0, root_counts=True, guide=None):
    """x [B, b, V] float32 logits; flat cost unless given."""
    B, b, V = x.shape
    tk = oracle.topk_marginals(x, K)
    cost = np.full((1, n_max + 1), 10.0, np.float32) if cost_row is None else cost_row
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, n_max, np.zeros(B, np.int32),
                           np.zeros(B, np.int32), cost, np.full(B, l_ar, np.float32),
                           root_counts=root_counts, guide=guide)
    return tk, tr


def count_trees_gf(b, K, n_max):
    """Number of prefix-closed trees (containing the root) of each size in the
    complete K-ary candidate tree of depth b: F_0 = x, F_h = x (1 + F_{h-1})^K."""
    F = np.zeros(n_max + 1, dtype=object)
    F[1] = 1
    for _ in range(b):
        base = np.zeros(n_max + 1, dtype=object)
        base[0] = 1
        base[1:] += F[1:]
        P = np.zeros(n_max + 1, dtype=object)
        P[0] = 1
        for _k in range(K):
            Q = np.zeros(n_max + 1, dtype=object)
            for i in range(n_max + 1):
                if P[i]:
                    for j in range(n_max + 1 - i):
                        Q[i + j] += P[i] * base[j]
            P = Q
        F = np.zeros(n_max + 1, dtype=object)
        F[1:] = P[:n_max]
    return [int(c) for c in F]


def brute_force_max(q_sorted, b, K, n_max):
    """Enumerate every prefix-closed tree of size <= n_max once (extension with
    exclusion) and return (max sum of rho per size, number of trees per size)."""
    best = [-1.0] * (n_max + 1)
    count = [0] * (n_max + 1)

    def rho(path):
        return math.prod(q_sorted[k][j] for k, j in enumerate(path))

    def children(path):
        return [path + (j,) for j in range(K)] if len(path) < b else []

    def rec(size, total, frontier):
        count[size] += 1
        best[size] = max(best[size], total)
        if size == n_max:
            return
        for i, c in enumerate(frontier):
            rec(size + 1, total + rho(c), frontier[i + 1:] + children(c))

    rec(1, 1.0, children(()))
    return best, count


@pytest.mark.parametrize("K,b,n_max,seed", [(3, 3, 8, 0), (2, 4, 10, 1), (3, 3, 8, 2), (2, 3, 7, 3)])
def test_best_first_matches_brute_force(K, b, n_max, seed):
    w = synth.workload(1, seed=0xBA5710 + 100 + seed)
    x = synth.drafter_logits(w)[:, :b, :]
    q, _, _ = ranked_q(x[0])
    best, count = brute_force_max(q[:, :K], b, K, n_max)
    assert count[1:] == count_trees_gf(b, K, n_max)[1:]
    tk, tr = run_oracle(x, K, n_max)
    assert tr.n_nodes[0] == n_max
    for N in range(1, n_max + 1):
        assert abs(tr.a_hat[0, N - 1] - best[N]) <= 1e-12 * best[N], (N, tr.a_hat[0, N - 1], best[N])


def test_tree_count_generating_function_value():
    # 8,210 prefix-closed trees of size <= 8 for K=3, b=3 (by the generating
    # function above; also what the enumeration reaches in the test before).
    assert sum(count_trees_gf(3, 3, 8)[1:]) == 8210


def _all_candidate_log_rho(logq_sorted, b, K):
    out = []
    acc = np.zeros(1)
    for d in range(b):
        acc = (acc[:, None] + logq_sorted[d, :K][None, :]).reshape(-1)
        out.append(acc)
    return out


def test_closed_form_top_n_candidates_cfg1():
    """rho(child) <= rho(parent), so the N-1 best candidates form a prefix-closed
    set: A_hat(T_N) = 1 + (sum of the N-1 largest rho over all 4,680 candidates)."""
    w = synth.workload(1)
    x = synth.drafter_logits(w)
    _, logq, _ = ranked_q(x[0])
    lrs = np.concatenate(_all_candidate_log_rho(logq, w.b, w.K))
    assert lrs.size == sum(w.K ** d for d in range(1, w.b + 1)) == 4680
    top = np.sort(np.exp(lrs))[::-1]
    tk, tr = run_oracle(x, w.K, w.n_max)
    for N in range(1, w.n_max + 1):
        want = 1.0 + top[: N - 1].sum()
        assert abs(tr.a_hat[0, N - 1] - want) <= 1e-12 * want
    # and the node set is exactly that top set
    paths = rank_paths(tr.parent[0], tr.rank[0], w.n_max)[1:]
    got = sorted(float(sum(logq[k, j] for k, j in enumerate(p))) for p in paths)
    assert np.allclose(sorted(np.sort(lrs)[::-1][: w.n_max - 1]), got, rtol=0, atol=1e-12)


def knapsack_max(q_sorted, b, K, n_max):
    """Tree-knapsack DP: g[d][n] = max relative mass of a size-n prefix-closed
    subtree hanging at a depth-d node (marginals are position-wise, so the same
    for every depth-d node).  Max-plus merge over the K children."""
    NEG = -np.inf
    g = [None] * (b + 1)
    g[b] = np.full(n_max + 1, NEG)
    g[b][1] = 1.0
    for d in range(b - 1, -1, -1):
        acc = np.full(n_max + 1, NEG)
        acc[0] = 0.0
        for j in range(K):
            child = np.full(n_max + 1, NEG)
            child[0] = 0.0
            child[1:] = q_sorted[d][j] * g[d + 1][1:]
            new = np.full(n_max + 1, NEG)
            for a in range(n_max + 1):
                if acc[a] == NEG:
                    continue
                for c in range(n_max + 1 - a):
                    if child[c] != NEG and acc[a] + child[c] > new[a + c]:
                        new[a + c] = acc[a] + child[c]
            acc = new
        g[d] = np.full(n_max + 1, NEG)
        g[d][1:] = 1.0 + acc[: n_max]
    return g[0]


def test_knapsack_dp_cfg1():
    w = synth.workload(1)
    x = synth.drafter_logits(w)
    q, _, _ = ranked_q(x[0])
    best = knapsack_max(q, w.b, w.K, w.n_max)
    tk, tr = run_oracle(x, w.K, w.n_max)
    for N in range(1, w.n_max + 1):
        assert abs(tr.a_hat[0, N - 1] - best[N]) <= 1e-12 * best[N]


def _threshold_dfs(logq, b, K, tau, eps=1e-9):
    found = {}

    def rec(d, lp, path):
        for j in range(K):
            v = lp + logq[d, j]
            if v < tau - eps:
                break
            found[path + (j,)] = v
            if d + 1 < b:
                rec(d + 1, v, path + (j,))

    rec(0, 0.0, ())
    return found


@pytest.mark.parametrize("cid", [2, 3])
def test_threshold_dfs_at_scale(cid):
    """Every candidate scoring above the tree's weakest node is in the tree, and
    the tree holds nothing below it (pruned enumeration, scores from scipy)."""
    w = synth.workload(cid, B=min(8, synth.WORKLOADS[cid].B))
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w),
                           synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
    f = synth.bf16_bits_to_f32(x)
    for r in range(w.B):
        _, logq, _ = ranked_q(f[r])
        n = tr.n_nodes[r]
        paths = rank_paths(tr.parent[r], tr.rank[r], n)[1:]
        tau = min(tr.log_rho[r, 1:n])
        found = _threshold_dfs(logq, w.b, w.K, tau)
        strict = {p for p, v in found.items() if v > tau + 1e-9}
        assert strict <= set(paths)
        assert set(paths) <= set(found)
        for p in paths:
            assert abs(found[p] - tr.log_rho[r, paths.index(p) + 1]) < 1e-9


@pytest.mark.parametrize("cid", [1, 2, 3, 4])
def test_invariants_and_controller(cid):
    """Structural invariants, and: the first-decrease stop rule returns the largest
    maximiser of S(N) over 1..n_max.  (Derived here, not on the pages: A_hat is
    concave and increasing and C is convex, non-decreasing and positive for these
    cost models, so once S decreases it keeps decreasing.)"""
    w = synth.workload(cid, B=min(8, synth.WORKLOADS[cid].B))
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = synth.root_tokens(w), synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    flat = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx,
                             np.full_like(cost, 7.0), lar)
    assert tr.flagged_pops == 0 and tr.flagged_stops == 0
    C = cost[0].astype(np.float64)
    for r in range(w.B):
        n = tr.n_nodes[r]
        check_tree(r, n, tr.parent[r], tr.depth[r], tr.pos_id[r], tr.token[r], tr.rank[r],
                   tr.log_rho[r], tr.anc_mask[r], tk.tok[r], ctx[r], roots[r], w.b, w.K, w.n_max)
        # the budgeted tree is a prefix of the unbudgeted best-first sequence
        nf = flat.n_nodes[r]
        assert n <= nf
        for a in ("parent", "rank", "token"):
            assert np.array_equal(getattr(tr, a)[r, :n], getattr(flat, a)[r, :n])
        S = flat.a_hat[r, :nf] * float(lar[r]) / C[1: nf + 1]
        best = S.max()
        n_star = 1 + max(i for i in range(nf) if S[i] == best)
        assert n == n_star, (r, n, n_star)
        assert np.allclose(tr.speedup[r, :n], S[:n], rtol=1e-14)
        # A_hat concave in N: increments rho_N non-increasing
        inc = np.diff(flat.a_hat[r, :nf])
        assert np.all(np.diff(inc) <= 1e-15)


def test_special_case_chain_k1():
    """K = 1: the tree is the rank-0 chain (the single-path greedy drafting the
    pages compare against)."""
    w = synth.workload(2)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, 1)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, 17, synth.root_tokens(w), synth.ctx_lens(w),
                           np.full((1, 18), 5.0, np.float32), synth.l_ar(w))
    assert tr.n_nodes[0] == 17
    assert tr.parent[0, 1:17].tolist() == list(range(16))
    assert tr.token[0, 1:17].tolist() == synth.spike_positions(w)[0].tolist()


def test_special_case_root_only():
    w = synth.workload(1)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, 1, [5], [9], np.full((1, 2), 3.0, np.float32),
                           [20.0])
    assert tr.n_nodes[0] == 1 and tr.token[0, 0] == 5 and tr.pos_id[0, 0] == 9
    assert tr.a_hat[0, 0] == 1.0 and tr.anc_mask[0, 0, 0] == 1


def test_flat_cost_fills_budget_cfg5():
    w = synth.workload(5, B=3)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w),
                           synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
    assert np.all(tr.n_nodes == 256)


def test_knee_cost_keeps_at_least_32():
    w = synth.workload(3, B=6)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w),
                           synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
    assert np.all(tr.n_nodes >= 32)


def test_golden_cat_dog():
    g = json.load(open(os.path.join(GOLDEN, "cat_dog.json")))
    for case in g["cases"]:
        rows = np.array([[math.log(p) for p in row] for row in case["q"]], np.float32)[None]
        b = rows.shape[1]
        K = rows.shape[2]
        n_max = len(case["expected"])
        tk, tr = run_oracle(rows, K, n_max)
        assert tr.n_nodes[0] == n_max
        for i, (path, rho) in enumerate(case["expected"]):
            got = rank_paths(tr.parent[0], tr.rank[0], n_max)[i]
            assert list(got) == path
            assert abs(math.exp(tr.log_rho[0, i]) - rho) < 1e-6
        assert abs(tr.a_hat[0, n_max - 1] - case["a_hat"]) < 1e-6
        assert b == len(case["q"])


def test_near_tie_flag_and_guide():
    """A depth-1 candidate and a depth-2 candidate within 1e-7 of each other are
    a flagged near tie; a guide is followed there and only there."""
    x_f = 1.0
    lse2 = math.log(1.0 + math.exp(-x_f))
    rows = np.array([[[0.0, -lse2, -30.0], [0.0, -x_f, -30.0]]], np.float32)
    tk, tr = run_oracle(rows, 2, 4)
    assert tr.flagged_pops >= 1
    own = (tr.n_nodes.copy(), tr.parent.copy(), tr.rank.copy())
    # swap the order of the two tied nodes 2 and 3 in a guide
    gp, gr = own[1].copy(), own[2].copy()
    gp[0, 2], gp[0, 3] = own[1][0, 3], own[1][0, 2]
    gr[0, 2], gr[0, 3] = own[2][0, 3], own[2][0, 2]
    tk, tr2 = run_oracle(rows, 2, 4, guide=(own[0], gp, gr))
    assert tr2.guided == 1
    assert tr2.parent[0, 2] == gp[0, 2] and tr2.rank[0, 2] == gr[0, 2]
    # a guide that departs at a step that is not a near tie is ignored
    gp2, gr2 = own[1].copy(), own[2].copy()
    gr2[0, 1] = 1
    tk, tr3 = run_oracle(rows, 2, 4, guide=(own[0], gp2, gr2))
    assert tr3.rank[0, 1] == own[2][0, 1]


def test_root_excluded_reading_runs():
    """The alternative reading (root not counted in N and A_hat) is available
    for comparison; with a flat cost it builds the same node sequence."""
    w = synth.workload(1)
    x = synth.drafter_logits(w)
    tk, a = run_oracle(x, w.K, w.n_max)
    tk, b_ = run_oracle(x, w.K, w.n_max, root_counts=False)
    n = a.n_nodes[0]
    assert b_.n_nodes[0] == n
    assert np.array_equal(a.parent[0, :n], b_.parent[0, :n])
    assert np.allclose(b_.a_hat[0, :n], a.a_hat[0, :n] - 1.0)
