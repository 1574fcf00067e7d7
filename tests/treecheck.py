"""Structural checks on an emitted draft tree (test infrastructure).

These hold for any correct best-first tree: prefix closure, the parent/child
relation of ranks and tokens, rho(child) <= rho(parent) (Bastion,
gist.science/nl/paper/2605.29727, Methodologie §1 "Pad-scoren"), and the
non-increasing pop sequence that makes A_hat(T_N) concave in N (§2 "Optimale
Constructie").
"""
import numpy as np


def rank_paths(parent, rank, n):
    """Rank tuple of each node's path (root = ())."""
    paths = [()]
    for i in range(1, n):
        paths.append(paths[parent[i]] + (int(rank[i]),))
    return paths


def check_tree(r, n, parent, depth, pos_id, token, rank, log_rho, anc_mask, topk_tok, ctx_len,
               root_token, b, K, n_max, tol=0.0):
    W = (n_max + 31) // 32
    assert 1 <= n <= n_max
    assert parent[0] == -1 and depth[0] == 0 and rank[0] == -1 and token[0] == root_token
    assert pos_id[0] == ctx_len
    seen = set()
    for i in range(1, n):
        p = parent[i]
        assert 0 <= p < i, (r, i, p)
        assert depth[i] == depth[p] + 1 <= b
        assert 0 <= rank[i] < K
        assert token[i] == topk_tok[depth[i] - 1][rank[i]]
        assert pos_id[i] == ctx_len + depth[i]
        assert (p, rank[i]) not in seen
        seen.add((p, rank[i]))
        assert log_rho[i] <= log_rho[p] + tol
        # pop order: non-increasing scores (concavity of A_hat in N)
        if i >= 2:
            assert log_rho[i] <= log_rho[i - 1] + tol, (r, i)
    # sibling ranks are a prefix 0..c-1 (a node's next child is its next-ranked token)
    kids = {}
    for i in range(1, n):
        kids.setdefault(int(parent[i]), []).append(int(rank[i]))
    for p, ks in kids.items():
        assert sorted(ks) == list(range(len(ks))), (r, p, ks)
    # ancestor-or-self masks, rebuilt by walking parents
    for i in range(n):
        want = np.zeros(W, np.uint32)
        j = i
        while j >= 0:
            want[j // 32] |= np.uint32(1 << (j % 32))
            j = parent[j] if j > 0 else -1
        assert np.array_equal(np.asarray(anc_mask[i], np.uint32), want), (r, i)
