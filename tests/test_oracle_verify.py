"""Pins for the oracle's greedy verification (no GPU).

Greedy (temperature 0) acceptance as evaluated on the pages (Bastion,
gist.science/nl/paper/2605.29727, "Experimentele Resultaten").  The accept
scan is checked against an independent sequential check that decodes token by
token with the target's greedy choice and looks each prefix up in a dictionary
of the tree's paths.
"""
import numpy as np
import pytest

import oracle
import synth


def _pipeline(cid, B=None):
    w = synth.workload(cid, **({"B": B} if B else {}))
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w),
                           synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
    return w, tk, tr


def sequential_ar_check(target_rows_f, n, parent, token, b):
    """Token-by-token greedy decode against a {token path: node} dictionary."""
    path_of = {(): 0}
    paths = [()]
    for i in range(1, n):
        paths.append(paths[parent[i]] + (int(token[i]),))
        path_of[paths[i]] = i
    prefix, accepted, nodes = (), [], [0]
    while True:
        node = path_of[prefix]
        t = int(np.argmax(target_rows_f[node]))  # library argmax: first maximum
        nxt = prefix + (t,)
        if nxt in path_of and len(accepted) < b:
            accepted.append(t)
            nodes.append(path_of[nxt])
            prefix = nxt
        else:
            return accepted, t, nodes


@pytest.mark.parametrize("cid,B", [(1, None), (2, None), (3, 8)])
def test_accept_scan_matches_sequential_check(cid, B):
    w, tk, tr = _pipeline(cid, B)
    tgt, planted = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    vf = oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    f = synth.bf16_bits_to_f32(tgt) if tgt.dtype == np.uint16 else tgt
    for r in range(w.B):
        n = tr.n_nodes[r]
        assert np.array_equal(vf.argmax[r, :n], np.argmax(f[r, :n], axis=-1))
        assert np.array_equal(vf.argmax[r, :n], planted[r, :n])
        acc, bonus, nodes = sequential_ar_check(f[r], n, tr.parent[r], tr.token[r], w.b)
        L = vf.accept_len[r]
        assert L == len(acc)
        assert vf.out_tokens[r, :L].tolist() == acc and vf.out_tokens[r, L] == bonus
        assert np.all(vf.out_tokens[r, L + 1:] == -1)
        assert vf.accept_nodes[r, : L + 1].tolist() == nodes
        assert np.all(vf.accept_nodes[r, L + 1:] == -1)


def test_full_agreement_accepts_rank0_chain():
    """If the target always agrees with the drafter's best token, the accepted
    path is the rank-0 chain as far as the tree holds it."""
    w, tk, tr = _pipeline(2)
    n = tr.n_nodes[0]
    tgt = np.zeros((1, w.n_max, w.V), np.uint16)
    for i in range(n):
        d = tr.depth[0, i]
        t = tk.tok[0, d, 0] if d < w.b else 0
        tgt[0, i, t] = synth.f64_to_bf16_bits(5.0)
    vf = oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    chain, cur = 0, 0
    while True:
        kids = [i for i in range(1, n) if tr.parent[0, i] == cur and tr.rank[0, i] == 0]
        if not kids:
            break
        cur = kids[0]
        chain += 1
    assert vf.accept_len[0] == chain


def test_all_plants_off_tree_accept_nothing():
    w, tk, tr = _pipeline(1)
    n = tr.n_nodes[0]
    tgt = np.zeros((1, w.n_max, w.V), np.float32)
    off = [v for v in range(w.V) if v not in set(tr.token[0, :n].tolist())][0]
    tgt[0, :, off] = 3.0
    vf = oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    assert vf.accept_len[0] == 0 and vf.out_tokens[0, 0] == off
    assert vf.accept_nodes[0].tolist() == [0] + [-1] * w.b


def test_argmax_ties_lowest_token_and_status():
    tgt = np.zeros((2, 1, 6), np.float32)
    tgt[0, 0, [2, 4]] = 1.0
    tgt[1, 0, 3] = np.nan
    vf = oracle.verify_greedy(tgt, 1, [1, 1], np.full((2, 1), -1), np.zeros((2, 1)))
    assert vf.argmax[0, 0] == 2
    assert vf.status[1] & oracle.ST_NONFINITE
