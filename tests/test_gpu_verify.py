"""GPU parity: greedy verification (C ABI) against the oracle, bit-exact
(argmaxes, accept lengths, accepted nodes, output tokens)."""
import numpy as np
import pytest

import oracle
import synth
from gpuhelp import compare_verify, gpu_verify, host, to_dev, to_pinned, workload_inputs

pytestmark = pytest.mark.gpu


def _tree(w):
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, c, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, c, lar)
    return tk, tr


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_verify_workloads(cuda_lib, cid):
    w = synth.workload(cid)
    tk, tr = _tree(w)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    g, st = gpu_verify(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    assert int(st.abs().sum()) == 0
    compare_verify(g, oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token), tr.n_nodes)


def test_verify_ties_and_ragged_vocab(cuda_lib):
    """Rows of equal maxima (lowest token wins), V = 151937, misaligned rows."""
    B, n_max, V, b = 2, 8, 151937, 4
    tgt = np.zeros((B, n_max, V), np.uint16)
    tgt[0, 0, [5, 90000]] = synth.f64_to_bf16_bits(3.0)
    tgt[0, 1, [151936, 151935]] = synth.f64_to_bf16_bits(1.0)
    tgt[1, :, 77] = synth.f64_to_bf16_bits(-1.0)   # all others 0 -> token 0 wins
    n_nodes = np.array([3, 8], np.int32)
    parent = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2, 3], np.int32), (B, 1))
    token = np.tile(np.array([9, 90000, 5, 151935, 0, 1, 2, 3], np.int32), (B, 1))
    g, st = gpu_verify(tgt, b, n_nodes, parent, token)
    ref = oracle.verify_greedy(tgt, b, n_nodes, parent, token)
    compare_verify(g, ref, n_nodes)
    assert host(g.argmax)[0, 0] == 5


def test_verify_f32_and_status(cuda_lib):
    from draft_tree_build_gb300 import bastion
    B, n_max, V, b = 3, 4, 1000, 2
    rng = np.random.default_rng(3)
    tgt = rng.normal(size=(B, n_max, V)).astype(np.float32)
    tgt[1, 0, 10] = np.nan
    n_nodes = np.array([2, 2, 0], np.int32)   # request 2: no valid tree
    parent = np.tile(np.array([-1, 0, 0, 0], np.int32), (B, 1))
    token = np.tile(np.array([1, 2, 3, 4], np.int32), (B, 1))
    g, st = gpu_verify(tgt, b, n_nodes, parent, token)
    s = host(st)
    assert s[0] == 0 and s[1] & bastion.STATUS_NONFINITE and s[2] & bastion.STATUS_BAD_TREE
    ref = oracle.verify_greedy(tgt[:1], b, n_nodes[:1], parent[:1], token[:1])
    assert host(g.accept_len)[0] == ref.accept_len[0]
    assert host(g.accept_len)[2] == 0 and np.all(host(g.out_tokens)[2] == -1)


def test_verify_requests_without_rows_between_others(cuda_lib):
    """Requests whose tree size is out of range read no rows and get empty
    results; the items of the others (found by searching the per-request
    item counts) are still every row of theirs, bit-exact."""
    from draft_tree_build_gb300 import bastion
    B, n_max, V, b = 6, 8, 5000, 3
    rng = np.random.default_rng(11)
    tgt = synth.f32_to_bf16_bits(rng.normal(size=(B, n_max, V)).astype(np.float32))
    n_nodes = np.array([0, 5, -1, 0, 8, n_max + 1], np.int32)
    parent = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2, 3], np.int32), (B, 1))
    token = rng.integers(0, V, size=(B, n_max)).astype(np.int32)
    g, st = gpu_verify(tgt, b, n_nodes, parent, token)
    s = host(st)
    ok = (n_nodes >= 1) & (n_nodes <= n_max)
    assert np.all((s[~ok] & bastion.STATUS_BAD_TREE) != 0) and np.all(s[ok] == 0)
    am, al, an, ot = host(g.argmax), host(g.accept_len), host(g.accept_nodes), host(g.out_tokens)
    for r in np.flatnonzero(ok):
        ref = oracle.verify_greedy(tgt[r:r + 1], b, n_nodes[r:r + 1], parent[r:r + 1], token[r:r + 1])
        n = int(n_nodes[r])
        assert np.array_equal(am[r, :n], ref.argmax[0, :n]), r
        assert al[r] == ref.accept_len[0] and np.array_equal(an[r], ref.accept_nodes[0])
        assert np.array_equal(ot[r], ref.out_tokens[0])
    for r in np.flatnonzero(~ok):
        assert al[r] == 0 and np.all(an[r] == -1) and np.all(ot[r] == -1)


def test_verify_full_agreement_chain(cuda_lib):
    w = synth.workload(2)
    tk, tr = _tree(w)
    n = int(tr.n_nodes[0])
    tgt = np.zeros((1, w.n_max, w.V), np.uint16)
    for i in range(n):
        d = tr.depth[0, i]
        tgt[0, i, tk.tok[0, d, 0] if d < w.b else 0] = synth.f64_to_bf16_bits(5.0)
    g, _ = gpu_verify(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    compare_verify(g, oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token), tr.n_nodes)


def test_verify_deterministic_and_reusable_workspace(cuda_lib):
    w = synth.workload(3, B=6)
    tk, tr = _tree(w)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    td = to_dev(tgt)
    a, _ = gpu_verify(None, w.b, tr.n_nodes, tr.parent, tr.token, target_dev=td)
    b_, _ = gpu_verify(None, w.b, tr.n_nodes, tr.parent, tr.token, target_dev=td)
    for f in ("argmax", "accept_len", "accept_nodes", "out_tokens"):
        assert np.array_equal(host(getattr(a, f)), host(getattr(b_, f)))


@pytest.mark.parametrize("cid", [1, 3])
def test_verify_reads_pinned_host_target(cuda_lib, cid):
    """Target logits left in pinned host memory: the sweep reads the tree's rows
    in place over the host link, with the results of the device-resident call."""
    w = synth.workload(cid)
    tk, tr = _tree(w)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    g, st = gpu_verify(tgt, w.b, tr.n_nodes, tr.parent, tr.token, target_dev=to_pinned(tgt))
    assert int(st.abs().sum()) == 0
    compare_verify(g, oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token), tr.n_nodes)


def test_verify_rejects_pageable_host_target(cuda_lib):
    """A pageable host tensor is refused by the binding before the library sees it."""
    import torch
    from draft_tree_build_gb300 import bastion
    tgt = np.zeros((1, 4, 64), np.float32)
    with pytest.raises(bastion.BastionError, match="pinned"):
        gpu_verify(tgt, 2, np.array([1], np.int32), np.full((1, 4), -1, np.int32),
                   np.zeros((1, 4), np.int32), target_dev=torch.from_numpy(tgt))
