"""GPU parity: best-first trees on a latent-mixture proposal (C ABI) against
the oracle.  Both sides form the scores in fp64 with the same operations, so
the tree topology, tokens and masks must match exactly (random fp32 branch
logits have no ties); log rho, A_hat and S are returned as float and must be
within 1e-6 relative of the oracle's fp64 values."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, host, to_dev

pytestmark = pytest.mark.gpu


def _branch_topk(B, Z, b, V, K, seed):
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=(B, Z, b, V)) * 2.0).astype(np.float32)
    tk = oracle.topk_marginals(x.reshape(B * Z * b, V), K)
    return (tk.logit.reshape(B, Z, b, K), tk.tok.reshape(B, Z, b, K), tk.lse.reshape(B, Z, b))


def _gpu(lg, tk, ls, pi, n_max, roots, ctx, cost, lar):
    from draft_tree_build_gb300 import bastion
    B = lg.shape[0]
    W = (n_max + 31) // 32
    out = {k: torch.full((B, n_max), -7, dtype=torch.int32, device=dev())
           for k in ("parent", "depth", "pos_id", "token")}
    for k in ("log_rho", "a_hat", "speedup"):
        out[k] = torch.full((B, n_max), float("nan"), dtype=torch.float32, device=dev())
    out["n_nodes"] = torch.zeros(B, dtype=torch.int32, device=dev())
    out["anc_mask"] = torch.zeros((B, n_max, W), dtype=torch.int32, device=dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    bastion.bastion_build_tree_mixture(
        to_dev(lg), to_dev(tk), to_dev(ls), to_dev(np.ascontiguousarray(pi, np.float64)), n_max,
        to_dev(roots), to_dev(ctx), to_dev(np.ascontiguousarray(cost, np.float32)), to_dev(lar),
        out["n_nodes"], out["parent"], out["depth"], out["pos_id"], out["token"], out["log_rho"],
        out["a_hat"], out["speedup"], out["anc_mask"], st)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}, host(st)


def _compare(g, ref):
    assert np.array_equal(g["n_nodes"], ref.n_nodes)
    for r in range(len(ref.n_nodes)):
        n = int(ref.n_nodes[r])
        for f in ("parent", "depth", "pos_id", "token"):
            assert np.array_equal(g[f][r, :n], getattr(ref, f)[r, :n]), (r, f)
        assert np.array_equal(g["anc_mask"][r, :n].view(np.uint32), ref.anc_mask[r, :n])
        for f in ("log_rho", "a_hat", "speedup"):
            want = getattr(ref, f)[r, :n]
            assert np.allclose(g[f][r, :n], want, rtol=1e-6, atol=1e-6), (r, f)
        assert np.all(g["parent"][r, n:] == -7)   # rows past the tree untouched


@pytest.mark.parametrize("Z,b,V,K,n_max,cost", [
    (1, 5, 300, 8, 40, "flat"),
    (3, 5, 300, 8, 40, "flat"),
    (2, 16, 2000, 32, 64, "workload"),
    (4, 16, 5000, 64, 128, "flat"),
])
def test_mixture_tree_matches_oracle(cuda_lib, Z, b, V, K, n_max, cost):
    B = 3 if n_max <= 64 else 2
    lg, tk, ls = _branch_topk(B, Z, b, V, K, Z * 100 + K)
    pi = np.random.default_rng(K).dirichlet(np.ones(Z), size=B)
    roots = np.arange(B, dtype=np.int32) + 11
    ctx = np.full(B, 40, np.int32)
    lar = np.full(B, 18.0, np.float32)
    c = (np.full((1, n_max + 1), 5.0, np.float32) if cost == "flat"
         else synth.cost_table(synth.workload(2, n_max=n_max)))
    g, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(st == 0)
    ref = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    _compare(g, ref)


def test_mixture_tree_zero_weight_branch_and_bad_cost(cuda_lib):
    """A branch of weight 0 contributes nothing (its log weight is -inf on both
    sides); a non-positive cost entry sets the status bit."""
    from draft_tree_build_gb300 import bastion
    B, Z, b, V, K, n_max = 2, 3, 6, 400, 8, 32
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 9)
    pi = np.array([[0.5, 0.0, 0.5], [0.2, 0.8, 0.0]])
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(st == 0)
    _compare(g, oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, c, lar))
    c[0, 7] = 0.0
    _, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(st & bastion.STATUS_BAD_COST)


def test_mixture_tree_bad_weight_sets_status(cuda_lib):
    """A negative or NaN branch weight sets the weight status bit on that
    request only; the others are built as the oracle builds them."""
    from draft_tree_build_gb300 import bastion
    B, Z, b, V, K, n_max = 3, 2, 5, 300, 8, 24
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 21)
    pi = np.array([[0.5, 0.5], [-0.25, 1.25], [np.nan, 1.0]])
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert st[0] == 0
    assert st[1] & bastion.STATUS_BAD_WEIGHT and st[2] & bastion.STATUS_BAD_WEIGHT
    ref = oracle.build_tree_mixture(lg[:1], tk[:1], ls[:1], pi[:1], n_max, roots[:1], ctx[:1], c, lar[:1])
    assert int(g["n_nodes"][0]) == int(ref.n_nodes[0])
    n = int(ref.n_nodes[0])
    assert np.array_equal(g["token"][0, :n], ref.token[0, :n])
