"""GPU parity: best-first trees on a latent-mixture proposal (C ABI) against
the oracle.

The kernel forms the per-branch path scores in fixed point and the mixture sum
over the branches in fp32: log rho is within (5 + Z/2) 2^-23 of exact.  Where
the oracle flags a near tie (a rival within 1e-5 in log rho, or a stop test
within 1e-5 of its boundary), either choice is correct, and the oracle is run
again with the GPU's tree as its guide, followed only at those steps and only
where the GPU's choice lies inside the band.  Outside them the tree topology,
tokens and ancestor masks must match exactly; log rho, A_hat and S are
returned as float and are compared within the kernel's error bound plus one
float rounding."""
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, host, to_dev

pytestmark = pytest.mark.gpu


def _branch_topk(B, Z, b, V, K, seed, scale=2.0):
    rng = np.random.default_rng(seed)
    x = (rng.normal(size=(B, Z, b, V)) * scale).astype(np.float32)
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
    Z, b, K = lg.shape[1:]
    ws = bastion.workspace(bastion.bastion_build_tree_mixture_workspace_bytes(B, Z, b, K, n_max), dev())
    bastion.bastion_build_tree_mixture(
        to_dev(lg), to_dev(tk), to_dev(ls), to_dev(np.ascontiguousarray(pi, np.float64)), n_max,
        to_dev(roots), to_dev(ctx), to_dev(np.ascontiguousarray(cost, np.float32)), to_dev(lar),
        out["n_nodes"], out["parent"], out["depth"], out["pos_id"], out["token"], out["log_rho"],
        out["a_hat"], out["speedup"], out["anc_mask"], ws, st)
    torch.cuda.synchronize()
    return {k: host(v) for k, v in out.items()}, host(st)


def _oracle_one(args):
    lg, tk, ls, pi, n_max, roots, ctx, cost, lar, g = args
    ref = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, cost, lar)
    if (ref.flagged_pops or ref.flagged_stops) and g is not None:
        ref = oracle.build_tree_mixture(lg, tk, ls, pi, n_max, roots, ctx, cost, lar, guide=g)
    return ref


def _guided(lg, tk, ls, pi, n_max, roots, ctx, cost, lar, g=None):
    """The oracle per request (threads: the library call releases the GIL),
    rerun with the GPU's tree as guide where it flags near ties; the results
    stacked, with the counters summed."""
    B = lg.shape[0]
    cost = np.ascontiguousarray(cost, np.float32).reshape(-1, n_max + 1)
    jobs = []
    for r in range(B):
        c = cost[r:r + 1] if cost.shape[0] == B and B > 1 else cost
        gr = None if g is None else (g["n_nodes"][r:r + 1], g["parent"][r:r + 1], g["token"][r:r + 1])
        jobs.append((lg[r:r + 1], tk[r:r + 1], ls[r:r + 1], pi[r:r + 1], n_max, roots[r:r + 1],
                     ctx[r:r + 1], c, lar[r:r + 1], gr))
    with ThreadPoolExecutor(max_workers=16) as ex:
        refs = list(ex.map(_oracle_one, jobs))
    cat = {f: np.concatenate([getattr(x, f) for x in refs]) for f in
           ("n_nodes", "parent", "depth", "pos_id", "token", "log_rho", "a_hat", "speedup", "anc_mask",
            "status")}
    out = oracle.MixTree(**cat)
    out.flagged_pops = sum(x.flagged_pops for x in refs)
    out.flagged_stops = sum(x.flagged_stops for x in refs)
    out.guided = sum(x.guided for x in refs)
    return out


def _compare(g, ref, Z):
    assert np.array_equal(g["n_nodes"], ref.n_nodes)
    eps = (5 + Z / 2) * 2.0 ** -23 + 2.0 ** -30
    for r in range(len(ref.n_nodes)):
        n = int(ref.n_nodes[r])
        for f in ("parent", "depth", "pos_id", "token"):
            assert np.array_equal(g[f][r, :n], getattr(ref, f)[r, :n]), (r, f)
        assert np.array_equal(g["anc_mask"][r, :n].view(np.uint32), ref.anc_mask[r, :n])
        lr = ref.log_rho[r, :n]
        assert np.all(np.abs(g["log_rho"][r, :n] - lr) <= eps + 2.0 ** -24 * np.abs(lr)), r
        # A_hat sums rho's of relative error <= eps + 2 ulp of expf, in fp32 with compensation
        rel = eps + 2.0 ** -22 + 2.0 ** -23
        for f in ("a_hat", "speedup"):
            want = getattr(ref, f)[r, :n]
            assert np.all(np.abs(g[f][r, :n] - want) <= (rel + 2.0 ** -23) * np.abs(want)), (r, f)
        assert np.all(g["parent"][r, n:] == -7)   # rows past the tree untouched


def _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar, max_guided=None):
    g, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(st == 0)
    ref = _guided(lg, tk, ls, pi, n_max, roots, ctx, c, lar, g)
    _compare(g, ref, lg.shape[1])
    if max_guided is not None:
        assert ref.guided <= max_guided
    return g, ref


@pytest.mark.parametrize("Z,b,V,K,n_max,cost", [
    (1, 5, 300, 8, 40, "flat"),
    (3, 5, 300, 8, 40, "flat"),
    (2, 16, 2000, 32, 64, "workload"),
    (4, 16, 5000, 64, 128, "flat"),
    (4, 16, 5000, 128, 128, "workload"),   # Z K = 512
    (8, 16, 3000, 64, 128, "flat"),        # Z = 8
    (32, 4, 600, 16, 64, "flat"),          # one lane per branch
    (3, 32, 400, 8, 256, "flat"),          # b = 32, n_max = 256
    (2, 2, 3000, 1024, 16, "flat"),        # K = 1024
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
    _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar, max_guided=2)


def test_mixture_tree_bench_shape_every_request(cuda_lib):
    """B = 32, Z = 4, b = 16, K = 64, n_max = 128: the branch top-64 lists of
    bf16 logits over a 151,936-token vocabulary (a shared N(0, 4) part plus a
    branch part N(0, 1)), every request against the guided oracle.  A flat
    cost table makes every tree fill the budget (the longest build); the
    batched workload's cost table stops them at its knee.  bf16 logits tie
    often: exact ties within a parent resolve by token on both sides, the
    rest are flagged."""
    B, Z, b, V, K, n_max = 32, 4, 16, 151936, 64, 128
    x, pi = synth.mixture_inputs(B, Z, b, V, seed=0xBA5710 + 7)
    tk = oracle.topk_marginals(x.reshape(B * Z * b, V), K)
    del x
    lg, tok, ls = (tk.logit.reshape(B, Z, b, K), tk.tok.reshape(B, Z, b, K), tk.lse.reshape(B, Z, b))
    w = synth.workload(3)
    roots, ctx = synth.root_tokens(w), synth.ctx_lens(w)
    flat = np.full((1, n_max + 1), 5.0, np.float32)
    g, ref = _run(lg, tok, ls, pi, n_max, roots, ctx, flat, synth.l_ar(w))
    assert ref.guided <= 8
    assert np.all(g["n_nodes"] == n_max)
    g, ref = _run(lg, tok, ls, pi, n_max, roots, ctx, synth.cost_table(w), synth.l_ar(w))
    assert ref.guided <= 8


def _tie_case():
    """Z = 2, pi = (1/2, 1/2), b = 2, K = 2, logits log p with lse = 0:
    rho (10) 1/2, (10,20) 1/4, then (11), (12) and (10,21) all 1/8."""
    tk = np.array([[[[10, 11], [20, 21]], [[10, 12], [20, 22]]]], np.int32)
    p = np.array([[[[0.5, 0.25], [0.5, 0.5]], [[0.5, 0.25], [0.5, 0.25]]]])
    return np.log(p).astype(np.float32), tk, np.zeros((1, 2, 2)), np.array([[0.5, 0.5]])


def test_mixture_tie_across_depths(cuda_lib):
    """Candidates at depths 1 and 2 tie mathematically (Z = 2): the oracle
    flags the pops and the GPU's order is one of the correct ones."""
    lg, tk, ls, pi = _tie_case()
    n_max = 6
    roots, ctx, lar = np.zeros(1, np.int32), np.zeros(1, np.int32), np.full(1, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g, ref = _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert ref.flagged_pops >= 2
    assert sorted(g["token"][0, :6].tolist()) == [0, 10, 11, 12, 20, 21]


def test_mixture_stop_on_the_boundary(cuda_lib):
    """rho C(1) = A_hat (C(2) - C(1)) exactly: either tree is correct."""
    lg, tk, ls, pi = _tie_case()
    n_max = 4
    roots, ctx, lar = np.zeros(1, np.int32), np.zeros(1, np.int32), np.full(1, 18.0, np.float32)
    c = np.array([[0.0, 2.0, 3.0, 3.0, 3.0]], np.float32)
    g, ref = _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert ref.flagged_stops >= 1
    assert int(g["n_nodes"][0]) in (1, 4)


def test_mixture_tree_steep_lists_take_the_log_domain_rescan(cuda_lib):
    """Ranked logits 23 nats apart (and -inf tails): after a node's first few
    children are taken, the rest lie more than 69 nats (2^-100) below its best
    and the kernel rescans it in the log domain.  A flat cost fills the budget,
    so such children do enter the tree."""
    B, Z, b, K, n_max = 2, 2, 2, 8, 80
    rng = np.random.default_rng(3)
    lg = np.empty((B, Z, b, K), np.float32)
    tk = np.empty((B, Z, b, K), np.int32)
    for r in range(B):
        for z in range(Z):
            for d in range(b):
                lg[r, z, d] = -23.0 * np.arange(K) - (3.5 * z + 0.25 * d + 0.125 * r)
                tk[r, z, d] = rng.permutation(40)[:K]
    lg[:, :, :, -1] = -np.inf                    # a masked tail entry
    ls = np.log(np.exp(lg.astype(np.float64)).sum(axis=-1) + 1e-3)
    pi = np.array([[0.6, 0.4], [0.25, 0.75]])
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g, ref = _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(g["n_nodes"] == n_max)
    # some node's child in the tree lies more than 100 ln 2 below that node's
    # first child (the scan that found it ran in the log domain)
    gap = 0.0
    for r in range(B):
        first = {}
        for i in range(1, n_max):
            p = int(ref.parent[r, i])
            first.setdefault(p, ref.log_rho[r, i])
            gap = max(gap, first[p] - ref.log_rho[r, i])
    assert gap > 100 * np.log(2.0)


def test_mixture_tree_per_request_cost(cuda_lib):
    B, Z, b, V, K, n_max = 4, 3, 8, 2000, 32, 64
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 31)
    pi = np.random.default_rng(5).dirichlet(np.ones(Z), size=B)
    base = synth.cost_table(synth.workload(2, n_max=n_max))
    c = (base * (1.0 + np.arange(B, dtype=np.float32)[:, None] / 3)).astype(np.float32)
    roots, ctx, lar = np.arange(B, dtype=np.int32), np.full(B, 9, np.int32), np.full(B, 18.0, np.float32)
    _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar, max_guided=2)


def test_mixture_tree_deterministic(cuda_lib):
    B, Z, b, V, K, n_max = 3, 4, 16, 5000, 64, 128
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 44)
    pi = np.random.default_rng(4).dirichlet(np.ones(Z), size=B)
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g1, _ = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    g2, _ = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    for k in g1:
        assert np.array_equal(g1[k], g2[k], equal_nan=True), k


def test_mixture_tree_zero_weight_branch_and_bad_cost(cuda_lib):
    """A branch of weight 0 contributes nothing (its log weight is -inf on both
    sides); a non-positive cost entry sets the status bit."""
    from draft_tree_build_gb300 import bastion
    B, Z, b, V, K, n_max = 2, 3, 6, 400, 8, 32
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 9)
    pi = np.array([[0.5, 0.0, 0.5], [0.2, 0.8, 0.0]])
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    c[0, 7] = 0.0
    _, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert np.all(st & bastion.STATUS_BAD_COST)


def test_mixture_tree_bad_weight_sets_status(cuda_lib):
    """A negative or NaN branch weight sets the weight status bit on that
    request only, and counts as weight 0 there."""
    from draft_tree_build_gb300 import bastion
    B, Z, b, V, K, n_max = 3, 2, 5, 300, 8, 24
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 21)
    pi = np.array([[0.5, 0.5], [-0.25, 1.25], [np.nan, 1.0]])
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    g, st = _gpu(lg, tk, ls, pi, n_max, roots, ctx, c, lar)
    assert st[0] == 0
    assert st[1] & bastion.STATUS_BAD_WEIGHT and st[2] & bastion.STATUS_BAD_WEIGHT
    pz = np.array([[0.5, 0.5], [0.0, 1.25], [0.0, 1.0]])
    ref = _guided(lg, tk, ls, pz, n_max, roots, ctx, c, lar, g)
    _compare(g, ref, Z)


@pytest.mark.parametrize("Z,K", [(4, 64), (2, 32), (12, 16)])
def test_mixture_tree_unranked_lists(cuda_lib, Z, K):
    """Branch lists given in no particular order (the ranks of every row
    shuffled): the kernel's scans cannot stop early on the sorted order and
    read every child; the tree is the oracle's, which never assumes the order."""
    B, b, V, n_max = 2, 8, 3000, 64
    lg, tk, ls = _branch_topk(B, Z, b, V, K, 70 + Z)
    rng = np.random.default_rng(Z)
    for r in range(B):
        for z in range(Z):
            for d in range(b):
                perm = rng.permutation(K)
                lg[r, z, d] = lg[r, z, d, perm]
                tk[r, z, d] = tk[r, z, d, perm]
    pi = rng.dirichlet(np.ones(Z), size=B)
    roots, ctx, lar = np.zeros(B, np.int32), np.zeros(B, np.int32), np.full(B, 18.0, np.float32)
    c = np.full((1, n_max + 1), 5.0, np.float32)
    _run(lg, tk, ls, pi, n_max, roots, ctx, c, lar, max_guided=2)
