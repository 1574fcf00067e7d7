"""GPU parity: best-first tree + online controller (C ABI) against the oracle.

Both sides take the same inputs (the oracle's top-K logits, tokens and fp64
lse).  Bit-exact: n_nodes, parent, depth, pos_id, token, rank, ancestor masks.
log rho within 1e-5 (absolute in log, i.e. 1e-5 relative in rho); A_hat and
S within 1e-5 relative.
"""
import numpy as np
import pytest

import oracle
import synth
from gpuhelp import compare_tree, gpu_tree, host, oracle_tree_guided, workload_inputs
from treecheck import check_tree

pytestmark = pytest.mark.gpu


def _case(w, K=None, n_max=None, cost=None):
    K = K or w.K
    n_max = n_max or w.n_max
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, K)
    roots, ctx, c, lar = workload_inputs(w)
    if cost is not None:
        c = cost
    elif n_max != w.n_max:
        c = np.array([[synth.cost_ms(N, w.cost) for N in range(n_max + 1)]], np.float32)
    g, st = gpu_tree(tk.logit, tk.tok, tk.lse, n_max, roots, ctx, c, lar)
    ref = oracle_tree_guided(tk.logit, tk.tok, tk.lse, n_max, roots, ctx, c, lar, g)
    assert ref.guided == 0, "GPU departed from the oracle at a near tie"
    compare_tree(g, ref)
    for r in range(w.B):
        n = int(ref.n_nodes[r])
        check_tree(r, n, host(g.parent)[r], host(g.depth)[r], host(g.pos_id)[r], host(g.token)[r],
                   host(g.rank)[r], host(g.log_rho)[r].astype(np.float64),
                   host(g.anc_mask)[r].view(np.uint32), tk.tok[r], ctx[r], roots[r], w.b, K, n_max,
                   tol=1e-6)
    return g, st, ref


@pytest.mark.parametrize("cid", [1, 2, 3, 4, 5])
def test_tree_workloads(cuda_lib, cid):
    g, st, ref = _case(synth.workload(cid))
    assert int(st.abs().sum()) == 0


def test_tree_chain_k1(cuda_lib):
    w = synth.workload(2)
    g, _, ref = _case(w, K=1, n_max=17, cost=np.full((1, 18), 4.0, np.float32))
    assert host(g.n_nodes)[0] == 17
    assert host(g.parent)[0, 1:17].tolist() == list(range(16))


def test_tree_root_only(cuda_lib):
    w = synth.workload(1)
    g, _, ref = _case(w, n_max=1, cost=np.full((1, 2), 4.0, np.float32))
    assert host(g.n_nodes)[0] == 1


def test_tree_b1_and_wide(cuda_lib):
    w = synth.workload(3, b=1, B=4)
    g, _, ref = _case(w, n_max=65, cost=np.full((1, 66), 4.0, np.float32))
    assert np.all(host(g.depth)[:, 1:65] == 1)


def test_tree_max_sizes(cuda_lib):
    """b = 32, K = 1024, n_max = 256, flat cost (fills the budget)."""
    w = synth.Workload(92, "max", B=3, b=32, V=4096, K=1024, n_max=256, dtype="bf16", l_ar_ms=15.0,
                       cost="flat", drafter="spike-geometric", p_agree="uniform", seed=4242)
    g, _, ref = _case(w)
    assert np.all(host(g.n_nodes) == 256)


def test_tree_ties_everywhere(cuda_lib):
    """All-equal logits: every candidate at a depth ties; the total order decides."""
    B, b, K = 2, 4, 6
    logit = np.zeros((B, b, K), np.float32)
    tok = np.tile(np.arange(K, dtype=np.int32), (B, b, 1))
    lse = np.full((B, b), np.log(1000.0))
    cost = np.full((1, 41), 3.0, np.float32)
    g, _ = gpu_tree(logit, tok, lse, 40, [1, 2], [0, 5], cost, [10.0, 10.0])
    ref = oracle.build_tree(logit, tok, lse, 40, [1, 2], [0, 5], cost, [10.0, 10.0])
    compare_tree(g, ref)


def test_tree_per_request_cost_and_bad_cost(cuda_lib):
    from draft_tree_build_gb300 import bastion
    w = synth.workload(3, B=4)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, c, lar = workload_inputs(w)
    cost = np.tile(c, (4, 1))
    cost[1] = 5.0 + 0.5 * np.arange(w.n_max + 1)   # steep: small tree
    cost[2, 7] = 0.0                               # not a valid cost
    g, st = gpu_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    ref = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    s = host(st)
    assert s[2] & bastion.STATUS_BAD_COST and s[0] == 0 and s[1] == 0
    assert np.array_equal(host(g.n_nodes)[[0, 1, 3]], ref.n_nodes[[0, 1, 3]])
    assert host(g.n_nodes)[1] < 32
