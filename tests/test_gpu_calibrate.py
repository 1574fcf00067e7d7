"""GPU parity: calibration of the verification cost model (C ABI) against the
oracle, and the calibrated table driving the tree build on the device."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import compare_tree, dev, host, oracle_tree_guided, to_dev, workload_inputs

pytestmark = pytest.mark.gpu

ROOF = dict(bytes0=16e9, bytes1=2.0e6, flops0=0.0, flops1=16e9, bw=8e9, peak=2.25e12)


def gpu_calibrate(n, t, roof, t_draft, n_max):
    from draft_tree_build_gb300 import bastion
    nd = torch.from_numpy(np.asarray(n, np.float32)).to(dev())
    td = torch.from_numpy(np.asarray(t, np.float32)).to(dev())
    cost = torch.zeros(n_max + 1, dtype=torch.float32, device=dev())
    par = torch.zeros(2, dtype=torch.float32, device=dev())
    st = torch.zeros(1, dtype=torch.int32, device=dev())
    bastion.bastion_calibrate_cost(nd, td, roof, t_draft, n_max, cost, par, st)
    torch.cuda.synchronize()
    return cost, host(par), int(host(st)[0])


@pytest.mark.parametrize("count", [7, 300, 100000])
def test_calibrate_matches_oracle(cuda_lib, count):
    rng = np.random.default_rng(count)
    n = rng.integers(1, 4000, size=count).astype(np.float32)
    r = np.maximum((ROOF["bytes0"] + ROOF["bytes1"] * n.astype(np.float64)) / ROOF["bw"],
                   ROOF["flops1"] * n.astype(np.float64) / ROOF["peak"])
    t = (1.2 * r + 0.5 + rng.normal(scale=0.05, size=count)).astype(np.float32)
    cost, par, st = gpu_calibrate(n, t, ROOF, 3.0, 256)
    ref, a, b = oracle.calibrate_cost(n.astype(np.float64), t.astype(np.float64), ROOF, 3.0, 256)
    assert st == 0
    assert par[0] == pytest.approx(a, rel=1e-6) and par[1] == pytest.approx(b, rel=1e-5, abs=1e-6)
    assert np.allclose(host(cost), ref, rtol=1e-6)


def test_calibrated_table_drives_the_tree_build(cuda_lib):
    """Calibrating from noise-free samples of the serving workload's cost model
    gives its table on the device; the tree build reading that table in place
    produces the oracle's trees."""
    from draft_tree_build_gb300 import bastion
    w = synth.workload(5, B=4)
    r = dict(bytes0=16e9, bytes1=0.0, flops0=0.0, flops1=16e9, bw=8e9, peak=2.25e12)
    n = np.array([1, 50, 200, 281, 282, 256, 1000], np.float32)
    t = np.array([synth.cost_ms(int(k), w.cost) for k in n], np.float64) - 3.0
    cost, par, st = gpu_calibrate(n, t, r, 3.0, w.n_max)
    assert st == 0
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, _, lar = workload_inputs(w)
    table = host(cost).reshape(1, -1)
    ref = oracle_tree_guided(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, table, lar)
    # the GPU tree from the same top-K inputs, reading the calibrated table in place
    tree = bastion.alloc_tree(w.B, w.n_max, dev())
    status = torch.zeros(w.B, dtype=torch.int32, device=dev())
    bastion.bastion_build_tree(to_dev(tk.logit), to_dev(tk.tok), to_dev(tk.lse), w.n_max, to_dev(roots),
                               to_dev(ctx), cost.view(1, -1), to_dev(lar), tree.n_nodes, tree.parent,
                               tree.depth, tree.pos_id, tree.token, tree.rank, tree.log_rho, tree.a_hat,
                               tree.speedup, tree.anc_mask, status)
    torch.cuda.synchronize()
    assert int(status.abs().sum()) == 0
    ref = oracle_tree_guided(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, table, lar, tree)
    compare_tree(tree, ref)


def test_calibrate_flags_bad_samples(cuda_lib):
    from draft_tree_build_gb300 import bastion
    _, _, st = gpu_calibrate([1, 2, 3], [1.0, float("nan"), 2.0], ROOF, 1.0, 8)
    assert st & bastion.STATUS_BAD_COST
    # a negative intercept large enough to make C(N) negative
    _, _, st = gpu_calibrate([1, 2000], [-50.0, -40.0], ROOF, 0.0, 8)
    assert st & bastion.STATUS_BAD_COST
