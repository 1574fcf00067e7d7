"""GPU parity of the whole tree step (K1 -> K2 -> K4 through the C ABI, on the
GPU's own intermediate results) against the oracle's whole step, at full
workload sizes and in the same launch configuration the bench times."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import compare_topk, compare_verify, compare_tree, dev, host, oracle_tree_guided, to_dev, \
    workload_inputs

pytestmark = pytest.mark.gpu


def _step(w, graph=False, chunks=1, cost_per_request=False):
    from draft_tree_build_gb300 import bastion
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    if cost_per_request:  # request r's costs scaled by 1 + r/4: trees differ across requests
        cost = (cost * (1.0 + np.arange(w.B, dtype=np.float32)[:, None] / 4)).astype(np.float32)
    step = bastion.TreeStep(w.B, w.b, w.V, w.K, w.n_max, dev(), torch.from_numpy(roots),
                            torch.from_numpy(ctx), torch.from_numpy(cost), torch.from_numpy(lar))
    xd = to_dev(x)
    # the target rows are planted from the oracle's tree (never from the GPU's)
    ref_tree = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, ref_tree.n_nodes, ref_tree.depth, tk.tok)
    td = to_dev(tgt)
    if graph:
        g = step.capture(xd, td, chunks=chunks)
        step.status.zero_()
        g.replay()
    elif chunks > 1:
        step.run_chunked(xd, td, chunks)
    else:
        step.run(xd, td)
    torch.cuda.synchronize()
    assert int(step.status.abs().sum()) == 0
    compare_topk(step.topk, tk)
    ref = oracle_tree_guided(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar, step.tree)
    assert ref.guided == 0
    compare_tree(step.tree, ref)
    vf = oracle.verify_greedy(tgt, w.b, ref.n_nodes, ref.parent, ref.token)
    compare_verify(step.ver, vf, ref.n_nodes)
    return step, vf


@pytest.mark.parametrize("cid", [1, 2])
def test_pipeline_small(cuda_lib, cid):
    _step(synth.workload(cid))


def test_pipeline_batched_qwen3_vocab_graph(cuda_lib):
    """B=32, b=16, V=151936, K=64, N_max=128: replayed from a CUDA graph as in the bench."""
    step, vf = _step(synth.workload(3), graph=True)
    assert vf.accept_len.max() >= 1


def test_pipeline_graph_replayed_many_times(cuda_lib):
    """The step replayed 50 times from two graphs on two alternating inputs: the
    verify workspace returns to zero after every replay, and the results stay
    the oracle's."""
    from draft_tree_build_gb300 import bastion
    w = synth.workload(3)
    x = synth.drafter_logits(w)
    x2 = synth.drafter_logits(synth.workload(3, seed=w.seed + 17))
    roots, ctx, cost, lar = workload_inputs(w)
    step = bastion.TreeStep(w.B, w.b, w.V, w.K, w.n_max, dev(), torch.from_numpy(roots),
                            torch.from_numpy(ctx), torch.from_numpy(cost), torch.from_numpy(lar))
    xs = [to_dev(x), to_dev(x2)]
    td = torch.zeros((w.B, w.n_max, w.V), dtype=xs[0].dtype, device=dev())
    graphs = [step.capture(xs[i], td) for i in range(2)]
    for i in range(50):
        graphs[i & 1].replay()
    torch.cuda.synchronize()
    assert int(step.ws_verify.abs().sum()) == 0
    assert int(step.status.abs().sum()) == 0
    tk = oracle.topk_marginals(x2, w.K)   # replay 49 ran on the second input
    compare_topk(step.topk, tk)
    ref = oracle_tree_guided(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar, step.tree)
    compare_tree(step.tree, ref)


def test_pipeline_serving_llama_vocab(cuda_lib):
    """B=64, b=16, V=128256, K=64, N_max=256 (every tree fills the budget)."""
    step, vf = _step(synth.workload(5))
    assert np.all(host(step.tree.n_nodes) == 256)


@pytest.mark.parametrize("chunks", [2, 3, 4])
def test_pipeline_chunked_graph(cuda_lib, chunks):
    """The batch split into request chunks on forked streams inside the graph
    (three chunks leave unequal slices of 32 requests)."""
    _step(synth.workload(3), graph=True, chunks=chunks)


@pytest.mark.parametrize("cost_per_request", [False, True])
def test_pipeline_chunked_eager(cuda_lib, cost_per_request):
    """Chunks on streams without a graph; B=5 in four chunks (1, 1, 1, 2
    requests), with a shared and a per-request cost table."""
    _step(synth.workload(3, B=5), chunks=4, cost_per_request=cost_per_request)
