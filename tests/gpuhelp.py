"""Helpers for the GPU parity tests: numpy <-> torch marshalling and the
oracle-side reference runs (test infrastructure)."""
import numpy as np
import torch

import oracle
import synth


def dev():
    return torch.device("cuda:0")


def to_dev(a: np.ndarray) -> torch.Tensor:
    """numpy float32 / uint16 (bf16 bits) / int32 / float64 -> CUDA tensor."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev())
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev())


def to_pinned(a: np.ndarray) -> torch.Tensor:
    """numpy float32 / uint16 (bf16 bits) -> pinned (page-locked) host tensor."""
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).pin_memory()
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def gpu_topk(x: np.ndarray, K: int, x_dev=None):
    from draft_tree_build_gb300 import bastion
    xd = to_dev(x) if x_dev is None else x_dev
    B, b, V = xd.shape
    t = bastion.alloc_topk(B, b, K, dev())
    ws = bastion.workspace(bastion.bastion_topk_marginals_workspace_bytes(B, b, V, K), dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    bastion.bastion_topk_marginals(xd, K, t.logq, t.logit, t.tok, t.lse, ws, st)
    torch.cuda.synchronize()
    return t, st


def gpu_tree(logit, tok, lse, n_max, roots, ctx, cost, lar):
    from draft_tree_build_gb300 import bastion
    lg = logit if isinstance(logit, torch.Tensor) else to_dev(np.asarray(logit, np.float32))
    tk = tok if isinstance(tok, torch.Tensor) else to_dev(np.asarray(tok, np.int32))
    ls = lse if isinstance(lse, torch.Tensor) else to_dev(np.asarray(lse, np.float64))
    B = lg.shape[0]
    tr = bastion.alloc_tree(B, n_max, dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    bastion.bastion_build_tree(lg, tk, ls, n_max, to_dev(np.asarray(roots, np.int32)),
                               to_dev(np.asarray(ctx, np.int32)), to_dev(np.asarray(cost, np.float32)),
                               to_dev(np.asarray(lar, np.float32)), tr.n_nodes, tr.parent, tr.depth,
                               tr.pos_id, tr.token, tr.rank, tr.log_rho, tr.a_hat, tr.speedup,
                               tr.anc_mask, st)
    torch.cuda.synchronize()
    return tr, st


def gpu_verify(target, b, n_nodes, parent, token, target_dev=None):
    from draft_tree_build_gb300 import bastion
    td = to_dev(target) if target_dev is None else target_dev
    B, n_max, V = td.shape
    v = bastion.alloc_verify(B, n_max, b, dev())
    ws = bastion.workspace(bastion.bastion_verify_greedy_workspace_bytes(B, n_max, V), dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    nn = n_nodes if isinstance(n_nodes, torch.Tensor) else to_dev(np.asarray(n_nodes, np.int32))
    pa = parent if isinstance(parent, torch.Tensor) else to_dev(np.asarray(parent, np.int32))
    tk = token if isinstance(token, torch.Tensor) else to_dev(np.asarray(token, np.int32))
    bastion.bastion_verify_greedy(td, b, nn, pa, tk, v.argmax, v.accept_len, v.accept_nodes,
                                  v.out_tokens, ws, st)
    torch.cuda.synchronize()
    assert int(ws.abs().sum()) == 0, "workspace not left zeroed"
    return v, st


def compare_topk(g, ref: "oracle.TopK", lse_atol=2e-6):
    assert np.array_equal(host(g.tok), ref.tok)
    assert np.array_equal(host(g.logit), ref.logit)
    fin = np.isfinite(ref.lse)
    assert np.all(np.abs(host(g.lse)[fin] - ref.lse[fin]) <= lse_atol), np.abs(host(g.lse)[fin] - ref.lse[fin]).max()
    lq, rl = host(g.logq), ref.logq
    ok = np.isfinite(rl)
    assert np.all(np.abs(lq[ok] - rl[ok]) <= lse_atol + 1e-6 * np.abs(rl[ok]))
    assert np.array_equal(np.isneginf(lq), np.isneginf(rl))


def compare_tree(g, ref: "oracle.Tree", W=None):
    n_g = host(g.n_nodes)
    assert np.array_equal(n_g, ref.n_nodes), (n_g, ref.n_nodes)
    B = len(n_g)
    for r in range(B):
        n = int(ref.n_nodes[r])
        for name in ("parent", "depth", "pos_id", "token", "rank"):
            a, b_ = host(getattr(g, name))[r, :n], getattr(ref, name)[r, :n]
            assert np.array_equal(a, b_), (name, r, a, b_)
        assert np.array_equal(host(g.anc_mask)[r, :n].view(np.uint32), ref.anc_mask[r, :n])
        lr = host(g.log_rho)[r, :n].astype(np.float64)
        assert np.all(np.abs(lr - ref.log_rho[r, :n]) <= 1e-5), np.abs(lr - ref.log_rho[r, :n]).max()
        for name in ("a_hat", "speedup"):
            a = host(getattr(g, name))[r, :n].astype(np.float64)
            b_ = getattr(ref, name)[r, :n]
            assert np.all(np.abs(a - b_) <= 1e-5 * np.abs(b_)), (name, r)


def oracle_tree_guided(logit, tok, lse, n_max, roots, ctx, cost, lar, g=None):
    """Oracle tree; when it flags near ties and a GPU tree is given, rerun with
    the GPU tree as the guide (followed only at the flagged steps)."""
    ref = oracle.build_tree(logit, tok, lse, n_max, roots, ctx, cost, lar)
    if (ref.flagged_pops or ref.flagged_stops) and g is not None:
        ref = oracle.build_tree(logit, tok, lse, n_max, roots, ctx, cost, lar,
                                guide=(host(g.n_nodes), host(g.parent), host(g.rank)))
    return ref


def compare_verify(g, ref: "oracle.Verify", n_nodes):
    am = host(g.argmax)
    for r in range(len(n_nodes)):
        n = int(n_nodes[r])
        assert np.array_equal(am[r, :n], ref.argmax[r, :n]), r
    assert np.array_equal(host(g.accept_len), ref.accept_len)
    assert np.array_equal(host(g.accept_nodes), ref.accept_nodes)
    assert np.array_equal(host(g.out_tokens), ref.out_tokens)


def workload_inputs(w):
    return synth.root_tokens(w), synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w)
