"""GPU parity: stochastic tree verification (C ABI) against the oracle.

The draws are integers decided by floating point: the kernel forms the
cumulative weights in fp32 (compensated across items) with fp32 exponentials
and log2(e)/T rounded to float, the oracle in fp64.  Where the oracle's draw
lies within MARGIN of the row's total from a neighbouring token's interval, the
GPU may take that neighbour; everywhere else the draw must be identical.  The
walk is then checked exactly against the greedy walk over the GPU's own draws.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, host, to_dev, to_pinned, workload_inputs

pytestmark = pytest.mark.gpu

MARGIN = 4e-6


def gpu_sample(target, b, T, u, n_nodes, parent, token, target_dev=None):
    from draft_tree_build_gb300 import bastion
    td = to_dev(target) if target_dev is None else target_dev
    B, n_max, V = td.shape
    out = {k: torch.full(s, -7, dtype=torch.int32, device=dev())
           for k, s in (("sampled", (B, n_max)), ("accept_len", (B,)), ("accept_nodes", (B, b + 1)),
                        ("out_tokens", (B, b + 1)))}
    ws = bastion.workspace(bastion.bastion_verify_sample_workspace_bytes(B, n_max, V), dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    ud = torch.from_numpy(np.ascontiguousarray(u, np.float64)).to(dev())
    args = [to_dev(np.asarray(x, np.int32)) for x in (n_nodes, parent, token)]
    bastion.bastion_verify_sample(td, b, T, ud, *args, out["sampled"], out["accept_len"],
                                  out["accept_nodes"], out["out_tokens"], ws, st)
    torch.cuda.synchronize()
    assert int(ws[: B * n_max * 8].abs().sum()) == 0, "row keys not left zeroed"
    return {k: host(v) for k, v in out.items()}, host(st)


def _neighbours(row_w, y):
    """Tokens adjacent to y among those with weight."""
    nz = np.flatnonzero(row_w > 0)
    k = np.searchsorted(nz, y)
    return {int(nz[j]) for j in (k - 1, k, k + 1) if 0 <= j < len(nz)}


def walk(draws, n, parent, token, b):
    cur, out, nodes = 0, [], [0]
    while len(out) < b:
        nxt = [c for c in range(1, n) if parent[c] == cur and token[c] == draws[cur]]
        if not nxt:
            break
        out.append(int(draws[cur]))
        cur = nxt[0]
        nodes.append(cur)
    return len(out), nodes, out + [int(draws[cur])]


def check(g, ref, tgt_f64, T, n_nodes, parent, token, b):
    """Draws: identical, or a neighbour where the oracle's margin is small;
    the walk: exactly the greedy walk over the GPU's draws."""
    B = len(n_nodes)
    flagged = 0
    for r in range(B):
        n = int(n_nodes[r])
        for i in range(n):
            y, yr = int(g["sampled"][r, i]), int(ref.sampled[r, i])
            if y == yr:
                continue
            assert ref.margin[r, i] < MARGIN, (r, i, y, yr, ref.margin[r, i])
            x = tgt_f64[r, i]
            w = np.where(np.isfinite(x), np.exp((x - x[np.isfinite(x)].max()) / T), 0.0)
            assert y in _neighbours(w, yr), (r, i, y, yr)
            flagged += 1
        L, nodes, toks = walk(g["sampled"][r], n, parent[r], token[r], b)
        assert g["accept_len"][r] == L
        assert list(g["accept_nodes"][r, : L + 1]) == nodes and np.all(g["accept_nodes"][r, L + 1:] == -1)
        assert list(g["out_tokens"][r, : L + 1]) == toks and np.all(g["out_tokens"][r, L + 1:] == -1)
    return flagged


def _as_f64(tgt):
    if tgt.dtype == np.uint16:
        return (tgt.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return tgt.astype(np.float64)


def _random_tree(rng, B, n_max, V):
    n_nodes = rng.integers(1, n_max + 1, size=B).astype(np.int32)
    parent = np.full((B, n_max), -1, np.int32)
    token = np.zeros((B, n_max), np.int32)
    for r in range(B):
        for i in range(1, n_nodes[r]):
            parent[r, i] = rng.integers(0, i)
            token[r, i] = rng.integers(0, V)
    return n_nodes, parent, token


@pytest.mark.parametrize("V,dtype,T", [(1024, "f32", 1.0), (5000, "bf16", 0.7), (151937, "bf16", 1.5),
                                       (40000, "f32", 1.0), (17, "bf16", 1.0)])
def test_sample_small(cuda_lib, V, dtype, T):
    """Random trees whose draws are made to hit tree tokens: each node row has
    a few strong tokens, among them the tokens of its children."""
    rng = np.random.default_rng(V)
    B, n_max, b = 3, 8, 4
    n_nodes, parent, token = _random_tree(rng, B, n_max, V)
    x = rng.normal(size=(B, n_max, V))
    for r in range(B):
        for i in range(1, n_nodes[r]):
            x[r, parent[r, i], token[r, i]] = 6.0
    if dtype == "f32":
        tgt = x.astype(np.float32)
    else:
        tgt = synth.host_array((B, n_max, V), "bf16")
        tgt[...] = (x.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    u = rng.random((B, n_max))
    g, st = gpu_sample(tgt, b, T, u, n_nodes, parent, token)
    assert np.all(st == 0)
    ref = oracle.verify_sample(tgt, b, T, u, n_nodes, parent, token)
    check(g, ref, _as_f64(tgt), T, n_nodes, parent, token, b)


def test_sample_batched_qwen3_vocab(cuda_lib):
    """B=32, b=16, V=151936, N_max=128 at T = 1: oracle trees, planted target
    rows, seeded uniforms."""
    w = synth.workload(3)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    u = synth.verify_uniforms(w)
    g, st = gpu_sample(tgt, w.b, 1.0, u, tr.n_nodes, tr.parent, tr.token)
    assert np.all(st == 0)
    ref = oracle.verify_sample(tgt, w.b, 1.0, u, tr.n_nodes, tr.parent, tr.token)
    flagged = check(g, ref, _as_f64(tgt), 1.0, tr.n_nodes, tr.parent, tr.token, w.b)
    assert flagged <= 8


def test_sample_reads_pinned_host_target(cuda_lib):
    """The batched workload with its target logits in pinned host memory, read in
    place: the draws and walks of the device-resident call."""
    w = synth.workload(3)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    u = synth.verify_uniforms(w)
    g_dev, _ = gpu_sample(tgt, w.b, 1.0, u, tr.n_nodes, tr.parent, tr.token)
    g_host, st = gpu_sample(tgt, w.b, 1.0, u, tr.n_nodes, tr.parent, tr.token, target_dev=to_pinned(tgt))
    assert np.all(st == 0)
    for k in g_dev:
        assert np.array_equal(g_dev[k], g_host[k]), k


def test_sample_low_temperature_is_greedy(cuda_lib):
    """T -> 0 draws the argmax: the results equal the greedy kernel's."""
    from gpuhelp import gpu_verify
    w = synth.workload(3, B=4)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    td = to_dev(tgt)
    g, st = gpu_sample(None, w.b, 1e-3, np.random.default_rng(1).random((w.B, w.n_max)), tr.n_nodes,
                       tr.parent, tr.token, target_dev=td)
    gv, _ = gpu_verify(None, w.b, tr.n_nodes, tr.parent, tr.token, target_dev=td)
    for r in range(w.B):
        n = tr.n_nodes[r]
        assert np.array_equal(g["sampled"][r, :n], host(gv.argmax)[r, :n])
    assert np.array_equal(g["accept_len"], host(gv.accept_len))
    assert np.array_equal(g["out_tokens"], host(gv.out_tokens))


def test_sample_status_rows(cuda_lib):
    from draft_tree_build_gb300 import bastion
    B, n_max, V, b = 3, 2, 3000, 1
    tgt = np.random.default_rng(2).normal(size=(B, n_max, V)).astype(np.float32)
    tgt[1, 0, 17] = np.nan
    tgt[2, 1, :] = -np.inf
    n_nodes = np.array([2, 2, 2], np.int32)
    parent = np.array([[-1, 0]] * B, np.int32)
    token = np.array([[0, 5]] * B, np.int32)
    g, st = gpu_sample(tgt, b, 1.0, np.full((B, n_max), 0.5), n_nodes, parent, token)
    assert st[0] == 0 and st[1] & bastion.STATUS_NONFINITE and st[2] & bastion.STATUS_EMPTY_ROW
    assert g["sampled"][2, 1] == 0


def test_sample_deterministic(cuda_lib):
    w = synth.workload(2)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    td = to_dev(tgt)
    u = synth.verify_uniforms(w)
    a, _ = gpu_sample(None, w.b, 0.8, u, tr.n_nodes, tr.parent, tr.token, target_dev=td)
    c, _ = gpu_sample(None, w.b, 0.8, u, tr.n_nodes, tr.parent, tr.token, target_dev=td)
    for k in a:
        assert np.array_equal(a[k], c[k])
