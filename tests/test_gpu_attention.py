"""GPU parity: tree-masked GQA attention (tcgen05 kernel, C ABI) against the
fp64 oracle; bf16 output within 2e-2 absolute.  Rows past n_nodes untouched."""
import math
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, host, to_dev, workload_inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2


def _attn_inputs(B, n_max, Hq, Hkv, ctx, seed, D=128):
    w = synth.Workload(93, "attn", B=B, b=16, V=8, K=1, n_max=n_max, dtype="bf16", l_ar_ms=1.0,
                       cost="flat", drafter="spike-linear", p_agree="const0.7", ctx=ctx, Hq=Hq,
                       Hkv=Hkv, D=D, seed=seed)
    return synth.attention_inputs(w)


def _run(q, k, v, ctx_len, n_nodes, anc_mask, scale=None):
    from draft_tree_build_gb300 import bastion
    B, n_max, Hq, D = q.shape
    L_cap, Hkv = k.shape[1], k.shape[2]
    scale = scale or 1.0 / math.sqrt(D)
    out = torch.full((B, n_max, Hq, D), 7.0, dtype=torch.bfloat16, device=dev())
    ws = bastion.workspace(bastion.bastion_tree_attention_workspace_bytes(B, n_max, Hq, Hkv, D, L_cap), dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    bastion.bastion_tree_attention(to_dev(q), to_dev(k), to_dev(v), to_dev(np.asarray(ctx_len, np.int32)),
                                   to_dev(np.asarray(n_nodes, np.int32)),
                                   to_dev(np.asarray(anc_mask, np.uint32).view(np.int32)), scale, out, ws, st)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), host(st)


def _trees(B, n_max, seed, flat=True):
    w = synth.workload(2, B=B, n_max=n_max, seed=seed)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    cost = np.full((1, n_max + 1), 5.0, np.float32) if flat else synth.cost_table(w)
    return oracle.build_tree(tk.logit, tk.tok, tk.lse, n_max, np.zeros(B, np.int32),
                             np.zeros(B, np.int32), cost, np.full(B, 18.0, np.float32))


def _oracle_rows(q, k, v, ctx, tr, sel):
    """The oracle's rows for sel, split over host threads (the oracle is a C
    function called through ctypes, which releases the GIL while it runs)."""
    D = q.shape[-1]
    sel = np.ascontiguousarray(sel, np.int32).reshape(-1, 3)
    nt = max(1, min(len(sel) // 256, os.cpu_count() or 1))
    run = lambda s: oracle.tree_attention(q, k, v, ctx, tr.n_nodes, tr.anc_mask,  # noqa: E731
                                          1 / math.sqrt(D), sel=s)
    if nt == 1:
        return run(sel)
    with ThreadPoolExecutor(nt) as ex:
        return np.concatenate(list(ex.map(run, np.array_split(sel, nt))))


def _check_rows(out, q, k, v, ctx, tr, sel):
    ref = _oracle_rows(q, k, v, ctx, tr, sel)
    sel = np.asarray(sel).reshape(-1, 3)
    got = out[sel[:, 0], sel[:, 1], sel[:, 2]]
    err = np.abs(got - ref).max()
    assert err < TOL, err


def test_attention_small_all_rows(cuda_lib):
    B, n_max, Hq, Hkv, ctx = 2, 40, 8, 2, 300
    tr = _trees(B, n_max, 11)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 5)
    ctxs = np.array([ctx, 257], np.int32)
    out, st = _run(q, k, v, ctxs, tr.n_nodes, tr.anc_mask)
    assert np.all(st == 0)
    sel = [(r, i, h) for r in range(B) for i in range(int(tr.n_nodes[r])) for h in range(Hq)]
    _check_rows(out, q, k, v, ctxs, tr, sel)


def test_attention_rows_past_tree_untouched(cuda_lib):
    B, n_max, Hq, Hkv, ctx = 1, 64, 4, 1, 130
    tr = _trees(B, n_max, 12, flat=False)   # budgeted: n_nodes < n_max
    n = int(tr.n_nodes[0])
    assert n < n_max
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 6)
    out, _ = _run(q, k, v, [ctx], tr.n_nodes, tr.anc_mask)
    assert np.all(out[0, n:] == 7.0)
    _check_rows(out, q, k, v, [ctx], tr, [(0, i, h) for i in range(n) for h in range(Hq)])


def test_attention_chain_no_context_is_causal(cuda_lib):
    """ctx_len = 0 with a chain tree: plain causal self-attention."""
    B, n, Hq, Hkv = 1, 100, 4, 2
    W = (n + 31) // 32
    mask = np.zeros((1, n, W), np.uint32)
    for i in range(n):
        for j in range(i + 1):
            mask[0, i, j // 32] |= np.uint32(1 << (j % 32))
    q, k, v = _attn_inputs(B, n, Hq, Hkv, 0, 7)
    out, _ = _run(q, k, v, [0], [n], mask)
    qf = torch.from_numpy(synth.bf16_bits_to_f32(q[0]).astype(np.float64)).permute(1, 0, 2)[None]
    kf = torch.from_numpy(synth.bf16_bits_to_f32(k[0]).astype(np.float64)).repeat_interleave(2, 1).permute(1, 0, 2)[None]
    vf = torch.from_numpy(synth.bf16_bits_to_f32(v[0]).astype(np.float64)).repeat_interleave(2, 1).permute(1, 0, 2)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qf, kf, vf, is_causal=True)[0].permute(1, 0, 2)
    assert np.abs(out[0] - ref.numpy()).max() < TOL


@pytest.mark.parametrize("Hq,Hkv", [(32, 4), (8, 8), (16, 8)])
def test_attention_group_sizes(cuda_lib, Hq, Hkv):
    B, n_max, ctx = 2, 33, 200
    tr = _trees(B, n_max, 13)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 8)
    out, _ = _run(q, k, v, [ctx, ctx], tr.n_nodes, tr.anc_mask)
    rng = np.random.default_rng(0)
    sel = [(int(r), int(i), int(h)) for r, i, h in zip(rng.integers(0, B, 64), rng.integers(0, n_max, 64),
                                                       rng.integers(0, Hq, 64))]
    _check_rows(out, q, k, v, [ctx, ctx], tr, sel)


def test_attention_full_size_qwen3_layer(cuda_lib):
    """B=8, 32/8 heads, d=128, ctx 4096, N=64 trees from the single-request recipe."""
    w = synth.workload(4)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, c, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, c, lar)
    assert np.all(tr.n_nodes == 64)
    q, k, v = synth.attention_inputs(w)
    out, st = _run(q, k, v, ctx, tr.n_nodes, tr.anc_mask)
    assert np.all(st == 0)
    # every (request, node, head) row: 128 CTAs of 33 key tiles each
    sel = [(r, i, h) for r in range(w.B) for i in range(64) for h in range(32)]
    _check_rows(out, q, k, v, ctx, tr, sel)


def test_attention_kv_overflow_flag(cuda_lib):
    from draft_tree_build_gb300 import bastion
    B, n_max, Hq, Hkv, ctx = 1, 16, 4, 1, 100
    tr = _trees(B, n_max, 14)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 9)
    _, st = _run(q, k, v, [ctx + 5], tr.n_nodes, tr.anc_mask)   # ctx + n > L_cap
    assert st[0] & bastion.STATUS_KV_OVERFLOW


def test_attention_serving_size_sampled_rows(cuda_lib):
    """The serving step's attention shape: 64 requests, 256-node trees, 32/8
    heads, d=128, a 16,384-token context; sampled rows and every row of one
    request against the oracle.
    The trees come from the oracle (a small-vocabulary drafter, flat cost)."""
    B, n_max, Hq, Hkv, ctx = 64, 256, 32, 8, 16384
    w = synth.Workload(94, "trees", B=B, b=16, V=1024, K=64, n_max=n_max, dtype="bf16", l_ar_ms=15.0,
                       cost="flat", drafter="spike-geometric", p_agree="uniform", seed=777)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    cost = np.full((1, n_max + 1), 6.0, np.float32)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, n_max, np.zeros(B, np.int32),
                           np.full(B, ctx, np.int32), cost, np.full(B, 15.0, np.float32))
    assert np.all(tr.n_nodes == n_max)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 31)
    out, st = _run(q, k, v, np.full(B, ctx, np.int32), tr.n_nodes, tr.anc_mask)
    assert np.all(st == 0)
    rng = np.random.default_rng(5)
    sel = [(int(r), int(i), int(h)) for r, i, h in zip(rng.integers(0, B, 160),
                                                       rng.integers(0, n_max, 160), rng.integers(0, Hq, 160))]
    sel += [(0, 0, h) for h in range(0, 32, 4)] + [(B - 1, n_max - 1, h) for h in range(0, 32, 4)]
    # and every (node, head) row of one whole request (the CTAs of its 8 KV heads)
    rw = 37
    sel += [(rw, i, h) for i in range(n_max) for h in range(Hq)]
    _check_rows(out, q, k, v, np.full(B, ctx, np.int32), tr, sel)


def _to_bf16(x):
    """float -> bf16 bits, round to nearest even (test input construction)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def test_attention_late_max_jump_rescales(cuda_lib):
    """Context keys far into the context whose scores exceed every earlier one
    by more than 2^8 in log2 units for every row (keys 700 and 900, tiles 5 and
    7): the tile taken against the old reference max must be redone with the
    new one and the accumulator rescaled, twice."""
    B, n_max, Hq, Hkv, ctx = 1, 24, 4, 1, 1000
    tr = _trees(B, n_max, 15)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, ctx, 10)
    D = q.shape[-1]
    rng = np.random.default_rng(3)
    u = rng.normal(size=D)
    u /= np.linalg.norm(u)
    qf = synth.bf16_bits_to_f32(q).astype(np.float64) + 3.0 * u   # every row shares a component on u
    kf = synth.bf16_bits_to_f32(k).astype(np.float64)
    kf[0, 700, 0] = 40.0 * u    # ~15 log2 units above the earlier scores
    kf[0, 900, 0] = 80.0 * u    # ~15 more
    q2, k2 = _to_bf16(qf), _to_bf16(kf)
    out, st = _run(q2, k2, v, [ctx], tr.n_nodes, tr.anc_mask)
    assert st[0] == 0
    _check_rows(out, q2, k2, v, [ctx], tr, [(0, i, h) for i in range(int(tr.n_nodes[0])) for h in range(Hq)])


def test_attention_context_tile_boundaries(cuda_lib):
    """Context lengths 0, 1, 127, 128, 129 and 255 in one batch: the tree's
    keys start inside, at and just past a 128-key tile boundary."""
    ctxs = np.array([0, 1, 127, 128, 129, 255], np.int32)
    B, n_max, Hq, Hkv = len(ctxs), 20, 8, 2
    tr = _trees(B, n_max, 16)
    q, k, v = _attn_inputs(B, n_max, Hq, Hkv, int(ctxs.max()), 11)
    out, st = _run(q, k, v, ctxs, tr.n_nodes, tr.anc_mask)
    assert np.all(st == 0)
    sel = [(r, i, h) for r in range(B) for i in range(int(tr.n_nodes[r])) for h in range(Hq)]
    _check_rows(out, q, k, v, ctxs, tr, sel)
