"""Pins for the oracle's tree-masked GQA attention (no GPU).

The target verifies the whole draft tree in one parallel forward (Bastion,
gist.science/nl/paper/2605.29727, "Probleemstelling"); each tree token attends
to the committed context and to its own root path.  Special cases reduce to the
library's scaled-dot-product attention (torch, fp64 on CPU).
"""
import math

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")


def _f64(bits):
    return torch.from_numpy(synth.bf16_bits_to_f32(bits).astype(np.float64))


def _sdpa(q, k, v, mask, scale, G):
    """q [N, Hq, D], k/v [L, Hkv, D] -> [N, Hq, D] via torch sdpa (fp64)."""
    qh = q.permute(1, 0, 2)[None]
    kh = k.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    vh = v.repeat_interleave(G, dim=1).permute(1, 0, 2)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qh, kh, vh, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2)


def _rand_inputs(B, n_max, Hq, Hkv, D, L_cap, seed):
    w = synth.Workload(90, "t", B=B, b=16, V=8, K=1, n_max=n_max, dtype="bf16", l_ar_ms=1,
                       cost="flat", drafter="spike-linear", p_agree="const0.7", ctx=L_cap - n_max,
                       Hq=Hq, Hkv=Hkv, D=D, seed=seed)
    return synth.attention_inputs(w)


def _chain_mask(n, n_max):
    W = (n_max + 31) // 32
    m = np.zeros((n_max, W), np.uint32)
    for i in range(n):
        for j in range(i + 1):
            m[i, j // 32] |= np.uint32(1 << (j % 32))
    return m


def test_chain_without_context_is_causal_attention():
    B, n, Hq, Hkv, D = 1, 40, 8, 2, 64
    q, k, v = _rand_inputs(B, n, Hq, Hkv, D, n, 3)
    mask = _chain_mask(n, n)[None]
    sc = 1 / math.sqrt(D)
    out = oracle.tree_attention(q, k, v, [0], [n], mask, sc).reshape(n, Hq, D)
    ref = _sdpa(_f64(q[0]), _f64(k[0]), _f64(v[0]),
                torch.ones(n, n, dtype=torch.bool).tril(), sc, Hq // Hkv)
    assert np.allclose(out, ref.numpy(), atol=1e-12)


def test_single_query_is_decode_attention():
    ctx, Hq, Hkv, D = 300, 4, 1, 128
    q, k, v = _rand_inputs(1, 1, Hq, Hkv, D, ctx + 1, 4)
    mask = np.ones((1, 1, 1), np.uint32)
    sc = 1 / math.sqrt(D)
    out = oracle.tree_attention(q, k, v, [ctx], [1], mask, sc).reshape(1, Hq, D)
    ref = _sdpa(_f64(q[0]), _f64(k[0]), _f64(v[0]), None, sc, Hq)
    assert np.allclose(out, ref.numpy(), atol=1e-12)


def test_tree_mask_from_parent_pointers():
    """General tree with context; the expected visibility is rebuilt from the
    oracle tree's parent pointers (not from its bitmask words)."""
    w = synth.workload(2)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, [0], [50],
                           np.full((1, w.n_max + 1), 5.0, np.float32), [18.0])
    n = int(tr.n_nodes[0])
    ctx, Hq, Hkv, D = 50, 8, 2, 128
    q, k, v = _rand_inputs(1, w.n_max, Hq, Hkv, D, ctx + w.n_max, 5)
    sc = 1 / math.sqrt(D)
    out = oracle.tree_attention(q, k, v, [ctx], [n], tr.anc_mask, sc).reshape(n, Hq, D)
    vis = torch.zeros(n, ctx + n, dtype=torch.bool)
    vis[:, :ctx] = True
    for i in range(n):
        j = i
        while j >= 0:
            vis[i, ctx + j] = True
            j = int(tr.parent[0, j]) if j > 0 else -1
    ref = _sdpa(_f64(q[0, :n]), _f64(k[0, : ctx + n]), _f64(v[0, : ctx + n]), vis, sc, Hq // Hkv)
    assert np.allclose(out, ref.numpy(), atol=1e-12)
    # selected rows equal the full computation
    sel = np.array([[0, 3, 1], [0, n - 1, 7]])
    part = oracle.tree_attention(q, k, v, [ctx], [n], tr.anc_mask, sc, sel=sel)
    assert np.array_equal(part[0], out[3, 1]) and np.array_equal(part[1], out[n - 1, 7])


def _small_tree(ctx):
    w = synth.workload(2, n_max=24)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    return oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, [0], [ctx],
                             np.full((1, w.n_max + 1), 5.0, np.float32), [18.0])


def _visible(tr, ctx, i):
    """Key slots query i sees: the context and its root path (from parent pointers)."""
    keys = list(range(ctx))
    j = i
    while j >= 0:
        keys.append(ctx + j)
        j = int(tr.parent[0, j]) if j > 0 else -1
    return sorted(keys)


def test_zero_scale_averages_the_visible_values():
    """scale = 0 makes every visible key equally likely: each output is the
    mean of the value rows the query sees (a closed form)."""
    ctx, Hq, Hkv, D = 37, 4, 2, 128
    tr = _small_tree(ctx)
    n = int(tr.n_nodes[0])
    q, k, v = _rand_inputs(1, 24, Hq, Hkv, D, ctx + 24, 21)
    out = oracle.tree_attention(q, k, v, [ctx], [n], tr.anc_mask, 0.0).reshape(n, Hq, D)
    vf = synth.bf16_bits_to_f32(v[0]).astype(np.float64)
    for i in range(n):
        keys = _visible(tr, ctx, i)
        for h in range(Hq):
            assert np.allclose(out[i, h], vf[keys, h // (Hq // Hkv)].mean(0), atol=1e-13)


def test_context_permutation_invariance():
    """Permuting the context slots of K and V together leaves every output
    unchanged: attention is a weighted mean over a set."""
    ctx, Hq, Hkv, D = 50, 8, 2, 128
    tr = _small_tree(ctx)
    n = int(tr.n_nodes[0])
    q, k, v = _rand_inputs(1, 24, Hq, Hkv, D, ctx + 24, 22)
    perm = np.random.default_rng(0).permutation(ctx)
    k2, v2 = k.copy(), v.copy()
    k2[0, :ctx], v2[0, :ctx] = k[0, perm], v[0, perm]
    sc = 1 / math.sqrt(D)
    a = oracle.tree_attention(q, k, v, [ctx], [n], tr.anc_mask, sc)
    b = oracle.tree_attention(q, k2, v2, [ctx], [n], tr.anc_mask, sc)
    assert np.allclose(a, b, atol=1e-14)


def test_dominant_key_returns_its_value():
    """One context key whose score exceeds every other by > 60 (natural log
    units) for every query: each output is that key's value row."""
    ctx, Hq, Hkv, D = 40, 4, 1, 128
    tr = _small_tree(ctx)
    n = int(tr.n_nodes[0])
    q, k, v = _rand_inputs(1, 24, Hq, Hkv, D, ctx + 24, 23)
    u = np.zeros(D)
    u[5] = 1.0
    qf = synth.bf16_bits_to_f32(q).astype(np.float64)
    qf[..., 5] = 4.0                                   # every query has a large component on u
    kf = synth.bf16_bits_to_f32(k).astype(np.float64)
    kf[0, 17, 0] = 256.0 * u                           # score 1024 / sqrt(128) ~ 90
    to_bits = lambda a: (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)
    q2, k2 = to_bits(qf), to_bits(kf)                  # all values exact in bf16 or truncated alike
    sc = 1 / math.sqrt(D)
    s = np.einsum("nhd,ld->nhl", synth.bf16_bits_to_f32(q2[0]).astype(np.float64),
                  synth.bf16_bits_to_f32(k2[0, :, 0]).astype(np.float64)) * sc
    assert np.all(s[..., 17] - np.delete(s, 17, axis=-1).max(-1) > 60)
    out = oracle.tree_attention(q2, k2, v, [ctx], [n], tr.anc_mask, sc).reshape(n, Hq, D)
    vrow = synth.bf16_bits_to_f32(v[0, 17, 0]).astype(np.float64)
    assert np.allclose(out, np.broadcast_to(vrow, out.shape), atol=1e-12)
