"""Pins for the oracle's stochastic verification (no GPU).

The pages evaluate greedy decoding only (Bastion, gist.science/nl/paper/
2605.29727, "Experimentele Resultaten"); the reading for temperature T > 0 is
the plainest lossless one: each node's token is a draw from softmax(l / T) by
inverse transform with the caller's uniform, and the walk is the greedy walk
with the drawn tokens.  The pins below check the draw against the definition of
the distribution (counts of a uniform grid of draws), its limits, and the walk
against the greedy oracle.
"""
import numpy as np
import pytest

import oracle
import synth


def _draws(row, T, us, dtype="f32"):
    """Draw once per uniform from one logit row (float64 values given)."""
    n = len(us)
    if dtype == "f32":
        tgt = np.broadcast_to(np.asarray(row, np.float32), (1, n, len(row))).copy()
    else:
        bits = np.array([synth.f64_to_bf16_bits(v) for v in row], np.uint16)
        tgt = np.broadcast_to(bits, (1, n, len(row))).copy()
    par = np.full((1, n), -1, np.int32)
    tok = np.full((1, n), -1, np.int32)
    return oracle.verify_sample(tgt, 1, T, np.asarray(us, np.float64).reshape(1, n), [n], par, tok)


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_grid_of_uniforms_draws_the_softmax(T, dtype):
    """With u on a uniform grid of N points, each token is drawn for a fraction
    of the grid within 1/N of its softmax probability."""
    row = [1.5, -2.0, 0.25, -np.inf, 3.0, 0.0, -0.75, 3.0]
    N = 4000
    r = _draws(row, T, (np.arange(N) + 0.5) / N, dtype)
    x = np.array(row, np.float64)
    p = np.exp((x - x[np.isfinite(x)].max()) / T)
    p[~np.isfinite(x)] = 0.0
    p /= p.sum()
    freq = np.bincount(r.sampled[0], minlength=len(row)) / N
    assert np.all(np.abs(freq - p) <= 1.0 / N + 1e-12), (freq, p)
    assert freq[3] == 0.0  # a -inf logit is never drawn
    assert np.all(r.margin[0] >= 0.0) and np.all(r.margin[0] <= 0.5)


def test_extreme_uniforms_and_empty_rows():
    row = [-np.inf, 0.5, -1.0, 2.0, -np.inf]
    r = _draws(row, 1.0, [0.0, np.nextafter(1.0, 0.0)])
    assert r.sampled[0, 0] == 1      # u = 0: the first token with weight
    assert r.sampled[0, 1] == 3      # u -> 1: the last token with weight
    r = _draws([-np.inf] * 6, 1.0, [0.3])
    assert r.status[0] & 2 and r.sampled[0, 0] == 0
    r = _draws([0.0, np.nan, 1.0], 1.0, [0.3])
    assert r.status[0] & 1


def test_temperature_scales_the_logits():
    """Sampling l at T = 2 equals sampling l / 2 at T = 1 (exact halves)."""
    rng = np.random.default_rng(5)
    row = (rng.normal(size=257) * 4).astype(np.float32)
    us = rng.random(300)
    a = _draws(row, 2.0, us)
    b = _draws(row / 2, 1.0, us)
    assert np.array_equal(a.sampled, b.sampled)


@pytest.mark.parametrize("cid", [1, 3])
def test_low_temperature_is_the_greedy_walk(cid):
    """As T -> 0 every draw is the argmax (unique maxima: planted), and the
    walk, accepted nodes and bonus are the greedy oracle's."""
    w = synth.workload(cid, **({"B": 3} if cid == 3 else {}))
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w),
                           synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    g = oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    u = np.random.default_rng(11).random((w.B, w.n_max))
    s = oracle.verify_sample(tgt, w.b, 1e-3, u, tr.n_nodes, tr.parent, tr.token)
    for r in range(w.B):
        n = tr.n_nodes[r]
        assert np.array_equal(s.sampled[r, :n], g.argmax[r, :n])
    assert np.array_equal(s.accept_len, g.accept_len)
    assert np.array_equal(s.accept_nodes, g.accept_nodes)
    assert np.array_equal(s.out_tokens, g.out_tokens)


def test_walk_follows_the_draws():
    """A hand-built tree: root 0 with children tokens 5 (node 1) and 7 (node 2);
    node 1 has a child token 9 (node 3).  The draws at nodes 0 and 1 are forced
    by one-hot rows; the walk accepts 5 then 9 and emits node 3's draw."""
    V, n = 16, 4
    tgt = np.full((1, n, V), -np.inf, np.float32)
    tgt[0, 0, 5] = 0.0
    tgt[0, 1, 9] = 0.0
    tgt[0, 2, 2] = 0.0
    tgt[0, 3, [1, 4]] = 0.0   # node 3: two equal tokens, u picks the second
    par = np.array([[-1, 0, 0, 1]], np.int32)
    tok = np.array([[-1, 5, 7, 9]], np.int32)
    u = np.array([[0.5, 0.5, 0.5, 0.75]])
    s = oracle.verify_sample(tgt, 3, 1.0, u, [n], par, tok)
    assert list(s.sampled[0]) == [5, 9, 2, 4]
    assert s.accept_len[0] == 2
    assert list(s.accept_nodes[0]) == [0, 1, 3, -1]
    assert list(s.out_tokens[0]) == [5, 9, 4, -1]
