"""Pins for the oracle's fused drafter LM-head + top-K (no GPU).

One drafter forward pass yields the position-wise marginals q_k = softmax(l_k)
(Bastion, gist.science/nl/paper/2605.29727, "Methodologie" §1); with the
drafter's output embedding W [V, H] and final hidden states h_k, l_k = W h_k.
The oracle forms the logits with plain loops in fp64 and ranks them as the
top-K oracle does.  The pins below tie it to a library matmul, to the already
pinned top-K oracle (identity embedding), and to invariances and a closed form
of the product.
"""
import numpy as np
import pytest

import oracle
import synth


def _bf16(x):
    """float -> bf16 bits, round to nearest even (test input construction)."""
    b = np.ascontiguousarray(x, np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


def _inputs(rows, H, V, seed, dtype="bf16"):
    rng = np.random.default_rng(seed)
    h = rng.normal(size=(rows, H)) * (2.0 / np.sqrt(H))
    w = rng.normal(size=(V, H))
    if dtype == "bf16":
        return _bf16(h), _bf16(w)
    return h.astype(np.float32), w.astype(np.float32)


def _f64(a):
    return synth.bf16_bits_to_f32(a).astype(np.float64) if a.dtype == np.uint16 else a.astype(np.float64)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_logits_match_library_matmul(dtype):
    h, w = _inputs(6, 96, 500, 1, dtype)
    _, logits = oracle.lm_head_topk(h, w, 16)
    ref = _f64(h) @ _f64(w).T
    assert np.allclose(logits, ref, rtol=1e-13, atol=1e-13)


def test_identity_embedding_reduces_to_the_topk_oracle():
    """W = the first V rows of the identity: the logits are the hidden states
    themselves, so every output equals the top-K oracle's on h."""
    rows, H, V, K = 5, 300, 256, 32
    h, _ = _inputs(rows, H, V, 2)
    w = _bf16(np.eye(V, H))
    tk, _ = oracle.lm_head_topk(h, w, K)
    ref = oracle.topk_marginals(np.ascontiguousarray(h[:, :V]), K)
    assert np.array_equal(tk.tok, ref.tok)
    assert np.array_equal(tk.logit, ref.logit) and np.array_equal(tk.logq, ref.logq)
    assert np.array_equal(tk.lse, ref.lse)


def test_permuting_the_vocabulary_permutes_the_tokens():
    rows, H, V, K = 4, 64, 700, 20
    h, w = _inputs(rows, H, V, 3)
    perm = np.random.default_rng(0).permutation(V)   # row v of w becomes row perm[v]
    w2 = np.empty_like(w)
    w2[perm] = w
    a, _ = oracle.lm_head_topk(h, w, K)
    b, _ = oracle.lm_head_topk(h, w2, K)
    assert np.array_equal(b.tok, perm[a.tok])
    assert np.array_equal(a.logit, b.logit)
    assert np.allclose(a.lse, b.lse, rtol=0, atol=1e-12)


def test_powers_of_two_move_between_the_factors():
    """(2 h) . (w / 2) = h . w exactly: every output is bit-identical."""
    h, w = _inputs(3, 128, 400, 4, "f32")
    a, la = oracle.lm_head_topk(h, w, 8)
    b, lb = oracle.lm_head_topk(h * np.float32(2), w * np.float32(0.5), 8)
    assert np.array_equal(la, lb)
    assert np.array_equal(a.tok, b.tok) and np.array_equal(a.lse, b.lse)


def test_aligned_hidden_state_picks_its_row():
    """Unit-norm embedding rows and h = c w[v*]: by Cauchy-Schwarz v* has the
    largest logit, c |w[v*]|^2, and every other logit is c w[v] . w[v*] < that."""
    H, V, c = 64, 300, 9.0
    rng = np.random.default_rng(5)
    w = rng.normal(size=(V, H))
    w /= np.linalg.norm(w, axis=1, keepdims=True)
    w = w.astype(np.float32)
    vstar = 123
    h = (c * w[vstar].astype(np.float64)).astype(np.float32)[None]
    tk, logits = oracle.lm_head_topk(h, w, 5)
    assert tk.tok[0, 0] == vstar
    wv = w[vstar].astype(np.float64)
    assert logits[0, vstar] == pytest.approx(float(h[0].astype(np.float64) @ wv), rel=1e-15)
    assert np.all(np.delete(logits[0], vstar) < logits[0, vstar])


def test_bad_arguments():
    h, w = _inputs(2, 16, 10, 6)
    with pytest.raises(ValueError):
        oracle.lm_head_topk(h, w, 11)   # K > V
    with pytest.raises(TypeError):
        oracle.lm_head_topk(h.astype(np.float32), w, 4)
