"""Pins for the oracle's softmax + top-K marginals (no GPU).

The marginals q_k are the block-diffusion drafter's position-wise distributions
(Bastion, gist.science/nl/paper/2605.29727, Methodologie §1); q_k = softmax(l_k).
"""
import math

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
import synth


def _f(x):
    return synth.bf16_bits_to_f32(x) if x.dtype == np.uint16 else x


def test_lse_matches_library_logsumexp():
    w = synth.workload(1)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    ref = logsumexp(x.astype(np.float64), axis=-1)
    assert np.allclose(tk.lse, ref, rtol=0, atol=1e-12)
    rng = np.random.default_rng(5)
    y = (rng.normal(size=(6, 300)) * 5).astype(np.float32)
    y[2, ::3] = -np.inf
    tk = oracle.topk_marginals(y, 10)
    assert np.allclose(tk.lse, logsumexp(y.astype(np.float64), axis=-1), rtol=0, atol=1e-12)


def test_ranks_match_library_sort():
    w = synth.workload(2)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    f = _f(x)[0]
    for k in range(w.b):
        order = np.lexsort((np.arange(w.V), -f[k].astype(np.float64)))[: w.K]
        assert np.array_equal(tk.tok[0, k], order)
        assert np.array_equal(tk.logit[0, k], f[k][order])
        assert np.allclose(tk.logq[0, k], (f[k][order] - tk.lse[0, k]).astype(np.float32), rtol=0, atol=0)


def test_bf16_ties_rank_by_lowest_token():
    x = np.full((1, 64), synth.f64_to_bf16_bits(1.5), np.uint16)
    x[0, 40] = synth.f64_to_bf16_bits(2.0)
    tk = oracle.topk_marginals(x, 8)
    assert tk.tok[0].tolist() == [40, 0, 1, 2, 3, 4, 5, 6]


def test_uniform_logits_closed_form():
    V = 1000
    x = np.zeros((3, V), np.float32)
    tk = oracle.topk_marginals(x, 5)
    assert np.allclose(tk.lse, math.log(V), atol=1e-13)
    assert np.all(tk.tok == np.arange(5))
    assert np.allclose(tk.logq, np.float32(-math.log(V)))


def test_cat_dog_marginal():
    # The pages' branching example: next word 'kat' with 80%, 'hond' with 20%
    # (Bastion, analogy part, "De Boom van Mogelijkheden").
    x = np.array([[math.log(0.8), math.log(0.2), -np.inf, -np.inf]], np.float32)
    tk = oracle.topk_marginals(x, 2)
    assert tk.tok[0].tolist() == [0, 1]
    assert np.allclose(np.exp(tk.logq[0]), [0.8, 0.2], rtol=1e-6)


def test_planted_top1_probability_closed_form():
    """The spike logit is set from the lognormal mean E[exp(2z)] = e^2, so the
    top-1 probability must come back near the planted p_k = 0.95 - 0.04k.
    Sum of V-1 lognormals has relative std sqrt(e^4-1)/sqrt(V-1) ~ 1.9%; the bf16
    rounding of a logit near 17 moves the odds by at most 2^-4 in log."""
    w = synth.workload(2)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    q1 = np.exp(tk.logq[0, :, 0].astype(np.float64))
    p = 0.95 - 0.04 * np.arange(w.b)
    lodds_err = np.abs(np.log(q1 / (1 - q1)) - np.log(p / (1 - p)))
    bound = 2 ** -4 + 5 * math.sqrt(math.e ** 4 - 1) / math.sqrt(w.V - 1)
    assert np.all(lodds_err < bound), lodds_err
    assert np.all(tk.tok[0, :, 0] == synth.spike_positions(w)[0])


def test_probabilities_sum_to_one():
    w = synth.workload(1)
    x = synth.drafter_logits(w).astype(np.float64)
    tk = oracle.topk_marginals(x.astype(np.float32), w.K)
    q = softmax(x, axis=-1)
    assert np.allclose(q.sum(-1), 1.0, atol=1e-12)
    # top-K log q agree with the library softmax
    for k in range(w.b):
        assert np.allclose(np.exp(tk.logq[0, k].astype(np.float64)), q[0, k][tk.tok[0, k]], rtol=2e-7)


def test_neg_inf_ranked_last_and_status():
    y = np.array([[-np.inf, 1.0, -np.inf, 0.5, -np.inf]], np.float32)
    tk = oracle.topk_marginals(y, 4)
    assert tk.tok[0].tolist() == [1, 3, 0, 2]
    assert np.isneginf(tk.logq[0, 2:]).all()
    assert tk.status[0] == 0
    y2 = np.array([[0.0, np.nan, 1.0], [0.0, np.inf, 1.0], [-np.inf, -np.inf, -np.inf]], np.float32)
    tk2 = oracle.topk_marginals(y2, 2)
    assert tk2.status[0] & oracle.ST_NONFINITE
    assert tk2.status[1] & oracle.ST_NONFINITE
    assert tk2.status[2] & oracle.ST_EMPTY_ROW


def test_bad_arguments_rejected():
    with pytest.raises(ValueError):
        oracle.topk_marginals(np.zeros((1, 4), np.float32), 5)
