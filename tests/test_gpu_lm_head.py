"""GPU parity: the fused drafter LM-head + top-K marginals (tcgen05 GEMM with
the top-K in its epilogue, C ABI) against the oracle, which forms the logits
W h in fp64 and ranks them exactly.

The GPU's logits are fp32 sums of the bf16 products accumulated on the tensor
cores, so each may differ from the exact one by the accumulation's rounding.
The library states the bound eps_v = 2^-16 sum_i |W[v,i] h[i]|; the test
checks, per row: every returned logit within eps of the exact logit of its
token; the ranking ordered by (returned logit desc, token asc); the returned
set a valid top K of the exact logits within 2 eps; the exact tokens wherever
the oracle's ranked logits are further apart than 2 eps from both neighbours;
lse within eps + 2e-6; log q = logit - lse."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, host, to_dev

pytestmark = pytest.mark.gpu

EPS_FRAC = 2.0 ** -16


@pytest.fixture(autouse=True, params=["1", "2", "4"])
def lm_cluster(request, monkeypatch):
    """Every case with the W tiles loaded per CTA, and multicast to clusters of
    two and four CTAs (where the M-tiles divide)."""
    monkeypatch.setenv("BASTION_LMHEAD_CLUSTER", request.param)
    return request.param


def _gpu(hidden, weight, K):
    from draft_tree_build_gb300 import bastion
    B, b, H = hidden.shape
    V = weight.shape[0]
    hd, wd = to_dev(hidden), to_dev(weight)
    t = bastion.alloc_topk(B, b, K, dev())
    ws = bastion.workspace(bastion.bastion_lm_head_topk_workspace_bytes(B, b, V, K), dev())
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    bastion.bastion_lm_head_topk(hd, wd, K, t.logq, t.logit, t.tok, t.lse, ws, st)
    torch.cuda.synchronize()
    return t, host(st)


def _check(t, hidden, weight, K, rows):
    """Compares the GPU's rows (flat indices into [B*b]) with the oracle's."""
    B, b, H = hidden.shape
    h2 = hidden.reshape(B * b, H)[rows]
    ref, logits = oracle.lm_head_topk(h2, weight, K)
    hf = synth.bf16_bits_to_f32(h2).astype(np.float64)
    wf = synth.bf16_bits_to_f32(weight).astype(np.float64)
    absdot = np.abs(hf) @ np.abs(wf).T           # [n, V]: sum_i |W[v,i] h[i]|
    g_tok = host(t.tok).reshape(B * b, K)[rows]
    g_lg = host(t.logit).reshape(B * b, K)[rows].astype(np.float64)
    g_lq = host(t.logq).reshape(B * b, K)[rows].astype(np.float64)
    g_lse = host(t.lse).reshape(B * b)[rows]
    worst = 0.0
    for q in range(len(rows)):
        ex = logits[q]
        eps = EPS_FRAC * absdot[q]
        emax = float(eps.max())
        err = np.abs(g_lg[q] - ex[g_tok[q]])
        worst = max(worst, float((err / absdot[q][g_tok[q]]).max()))
        assert np.all(err <= eps[g_tok[q]]), (q, err.max())
        # ordered by (returned logit desc, token asc)
        for i in range(K - 1):
            assert (g_lg[q, i] > g_lg[q, i + 1]) or (g_lg[q, i] == g_lg[q, i + 1] and g_tok[q, i] < g_tok[q, i + 1])
        # a valid top K of the exact logits within 2 eps
        kth = float(ref.logit[q, K - 1])
        assert np.all(ex[g_tok[q]] >= kth - 2 * emax)
        must = np.nonzero(ex > kth + 2 * emax)[0]
        assert set(must.tolist()) <= set(g_tok[q].tolist())
        # exact tokens where the oracle's neighbours are further than 2 eps
        rl = ref.logit[q].astype(np.float64)
        nxt = np.sort(ex)[::-1][K] if len(ex) > K else -np.inf
        for i in range(K):
            gap_up = rl[i - 1] - rl[i] if i > 0 else np.inf
            gap_dn = rl[i] - (rl[i + 1] if i + 1 < K else nxt)
            if gap_up > 2 * emax and gap_dn > 2 * emax:
                assert g_tok[q, i] == ref.tok[q, i], (q, i)
        assert abs(g_lse[q] - ref.lse[q]) <= emax + 2e-6, (q, g_lse[q] - ref.lse[q])
        assert np.all(np.abs(g_lq[q] - (g_lg[q] - g_lse[q])) <= 1e-5 + 1e-6 * np.abs(g_lq[q]))
    print(f"largest |logit error| / sum|w h|: {worst:.3e} (bound {EPS_FRAC:.3e})")
    return worst


@pytest.mark.parametrize("B,b,H,V,K", [
    (2, 5, 256, 5000, 16),      # one M-tile, 20 N-tiles, a ragged last tile
    (5, 26, 64, 1000, 64),      # 130 rows: two M-tiles, the second of 2 rows; one 64-column chunk
    (1, 3, 128, 64, 64),        # K = V: every token
    (3, 16, 1024, 32000, 8),    # more N-tiles than CTAs per M-tile
    (8, 16, 512, 151936, 64),   # the Qwen3 vocabulary, one M-tile
])
def test_lm_head_all_rows(cuda_lib, B, b, H, V, K):
    hidden, weight = synth.lm_head_inputs(B, b, H, V, seed=B * 1000 + H + V)
    t, st = _gpu(hidden, weight, K)
    assert np.all(st == 0)
    _check(t, hidden, weight, K, np.arange(B * b))


def test_lm_head_batched_workload_shape_sampled_rows(cuda_lib):
    """The batched workload's drafter: 32 requests x 16 positions, hidden size
    4096 (Qwen3-8B), vocabulary 151,936, top-64; rows from all four M-tiles
    and their edges compared with the oracle one by one."""
    B, b, H, V, K = 32, 16, 4096, 151936, 64
    hidden, weight = synth.lm_head_inputs(B, b, H, V, seed=4242)
    t, st = _gpu(hidden, weight, K)
    assert np.all(st == 0)
    _check(t, hidden, weight, K, np.array([0, 1, 127, 128, 255, 256, 300, 383, 384, 511]))


def test_lm_head_planted_rows(cuda_lib):
    """W rows equal to a hidden state (scaled) win that row: the planted token
    is rank 0 with the logit sum h_i^2 s (exact in fp32 here)."""
    B, b, H, V, K = 1, 4, 256, 3000, 8
    hidden, weight = synth.lm_head_inputs(B, b, H, V, seed=77)
    plant = [17, 2999, 1024, 512]
    for k, v in enumerate(plant):
        weight[v] = hidden[0, k]   # bf16 bits copied: W[v] = h_k
    t, st = _gpu(hidden, weight, K)
    assert np.all(host(t.tok)[0, :, 0] == np.array(plant))
    _check(t, hidden, weight, K, np.arange(B * b))


def test_lm_head_deterministic(cuda_lib):
    hidden, weight = synth.lm_head_inputs(2, 8, 512, 20000, seed=5)
    a, _ = _gpu(hidden, weight, 32)
    c, _ = _gpu(hidden, weight, 32)
    for f in ("logit", "tok", "lse", "logq"):
        assert np.array_equal(host(getattr(a, f)), host(getattr(c, f)))
