"""GPU parity: softmax + top-K marginals (C ABI) against the CPU oracle.

Bit-exact: kept tokens and logits.  lse and log q: within 2e-6 absolute (the
kernels sum exp in fp32 per thread, compensated, and take the log in fp64).
"""
import numpy as np
import pytest

import oracle
import synth
from gpuhelp import compare_topk, gpu_topk, host, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True, params=["stream", "cluster"])
def topk_path(request, monkeypatch):
    """Every case runs on both kernels: one CTA per row streaming the row
    (the default from two rows per SM) and a cluster of CTAs per row."""
    monkeypatch.setenv("BASTION_TOPK_PATH", request.param)
    return request.param


@pytest.mark.parametrize("cid", [1, 2, 3])
def test_topk_workloads(cuda_lib, cid):
    w = synth.workload(cid)
    x = synth.drafter_logits(w)
    g, st = gpu_topk(x, w.K)
    assert int(st.abs().sum()) == 0
    compare_topk(g, oracle.topk_marginals(x, w.K))


def test_topk_full_size_llama_vocab(cuda_lib):
    w = synth.workload(5)
    x = synth.drafter_logits(w)
    g, st = gpu_topk(x, w.K)
    assert int(st.abs().sum()) == 0
    compare_topk(g, oracle.topk_marginals(x, w.K))


@pytest.mark.parametrize("V,K,dtype", [(1023, 8, "f32"), (151937, 64, "bf16"), (1023, 1023, "bf16"),
                                       (5000, 1024, "f32"), (17, 3, "bf16"), (8, 8, "f32"),
                                       (151936, 1024, "bf16"), (40000, 200, "f32")])
def test_topk_ragged_vocab_and_large_k(cuda_lib, V, K, dtype):
    w = synth.Workload(91, "ragged", B=2, b=3, V=V, K=min(K, V), n_max=8, dtype=dtype, l_ar_ms=1.0,
                       cost="flat", drafter="spike-geometric", p_agree="uniform", seed=1234 + V)
    x = synth.drafter_logits(w)
    g, _ = gpu_topk(x, w.K)
    compare_topk(g, oracle.topk_marginals(x, w.K))


def test_topk_misaligned_row_stride(cuda_lib):
    """Rows at a stride that is not a multiple of 16 bytes (ld = V + 3)."""
    V, ld = 20001, 20004
    full = synth.host_array((2, 4, ld), "bf16")
    synth.fill_normal(full.ctypes.data, full.size, "bf16", 2.0, 77, 1)
    xd = to_dev(full)[:, :, :V]
    g, _ = gpu_topk(None, 16, x_dev=xd)
    compare_topk(g, oracle.topk_marginals(np.ascontiguousarray(full[:, :, :V]), 16))


def test_topk_all_equal_logits(cuda_lib):
    """Ties everywhere: the K lowest token ids, log q = -log V."""
    x = np.zeros((1, 4, 151936), np.uint16)
    g, _ = gpu_topk(x, 64)
    ref = oracle.topk_marginals(x, 64)
    compare_topk(g, ref)
    assert np.array_equal(host(g.tok)[0, 0], np.arange(64))


def test_topk_neg_inf_and_sparse_rows(cuda_lib):
    V = 30000
    x = np.full((1, 3, V), synth.f64_to_bf16_bits(-np.inf), np.uint16)
    x[0, 0, 123] = synth.f64_to_bf16_bits(1.0)
    x[0, 0, 29999] = synth.f64_to_bf16_bits(0.5)
    x[0, 1, ::7] = synth.f64_to_bf16_bits(2.0)
    x[0, 2, :] = synth.f64_to_bf16_bits(0.25)
    x[0, 2, 15000:] = synth.f64_to_bf16_bits(-np.inf)
    g, st = gpu_topk(x, 8)
    assert int(st[0]) == 0
    compare_topk(g, oracle.topk_marginals(x, 8))


def test_topk_nonfinite_sets_status(cuda_lib):
    from draft_tree_build_gb300 import bastion
    x = np.zeros((3, 2, 4096), np.float32)
    x[1, 1, 100] = np.nan
    x[2, 0, 7] = np.inf
    g, st = gpu_topk(x, 4)
    s = host(st)
    assert s[0] == 0
    assert s[1] & bastion.STATUS_NONFINITE and s[2] & bastion.STATUS_NONFINITE


def test_topk_deterministic(cuda_lib):
    w = synth.workload(3, B=8)
    x = synth.drafter_logits(w)
    xd = to_dev(x)
    a, _ = gpu_topk(None, w.K, x_dev=xd)
    b, _ = gpu_topk(None, w.K, x_dev=xd)
    for f in ("logq", "logit", "tok", "lse"):
        assert np.array_equal(host(getattr(a, f)), host(getattr(b, f)))


@pytest.mark.parametrize("V,dtype", [(151936, "f32"), (262144, "bf16"), (600000, "bf16"), (300000, "f32")])
def test_topk_wide_rows(cuda_lib, V, dtype):
    """Rows that need 16 slices per row, 16 vectors per thread, or the
    one-CTA-per-row exact path."""
    w = synth.Workload(92, "wide", B=1, b=3, V=V, K=64, n_max=8, dtype=dtype, l_ar_ms=1.0,
                       cost="flat", drafter="spike-geometric", p_agree="uniform", seed=4321 + V)
    x = synth.drafter_logits(w)
    g, st = gpu_topk(x, w.K)
    assert int(st.abs().sum()) == 0
    compare_topk(g, oracle.topk_marginals(x, w.K))


def test_topk_ascending_row_overflows_list(cuda_lib):
    """Logits increasing with the token id: the row threshold leaves more than
    the list holds, so the exact selection over the row takes over."""
    V = 151936
    x = np.empty((1, 2, V), np.float32)
    x[0, 0] = np.linspace(-8.0, 8.0, V, dtype=np.float32)
    x[0, 1] = x[0, 0][::-1]
    g, st = gpu_topk(x, 64)
    assert int(st[0]) == 0
    ref = oracle.topk_marginals(x, 64)
    compare_topk(g, ref)
    assert np.array_equal(host(g.tok)[0, 0], np.arange(V - 1, V - 65, -1))


def test_topk_ties_at_threshold(cuda_lib):
    """Many elements equal to the K-th value: lowest token ids win."""
    V = 65536
    x = np.full((1, 2, V), synth.f64_to_bf16_bits(-3.0), np.uint16)
    x[0, 0, ::97] = synth.f64_to_bf16_bits(1.0)   # 676 ties for 64 places
    x[0, 1, 5::1000] = synth.f64_to_bf16_bits(2.0)  # 66 distinct-position leaders
    x[0, 1, 7::1000] = synth.f64_to_bf16_bits(1.5)
    g, _ = gpu_topk(x, 64)
    compare_topk(g, oracle.topk_marginals(x, 64))
    assert np.array_equal(host(g.tok)[0, 0], np.arange(0, 97 * 64, 97))
