"""The non-allocating greedy-verify entry point, for callers that cannot
allocate device memory (it uses a fixed scratch array inside the library).

Called through the C ABI twice in a row on different inputs; each result must
equal what the workspace-taking entry point returns for the same inputs, and
what the CPU oracle returns (integers, so exactly).  This file is named to be
collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpuhelp import dev, gpu_verify, host, to_dev, workload_inputs

pytestmark = pytest.mark.gpu


def _inputs(cid, **over):
    w = synth.workload(cid, **over)
    x = synth.drafter_logits(w)
    tk = oracle.topk_marginals(x, w.K)
    roots, ctx, cost, lar = workload_inputs(w)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots, ctx, cost, lar)
    tgt, _ = synth.target_logits(w, tr.n_nodes, tr.depth, tk.tok)
    vf = oracle.verify_greedy(tgt, w.b, tr.n_nodes, tr.parent, tr.token)
    return w, tr, tgt, vf


def _noalloc(L, td, b, nn, pa, tk):
    B, n_max, V = td.shape
    out = [torch.full((B, n_max), -7, dtype=torch.int32, device=dev()),
           torch.zeros(B, dtype=torch.int32, device=dev()),
           torch.zeros(B, b + 1, dtype=torch.int32, device=dev()),
           torch.zeros(B, b + 1, dtype=torch.int32, device=dev())]
    st = torch.zeros(B, dtype=torch.int32, device=dev())
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    dtype = 1 if td.dtype == torch.bfloat16 else 0
    rc = L.bastion_verify_greedy_noalloc(p(td), dtype, B, n_max, V, td.stride(1), b, p(nn), p(pa), p(tk),
                                         p(out[0]), p(out[1]), p(out[2]), p(out[3]), p(st),
                                         ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert rc == 0, rc
    return out, st


def test_noalloc_matches_workspace_entry_point_twice(cuda_lib):
    L = cuda_lib.lib()
    cases = [_inputs(3), _inputs(1), _inputs(2, B=3, seed=99)]
    for w, tr, tgt, vf in cases:
        td = to_dev(tgt)
        nn, pa, tk = (to_dev(np.ascontiguousarray(a, np.int32)) for a in (tr.n_nodes, tr.parent, tr.token))
        ref, st_ref = gpu_verify(None, w.b, nn, pa, tk, target_dev=td)
        got, st = _noalloc(L, td, w.b, nn, pa, tk)
        assert np.array_equal(host(st), host(st_ref))
        for i in range(w.B):
            n = int(tr.n_nodes[i])
            assert np.array_equal(host(got[0])[i, :n], host(ref.argmax)[i, :n])
            assert np.array_equal(host(got[0])[i, :n], vf.argmax[i, :n])
        assert np.array_equal(host(got[1]), host(ref.accept_len))
        assert np.array_equal(host(got[2]), host(ref.accept_nodes))
        assert np.array_equal(host(got[3]), host(ref.out_tokens))
        # and the CPU oracle's walk
        assert np.array_equal(host(got[1]), vf.accept_len)
        assert np.array_equal(host(got[2]), vf.accept_nodes)
        assert np.array_equal(host(got[3]), vf.out_tokens)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    L = cuda_lib.lib()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check fails first
    # 128 requests x 256 nodes = 32768 rows > 16384
    rc = L.bastion_verify_greedy_noalloc(fake, 1, 128, 256, 1000, 1000, 4, fake, fake, fake, fake, fake,
                                         fake, fake, fake, None)
    assert rc == -2
