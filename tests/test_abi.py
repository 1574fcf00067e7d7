"""The C ABI library loads and exports every symbol the header declares, and
rejects bad arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _header_functions():
    src = open(os.path.join(ROOT, "include", "bastion.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(bastion_\w+)\s*\(", src)


@pytest.fixture(scope="module")
def L():
    from draft_tree_build_gb300 import bastion
    return bastion.lib()


def test_exports_every_declared_symbol(L):
    from draft_tree_build_gb300 import bastion
    names = _header_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(bastion.SYMBOLS)


def _header_arg_counts():
    src = open(os.path.join(ROOT, "include", "bastion.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"\b(bastion_\w+)\s*\(([^)]*)\)\s*;", src):
        args = m.group(2).strip()
        out[m.group(1)] = 0 if args in ("", "void") else args.count(",") + 1
    return out


def test_binding_argtypes_match_header(L):
    counts = _header_arg_counts()
    assert len(counts) == 17
    for name, n in counts.items():
        assert len(getattr(L, name).argtypes) == n, name


def test_version_and_strings(L):
    assert L.bastion_version().startswith(b"bastion-gb300")
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 1, 2, 4, 8, 16, 32, 1 << 30):
        assert L.bastion_status_string(code) != b"unknown code"


def test_host_checks_reject_before_launch(L):
    vp = ctypes.c_void_p
    fake = vp(0x10000)  # never dereferenced: every call below fails a host check
    ws = vp(0x100000)
    # null pointers
    assert L.bastion_topk_marginals(None, 1, 1, 1, 8, 8, 1, None, fake, fake, fake, ws, 1 << 20, fake, None) == -1
    # bad dtype
    assert L.bastion_topk_marginals(fake, 7, 1, 1, 8, 8, 1, None, fake, fake, fake, ws, 1 << 20, fake, None) == -3
    # K > V, b > 32, ld < V
    assert L.bastion_topk_marginals(fake, 1, 1, 1, 8, 8, 9, None, fake, fake, fake, ws, 1 << 20, fake, None) == -2
    assert L.bastion_topk_marginals(fake, 1, 1, 33, 8, 8, 1, None, fake, fake, fake, ws, 1 << 20, fake, None) == -2
    assert L.bastion_topk_marginals(fake, 1, 1, 1, 8, 7, 1, None, fake, fake, fake, ws, 1 << 20, fake, None) == -2
    # misaligned logits / workspace
    assert L.bastion_topk_marginals(vp(0x10001), 1, 1, 1, 8, 8, 1, None, fake, fake, fake, ws, 1 << 20, fake, None) == -4
    assert L.bastion_topk_marginals(fake, 1, 1, 1, 8, 8, 1, None, fake, fake, fake, vp(0x100010), 1 << 20, fake, None) == -4
    # workspace too small
    assert L.bastion_topk_marginals(fake, 1, 1, 1, 8, 8, 1, None, fake, fake, fake, ws, 16, fake, None) == -5
    # tree: n_max > 256
    args = [fake] * 3 + [1, 4, 8, 257] + [fake] * 3 + [0, fake] + [fake] * 11 + [None]
    assert L.bastion_build_tree(*args) == -2
    # lm head: H not a multiple of 64 -> unsupported; K > 64 -> size; misaligned weight; small workspace
    lm = [fake, fake, 2, 4, 4096, 1000, 8, None, fake, fake, fake, ws, 1 << 24, fake, None]
    lm[4] = 4000
    assert L.bastion_lm_head_topk(*lm) == -6
    lm[4], lm[6] = 4096, 65
    assert L.bastion_lm_head_topk(*lm) == -2
    lm[6], lm[1] = 8, vp(0x10008)
    assert L.bastion_lm_head_topk(*lm) == -4
    lm[1], lm[12] = fake, 16
    assert L.bastion_lm_head_topk(*lm) == -5
    lm[12], lm[0] = 1 << 24, None
    assert L.bastion_lm_head_topk(*lm) == -1
    # attention: D != 128 -> unsupported; Hq % Hkv -> size
    base = [fake, fake, fake, 1, 16, 32, 8, 64, 256, fake, fake, fake, ctypes.c_float(0.1), fake, ws, 1 << 20, fake, None]
    assert L.bastion_tree_attention(*base) == -6
    base[6], base[7] = 5, 128
    assert L.bastion_tree_attention(*base) == -2
    # attention: a scale that is not finite and positive -> size; G = 3 -> unsupported
    base[6] = 8
    for bad in (0.0, -0.1, float("nan"), float("inf")):
        base[12] = ctypes.c_float(bad)
        assert L.bastion_tree_attention(*base) == -2
    base[12], base[5], base[6] = ctypes.c_float(0.1), 24, 8
    assert L.bastion_tree_attention(*base) == -6
    # mixture tree: Z > 32, K > 1024, b > 32, n_max > 256; misaligned pi; null pi
    mx = [fake] * 4 + [1, 33, 4, 8, 16] + [fake] * 3 + [0, fake] + [fake] * 9 + [ws, 1 << 30, fake, None]
    assert L.bastion_build_tree_mixture(*mx) == -2
    mx[5], mx[7] = 2, 1025
    assert L.bastion_build_tree_mixture(*mx) == -2
    mx[7], mx[6] = 8, 33
    assert L.bastion_build_tree_mixture(*mx) == -2
    mx[6], mx[8] = 4, 257
    assert L.bastion_build_tree_mixture(*mx) == -2
    mx[8], mx[3] = 16, vp(0x10004)
    assert L.bastion_build_tree_mixture(*mx) == -4
    mx[3] = None
    assert L.bastion_build_tree_mixture(*mx) == -1
    # mixture tree: workspace misaligned, too small, null
    mx[3] = fake
    mx[23] = vp(0x100010)
    assert L.bastion_build_tree_mixture(*mx) == -4
    mx[23], mx[24] = ws, L.bastion_build_tree_mixture_workspace_bytes(1, 2, 4, 8, 16) - 1
    assert L.bastion_build_tree_mixture(*mx) == -5
    mx[23], mx[24] = None, 1 << 30
    assert L.bastion_build_tree_mixture(*mx) == -1
    mx[23] = ws
    # the workspace size: per request, none for sizes out of range
    one = L.bastion_build_tree_mixture_workspace_bytes(1, 4, 16, 64, 128)
    assert one > 0 and one % 256 == 0
    assert L.bastion_build_tree_mixture_workspace_bytes(32, 4, 16, 64, 128) == 32 * one
    assert L.bastion_build_tree_mixture_workspace_bytes(1, 33, 16, 64, 128) == 0
    # mixture tree: tables larger than shared memory -> unsupported
    mx[5], mx[6], mx[7], mx[8] = 8, 32, 256, 256
    assert L.bastion_build_tree_mixture(*mx) == -6
    # verify: B > 4096
    assert L.bastion_verify_greedy(fake, 1, 5000, 4, 8, 8, 4, fake, fake, fake, fake, fake, fake, fake, ws, 1 << 20, fake, None) == -2
    # stochastic verify: temperature <= 0 or NaN; misaligned uniforms; null uniforms
    sv = [fake, 1, 2, 4, 8, 8, 4, ctypes.c_float(0.0), fake] + [fake] * 7 + [ws, 1 << 20, fake, None]
    assert L.bastion_verify_sample(*sv) == -2
    sv[7] = ctypes.c_float(float("nan"))
    assert L.bastion_verify_sample(*sv) == -2
    sv[7], sv[8] = ctypes.c_float(1.0), vp(0x10004)
    assert L.bastion_verify_sample(*sv) == -4
    sv[8] = None
    assert L.bastion_verify_sample(*sv) == -1
    sv[8] = fake
    sv[17] = 16
    assert L.bastion_verify_sample(*sv) == -5
    # calibration: no samples, n_max > 256, bw = 0, a NaN constant, misaligned table
    d = ctypes.c_double
    cal = [fake, fake, 8] + [d(1.0)] * 7 + [16, fake, fake, fake, None]
    assert L.bastion_calibrate_cost(*(cal[:2] + [0] + cal[3:])) == -2
    assert L.bastion_calibrate_cost(*(cal[:10] + [257] + cal[11:])) == -2
    assert L.bastion_calibrate_cost(*(cal[:7] + [d(0.0)] + cal[8:])) == -2
    assert L.bastion_calibrate_cost(*(cal[:3] + [d(float("nan"))] + cal[4:])) == -2
    assert L.bastion_calibrate_cost(*(cal[:11] + [vp(0x10002)] + cal[12:])) == -4
    assert L.bastion_calibrate_cost(*(cal[:12] + [None] + cal[13:])) == -1


def test_workspace_queries(L):
    assert L.bastion_topk_marginals_workspace_bytes(32, 16, 151936, 64) > 0
    assert L.bastion_topk_marginals_workspace_bytes(1, 1, 8, 9) == 0
    assert L.bastion_verify_greedy_workspace_bytes(32, 128, 151936) >= 32 * 128 * 8
    assert L.bastion_verify_sample_workspace_bytes(32, 128, 151936) >= 32 * 128 * (8 + 75 * 16)
    assert L.bastion_verify_sample_workspace_bytes(1, 257, 8) == 0
    assert L.bastion_tree_attention_workspace_bytes(8, 64, 32, 8, 128, 4160) > 0


def test_mixture_binding_rejects_wrong_dtypes_and_shapes(L):
    """The binding checks dtypes and shapes before the library reads the bytes
    (CPU tensors: the check fails before any pointer is passed)."""
    import torch
    from draft_tree_build_gb300 import bastion
    B, Z, b, K, n_max = 2, 3, 4, 8, 16
    lg = torch.zeros(B, Z, b, K)
    tk = torch.zeros(B, Z, b, K, dtype=torch.int32)
    ls = torch.zeros(B, Z, b, dtype=torch.float64)
    pi = torch.full((B, Z), 1.0 / Z, dtype=torch.float64)
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)  # noqa: E731
    f32 = lambda *s: torch.zeros(*s)  # noqa: E731
    rest = (n_max, i32(B), i32(B), f32(1, n_max + 1), f32(B), i32(B), i32(B, n_max), i32(B, n_max),
            i32(B, n_max), i32(B, n_max), f32(B, n_max), f32(B, n_max), f32(B, n_max),
            i32(B, n_max, 1), torch.zeros(1 << 20, dtype=torch.uint8), i32(B))
    with pytest.raises(bastion.BastionError, match="lse"):
        bastion.bastion_build_tree_mixture(lg, tk, ls.float(), pi, *rest)
    with pytest.raises(bastion.BastionError, match="pi"):
        bastion.bastion_build_tree_mixture(lg, tk, ls, pi.float(), *rest)
    with pytest.raises(bastion.BastionError, match="topk_tok"):
        bastion.bastion_build_tree_mixture(lg, tk.long(), ls, pi, *rest)
    with pytest.raises(bastion.BastionError, match="must match"):
        bastion.bastion_build_tree_mixture(lg, tk, ls[:, :, :2].contiguous(), pi, *rest)
    with pytest.raises(bastion.BastionError, match="cost_ms"):
        bastion.bastion_build_tree_mixture(lg, tk, ls, pi, n_max, i32(B), i32(B), f32(1, n_max), *rest[4:])
