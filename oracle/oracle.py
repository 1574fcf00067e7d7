"""ctypes wrapper of the fp64 C++ oracle (``oracle.cpp``).  TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
use this module.  It marshals numpy arrays into the plain C functions; all of
the arithmetic is in ``oracle.cpp``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

ST_NONFINITE = 1
ST_EMPTY_ROW = 2
ST_BAD_COST = 4


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "oracle.cpp")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off",
                           "-fno-fast-math", src, "-o", tmp])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, dbl = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_topk_marginals.argtypes = [vp, i32, i32, i32, i64, i32, vp, vp, vp, vp, vp]
        L.oracle_topk_marginals.restype = i32
        L.oracle_lm_head_topk.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, vp]
        L.oracle_lm_head_topk.restype = i32
        L.oracle_build_tree_mixture.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp,
                                                i32, vp, vp, vp, vp] + [vp] * 10 + [vp, vp, vp]
        L.oracle_build_tree_mixture.restype = i32
        L.oracle_build_tree.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, i32, vp, i32,
                                        vp, vp, vp] + [vp] * 11 + [vp, vp, vp]
        L.oracle_build_tree.restype = i32
        L.oracle_verify_greedy.argtypes = [vp, i32, i32, i32, i32, i64, i32, vp, vp, vp,
                                           vp, vp, vp, vp, vp]
        L.oracle_verify_greedy.restype = i32
        L.oracle_verify_sample.argtypes = [vp, i32, i32, i32, i32, i64, i32, dbl, vp, vp, vp, vp,
                                           vp, vp, vp, vp, vp, vp]
        L.oracle_verify_sample.restype = i32
        L.oracle_calibrate_cost.argtypes = [vp, vp, i32] + [dbl] * 7 + [i32, vp, vp]
        L.oracle_calibrate_cost.restype = i32
        L.oracle_tree_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i64, vp, vp, vp,
                                            dbl, vp, i64, vp]
        L.oracle_tree_attention.restype = i64
        _lib = L
    return _lib


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return 0
    if a.dtype == np.uint16:
        return 1
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


@dataclass
class TopK:
    logq: np.ndarray      # float32 [..., K]  log q = l - lse, rounded once
    logit: np.ndarray     # float32 [..., K]  the K best logits as given
    tok: np.ndarray       # int32 [..., K]
    lse: np.ndarray       # float64 [...]
    status: np.ndarray    # int32 [...]


def topk_marginals(logits: np.ndarray, K: int) -> TopK:
    """logits [..., V] (float32 or bf16 bits as uint16), contiguous."""
    logits = np.ascontiguousarray(logits)
    lead, V = logits.shape[:-1], logits.shape[-1]
    rows = int(np.prod(lead)) if lead else 1
    logq = np.empty(lead + (K,), np.float32)
    logit = np.empty(lead + (K,), np.float32)
    tok = np.empty(lead + (K,), np.int32)
    lse = np.empty(lead, np.float64)
    st = np.empty(lead, np.int32)
    rc = lib().oracle_topk_marginals(_p(logits), _dtype_code(logits), rows, V, V, K, _p(logq),
                                     _p(logit), _p(tok), _p(lse), _p(st))
    if rc != 0:
        raise ValueError("oracle_topk_marginals: bad arguments")
    return TopK(logq, logit, tok, lse, st)


@dataclass
class MixTree:
    n_nodes: np.ndarray   # int32 [B]
    parent: np.ndarray    # int32 [B, n_max]
    depth: np.ndarray
    pos_id: np.ndarray
    token: np.ndarray
    log_rho: np.ndarray   # float64 [B, n_max]
    a_hat: np.ndarray
    speedup: np.ndarray
    anc_mask: np.ndarray  # uint32 [B, n_max, W]
    status: np.ndarray
    flagged_pops: int = 0
    flagged_stops: int = 0
    guided: int = 0


def build_tree_mixture(topk_logit, topk_tok, lse, pi, n_max: int, root_token, ctx_len, cost_ms,
                       l_ar, guide=None) -> MixTree:
    """Best-first tree on the latent-mixture path score.  topk_logit/tok
    [B, Z, b, K]; lse [B, Z, b] fp64; pi [B, Z] (rows summing to 1); cost_ms
    [Bc, n_max+1] (Bc = 1 or B); guide: optional (n_nodes, parent, token) of
    another implementation's tree, followed only at near-tie steps."""
    lg = np.ascontiguousarray(topk_logit, dtype=np.float32)
    tk = np.ascontiguousarray(topk_tok, dtype=np.int32)
    ls = np.ascontiguousarray(lse, dtype=np.float64)
    pz = np.ascontiguousarray(pi, dtype=np.float64)
    B, Z, b, K = lg.shape
    cost = np.ascontiguousarray(cost_ms, dtype=np.float32).reshape(-1, n_max + 1)
    W = (n_max + 31) // 32
    out = MixTree(np.zeros(B, np.int32), np.full((B, n_max), -1, np.int32),
                  np.zeros((B, n_max), np.int32), np.zeros((B, n_max), np.int32),
                  np.zeros((B, n_max), np.int32), np.zeros((B, n_max)), np.zeros((B, n_max)),
                  np.zeros((B, n_max)), np.zeros((B, n_max, W), np.uint32), np.zeros(B, np.int32))
    g = [None, None, None]
    if guide is not None:
        g = [np.ascontiguousarray(x, dtype=np.int32) for x in guide]
    fp, fs, gd = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    rc = lib().oracle_build_tree_mixture(
        _p(lg), _p(tk), _p(ls), _p(pz), B, Z, b, K, n_max,
        _p(np.ascontiguousarray(root_token, dtype=np.int32)),
        _p(np.ascontiguousarray(ctx_len, dtype=np.int32)), _p(cost), int(cost.shape[0] == B and B > 1),
        _p(np.ascontiguousarray(l_ar, dtype=np.float32)), _p(g[0]), _p(g[1]), _p(g[2]),
        _p(out.n_nodes), _p(out.parent),
        _p(out.depth), _p(out.pos_id), _p(out.token), _p(out.log_rho), _p(out.a_hat),
        _p(out.speedup), _p(out.anc_mask), _p(out.status), ctypes.byref(fp), ctypes.byref(fs),
        ctypes.byref(gd))
    if rc != 0:
        raise ValueError("oracle_build_tree_mixture: bad arguments")
    out.flagged_pops, out.flagged_stops, out.guided = fp.value, fs.value, gd.value
    return out


def lm_head_topk(hidden: np.ndarray, weight: np.ndarray, K: int):
    """Fused drafter LM-head + top-K: hidden [..., H] and weight [V, H], both
    float32 or bf16 bits (uint16).  Returns (TopK of the logits hidden . weight^T
    formed in fp64, the logits [..., V] in fp64)."""
    hidden = np.ascontiguousarray(hidden)
    weight = np.ascontiguousarray(weight)
    if hidden.dtype != weight.dtype:
        raise TypeError("hidden and weight must share a dtype")
    lead, H = hidden.shape[:-1], hidden.shape[-1]
    V = weight.shape[0]
    if weight.shape != (V, H):
        raise ValueError("weight must be [V, H]")
    rows = int(np.prod(lead)) if lead else 1
    logq = np.empty(lead + (K,), np.float32)
    logit = np.empty(lead + (K,), np.float32)
    tok = np.empty(lead + (K,), np.int32)
    lse = np.empty(lead, np.float64)
    st = np.empty(lead, np.int32)
    logits = np.empty(lead + (V,), np.float64)
    rc = lib().oracle_lm_head_topk(_p(hidden), _p(weight), _dtype_code(hidden), rows, H, V, K,
                                   _p(logq), _p(logit), _p(tok), _p(lse), _p(logits), _p(st))
    if rc != 0:
        raise ValueError("oracle_lm_head_topk: bad arguments")
    return TopK(logq, logit, tok, lse, st), logits


@dataclass
class Tree:
    n_nodes: np.ndarray   # int32 [B]
    parent: np.ndarray    # int32 [B, n_max]
    depth: np.ndarray
    pos_id: np.ndarray
    token: np.ndarray
    rank: np.ndarray
    log_rho: np.ndarray   # float64 [B, n_max]
    a_hat: np.ndarray
    speedup: np.ndarray
    anc_mask: np.ndarray  # uint32 [B, n_max, W]
    status: np.ndarray
    flagged_pops: int
    flagged_stops: int
    guided: int


def build_tree(topk_logit, topk_tok, lse, n_max: int, root_token, ctx_len, cost_ms, l_ar,
               root_counts: bool = True, guide=None) -> Tree:
    """topk_logit/tok [B, b, K]; lse [B, b] fp64; cost_ms [Bc, n_max+1] (Bc = 1 or B);
    guide: optional (n_nodes, parent, rank) of another implementation's tree,
    followed only at near-tie steps."""
    lg = np.ascontiguousarray(topk_logit, dtype=np.float32)
    tk = np.ascontiguousarray(topk_tok, dtype=np.int32)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    B, b, K = lg.shape
    W = (n_max + 31) // 32
    root_token = np.ascontiguousarray(root_token, dtype=np.int32)
    ctx_len = np.ascontiguousarray(ctx_len, dtype=np.int32)
    cost = np.ascontiguousarray(cost_ms, dtype=np.float32).reshape(-1, n_max + 1)
    per_req = 1 if cost.shape[0] == B and B > 1 else 0
    l_ar = np.ascontiguousarray(l_ar, dtype=np.float32)
    out_i = {k: np.full((B, n_max), -7, np.int32) for k in ("parent", "depth", "pos_id", "token", "rank")}
    out_d = {k: np.full((B, n_max), np.nan) for k in ("log_rho", "a_hat", "speedup")}
    mask = np.zeros((B, n_max, W), np.uint32)
    n_nodes = np.zeros(B, np.int32)
    st = np.zeros(B, np.int32)
    fp, fs, gd = ctypes.c_int32(0), ctypes.c_int32(0), ctypes.c_int32(0)
    g = [None, None, None]
    if guide is not None:
        g = [np.ascontiguousarray(x, dtype=np.int32) for x in guide]
    rc = lib().oracle_build_tree(
        _p(lg), _p(tk), _p(lse), B, b, K, n_max, _p(root_token), _p(ctx_len), _p(cost), per_req, _p(l_ar),
        1 if root_counts else 0, _p(g[0]), _p(g[1]), _p(g[2]),
        _p(n_nodes), _p(out_i["parent"]), _p(out_i["depth"]), _p(out_i["pos_id"]),
        _p(out_i["token"]), _p(out_i["rank"]), _p(out_d["log_rho"]), _p(out_d["a_hat"]),
        _p(out_d["speedup"]), _p(mask), _p(st), ctypes.byref(fp), ctypes.byref(fs),
        ctypes.byref(gd))
    if rc != 0:
        raise ValueError("oracle_build_tree: bad arguments")
    return Tree(n_nodes, out_i["parent"], out_i["depth"], out_i["pos_id"], out_i["token"],
                out_i["rank"], out_d["log_rho"], out_d["a_hat"], out_d["speedup"], mask, st,
                fp.value, fs.value, gd.value)


@dataclass
class Verify:
    argmax: np.ndarray        # int32 [B, n_max] (-1 past n_nodes)
    accept_len: np.ndarray    # int32 [B]
    accept_nodes: np.ndarray  # int32 [B, b+1]
    out_tokens: np.ndarray    # int32 [B, b+1]
    status: np.ndarray


def verify_greedy(target: np.ndarray, b: int, n_nodes, parent, token) -> Verify:
    """target [B, n_max, V] (float32 or bf16 bits); tree arrays [B, n_max]."""
    target = np.ascontiguousarray(target)
    B, n_max, V = target.shape
    n_nodes = np.ascontiguousarray(n_nodes, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    token = np.ascontiguousarray(token, dtype=np.int32)
    am = np.full((B, n_max), -1, np.int32)
    al = np.zeros(B, np.int32)
    an = np.zeros((B, b + 1), np.int32)
    ot = np.zeros((B, b + 1), np.int32)
    st = np.zeros(B, np.int32)
    rc = lib().oracle_verify_greedy(_p(target), _dtype_code(target), B, n_max, V, V, b,
                                    _p(n_nodes), _p(parent), _p(token), _p(am), _p(al), _p(an),
                                    _p(ot), _p(st))
    if rc != 0:
        raise ValueError("oracle_verify_greedy: bad arguments")
    return Verify(am, al, an, ot, st)


@dataclass
class VerifySample:
    sampled: np.ndarray       # int32 [B, n_max] the token drawn at each node (-1 past n_nodes)
    margin: np.ndarray        # float64 [B, n_max] distance of the draw to a neighbouring interval / S
    accept_len: np.ndarray    # int32 [B]
    accept_nodes: np.ndarray  # int32 [B, b+1]
    out_tokens: np.ndarray    # int32 [B, b+1]
    status: np.ndarray


def verify_sample(target: np.ndarray, b: int, T: float, u, n_nodes, parent, token) -> VerifySample:
    """Stochastic verification at temperature T with the uniforms u [B, n_max]
    (float64 in [0, 1)); target [B, n_max, V] (float32 or bf16 bits)."""
    target = np.ascontiguousarray(target)
    B, n_max, V = target.shape
    u = np.ascontiguousarray(u, dtype=np.float64).reshape(B, n_max)
    n_nodes = np.ascontiguousarray(n_nodes, dtype=np.int32)
    parent = np.ascontiguousarray(parent, dtype=np.int32)
    token = np.ascontiguousarray(token, dtype=np.int32)
    sm = np.full((B, n_max), -1, np.int32)
    mg = np.zeros((B, n_max), np.float64)
    al = np.zeros(B, np.int32)
    an = np.zeros((B, b + 1), np.int32)
    ot = np.zeros((B, b + 1), np.int32)
    st = np.zeros(B, np.int32)
    rc = lib().oracle_verify_sample(_p(target), _dtype_code(target), B, n_max, V, V, b, float(T),
                                    _p(u), _p(n_nodes), _p(parent), _p(token), _p(sm), _p(mg), _p(al),
                                    _p(an), _p(ot), _p(st))
    if rc != 0:
        raise ValueError("oracle_verify_sample: bad arguments")
    return VerifySample(sm, mg, al, an, ot, st)


def calibrate_cost(sample_n, sample_ms, roofline: dict, t_draft: float, n_max: int):
    """Least-squares calibration of T_verify = alpha roof(N) + beta; returns
    (cost table C(0..n_max) float64, alpha, beta).  roofline holds bytes0,
    bytes1, flops0, flops1, bw, peak (any consistent units giving ms)."""
    n = np.ascontiguousarray(sample_n, dtype=np.float64)
    t = np.ascontiguousarray(sample_ms, dtype=np.float64)
    cost = np.zeros(n_max + 1, np.float64)
    par = np.zeros(2, np.float64)
    r = roofline
    rc = lib().oracle_calibrate_cost(_p(n), _p(t), len(n), r["bytes0"], r["bytes1"], r["flops0"],
                                     r["flops1"], r["bw"], r["peak"], float(t_draft), n_max, _p(cost),
                                     _p(par))
    if rc != 0:
        raise ValueError("oracle_calibrate_cost: bad arguments")
    return cost, float(par[0]), float(par[1])


def tree_attention(q, k, v, ctx_len, n_nodes, anc_mask, scale: float, sel=None) -> np.ndarray:
    """q [B, n_max, Hq, D], k/v [B, L_cap, Hkv, D] as bf16 bits (uint16).
    Returns fp64 [n_rows, D] for the selected (r, i, h) triples, or for every
    (r, i < n_nodes[r], h) in that order when sel is None."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    B, n_max, Hq, D = q.shape
    L_cap, Hkv = k.shape[1], k.shape[2]
    ctx_len = np.ascontiguousarray(ctx_len, dtype=np.int32)
    n_nodes = np.ascontiguousarray(n_nodes, dtype=np.int32)
    anc_mask = np.ascontiguousarray(anc_mask, dtype=np.uint32)
    if sel is not None:
        sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 3)
        n_out = sel.shape[0]
    else:
        n_out = int(n_nodes.sum()) * Hq
    out = np.zeros((n_out, D), np.float64)
    cnt = lib().oracle_tree_attention(_p(q), _p(k), _p(v), B, n_max, Hq, Hkv, D, L_cap,
                                      _p(ctx_len), _p(n_nodes), _p(anc_mask), float(scale),
                                      _p(sel), 0 if sel is None else sel.shape[0], _p(out))
    if cnt < 0:
        raise ValueError("oracle_tree_attention: bad arguments")
    return out
