"""Python binding of the C ABI in ``include/bastion.h`` (ctypes; argument
marshalling only).  Every function takes CUDA tensors, passes their device
pointers and the current stream to ``libbastion.so``, and raises on a negative
return code.  All computation happens in the library's kernels; there is no
fallback path: if the library cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import _build

BASTION_F32 = 0
BASTION_BF16 = 1

STATUS_NONFINITE = 1
STATUS_EMPTY_ROW = 2
STATUS_BAD_COST = 4
STATUS_KV_OVERFLOW = 8
STATUS_BAD_TREE = 16
STATUS_BAD_WEIGHT = 32
STATUS_TIMEOUT = 1 << 30

# the exported C symbols, in header order
SYMBOLS = (
    "bastion_version", "bastion_status_string",
    "bastion_topk_marginals_workspace_bytes", "bastion_topk_marginals",
    "bastion_lm_head_topk_workspace_bytes", "bastion_lm_head_topk",
    "bastion_build_tree", "bastion_build_tree_mixture_workspace_bytes", "bastion_build_tree_mixture",
    "bastion_calibrate_cost",
    "bastion_tree_attention_workspace_bytes", "bastion_tree_attention",
    "bastion_verify_greedy_workspace_bytes", "bastion_verify_greedy",
    "bastion_verify_sample_workspace_bytes", "bastion_verify_sample",
    "bastion_verify_greedy_noalloc",
)


class BastionError(RuntimeError):
    pass


_lib = None


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True):
    """Load libbastion.so (building it in-tree first if it is missing or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    if build_if_missing and not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise BastionError(f"libbastion.so not found at {_build.LIB}; run __graft_entry__.build()")
    L = ctypes.CDLL(_build.LIB)
    vp, i32, i64, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    L.bastion_version.restype = ctypes.c_char_p
    L.bastion_version.argtypes = []
    L.bastion_status_string.restype = ctypes.c_char_p
    L.bastion_status_string.argtypes = [i32]
    L.bastion_topk_marginals_workspace_bytes.restype = sz
    L.bastion_topk_marginals_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.bastion_topk_marginals.restype = i32
    L.bastion_topk_marginals.argtypes = [vp, i32, i32, i32, i32, i64, i32, vp, vp, vp, vp, vp, sz, vp, vp]
    L.bastion_lm_head_topk_workspace_bytes.restype = sz
    L.bastion_lm_head_topk_workspace_bytes.argtypes = [i32, i32, i32, i32]
    L.bastion_lm_head_topk.restype = i32
    L.bastion_lm_head_topk.argtypes = [vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, vp, vp, sz, vp, vp]
    L.bastion_build_tree.restype = i32
    L.bastion_build_tree.argtypes = [vp, vp, vp, i32, i32, i32, i32, vp, vp, vp, i32, vp] + [vp] * 11 + [vp]
    L.bastion_build_tree_mixture_workspace_bytes.restype = sz
    L.bastion_build_tree_mixture_workspace_bytes.argtypes = [i32, i32, i32, i32, i32]
    L.bastion_build_tree_mixture.restype = i32
    L.bastion_build_tree_mixture.argtypes = [vp, vp, vp, vp, i32, i32, i32, i32, i32, vp, vp, vp, i32,
                                             vp] + [vp] * 9 + [vp, sz, vp, vp]
    L.bastion_calibrate_cost.restype = i32
    L.bastion_calibrate_cost.argtypes = [vp, vp, i32] + [ctypes.c_double] * 7 + [i32, vp, vp, vp, vp]
    L.bastion_tree_attention_workspace_bytes.restype = sz
    L.bastion_tree_attention_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i64]
    L.bastion_tree_attention.restype = i32
    L.bastion_tree_attention.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i64, vp, vp, vp, f32,
                                         vp, vp, sz, vp, vp]
    L.bastion_verify_greedy_workspace_bytes.restype = sz
    L.bastion_verify_greedy_workspace_bytes.argtypes = [i32, i32, i32]
    L.bastion_verify_greedy.restype = i32
    L.bastion_verify_greedy.argtypes = [vp, i32, i32, i32, i32, i64, i32, vp, vp, vp, vp, vp, vp, vp,
                                        vp, sz, vp, vp]
    L.bastion_verify_sample_workspace_bytes.restype = sz
    L.bastion_verify_sample_workspace_bytes.argtypes = [i32, i32, i32]
    L.bastion_verify_sample.restype = i32
    L.bastion_verify_sample.argtypes = [vp, i32, i32, i32, i32, i64, i32, f32, vp, vp, vp, vp, vp, vp,
                                        vp, vp, vp, sz, vp, vp]
    L.bastion_verify_greedy_noalloc.restype = i32
    L.bastion_verify_greedy_noalloc.argtypes = [vp, i32, i32, i32, i32, i64, i32, vp, vp, vp, vp, vp,
                                                vp, vp, vp, vp]
    _lib = L
    return L


def _p(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise BastionError("tensor must live on a CUDA device")
    return ctypes.c_void_p(t.data_ptr())


def _p_rows(t):
    """Target logits: a device tensor, or a pinned (page-locked) host tensor, which
    the verify kernels read in place over the host link (only the rows of the
    tree's nodes cross it)."""
    if t.is_cuda or (t.device.type == "cpu" and t.is_pinned()):
        return ctypes.c_void_p(t.data_ptr())
    raise BastionError("target logits must live on a CUDA device or in pinned host memory")


def _s(stream):
    st = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(st.cuda_stream)


def _dtype(t) -> int:
    if t.dtype == torch.float32:
        return BASTION_F32
    if t.dtype == torch.bfloat16:
        return BASTION_BF16
    raise BastionError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _check(rc: int, name: str):
    if rc != 0:
        raise BastionError(f"{name}: {bastion_status_string(rc)} ({rc})")


def _rows_view(x, dims):
    """Row stride (elements) of a [B, n, V] tensor whose last dim is contiguous and
    whose B*n rows are evenly strided."""
    if x.dim() != dims:
        raise BastionError(f"expected {dims} dims, got {tuple(x.shape)}")
    if x.stride(-1) != 1:
        raise BastionError("last dimension must be contiguous")
    ld = x.stride(-2)
    if x.shape[0] > 1 and x.stride(0) != ld * x.shape[1]:
        raise BastionError("rows must be evenly strided")
    return ld


# --------------------------------------------------------------------------- C ABI mirrors

def bastion_version() -> str:
    return lib().bastion_version().decode()


def bastion_status_string(code: int) -> str:
    return lib().bastion_status_string(int(code)).decode()


def bastion_topk_marginals_workspace_bytes(B: int, b: int, V: int, K: int) -> int:
    return int(lib().bastion_topk_marginals_workspace_bytes(B, b, V, K))


def bastion_topk_marginals(logits, K, topk_logq, topk_logit, topk_tok, lse, workspace, status,
                           stream=None):
    """logits [B, b, V] (fp32/bf16, last dim contiguous); outputs [B, b, K] / [B, b]."""
    B, b, V = logits.shape
    ld = _rows_view(logits, 3)
    rc = lib().bastion_topk_marginals(_p(logits), _dtype(logits), B, b, V, ld, int(K), _p(topk_logq),
                                      _p(topk_logit), _p(topk_tok), _p(lse), _p(workspace),
                                      workspace.numel() * workspace.element_size(), _p(status), _s(stream))
    _check(rc, "bastion_topk_marginals")


def bastion_lm_head_topk_workspace_bytes(B: int, b: int, V: int, K: int) -> int:
    return int(lib().bastion_lm_head_topk_workspace_bytes(B, b, V, K))


def bastion_lm_head_topk(hidden, weight, K, topk_logq, topk_logit, topk_tok, lse, workspace, status,
                         stream=None):
    """hidden [B, b, H] and weight [V, H], contiguous bfloat16; outputs as
    bastion_topk_marginals for the logits hidden . weight^T."""
    for name, t in (("hidden", hidden), ("weight", weight)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise BastionError(f"lm head: {name} must be contiguous bfloat16")
    B, b, H = hidden.shape
    V = weight.shape[0]
    if weight.dim() != 2 or weight.shape[1] != H:
        raise BastionError("lm head: weight must be [V, H] with the hidden size of hidden")
    rc = lib().bastion_lm_head_topk(_p(hidden), _p(weight), B, b, H, V, int(K), _p(topk_logq),
                                    _p(topk_logit), _p(topk_tok), _p(lse), _p(workspace),
                                    workspace.numel() * workspace.element_size(), _p(status), _s(stream))
    _check(rc, "bastion_lm_head_topk")


def bastion_build_tree(topk_logit, topk_tok, lse, n_max, root_token, ctx_len, cost_ms, l_ar,
                       n_nodes, parent, depth, pos_id, token, rank, log_rho, a_hat, speedup,
                       anc_mask, status, stream=None):
    B, b, K = topk_logit.shape
    per_req = 1 if (cost_ms.dim() == 2 and cost_ms.shape[0] == B and B > 1) else 0
    rc = lib().bastion_build_tree(_p(topk_logit), _p(topk_tok), _p(lse), B, b, K, int(n_max),
                                  _p(root_token), _p(ctx_len), _p(cost_ms), per_req, _p(l_ar),
                                  _p(n_nodes), _p(parent), _p(depth), _p(pos_id), _p(token), _p(rank),
                                  _p(log_rho), _p(a_hat), _p(speedup), _p(anc_mask), _p(status), _s(stream))
    _check(rc, "bastion_build_tree")


def bastion_build_tree_mixture_workspace_bytes(B: int, Z: int, b: int, K: int, n_max: int) -> int:
    return int(lib().bastion_build_tree_mixture_workspace_bytes(B, Z, b, K, n_max))


def bastion_build_tree_mixture(topk_logit, topk_tok, lse, pi, n_max, root_token, ctx_len, cost_ms, l_ar,
                               n_nodes, parent, depth, pos_id, token, log_rho, a_hat, speedup, anc_mask,
                               workspace, status, stream=None):
    """topk_logit/tok [B, Z, b, K], lse [B, Z, b] float64, pi [B, Z] float64 (contiguous);
    workspace: bastion_build_tree_mixture_workspace_bytes(B, Z, b, K, n_max) bytes."""
    B, Z, b, K = topk_logit.shape
    for t in (topk_logit, topk_tok, lse, pi):
        if not t.is_contiguous():
            raise BastionError("mixture tree inputs must be contiguous")
    # the library reads these bytes as the stated types; a wrong dtype would be read as garbage
    for name, t, dt in (("topk_logit", topk_logit, torch.float32), ("topk_tok", topk_tok, torch.int32),
                        ("lse", lse, torch.float64), ("pi", pi, torch.float64)):
        if t.dtype != dt:
            raise BastionError(f"mixture tree: {name} must be {dt}, got {t.dtype}")
    if tuple(topk_tok.shape) != (B, Z, b, K) or tuple(lse.shape) != (B, Z, b) or tuple(pi.shape) != (B, Z):
        raise BastionError("mixture tree: topk_tok [B,Z,b,K], lse [B,Z,b] and pi [B,Z] must match topk_logit")
    if cost_ms.numel() not in (n_max + 1, B * (n_max + 1)):
        raise BastionError("mixture tree: cost_ms must hold n_max + 1 entries, or n_max + 1 per request")
    per_req = 1 if (cost_ms.dim() == 2 and cost_ms.shape[0] == B and B > 1) else 0
    rc = lib().bastion_build_tree_mixture(_p(topk_logit), _p(topk_tok), _p(lse), _p(pi), B, Z, b, K,
                                          int(n_max), _p(root_token), _p(ctx_len), _p(cost_ms), per_req,
                                          _p(l_ar), _p(n_nodes), _p(parent), _p(depth), _p(pos_id),
                                          _p(token), _p(log_rho), _p(a_hat), _p(speedup), _p(anc_mask),
                                          _p(workspace), workspace.numel() * workspace.element_size(),
                                          _p(status), _s(stream))
    _check(rc, "bastion_build_tree_mixture")


def bastion_calibrate_cost(sample_n, sample_ms, roofline: dict, t_draft, n_max, cost_ms, params, status,
                           stream=None):
    """sample_n / sample_ms [n] float32 on the device; cost_ms [n_max + 1], params [2] float32.
    roofline: bytes0, bytes1, flops0, flops1, bw, peak (roof(N) in ms)."""
    r = roofline
    rc = lib().bastion_calibrate_cost(_p(sample_n), _p(sample_ms), int(sample_n.numel()), r["bytes0"],
                                      r["bytes1"], r["flops0"], r["flops1"], r["bw"], r["peak"],
                                      float(t_draft), int(n_max), _p(cost_ms), _p(params), _p(status),
                                      _s(stream))
    _check(rc, "bastion_calibrate_cost")


def bastion_tree_attention_workspace_bytes(B, n_max, Hq, Hkv, D, L_cap) -> int:
    return int(lib().bastion_tree_attention_workspace_bytes(B, n_max, Hq, Hkv, D, L_cap))


def bastion_tree_attention(q, k_cache, v_cache, ctx_len, n_nodes, anc_mask, scale, out, workspace,
                           status, stream=None):
    """q/out [B, n_max, Hq, D], k/v [B, L_cap, Hkv, D], bf16 contiguous."""
    B, n_max, Hq, D = q.shape
    L_cap, Hkv = k_cache.shape[1], k_cache.shape[2]
    for t in (q, k_cache, v_cache, out):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise BastionError("attention tensors must be contiguous bfloat16")
    rc = lib().bastion_tree_attention(_p(q), _p(k_cache), _p(v_cache), B, n_max, Hq, Hkv, D, L_cap,
                                      _p(ctx_len), _p(n_nodes), _p(anc_mask), float(scale), _p(out),
                                      _p(workspace), workspace.numel() * workspace.element_size(),
                                      _p(status), _s(stream))
    _check(rc, "bastion_tree_attention")


def bastion_verify_greedy_workspace_bytes(B: int, n_max: int, V: int) -> int:
    return int(lib().bastion_verify_greedy_workspace_bytes(B, n_max, V))


def bastion_verify_greedy(target_logits, b, n_nodes, parent, token, argmax, accept_len,
                          accept_nodes, out_tokens, workspace, status, stream=None):
    """target_logits [B, n_max, V] (fp32/bf16, last dim contiguous), on the device or in
    pinned host memory."""
    B, n_max, V = target_logits.shape
    ld = _rows_view(target_logits, 3)
    rc = lib().bastion_verify_greedy(_p_rows(target_logits), _dtype(target_logits), B, n_max, V, ld, int(b),
                                     _p(n_nodes), _p(parent), _p(token), _p(argmax), _p(accept_len),
                                     _p(accept_nodes), _p(out_tokens), _p(workspace),
                                     workspace.numel() * workspace.element_size(), _p(status), _s(stream))
    _check(rc, "bastion_verify_greedy")


def bastion_verify_sample_workspace_bytes(B: int, n_max: int, V: int) -> int:
    return int(lib().bastion_verify_sample_workspace_bytes(B, n_max, V))


def bastion_verify_sample(target_logits, b, temperature, uniforms, n_nodes, parent, token, sampled,
                          accept_len, accept_nodes, out_tokens, workspace, status, stream=None):
    """target_logits [B, n_max, V] (fp32/bf16, last dim contiguous); uniforms [B, n_max] float64."""
    B, n_max, V = target_logits.shape
    ld = _rows_view(target_logits, 3)
    if uniforms.dtype != torch.float64 or not uniforms.is_contiguous():
        raise BastionError("uniforms must be a contiguous float64 tensor")
    rc = lib().bastion_verify_sample(_p_rows(target_logits), _dtype(target_logits), B, n_max, V, ld, int(b),
                                     float(temperature), _p(uniforms), _p(n_nodes), _p(parent), _p(token),
                                     _p(sampled), _p(accept_len), _p(accept_nodes), _p(out_tokens),
                                     _p(workspace), workspace.numel() * workspace.element_size(),
                                     _p(status), _s(stream))
    _check(rc, "bastion_verify_sample")


def bastion_verify_greedy_noalloc(target_logits, b, n_nodes, parent, token, argmax, accept_len,
                                  accept_nodes, out_tokens, status, stream=None):
    """Same as bastion_verify_greedy without a workspace argument, for callers that
    cannot allocate device memory: the library uses a fixed 128 KiB scratch array
    of its own (B <= 4096, B * n_max <= 16384).  Calls that overlap on the GPU race
    on that array."""
    B, n_max, V = target_logits.shape
    ld = _rows_view(target_logits, 3)
    rc = lib().bastion_verify_greedy_noalloc(_p_rows(target_logits), _dtype(target_logits), B, n_max, V, ld,
                                             int(b), _p(n_nodes), _p(parent), _p(token), _p(argmax),
                                             _p(accept_len), _p(accept_nodes), _p(out_tokens), _p(status),
                                             _s(stream))
    _check(rc, "bastion_verify_greedy_noalloc")


# --------------------------------------------------------------------------- buffers

def workspace(nbytes: int, device) -> torch.Tensor:
    """A zero-filled, 256-byte aligned workspace (torch allocations are)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


@dataclass
class TopK:
    logq: torch.Tensor
    logit: torch.Tensor
    tok: torch.Tensor
    lse: torch.Tensor


@dataclass
class Tree:
    n_nodes: torch.Tensor
    parent: torch.Tensor
    depth: torch.Tensor
    pos_id: torch.Tensor
    token: torch.Tensor
    rank: torch.Tensor
    log_rho: torch.Tensor
    a_hat: torch.Tensor
    speedup: torch.Tensor
    anc_mask: torch.Tensor


@dataclass
class Verify:
    argmax: torch.Tensor
    accept_len: torch.Tensor
    accept_nodes: torch.Tensor
    out_tokens: torch.Tensor


def alloc_topk(B, b, K, device) -> TopK:
    return TopK(torch.empty(B, b, K, dtype=torch.float32, device=device),
                torch.empty(B, b, K, dtype=torch.float32, device=device),
                torch.empty(B, b, K, dtype=torch.int32, device=device),
                torch.empty(B, b, dtype=torch.float64, device=device))


def alloc_tree(B, n_max, device) -> Tree:
    W = (n_max + 31) // 32
    i = lambda: torch.full((B, n_max), -7, dtype=torch.int32, device=device)  # noqa: E731
    f = lambda: torch.full((B, n_max), float("nan"), dtype=torch.float32, device=device)  # noqa: E731
    return Tree(torch.zeros(B, dtype=torch.int32, device=device), i(), i(), i(), i(), i(), f(), f(), f(),
                torch.zeros(B, n_max, W, dtype=torch.int32, device=device))


def alloc_verify(B, n_max, b, device) -> Verify:
    return Verify(torch.full((B, n_max), -7, dtype=torch.int32, device=device),
                  torch.zeros(B, dtype=torch.int32, device=device),
                  torch.zeros(B, b + 1, dtype=torch.int32, device=device),
                  torch.zeros(B, b + 1, dtype=torch.int32, device=device))


class TreeStep:
    """One tree step (top-K marginals -> best-first tree -> greedy verify) over
    preallocated device buffers; ``capture()`` records the launches in a CUDA
    graph so a step replays with one host call."""

    def __init__(self, B, b, V, K, n_max, device, root_token, ctx_len, cost_ms, l_ar):
        self.B, self.b, self.V, self.K, self.n_max = B, b, V, K, n_max
        self.device = device
        self.topk = alloc_topk(B, b, K, device)
        self.tree = alloc_tree(B, n_max, device)
        self.ver = alloc_verify(B, n_max, b, device)
        self.status = torch.zeros(B, dtype=torch.int32, device=device)
        self.ws_topk = workspace(bastion_topk_marginals_workspace_bytes(B, b, V, K), device)
        self.ws_verify = workspace(bastion_verify_greedy_workspace_bytes(B, n_max, V), device)
        self.root_token = root_token.to(device=device, dtype=torch.int32)
        self.ctx_len = ctx_len.to(device=device, dtype=torch.int32)
        self.cost_ms = cost_ms.to(device=device, dtype=torch.float32)
        self.l_ar = l_ar.to(device=device, dtype=torch.float32)
        self.graph = None

    def draft(self, drafter_logits, stream=None):
        """Steps 1-3: marginals, then the tree (its size decides which target rows exist)."""
        t, tr = self.topk, self.tree
        bastion_topk_marginals(drafter_logits, self.K, t.logq, t.logit, t.tok, t.lse, self.ws_topk,
                               self.status, stream)
        bastion_build_tree(t.logit, t.tok, t.lse, self.n_max, self.root_token, self.ctx_len,
                           self.cost_ms, self.l_ar, tr.n_nodes, tr.parent, tr.depth, tr.pos_id,
                           tr.token, tr.rank, tr.log_rho, tr.a_hat, tr.speedup, tr.anc_mask,
                           self.status, stream)

    def set_sampling(self, temperature, uniforms):
        """Verify at temperature T > 0 with the uniforms [B, n_max] (float64 in
        [0, 1), refreshed by the caller between steps); T = 0 returns to greedy."""
        self.temperature = float(temperature)
        if self.temperature > 0:
            self.uniforms = uniforms.to(device=self.device, dtype=torch.float64).contiguous()
            self.ws_sample = workspace(bastion_verify_sample_workspace_bytes(self.B, self.n_max, self.V),
                                       self.device)

    def verify(self, target_logits, stream=None):
        """Step 4: verification of the tree against the target's logits (greedy,
        or sampled at the temperature set by set_sampling)."""
        tr, v = self.tree, self.ver
        if getattr(self, "temperature", 0.0) > 0:
            bastion_verify_sample(target_logits, self.b, self.temperature, self.uniforms, tr.n_nodes,
                                  tr.parent, tr.token, v.argmax, v.accept_len, v.accept_nodes,
                                  v.out_tokens, self.ws_sample, self.status, stream)
            return
        bastion_verify_greedy(target_logits, self.b, tr.n_nodes, tr.parent, tr.token, v.argmax,
                              v.accept_len, v.accept_nodes, v.out_tokens, self.ws_verify,
                              self.status, stream)

    def run(self, drafter_logits, target_logits, stream=None):
        self.draft(drafter_logits, stream)
        self.verify(target_logits, stream)

    def run_chunked(self, drafter_logits, target_logits, chunks):
        """The same step with the batch split into request chunks on their own
        streams (forked from and joined to the current stream).  A chunk's
        top-K starts after the previous chunk's top-K, so one chunk's tree build
        (a serial chain per request) overlaps the other chunks' sweeps.
        Requests are independent, so the results equal run()'s."""
        B = self.B
        chunks = max(1, min(chunks, B))
        bounds = [B * c // chunks for c in range(chunks + 1)]
        if getattr(self, "_chunk_state", None) is None or len(self._chunk_state) != chunks:
            self._chunk_state = []
            for c in range(chunks):
                nb = bounds[c + 1] - bounds[c]
                self._chunk_state.append((torch.cuda.Stream(device=self.device),
                                          workspace(bastion_verify_greedy_workspace_bytes(nb, self.n_max, self.V),
                                                    self.device)))
        main = torch.cuda.current_stream(self.device)
        t, tr, v = self.topk, self.tree, self.ver
        per_req_cost = self.cost_ms.dim() == 2 and self.cost_ms.shape[0] == B and B > 1
        prev = None
        for c in range(chunks):
            c0, c1 = bounds[c], bounds[c + 1]
            st, ws_v = self._chunk_state[c]
            st.wait_stream(main)
            if prev is not None:
                st.wait_event(prev)
            with torch.cuda.stream(st):
                bastion_topk_marginals(drafter_logits[c0:c1], self.K, t.logq[c0:c1], t.logit[c0:c1],
                                       t.tok[c0:c1], t.lse[c0:c1], self.ws_topk, self.status[c0:c1], st)
                prev = torch.cuda.Event()
                prev.record(st)
                cost = self.cost_ms[c0:c1] if per_req_cost else self.cost_ms
                bastion_build_tree(t.logit[c0:c1], t.tok[c0:c1], t.lse[c0:c1], self.n_max,
                                   self.root_token[c0:c1], self.ctx_len[c0:c1], cost, self.l_ar[c0:c1],
                                   tr.n_nodes[c0:c1], tr.parent[c0:c1], tr.depth[c0:c1], tr.pos_id[c0:c1],
                                   tr.token[c0:c1], tr.rank[c0:c1], tr.log_rho[c0:c1], tr.a_hat[c0:c1],
                                   tr.speedup[c0:c1], tr.anc_mask[c0:c1], self.status[c0:c1], st)
                bastion_verify_greedy(target_logits[c0:c1], self.b, tr.n_nodes[c0:c1], tr.parent[c0:c1],
                                      tr.token[c0:c1], v.argmax[c0:c1], v.accept_len[c0:c1],
                                      v.accept_nodes[c0:c1], v.out_tokens[c0:c1], ws_v,
                                      self.status[c0:c1], st)
        for c in range(chunks):
            main.wait_stream(self._chunk_state[c][0])

    def capture(self, drafter_logits, target_logits, chunks=1):
        """Records one step in a CUDA graph (chunks > 1: run_chunked)."""
        def step():
            if chunks > 1:
                self.run_chunked(drafter_logits, target_logits, chunks)
            else:
                self.run(drafter_logits, target_logits)
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()  # warm (sets kernel attributes, creates the chunk streams)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        self.graph = g
        return g
