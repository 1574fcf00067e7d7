"""Input recipes for the five workloads of the BASTION draft-tree hot path.

Everything here produces *inputs*: drafter logits shaped like a block-diffusion
drafter's per-position logits, a supplied cost table C(N), per-request L_AR,
root tokens and context lengths, target logits with a planted argmax per tree
node, and the Q/K/V tensors of a tree-verification attention layer.  It holds
none of the method's arithmetic: no softmax, ranking, tree search or argmax.

Random numbers come from the counter-based generator in ``synth.c``; every
value is addressed by (seed, stream, index), so both sides of a parity check
get identical bytes however the work is split.

Method background (Bastion: Budget-Aware Speculative Decoding with
Tree-structured Block Diffusion Drafting, gist.science/nl/paper/2605.29727,
"Technische Samenvatting", Methodologie §1-§3): the drafter emits one marginal
q_k per block position in one forward pass; the tree is verified by the target
in parallel; the controller trades Â(T_N) against a calibrated latency C(N).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libsynth.so")

# stream ids (one per synthetic tensor)
S_DRAFT_NOISE = 1
S_SPIKE_POS = 2
S_SPIKE_P1 = 3
S_TARGET_NOISE = 4
S_PLANT = 5
S_ROOT = 6
S_CTX = 7
S_PAGREE = 8
S_Q = 9
S_K = 10
S_V = 11
S_VERIFY_U = 12
S_HIDDEN = 13
S_WEIGHT = 14
S_MIX_BASE = 15
S_MIX_BRANCH = 16
S_MIX_PI = 17

PLANT_VALUE = 12.0  # above any Box-Muller draw (|z| < 8.7 since u1 >= 2^-54)

BASE_SEED = 0xBA5710


def build(force: bool = False) -> str:
    """Compile libsynth.so (plain C, OpenMP, no FMA contraction)."""
    src = os.path.join(_HERE, "synth.c")
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                           "-ffp-contract=off", "-fno-fast-math", src, "-o", tmp, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_lib = None


def lib():
    global _lib
    if _lib is None:
        build()
        L = ctypes.CDLL(_LIB_PATH)
        u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        L.synth_splitmix64_next.argtypes = [ctypes.POINTER(u64)]
        L.synth_splitmix64_next.restype = u64
        L.synth_u64.argtypes = [u64, u64, u64]
        L.synth_u64.restype = u64
        L.synth_uniform.argtypes = [u64, u64, u64]
        L.synth_uniform.restype = dbl
        L.synth_normal.argtypes = [u64, u64, u64]
        L.synth_normal.restype = dbl
        L.synth_f64_to_bf16.argtypes = [dbl]
        L.synth_f64_to_bf16.restype = ctypes.c_uint16
        for name in ("synth_fill_normal_bf16", "synth_fill_normal_f32"):
            getattr(L, name).argtypes = [vp, i64, dbl, u64, u64, i64]
            getattr(L, name).restype = None
        for name in ("synth_fill_normal_rows_bf16", "synth_fill_normal_rows_f32"):
            getattr(L, name).argtypes = [vp, i64, i64, i64, dbl, u64, u64, i64]
            getattr(L, name).restype = None
        L.synth_fill_uniform.argtypes = [vp, i64, u64, u64, i64]
        L.synth_fill_uniform.restype = None
        _lib = L
    return _lib


# ----------------------------------------------------------------------------- primitives

def splitmix64_sequence(seed: int, n: int) -> list[int]:
    st = ctypes.c_uint64(seed)
    return [lib().synth_splitmix64_next(ctypes.byref(st)) for _ in range(n)]


def uniforms(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    out = np.empty(n, dtype=np.float64)
    if n:
        lib().synth_fill_uniform(out.ctypes.data, n, seed, stream, offset)
    return out


def normals(seed: int, stream: int, n: int, offset: int = 0) -> np.ndarray:
    return np.array([lib().synth_normal(seed, stream, offset + i) for i in range(n)])


def verify_uniforms(w: "Workload") -> np.ndarray:
    """float64 [B, n_max] in [0, 1): the draws of stochastic verification."""
    return uniforms(w.seed, S_VERIFY_U, w.B * w.n_max).reshape(w.B, w.n_max)


def f64_to_bf16_bits(x: float) -> int:
    return int(lib().synth_f64_to_bf16(float(x)))


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32)


def fill_normal(ptr: int, n: int, dtype: str, scale: float, seed: int, stream: int,
                offset: int = 0) -> None:
    """Fill n contiguous elements at a raw host pointer."""
    if dtype == "bf16":
        lib().synth_fill_normal_bf16(ptr, n, scale, seed, stream, offset)
    elif dtype == "f32":
        lib().synth_fill_normal_f32(ptr, n, scale, seed, stream, offset)
    else:
        raise ValueError(dtype)


def lm_head_inputs(B: int, b: int, H: int, V: int, seed: int):
    """Drafter final hidden states [B, b, H] ~ N(0, 1) and an output embedding
    [V, H] ~ N(0, 4/H), both bf16 bits (uint16): logits of standard deviation
    about 2, the drafter-logit scale of the batched workloads."""
    hidden = host_array((B, b, H), "bf16")
    weight = host_array((V, H), "bf16")
    fill_normal(hidden.ctypes.data, hidden.size, "bf16", 1.0, seed, S_HIDDEN)
    fill_normal(weight.ctypes.data, weight.size, "bf16", 2.0 / float(np.sqrt(H)), seed, S_WEIGHT)
    return hidden, weight


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to the nearest bf16 (ties to even), as uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)).astype(np.uint16)


def mixture_inputs(B: int, Z: int, b: int, V: int, seed: int):
    """Per-branch drafter logits of a latent-mixture proposal and its branch
    weights.  Logits [B, Z, b, V] as bf16 bits: a part shared by the branches,
    N(0, 2^2) (the drafter-logit scale of the batched workloads), plus a
    branch part N(0, 1), so that the branches' top lists overlap in part.
    Weights pi [B, Z] float64: normalised standard exponentials (a flat
    Dirichlet draw)."""
    base = np.empty((B, 1, b, V), np.float32)
    fill_normal(base.ctypes.data, base.size, "f32", 2.0, seed, S_MIX_BASE)
    dev = np.empty((B, Z, b, V), np.float32)
    fill_normal(dev.ctypes.data, dev.size, "f32", 1.0, seed, S_MIX_BRANCH)
    dev += base
    del base
    logits = f32_to_bf16_bits(dev)
    del dev
    e = -np.log(uniforms(seed, S_MIX_PI, B * Z).reshape(B, Z))
    return logits, e / e.sum(axis=1, keepdims=True)


def fill_normal_rows(ptr: int, rows: int, cols: int, ld: int, dtype: str, scale: float,
                     seed: int, stream: int, offset: int = 0) -> None:
    if dtype == "bf16":
        lib().synth_fill_normal_rows_bf16(ptr, rows, cols, ld, scale, seed, stream, offset)
    elif dtype == "f32":
        lib().synth_fill_normal_rows_f32(ptr, rows, cols, ld, scale, seed, stream, offset)
    else:
        raise ValueError(dtype)


# ----------------------------------------------------------------------------- workloads

@dataclass
class Workload:
    """One named workload: sizes, dtypes, cost model and the drafter/target recipe."""
    cid: int
    name: str
    B: int
    b: int
    V: int
    K: int
    n_max: int
    dtype: str                      # drafter / target logit dtype: "f32" or "bf16"
    l_ar_ms: float
    cost: str                       # cost model id
    drafter: str                    # drafter recipe id
    p_agree: str                    # plant recipe id
    ctx: int | None = None          # fixed context length (attention workloads)
    Hq: int = 32
    Hkv: int = 8
    D: int = 128
    seed: int = field(default=0)

    def __post_init__(self):
        if not self.seed:
            self.seed = BASE_SEED + self.cid

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def ld(self) -> int:
        return self.V

    @property
    def L_cap(self) -> int:
        return (self.ctx or 0) + self.n_max


WORKLOADS = {
    1: Workload(1, "tiny-b4-v1024-k8-n16-f32", B=1, b=4, V=1024, K=8, n_max=16, dtype="f32",
                l_ar_ms=20.0, cost="tiny", drafter="sigma-ramp", p_agree="const0.7"),
    2: Workload(2, "single-b16-v151936-k32-n64-bf16", B=1, b=16, V=151936, K=32, n_max=64,
                dtype="bf16", l_ar_ms=18.0, cost="knee32", drafter="spike-linear",
                p_agree="depth-linear"),
    3: Workload(3, "batch32-b16-v151936-k64-n128-bf16", B=32, b=16, V=151936, K=64, n_max=128,
                dtype="bf16", l_ar_ms=18.0, cost="knee32", drafter="spike-geometric",
                p_agree="uniform"),
    4: Workload(4, "attn-b8-n64-ctx4096-h32x8-d128-bf16", B=8, b=16, V=151936, K=32, n_max=64,
                dtype="bf16", l_ar_ms=18.0, cost="flat", drafter="spike-linear",
                p_agree="depth-linear", ctx=4096),
    5: Workload(5, "serve64-b16-v128256-k64-n256-ctx16384-bf16", B=64, b=16, V=128256, K=64,
                n_max=256, dtype="bf16", l_ar_ms=15.0, cost="roofline-flat281",
                drafter="spike-geometric", p_agree="uniform", ctx=16384),
}


def workload(cid: int, **over) -> Workload:
    w = WORKLOADS[cid]
    if over:
        d = dict(w.__dict__)
        d.update(over)
        w = Workload(**d)
    return w


def cost_ms(N: int, model: str) -> float:
    """C(N) = T_draft + T_verify(N) in ms for the supplied cost models."""
    if model == "tiny":
        return 3.0 + 20.0 + 0.1 * max(0, N - 8)
    if model == "knee32":
        return 2.5 + 18.0 + 0.04 * max(0, N - 32)
    if model == "flat":
        return 2.5 + 18.0
    if model == "roofline-flat281":
        # T_verify = max(16 GB / 8 TB/s, 2 * 8e9 * N flop / 2.25 PFLOP/s) + 1 ms
        return 3.0 + max(16e9 / 8e12, 2.0 * 8e9 * N / 2.25e15) * 1e3 + 1.0
    raise ValueError(model)


def cost_table(w: Workload) -> np.ndarray:
    """float32 [1, n_max+1]; entry N holds C(N)."""
    return np.array([[cost_ms(N, w.cost) for N in range(w.n_max + 1)]], dtype=np.float32)


def l_ar(w: Workload) -> np.ndarray:
    return np.full(w.B, w.l_ar_ms, dtype=np.float32)


def root_tokens(w: Workload) -> np.ndarray:
    u = uniforms(w.seed, S_ROOT, w.B)
    return np.minimum((u * w.V).astype(np.int64), w.V - 1).astype(np.int32)


def ctx_lens(w: Workload) -> np.ndarray:
    if w.ctx is not None:
        return np.full(w.B, w.ctx, dtype=np.int32)
    u = uniforms(w.seed, S_CTX, w.B)
    return (u * 4096).astype(np.int32)


def spike_positions(w: Workload) -> np.ndarray:
    u = uniforms(w.seed, S_SPIKE_POS, w.B * w.b).reshape(w.B, w.b)
    return np.minimum((u * w.V).astype(np.int64), w.V - 1)


def top1_targets(w: Workload) -> np.ndarray:
    """Planted top-1 probability per (request, depth index k=0..b-1)."""
    k = np.arange(w.b, dtype=np.float64)
    if w.drafter == "spike-linear":
        return np.tile(0.95 - 0.04 * k, (w.B, 1))
    if w.drafter == "spike-geometric":
        p1 = 0.3 + 0.69 * uniforms(w.seed, S_SPIKE_P1, w.B)
        return p1[:, None] * 0.9 ** k[None, :]
    raise ValueError(w.drafter)


def spike_logit(p: float, V: int, sigma: float) -> float:
    """Logit that gives the spike softmax probability ~p against V-1 noise logits
    sigma*z, using the lognormal mean E[exp(sigma z)] = exp(sigma^2/2) in place of
    the sample sum (closed form; no softmax of the actual row)."""
    return math.log(p / (1.0 - p)) + math.log(V - 1) + 0.5 * sigma * sigma


def fill_drafter(w: Workload, ptr: int, ld: int | None = None) -> None:
    """Write drafter logits [B, b, V] (row stride ld elements) at a host pointer."""
    ld = ld or w.V
    rows = w.B * w.b
    es = w.elem_bytes
    if w.drafter == "sigma-ramp":
        # l[k, v] = (1 + 0.5 k) z + h_k [v = s_k], h = (6, 4, 3, 2) for k = 0..3
        h = (6.0, 4.0, 3.0, 2.0)
        s = spike_positions(w)
        for r in range(w.B):
            for k in range(w.b):
                row = r * w.b + k
                sig = 1.0 + 0.5 * k
                fill_normal_rows(ptr + row * ld * es, 1, w.V, ld, w.dtype, sig, w.seed,
                                 S_DRAFT_NOISE, row * w.V)
                v = int(s[r, k])
                z = lib().synth_normal(w.seed, S_DRAFT_NOISE, row * w.V + v)
                _poke(ptr + (row * ld + v) * es, w.dtype, sig * z + h[k % len(h)])
        return
    sigma = 2.0
    fill_normal_rows(ptr, rows, w.V, ld, w.dtype, sigma, w.seed, S_DRAFT_NOISE, 0)
    s = spike_positions(w)
    p = top1_targets(w)
    for r in range(w.B):
        for k in range(w.b):
            row = r * w.b + k
            _poke(ptr + (row * ld + int(s[r, k])) * es, w.dtype, spike_logit(p[r, k], w.V, sigma))


def _poke(addr: int, dtype: str, value: float) -> None:
    if dtype == "bf16":
        ctypes.c_uint16.from_address(addr).value = f64_to_bf16_bits(value)
    else:
        ctypes.c_float.from_address(addr).value = value


def host_array(shape, dtype: str) -> np.ndarray:
    return np.empty(shape, dtype=np.float32 if dtype == "f32" else np.uint16)


def drafter_logits(w: Workload) -> np.ndarray:
    """numpy [B, b, V]: float32, or uint16 holding bf16 bits."""
    a = host_array((w.B, w.b, w.V), w.dtype)
    fill_drafter(w, a.ctypes.data)
    return a


def p_agree(w: Workload, depth_of_choice: int, r: int, pr: np.ndarray | None = None) -> float:
    """Probability that a node's planted target token is its best child.
    depth_of_choice is the depth of the token being chosen (node depth + 1)."""
    if w.p_agree == "const0.7":
        return 0.7
    if w.p_agree == "depth-linear":
        return 0.8 - 0.4 * (depth_of_choice - 1) / 15.0
    if w.p_agree == "uniform":
        if pr is None:
            pr = 0.3 + 0.6 * uniforms(w.seed, S_PAGREE, w.B)
        return float(pr[r])
    raise ValueError(w.p_agree)


def fill_target_noise(w: Workload, ptr: int, ld: int | None = None) -> None:
    """Target logits [B, n_max, V] of N(0,1) noise at a host pointer."""
    ld = ld or w.V
    fill_normal_rows(ptr, w.B * w.n_max, w.V, ld, w.dtype, 1.0, w.seed, S_TARGET_NOISE, 0)


def plant_tokens(w: Workload, n_nodes, depth, topk_tok) -> np.ndarray:
    """Token planted as the target argmax of each tree node ([B, n_max], -1 past n_nodes).

    Node i at depth d < b: with probability p_agree(d+1) its best child token
    (rank 0 of q_{d+1}), else a uniformly drawn rank 1..K-1 of q_{d+1}, so that
    sibling branches can be accepted.  A node at depth b draws uniformly over V.
    topk_tok is [B, b, K] (rank order per position), the tree arrays are
    [B, n_max]; they come from whichever side builds the tree.
    """
    n_nodes = np.asarray(n_nodes)
    depth = np.asarray(depth).reshape(w.B, w.n_max)
    topk_tok = np.asarray(topk_tok).reshape(w.B, w.b, w.K)
    u = uniforms(w.seed, S_PLANT, w.B * w.n_max * 2).reshape(w.B, w.n_max, 2)
    pr = 0.3 + 0.6 * uniforms(w.seed, S_PAGREE, w.B) if w.p_agree == "uniform" else None
    out = np.full((w.B, w.n_max), -1, dtype=np.int64)
    for r in range(w.B):
        for i in range(int(n_nodes[r])):
            d = int(depth[r, i])
            if d < w.b:
                if u[r, i, 0] < p_agree(w, d + 1, r, pr) or w.K == 1:
                    out[r, i] = topk_tok[r, d, 0]
                else:
                    j = 1 + min(int(u[r, i, 1] * (w.K - 1)), w.K - 2)
                    out[r, i] = topk_tok[r, d, j]
            else:
                out[r, i] = min(int(u[r, i, 1] * w.V), w.V - 1)
    return out


def plant_into(w: Workload, ptr: int, planted: np.ndarray, ld: int | None = None) -> None:
    ld = ld or w.V
    es = w.elem_bytes
    for r in range(w.B):
        for i in range(w.n_max):
            t = int(planted[r, i])
            if t >= 0:
                _poke(ptr + ((r * w.n_max + i) * ld + t) * es, w.dtype, PLANT_VALUE)


def target_logits(w: Workload, n_nodes, depth, topk_tok) -> tuple[np.ndarray, np.ndarray]:
    a = host_array((w.B, w.n_max, w.V), w.dtype)
    fill_target_noise(w, a.ctypes.data)
    planted = plant_tokens(w, n_nodes, depth, topk_tok)
    plant_into(w, a.ctypes.data, planted)
    return a, planted


def fill_attention(w: Workload, q_ptr: int, k_ptr: int, v_ptr: int) -> None:
    """Q [B, n_max, Hq, D], K/V caches [B, L_cap, Hkv, D], all N(0,1)/sqrt(D) as bf16."""
    sc = 1.0 / math.sqrt(w.D)
    fill_normal(q_ptr, w.B * w.n_max * w.Hq * w.D, "bf16", sc, w.seed, S_Q)
    n_kv = w.B * w.L_cap * w.Hkv * w.D
    fill_normal(k_ptr, n_kv, "bf16", sc, w.seed, S_K)
    fill_normal(v_ptr, n_kv, "bf16", sc, w.seed, S_V)


def attention_inputs(w: Workload):
    q = np.empty((w.B, w.n_max, w.Hq, w.D), dtype=np.uint16)
    k = np.empty((w.B, w.L_cap, w.Hkv, w.D), dtype=np.uint16)
    v = np.empty_like(k)
    fill_attention(w, q.ctypes.data, k.ctypes.data, v.ctypes.data)
    return q, k, v
