"""Benchmark of the draft-tree hot path on one or more GB300 GPUs.

One step = one tree step over a batch of requests: softmax + top-K marginals
over the drafter logits, best-first tree build with the online controller, and
greedy verification against the target logits (three launches, replayed from a
CUDA graph).  Default workload: 32 requests, block size 16, vocab 151,936,
top-64, tree budget 128, bf16 logits.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
        [--workload 1..5]
Multi-GPU: launched under torchrun; every rank runs an independent replica on
its own GPU (weak scaling), timed with a barrier and the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree steps/s (top-K+best-first+verify) B=32 V=151936; % HBM roofline"
UNIT = "tree steps/s"
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class Clocks:
    """nvidia-smi sampling in the background (SM clock, power, throttle reasons)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "power_w_max": max(power) if power else None, "reasons": sorted(reasons)}


def profiled_traffic(summary: str, source: str):
    """DRAM bytes per launch from a committed ncu summary, or None when the
    kernel source has changed since the counters were taken."""
    import hashlib
    try:
        text = open(os.path.join(ROOT, "profiles", summary)).read()
        digest = hashlib.sha256(open(os.path.join(ROOT, "draft_tree_build_gb300", "csrc", source), "rb").read()).hexdigest()
    except OSError:
        return None
    fields = dict(line.split(": ", 1) for line in text.splitlines() if ": " in line and line[:1].isalpha())
    if fields.get("kernel_source_sha256_16", "").strip() != digest[:16]:
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def dist_setup():
    import torch
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    else:
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int) -> float:
    """The largest x over the ranks (the slowest replica's time)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_rate(units_per_rank: float, elapsed_ms: float, ws: int) -> float:
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return ws * units_per_rank / (elapsed_ms * 1e-3)


def pinned_from(arr: np.ndarray):
    import torch
    t = torch.empty(arr.shape, dtype=torch.int16 if arr.dtype == np.uint16 else torch.float32,
                    pin_memory=True)
    t.numpy()[...] = arr.view(np.int16) if arr.dtype == np.uint16 else arr
    return t.view(torch.bfloat16) if arr.dtype == np.uint16 else t


# --------------------------------------------------------------------------- our arm

def step_config(w, mean_nodes: float, ws: int) -> dict:
    """The config dict of a tree-step line (both arms print the same one)."""
    return {"workload": w.name, "B": w.B, "b": w.b, "V": w.V, "K": w.K, "n_max": w.n_max,
            "logit_dtype": w.dtype, "seed": w.seed, "mean_tree_nodes": mean_nodes,
            "l2": "inputs larger than L2, two rotating device copies",
            "parallelism": f"replicas x{ws}"}


def run_ours(args, ws, rank, local, light=False):
    import torch

    import synth
    from draft_tree_build_gb300 import bastion

    dev = torch.device(f"cuda:{local}")
    w = synth.workload(args.workload)
    es = w.elem_bytes
    roots, ctx, cost, lar = synth.root_tokens(w), synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w)

    # inputs: drafter logits on the host (pinned), two device copies (rotated so
    # every step reads logits the previous step did not touch)
    x_host = synth.drafter_logits(w)
    x_pin = pinned_from(x_host)
    xs = [x_pin.to(dev, non_blocking=False) for _ in range(2)]
    step = bastion.TreeStep(w.B, w.b, w.V, w.K, w.n_max, dev, torch.from_numpy(roots),
                            torch.from_numpy(ctx), torch.from_numpy(cost), torch.from_numpy(lar))
    sampled = args.temperature > 0
    if sampled:  # stochastic verification with seeded uniforms
        step.set_sampling(args.temperature, torch.from_numpy(synth.verify_uniforms(w)))
    # the target rows are planted at the nodes of the tree this device builds
    tgt_tmp = torch.zeros((w.B, w.n_max, w.V), dtype=xs[0].dtype, device=dev)
    step.run(xs[0], tgt_tmp)
    torch.cuda.synchronize()
    n_nodes = step.tree.n_nodes.cpu().numpy()
    depth = step.tree.depth.cpu().numpy()
    topk_tok = step.topk.tok.cpu().numpy()
    del tgt_tmp
    t_host = synth.host_array((w.B, w.n_max, w.V), w.dtype)
    synth.fill_target_noise(w, t_host.ctypes.data)
    synth.plant_into(w, t_host.ctypes.data, synth.plant_tokens(w, n_nodes, depth, topk_tok))
    t_pin = pinned_from(t_host)
    ts = [t_pin.to(dev) for _ in range(2)]

    bytes_k1 = w.B * w.b * w.V * es
    bytes_k4 = int(n_nodes.sum()) * w.V * es
    bytes_step = bytes_k1 + bytes_k4

    if args.profile_kernel:  # a few direct launches of one kernel, for a profiler
        t, tr, v = step.topk, step.tree, step.ver
        for i in range(args.launches):
            xd, td = xs[i & 1], ts[i & 1]
            if args.profile_kernel in ("topk", "step"):
                bastion.bastion_topk_marginals(xd, w.K, t.logq, t.logit, t.tok, t.lse, step.ws_topk,
                                               step.status)
            if args.profile_kernel in ("tree", "step"):
                bastion.bastion_build_tree(t.logit, t.tok, t.lse, w.n_max, step.root_token, step.ctx_len,
                                           step.cost_ms, step.l_ar, tr.n_nodes, tr.parent, tr.depth,
                                           tr.pos_id, tr.token, tr.rank, tr.log_rho, tr.a_hat,
                                           tr.speedup, tr.anc_mask, step.status)
            if args.profile_kernel in ("verify", "step"):
                step.verify(td)
        torch.cuda.synchronize()
        assert int(step.status.abs().sum()) == 0, "device status bits set"
        return None

    graphs = [step.capture(xs[i], ts[i], chunks=args.chunks) for i in range(2)]
    stream = torch.cuda.current_stream()

    # warm-up (W steps, then, for long runs, ~1 s more so the clocks settle)
    for i in range(args.warmup):
        graphs[i & 1].replay()
    torch.cuda.synchronize()
    t_end = time.time() + (1.0 if args.steps >= 100 else 0.0)
    i = 0
    while time.time() < t_end:
        for _ in range(50):
            graphs[i & 1].replay()
            i += 1
        torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        graphs[i & 1].replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    # keep the GPU busy a little longer so the clock samples cover the region
    for i in range(min(args.steps, 200)):
        graphs[i & 1].replay()
    torch.cuda.synchronize()
    clk = clocks.stop()

    # per-kernel durations: the same steps launched directly with events between
    P = min(args.steps, 100)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(P)]
    t, tr, v = step.topk, step.tree, step.ver
    for p in range(P):
        xd, td = xs[p & 1], ts[p & 1]
        evs[p][0].record(stream)
        bastion.bastion_topk_marginals(xd, w.K, t.logq, t.logit, t.tok, t.lse, step.ws_topk, step.status)
        evs[p][1].record(stream)
        bastion.bastion_build_tree(t.logit, t.tok, t.lse, w.n_max, step.root_token, step.ctx_len,
                                   step.cost_ms, step.l_ar, tr.n_nodes, tr.parent, tr.depth, tr.pos_id,
                                   tr.token, tr.rank, tr.log_rho, tr.a_hat, tr.speedup, tr.anc_mask,
                                   step.status)
        evs[p][2].record(stream)
        step.verify(td)
        evs[p][3].record(stream)
    torch.cuda.synchronize()
    k1 = statistics.mean(evs[p][0].elapsed_time(evs[p][1]) for p in range(P))
    k2 = statistics.mean(evs[p][1].elapsed_time(evs[p][2]) for p in range(P))
    k4 = statistics.mean(evs[p][2].elapsed_time(evs[p][3]) for p in range(P))
    # steps 1-3 as the step runs them (one fused launch where it applies)
    fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(P)]
    for p in range(P):
        fev[p][0].record(stream)
        step.draft(xs[p & 1])
        fev[p][1].record(stream)
    torch.cuda.synchronize()
    k12 = statistics.mean(a_.elapsed_time(b_) for a_, b_ in fev)
    assert int(step.status.abs().sum()) == 0, "device status bits set"
    hbm, peak_kind = peaks()
    ms_step = elapsed_ms / args.steps
    vname = "verify_sample" if sampled else "verify_greedy"
    kern = {"topk_marginals": {"ms": k1, "bytes": bytes_k1, "gbs": bytes_k1 / (k1 * 1e-3) / 1e9},
            "build_tree": {"ms": k2, "bytes": w.B * w.b * w.K * 16},
            "draft_tree": {"ms": k12, "bytes": bytes_k1, "gbs": bytes_k1 / (k12 * 1e-3) / 1e9,
                           "note": "steps 1-3 as the step launches them"},
            vname: {"ms": k4, "bytes": bytes_k4, "gbs": bytes_k4 / (k4 * 1e-3) / 1e9}}
    dom = max(("topk_marginals", vname), key=lambda k: kern[k]["ms"])
    if light:  # one line of the workloads table: no end-to-end leg
        ach = kern[dom]["gbs"]
        return {"workload": w.name, "value": aggregate_rate(args.steps, elapsed_ms, ws), "unit": UNIT,
                "steps": args.steps, "ms_per_step": ms_step, "mean_tree_nodes": float(n_nodes.mean()),
                "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                             "frac": ach / hbm, "peak_source": f"{peak_kind} copy bandwidth",
                             "step_frac": bytes_step / (ms_step * 1e-3) / 1e9 / hbm,
                             "bytes_per_step": bytes_step},
                "kernels": kern, "clocks": clk}

    # end to end through the public API with host buffers (pinned), per step:
    # H2D of the drafter logits (copy engine); the tree; verification reading
    # the target logits of the tree's nodes in place from pinned host memory
    # (only those rows cross the link, sized on the device: no host round trip
    # between the tree and its verification); D2H of the results
    E = max(3, min(args.steps, 20))
    out_host = torch.empty((w.B, w.b + 1), dtype=torch.int32, pin_memory=True)
    acc_host = torch.empty((w.B,), dtype=torch.int32, pin_memory=True)
    xin = torch.empty_like(xs[0])

    def e2e_step():
        xin.copy_(x_pin, non_blocking=True)
        step.draft(xin)
        step.verify(t_pin)
        out_host.copy_(step.ver.out_tokens, non_blocking=True)
        acc_host.copy_(step.ver.accept_len, non_blocking=True)

    acc_graph = step.ver.accept_len.cpu()  # from the graph replays above
    e2e_step()
    torch.cuda.synchronize()
    assert torch.equal(acc_host, acc_graph), "end-to-end result differs from the device-resident one"
    barrier(ws)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(E):
        e2e_step()
    f1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(f0.elapsed_time(f1), ws) / E
    h2d = x_pin.numel() * x_pin.element_size() + int(n_nodes.sum()) * w.V * es
    d2h = out_host.numel() * 4 + acc_host.numel() * 4
    # the host link's own rate: pinned host-to-device copies of the drafter logits
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for _ in range(5):
        xin.copy_(x_pin, non_blocking=True)
    l1.record(stream)
    torch.cuda.synchronize()
    link_gbs = 5 * x_pin.numel() * x_pin.element_size() / (l0.elapsed_time(l1) * 1e-3) / 1e9

    # the cost model's calibration on the device (1,024 observed samples), timed alone
    cal_n = torch.from_numpy(np.linspace(1, w.n_max, 1024).astype(np.float32)).to(dev)
    cal_t = torch.from_numpy((2.0 + 0.01 * np.linspace(1, w.n_max, 1024)).astype(np.float32)).to(dev)
    cal_c = torch.zeros(w.n_max + 1, dtype=torch.float32, device=dev)
    cal_p = torch.zeros(2, dtype=torch.float32, device=dev)
    cal_s = torch.zeros(1, dtype=torch.int32, device=dev)
    roof8b = dict(bytes0=16e9, bytes1=2.0e6, flops0=0.0, flops1=16e9, bw=8e9, peak=2.25e12)
    for _ in range(10):
        bastion.bastion_calibrate_cost(cal_n, cal_t, roof8b, 2.5, w.n_max, cal_c, cal_p, cal_s)
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for _ in range(P):
        bastion.bastion_calibrate_cost(cal_n, cal_t, roof8b, 2.5, w.n_max, cal_c, cal_p, cal_s)
    c1.record(stream)
    torch.cuda.synchronize()
    k_cal = c0.elapsed_time(c1) / P
    assert int(cal_s.item()) == 0

    kern["calibrate_cost"] = {"ms": k_cal, "samples": 1024, "note": "outside the step"}
    ach = kern[dom]["gbs"]
    res = {
        "metric": (METRIC if not sampled else
                   METRIC.replace("+verify)", f"+sampled verify, T={args.temperature:g})")),
        "value": aggregate_rate(args.steps, elapsed_ms, ws), "unit": UNIT,
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": step_config(w, float(n_nodes.mean()), ws),
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                     "frac": ach / hbm, "peak_source": f"{peak_kind} copy bandwidth",
                     "traffic": (profiled_traffic(*{"topk_marginals": ("topk_marginals_b32_v151936.md",
                                                                       "topk_marginals.cu"),
                                                    "verify_greedy": ("verify_greedy_b32_v151936.md",
                                                                      "verify_greedy.cu"),
                                                    "verify_sample": ("verify_sample_b32_v151936.md",
                                                                      "verify_sample.cu")}[dom])
                                 if w.cid == 3 else None),
                     "step_frac": bytes_step / (ms_step * 1e-3) / 1e9 / hbm,
                     "bytes_per_step": bytes_step},
        "kernels": kern,
        "clocks": clk,
        "e2e": {"value": aggregate_rate(1, e2e_ms, ws), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "h2d_gbs": h2d / (e2e_ms * 1e-3) / 1e9,
                "link_copy_gbs": link_gbs,
                "note": "target rows read in place from pinned host memory by the verify sweep"},
        # top-K, tree, verify sweep, (sampled: the draws,) verify finish
        "gpu_launches": (5 if sampled else 4) * args.steps,
    }
    return res


def run_with_attention(args, ws, rank, local, light=False):
    """Workload 4: one tree-masked GQA attention call per step (8 requests, 32/8
    heads, d 128, ctx 4096, trees of 64 nodes).  Workload 5: the full serving
    step, top-K + tree + attention + verify (64 requests, vocab 128,256, trees of
    256 nodes over a 16,384-token cache)."""
    import torch

    import synth
    from draft_tree_build_gb300 import bastion

    dev = torch.device(f"cuda:{local}")
    w = synth.workload(args.workload)
    es = w.elem_bytes
    roots, ctx, cost, lar = synth.root_tokens(w), synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w)
    x_host = synth.drafter_logits(w)
    x_pin = pinned_from(x_host)
    xd = x_pin.to(dev)
    step = bastion.TreeStep(w.B, w.b, w.V, w.K, w.n_max, dev, torch.from_numpy(roots),
                            torch.from_numpy(ctx), torch.from_numpy(cost), torch.from_numpy(lar))
    tgt_tmp = torch.zeros((w.B, w.n_max, 1 if args.workload == 4 else w.V), dtype=xd.dtype, device=dev)
    if args.workload == 4:
        # the tree only: run steps 1-3
        t, tr = step.topk, step.tree
        bastion.bastion_topk_marginals(xd, w.K, t.logq, t.logit, t.tok, t.lse, step.ws_topk, step.status)
        bastion.bastion_build_tree(t.logit, t.tok, t.lse, w.n_max, step.root_token, step.ctx_len,
                                   step.cost_ms, step.l_ar, tr.n_nodes, tr.parent, tr.depth, tr.pos_id,
                                   tr.token, tr.rank, tr.log_rho, tr.a_hat, tr.speedup, tr.anc_mask,
                                   step.status)
    else:
        step.run(xd, tgt_tmp)
    torch.cuda.synchronize()
    n_nodes = step.tree.n_nodes.cpu().numpy()
    depth = step.tree.depth.cpu().numpy()
    topk_tok = step.topk.tok.cpu().numpy()
    del tgt_tmp
    if args.workload == 5:
        t_host = synth.host_array((w.B, w.n_max, w.V), w.dtype)
        synth.fill_target_noise(w, t_host.ctypes.data)
        synth.plant_into(w, t_host.ctypes.data, synth.plant_tokens(w, n_nodes, depth, topk_tok))
        td = pinned_from(t_host).to(dev)
        del t_host
    q = torch.empty((w.B, w.n_max, w.Hq, w.D), dtype=torch.int16, pin_memory=True)
    k = torch.empty((w.B, w.L_cap, w.Hkv, w.D), dtype=torch.int16, pin_memory=True)
    v = torch.empty_like(k)
    synth.fill_attention(w, q.data_ptr(), k.data_ptr(), v.data_ptr())
    qd, kd, vd = (t.view(torch.bfloat16).to(dev) for t in (q, k, v))
    del q, k, v
    out = torch.empty((w.B, w.n_max, w.Hq, w.D), dtype=torch.bfloat16, device=dev)
    ws_attn = bastion.workspace(bastion.bastion_tree_attention_workspace_bytes(
        w.B, w.n_max, w.Hq, w.Hkv, w.D, w.L_cap), dev)
    ctx_d = torch.from_numpy(ctx).to(dev)
    scale = 1.0 / math.sqrt(w.D)
    stream = torch.cuda.current_stream()
    tr = step.tree

    def attn():
        bastion.bastion_tree_attention(qd, kd, vd, ctx_d, tr.n_nodes, tr.anc_mask, scale, out, ws_attn,
                                       step.status)

    def full():
        t, v_ = step.topk, step.ver
        bastion.bastion_topk_marginals(xd, w.K, t.logq, t.logit, t.tok, t.lse, step.ws_topk, step.status)
        bastion.bastion_build_tree(t.logit, t.tok, t.lse, w.n_max, step.root_token, step.ctx_len,
                                   step.cost_ms, step.l_ar, tr.n_nodes, tr.parent, tr.depth, tr.pos_id,
                                   tr.token, tr.rank, tr.log_rho, tr.a_hat, tr.speedup, tr.anc_mask,
                                   step.status)
        attn()
        bastion.bastion_verify_greedy(td, w.b, tr.n_nodes, tr.parent, tr.token, v_.argmax, v_.accept_len,
                                      v_.accept_nodes, v_.out_tokens, step.ws_verify, step.status)

    body = attn if args.workload == 4 else full
    body()
    torch.cuda.synchronize()
    if args.profile_kernel:  # a few direct launches, for a profiler
        for _ in range(args.launches):
            attn() if args.profile_kernel == "attn" else full()
        torch.cuda.synchronize()
        return None
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        body()
    for _ in range(args.warmup):
        g.replay()
    torch.cuda.synchronize()
    t_end = time.time() + (1.0 if args.steps >= 100 else 0.0)
    while time.time() < t_end:
        for _ in range(10):
            g.replay()
        torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    for _ in range(min(args.steps, 50)):
        g.replay()
    torch.cuda.synchronize()
    clk = clocks.stop()
    # attention kernel alone, events around each launch
    P = min(args.steps, 50)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(P)]
    for a_, b_ in evs:
        a_.record(stream)
        attn()
        b_.record(stream)
    torch.cuda.synchronize()
    t_attn = statistics.mean(a_.elapsed_time(b_) for a_, b_ in evs)
    assert int(step.status.abs().sum()) == 0, "device status bits set"

    hbm, peak_kind = peaks()
    pk = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))) if peak_kind == "measured" else {}
    # a kernel of milliseconds launched back to back runs under the power cap:
    # the sustained figure; a short one, timed alone: the burst figure
    long_kernel = t_attn >= 1.0
    tf_peak = float(pk.get("bf16_tflops_sustained" if long_kernel else "bf16_tflops",
                           1700.0 if long_kernel else 1900.0))
    tf_kind = f"{peak_kind} bf16 ({'sustained' if long_kernel else 'burst'})"
    G = w.Hq // w.Hkv
    vis_pairs = 0  # visible (query row, key) pairs per KV head: context + own root path
    for r in range(w.B):
        n = int(n_nodes[r])
        vis_pairs += n * int(ctx[r]) + int((depth[r, :n] + 1).sum())
    flops = 4.0 * w.D * G * w.Hkv * vis_pairs
    bytes_attn = (w.B * w.Hkv * (int(ctx.mean()) + w.n_max) * w.D * 2 * 2
                  + 2 * w.B * w.n_max * w.Hq * w.D * 2)
    t_mem = bytes_attn / (hbm * 1e9)
    t_tc = flops / (tf_peak * 1e12)
    bound = "hbm" if t_mem >= t_tc else "tensor"
    ms_step = elapsed_ms / args.steps
    if bound == "hbm":
        roof = {"bound": "hbm", "kernel": "tree_attention", "achieved": bytes_attn / (t_attn * 1e-3) / 1e9,
                "peak": hbm, "unit": "GB/s", "peak_source": f"{peak_kind} copy bandwidth"}
    else:
        roof = {"bound": "tensor", "kernel": "tree_attention", "achieved": flops / (t_attn * 1e-3) / 1e12,
                "peak": tf_peak, "unit": "TFLOP/s", "peak_source": tf_kind}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = (profiled_traffic("tree_attention_b8_ctx4096_n64.md", "tree_attention.cu")
                       if args.workload == 4 else None)
    roof["roofline_us"] = max(t_mem, t_tc) * 1e6
    roof["attn_bytes"] = bytes_attn
    roof["attn_flops"] = flops
    metric = ("tree-attention calls/s (B=8, 32/8 heads, d=128, ctx 4096, N=64)" if args.workload == 4
              else "full tree steps/s (top-K+best-first+attention+verify) B=64 V=128256 ctx 16384 N=256")
    if light:  # one line of the workloads table
        return {"workload": w.name, "metric": metric, "value": aggregate_rate(args.steps, elapsed_ms, ws),
                "unit": "calls/s" if args.workload == 4 else "steps/s", "steps": args.steps,
                "ms_per_step": ms_step, "mean_tree_nodes": float(n_nodes.mean()), "roofline": roof,
                "kernels": {"tree_attention": {"ms": t_attn}}, "clocks": clk}
    return {
        "metric": metric, "value": aggregate_rate(args.steps, elapsed_ms, ws),
        "unit": "calls/s" if args.workload == 4 else "steps/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16-in/f32-acc", "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "n_max": w.n_max, "ctx": w.ctx, "Hq": w.Hq, "Hkv": w.Hkv,
                   "D": w.D, "mean_tree_nodes": float(n_nodes.mean()),
                   "l2": "inputs larger than L2", "parallelism": f"replicas x{ws}"},
        "roofline": roof, "kernels": {"tree_attention": {"ms": t_attn}}, "clocks": clk,
        "gpu_launches": (1 if args.workload == 4 else 5) * args.steps,  # + attention
    }


# --------------------------------------------------------------------------- oracle legs

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


class OracleStep:
    """The oracle's tree step (top-K of a request's b rows, its tree, the
    verification of its target rows), request by request.  The target rows are
    planted at the oracle's own trees, outside any timing.  The oracle is C
    called through ctypes, which releases the GIL: a thread pool runs requests
    on several host cores at once."""

    def __init__(self, args, w):
        import oracle
        import synth
        self.args, self.w = args, w
        self.pre = (synth.root_tokens(w), synth.ctx_lens(w), synth.cost_table(w), synth.l_ar(w))
        self.x = synth.drafter_logits(w)
        tk_all = oracle.topk_marginals(self.x, w.K)
        tr_all = oracle.build_tree(tk_all.logit, tk_all.tok, tk_all.lse, w.n_max, *self.pre)
        self.mean_nodes = float(tr_all.n_nodes.mean())
        self.tgt, _ = synth.target_logits(w, tr_all.n_nodes, tr_all.depth, tk_all.tok)
        self.u = synth.verify_uniforms(w)

    def request(self, r):
        import oracle
        w, (roots, ctx, cost, lar) = self.w, self.pre
        tk = oracle.topk_marginals(self.x[r:r + 1], w.K)
        tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, roots[r:r + 1], ctx[r:r + 1],
                               cost, lar[r:r + 1])
        if self.args.temperature > 0:
            oracle.verify_sample(self.tgt[r:r + 1], w.b, self.args.temperature, self.u[r:r + 1],
                                 tr.n_nodes, tr.parent, tr.token)
        else:
            oracle.verify_greedy(self.tgt[r:r + 1], w.b, tr.n_nodes, tr.parent, tr.token)

    def step(self, pool=None):
        """One whole step: every request of the batch."""
        if pool is None:
            for r in range(self.w.B):
                self.request(r)
        else:
            list(pool.map(self.request, range(self.w.B)))


def cpu_baseline(args, budget_s=12.0):
    """Times the oracle as it stands on the host cores, on a bounded sample of
    the bench workload: whole requests on one thread for half the budget, then
    whole steps with the requests split over every host core for the other
    half.  The all-cores figure is the line's value."""
    from concurrent.futures import ThreadPoolExecutor

    import synth
    w = synth.workload(args.workload)
    o = OracleStep(args, w)
    t0 = time.perf_counter()
    done = 0
    while True:
        o.request(done % w.B)
        done += 1
        if time.perf_counter() - t0 > budget_s / 2:
            break
    dt1 = time.perf_counter() - t0
    single = 1.0 / (dt1 / done * w.B)
    n = host_cores()
    with ThreadPoolExecutor(n) as pool:
        o.step(pool)
        t0 = time.perf_counter()
        steps = 0
        while True:
            o.step(pool)
            steps += 1
            if time.perf_counter() - t0 > budget_s / 2:
                break
        dt = time.perf_counter() - t0
    return {"value": steps / dt, "unit": UNIT, "cores": n, "kind": "oracle", "nproc": n,
            "sample": f"{steps} whole {w.B}-request steps (top-K of 16 rows, tree, verify of its rows, "
                      f"per request) of the {w.name} workload in {dt:.1f} s, requests split over "
                      f"{n} host threads",
            "single_thread": {"value": single, "unit": UNIT, "cores": 1,
                              "sample": f"{done} whole requests in {dt1:.1f} s on one thread, "
                                        f"scaled to a {w.B}-request step"}}


def run_reference(args, ws, rank):
    """Reference arm: the oracle, as it stands, on the host cores; each step is
    one whole step of the workload (every request), the requests split over
    all host cores."""
    from concurrent.futures import ThreadPoolExecutor

    import synth
    w = synth.workload(args.workload)
    o = OracleStep(args, w)
    n = host_cores()
    with ThreadPoolExecutor(n) as pool:
        for _ in range(args.warmup):
            o.step(pool)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            o.step(pool)
        dt = time.perf_counter() - t0
    val = args.steps / dt
    metric = METRIC if args.temperature <= 0 else METRIC.replace(
        "+verify)", f"+sampled verify, T={args.temperature:g})")
    return {"impl": "reference", "metric": metric, "value": val, "unit": UNIT, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": step_config(w, o.mean_nodes, ws),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": n, "kind": "oracle", "nproc": n,
                             "sample": f"each step one whole {w.B}-request step (top-K, tree, verify "
                                       f"per request), the requests split over {n} host threads"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_lm_head(args, ws, rank, local, light=True):
    """The fused drafter LM-head + top-K on the batched workload's drafter: the
    32 x 16 final hidden states (hidden size 4,096, Qwen3-8B) times an output
    embedding of 151,936 rows, top-64 per row; tensor-bound (0.64 TFLOP per
    call), against the sustained bf16 peak (a kernel of ~0.6 ms launched back
    to back runs under the power cap)."""
    import torch

    import synth
    from draft_tree_build_gb300 import bastion

    dev = torch.device(f"cuda:{local}")
    B, b, H, V, K = 32, 16, 4096, 151936, 64
    hid, w = synth.lm_head_inputs(B, b, H, V, seed=0xBA5710 + 6)
    hd = torch.from_numpy(hid.view(np.int16)).view(torch.bfloat16).to(dev)
    wd = torch.from_numpy(w.view(np.int16)).view(torch.bfloat16).to(dev)
    del hid, w
    t = bastion.alloc_topk(B, b, K, dev)
    wsp = bastion.workspace(bastion.bastion_lm_head_topk_workspace_bytes(B, b, V, K), dev)
    st = torch.zeros(B, dtype=torch.int32, device=dev)

    def call():
        bastion.bastion_lm_head_topk(hd, wd, K, t.logq, t.logit, t.tok, t.lse, wsp, st)

    if args.profile_kernel:
        for _ in range(args.launches):
            call()
        torch.cuda.synchronize()
        return None
    steps, warm = (20, 3) if light else (args.steps, args.warmup)
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    clk = clocks.stop()
    assert int(st.abs().sum()) == 0, "device status bits set"
    ms = elapsed_ms / steps
    flops = 2.0 * B * b * H * V
    pk_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    pk = json.load(open(pk_path)) if os.path.exists(pk_path) else {}
    peak = float(pk.get("bf16_tflops_sustained", 1700.0))
    kind = "measured" if pk else "fallback"
    ach = flops / (ms * 1e-3) / 1e12
    return {"workload": f"lmhead-b{B}x{b}-h{H}-v{V}-k{K}-bf16",
            "metric": "fused drafter LM-head + top-K calls/s (512 x 4096 x 151936, top-64)",
            "value": aggregate_rate(steps, elapsed_ms, ws), "unit": "calls/s", "steps": steps,
            "ms_per_step": ms,
            "roofline": {"bound": "tensor", "kernel": "lm_head_topk", "achieved": ach, "peak": peak,
                         "unit": "TFLOP/s", "frac": ach / peak, "peak_source": f"{kind} bf16 (sustained)",
                         "flops": flops},
            "clocks": clk}


def run_mixture(args, ws, rank, local, light=True):
    """Best-first trees on a latent-mixture proposal (DBlast's dependent block
    proposal, Bastion's controller): B = 32 requests, Z = 4 branches, b = 16
    positions, the top-64 of each branch's bf16 logits over 151,936 tokens
    (found by the top-K kernel before the timed region), n_max = 128 and a flat
    cost table, so every tree fills the budget: the longest build.  The build
    is one warp's sequence of pops per request, bound by latency; the HBM
    figure relates the inputs it reads to the call's time."""
    import torch

    import synth
    from draft_tree_build_gb300 import bastion

    dev = torch.device(f"cuda:{local}")
    B, Z, b, V, K, n_max = 32, 4, 16, 151936, 64, 128
    x, pi = synth.mixture_inputs(B, Z, b, V, seed=0xBA5710 + 7)
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).to(dev).view(B * Z, b, V)
    del x
    t = bastion.alloc_topk(B * Z, b, K, dev)
    st = torch.zeros(B * Z, dtype=torch.int32, device=dev)
    wsp = bastion.workspace(bastion.bastion_topk_marginals_workspace_bytes(B * Z, b, V, K), dev)
    bastion.bastion_topk_marginals(xd, K, t.logq, t.logit, t.tok, t.lse, wsp, st)
    torch.cuda.synchronize()
    del xd, wsp
    lg, tk, ls = t.logit.view(B, Z, b, K), t.tok.view(B, Z, b, K), t.lse.view(B, Z, b)
    pid = torch.from_numpy(np.ascontiguousarray(pi)).to(dev)
    w = synth.workload(3)
    roots = torch.from_numpy(synth.root_tokens(w)).to(dev)
    ctx = torch.from_numpy(synth.ctx_lens(w)).to(dev)
    lar = torch.from_numpy(synth.l_ar(w)).to(dev)
    cost = torch.full((n_max + 1,), 5.0, dtype=torch.float32, device=dev)
    tr = bastion.alloc_tree(B, n_max, dev)
    wsm = bastion.workspace(bastion.bastion_build_tree_mixture_workspace_bytes(B, Z, b, K, n_max), dev)

    def call():
        bastion.bastion_build_tree_mixture(lg, tk, ls, pid, n_max, roots, ctx, cost, lar, tr.n_nodes,
                                           tr.parent, tr.depth, tr.pos_id, tr.token, tr.log_rho,
                                           tr.a_hat, tr.speedup, tr.anc_mask, wsm, st[:B])

    if args.profile_kernel:
        for _ in range(args.launches):
            call()
        torch.cuda.synchronize()
        return None
    steps, warm = (200, 10) if light else (args.steps, args.warmup)
    for _ in range(warm):
        call()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        call()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    elapsed_ms = max_over_ranks(e0.elapsed_time(e1), ws)
    clk = clocks.stop()
    assert int(st.abs().sum()) == 0, "device status bits set"
    assert int(tr.n_nodes.min()) == n_max
    ms = elapsed_ms / steps
    # inputs read per call: logits, tokens (4 B each per entry), lse, pi, cost
    nbytes = B * Z * b * K * 8 + B * Z * b * 8 + B * Z * 8 + (n_max + 1) * 4
    hbm, peak_kind = peaks()
    ach = nbytes / (ms * 1e-3) / 1e9
    return {"workload": f"mixture-b{B}-z{Z}-b{b}-k{K}-n{n_max}-flat",
            "metric": "latent-mixture tree builds/s (32 requests, Z=4, K=64, n_max=128, every tree full)",
            "value": aggregate_rate(steps, elapsed_ms, ws), "unit": "calls/s", "steps": steps,
            "ms_per_step": ms, "us_per_call": ms * 1e3,
            "roofline": {"bound": "hbm", "kernel": "build_tree_mixture", "achieved": ach, "peak": hbm,
                         "unit": "GB/s", "frac": ach / hbm, "peak_source": f"{peak_kind} copy bandwidth",
                         "note": "sequential pops per request on one SM (four warps): latency-bound, not HBM-bound"},
            "clocks": clk}


# steps and warm-up of each other workload's line: microsecond steps get many
# repetitions, the millisecond serving step a few
SUB_STEPS = {1: (500, 20), 2: (500, 20), 4: (200, 10), 5: (10, 3)}


def other_workloads(args, ws, rank, local) -> dict:
    """The other four workloads, each measured like the headline (graph replay,
    CUDA events, max over ranks) with its dominant kernel's roofline: the
    latency cases (1, 2), the attention layer (4) and the serving step (5)."""
    import gc

    import torch
    out = {}
    for wid in (1, 2, 4, 5):
        sub = argparse.Namespace(**vars(args))
        sub.workload = wid
        sub.steps, sub.warmup = SUB_STEPS[wid]
        sub.chunks = 1
        r = (run_with_attention if wid in (4, 5) else run_ours)(sub, ws, rank, local, light=True)
        out[str(wid)] = r
        gc.collect()
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    out["lm_head"] = run_lm_head(args, ws, rank, local, light=True)
    gc.collect()
    torch.cuda.empty_cache()
    out["mixture"] = run_mixture(args, ws, rank, local, light=True)
    gc.collect()
    torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", type=int, default=3, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lm-head", action="store_true",
                    help="only the fused drafter LM-head + top-K line")
    ap.add_argument("--no-workloads", action="store_true",
                    help="the headline line only (no table of the other four workloads)")
    ap.add_argument("--mixture", action="store_true",
                    help="only the latent-mixture tree line")
    ap.add_argument("--profile-kernel", choices=["topk", "tree", "verify", "step", "attn", "lmhead",
                                                 "mixture"],
                    help="launch one kernel (or the step) --launches times and exit, for ncu")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--temperature", type=float, default=0.0,
                    help="verify by sampling at this temperature (0: greedy, the headline)")
    ap.add_argument("--chunks", type=int, default=1,
                    help="request chunks of the step on forked streams inside the graph")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        ws = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return
        steps = args.steps
        res = run_reference(args, ws, rank)
        print(json.dumps(res), flush=True)
        return

    ws, rank, local = dist_setup()
    if args.mixture or args.profile_kernel == "mixture":
        res = run_mixture(args, ws, rank, local, light=False)
        if res is None:
            print("profile launches done", flush=True)
        elif rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.lm_head or args.profile_kernel == "lmhead":
        res = run_lm_head(args, ws, rank, local, light=False)
        if res is None:
            print("profile launches done", flush=True)
        elif rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.workload in (4, 5):
        res = run_with_attention(args, ws, rank, local)
    else:
        res = run_ours(args, ws, rank, local)
    if (res is not None and args.workload == 3 and not args.no_workloads and not args.profile_kernel
            and args.temperature <= 0):
        res["workloads"] = other_workloads(args, ws, rank, local)
    if res is None:
        print("profile launches done", flush=True)
    elif rank == 0:
        if ws == 1 and not args.no_cpu_baseline and args.workload not in (4, 5):
            res["cpu_baseline"] = cpu_baseline(args)
        print(json.dumps(res), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
