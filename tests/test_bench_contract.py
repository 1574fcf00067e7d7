"""The benchmark's reference arm (the oracle timed on the host) keeps the
one-line JSON contract, on the CPU: the keys, their types, and that ranks other
than 0 print nothing and exit 0."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*args, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, env=e,
                          capture_output=True, text=True, timeout=600)


def test_reference_arm_line():
    r = _bench("--impl", "reference", "--workload", "1", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference"
    for k in ("metric", "unit", "dtype", "data", "scaling"):
        assert isinstance(d[k], str) and d[k]
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"]["workload"] == "tiny-b4-v1024-k8-n16-f32"
    # the same config dict as the GPU arm's line for this workload
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synth
    w = synth.workload(1)
    tk = oracle.topk_marginals(synth.drafter_logits(w), w.K)
    tr = oracle.build_tree(tk.logit, tk.tok, tk.lse, w.n_max, synth.root_tokens(w), synth.ctx_lens(w),
                           synth.cost_table(w), synth.l_ar(w))
    assert d["config"] == bench.step_config(w, float(tr.n_nodes.mean()), 1)
    # whole steps: the timed steps fit in the run
    assert d["ms_per_step"] * d["steps"] < 60e3
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    r = _bench("--impl", "reference", "--workload", "1", "--steps", "1", "--warmup", "3",
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_cpu_baseline_reports_single_thread_and_all_cores():
    import argparse
    sys.path.insert(0, ROOT)
    import bench
    args = argparse.Namespace(workload=1, temperature=0.0)
    cb = bench.cpu_baseline(args, budget_s=0.4)
    assert cb["kind"] == "oracle" and cb["value"] > 0 and cb["unit"] == bench.UNIT
    assert cb["cores"] == cb["nproc"] == bench.host_cores() >= 1
    st = cb["single_thread"]
    assert st["cores"] == 1 and st["value"] > 0 and st["sample"]
