"""Pins for the oracle's calibration of the verification cost model (no GPU).

Bastion (gist.science/nl/paper/2605.29727), "Methodologie" §3,
"Latentiemodellering": T_verify(N) comes from a roofline model of memory
bandwidth and compute, calibrated with observed runtimes.  Reading: the
calibration is the least-squares line T_verify = alpha roof(N) + beta, and the
controller's table is C(N) = t_draft + T_verify(N).
"""
import numpy as np
import pytest

import oracle
import synth

# an 8B-parameter target in bf16: 16 GB of weights, 2 * 8e9 flop per token;
# units: bytes per ms and flop per ms, so roof() is in ms
ROOF = dict(bytes0=16e9, bytes1=2.0e6, flops0=0.0, flops1=16e9, bw=8e9, peak=2.25e12)


def roof(n, r=ROOF):
    n = np.asarray(n, np.float64)
    return np.maximum((r["bytes0"] + r["bytes1"] * n) / r["bw"], (r["flops0"] + r["flops1"] * n) / r["peak"])


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (1.3, 0.4), (0.8, 2.5)])
def test_noise_free_samples_recover_the_line(alpha, beta):
    n = np.array([1, 16, 64, 256, 1024, 2048, 4096], np.float64)  # both sides of the kink
    cost, a, b = oracle.calibrate_cost(n, alpha * roof(n) + beta, ROOF, 3.0, 256)
    assert a == pytest.approx(alpha, rel=1e-12) and b == pytest.approx(beta, rel=1e-12, abs=1e-12)


def test_noisy_samples_match_library_polyfit():
    rng = np.random.default_rng(4)
    n = rng.integers(1, 4000, size=200).astype(np.float64)
    t = 1.15 * roof(n) + 0.7 + rng.normal(scale=0.05, size=n.size)
    _, a, b = oracle.calibrate_cost(n, t, ROOF, 0.0, 8)
    pa, pb = np.polyfit(roof(n), t, 1)
    assert a == pytest.approx(pa, rel=1e-9) and b == pytest.approx(pb, rel=1e-9)


def test_no_spread_keeps_the_roofline_slope():
    n = np.full(5, 32.0)
    t = np.array([2.5, 2.6, 2.4, 2.55, 2.45])
    _, a, b = oracle.calibrate_cost(n, t, ROOF, 0.0, 8)
    assert a == 1.0 and b == pytest.approx(float(np.mean(t - roof(n))), rel=1e-12)


def test_table_is_flat_then_linear_past_the_kink():
    """Memory-bound until the token flops pass the weight bytes' time, then a
    slope of alpha * flops1 / peak per node."""
    n = np.array([1, 100, 2000, 4000], np.float64)
    cost, a, b = oracle.calibrate_cost(n, 1.2 * roof(n) + 0.3, ROOF, 2.0, 3000)
    kink = int(np.ceil((ROOF["bytes0"] / ROOF["bw"]) * ROOF["peak"] / (ROOF["flops1"] - ROOF["bytes1"] * ROOF["peak"] / ROOF["bw"])))
    d = np.diff(cost)
    assert np.allclose(d[: kink - 2], 1.2 * ROOF["bytes1"] / ROOF["bw"], rtol=1e-9)
    assert np.allclose(d[kink + 1:], 1.2 * ROOF["flops1"] / ROOF["peak"], rtol=1e-9)
    assert cost[0] == pytest.approx(2.0 + 1.2 * roof(0) + 0.3)


def test_reproduces_the_serving_workload_cost_table():
    """The serving workload's cost model (T_draft 3 ms, roofline of an 8B target
    on 8 TB/s and 2.25 PFLOP/s, plus 1 ms) is the calibrated table with
    alpha = 1, beta = 1 from noise-free samples of itself."""
    w = synth.workload(5)
    r = dict(bytes0=16e9, bytes1=0.0, flops0=0.0, flops1=16e9, bw=8e9, peak=2.25e12)
    n = np.array([1, 50, 200, 281, 282, 256, 1000], np.float64)
    t = np.array([synth.cost_ms(int(k), w.cost) for k in n]) - 3.0
    cost, a, b = oracle.calibrate_cost(n, t, r, 3.0, w.n_max)
    assert a == pytest.approx(1.0, rel=1e-12) and b == pytest.approx(1.0, rel=1e-12)
    assert np.allclose(cost.astype(np.float32), synth.cost_table(w)[0], rtol=1e-6)
