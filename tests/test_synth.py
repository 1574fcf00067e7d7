"""Pins for the seeded input generator (no GPU)."""
import math
from fractions import Fraction

import numpy as np
import pytest

import synth


def test_splitmix64_published_values():
    # Published splitmix64 outputs for seed 1234567 (Vigna's reference C code).
    assert synth.splitmix64_sequence(1234567, 5) == [
        6457827717110365317, 3203168211198807973, 9817491932198370423,
        4593380528125082431, 16408922859458223821]


def test_counter_addressing_is_order_free():
    a = synth.uniforms(7, 3, 100)
    b = np.concatenate([synth.uniforms(7, 3, 40), synth.uniforms(7, 3, 60, offset=40)])
    assert np.array_equal(a, b)
    assert np.all((a > 0) & (a < 1))
    z = synth.normals(7, 3, 50)
    buf = np.empty(50, np.float32)
    synth.fill_normal(buf.ctypes.data, 50, "f32", 1.0, 7, 3)
    assert np.array_equal(buf, z.astype(np.float32))


def test_normal_moments_and_shape():
    from scipy import stats
    z = np.empty(200000, np.float32)
    synth.fill_normal(z.ctypes.data, z.size, "f32", 1.0, 11, 1)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    assert stats.kstest(z[:20000], "norm").pvalue > 1e-3
    assert np.abs(z).max() < 8.7  # Box-Muller bound with u1 >= 2^-54


def _bf16_exact(x: float) -> int:
    """Reference RNE rounding of a double to bf16, in exact rational arithmetic."""
    if math.isnan(x):
        return 0x7FC0
    sign = 0x8000 if math.copysign(1.0, x) < 0 else 0
    a = abs(x)
    if math.isinf(a):
        return sign | 0x7F80
    if a == 0:
        return sign
    fa = Fraction(a)
    e = math.frexp(a)[1]
    q = Fraction(2) ** max(e - 8, -133)
    n = fa / q
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    y = fl * q
    if y > Fraction(3.3895313892515355e38):
        return sign | 0x7F80
    import struct
    bits = struct.unpack("<I", struct.pack("<f", float(y)))[0]
    return sign | ((bits >> 16) & 0x7FFF)


def test_bf16_round_to_nearest_even():
    rng = np.random.default_rng(0)
    xs = list(rng.normal(size=2000) * 10.0 ** rng.integers(-40, 39, size=2000))
    # halfway cases and edges
    xs += [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 2 ** -130, 2 ** -134, 2 ** -133 * 1.5,
           3.4e38, 3.3961e38, 0.0, -0.0, float("inf"), -float("inf"), 12.0, 16.87]
    for x in xs:
        assert synth.f64_to_bf16_bits(x) == _bf16_exact(float(x)), x
    assert synth.f64_to_bf16_bits(float("nan")) == 0x7FC0


def test_bf16_matches_torch_on_float_values():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(1)
    x = (rng.normal(size=5000) * 30).astype(np.float32)
    ours = np.array([synth.f64_to_bf16_bits(float(v)) for v in x], dtype=np.uint16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_cost_models():
    # tiny: 3 + 20 + 0.1 max(0, N-8); knee32: 2.5 + 18 + 0.04 max(0, N-32)
    assert synth.cost_ms(8, "tiny") == 23.0 and abs(synth.cost_ms(10, "tiny") - 23.2) < 1e-12
    assert synth.cost_ms(32, "knee32") == 20.5 and abs(synth.cost_ms(42, "knee32") - 20.9) < 1e-12
    c5 = [synth.cost_ms(N, "roofline-flat281") for N in range(1, 300)]
    assert all(c == 6.0 for c in c5[:281]) and c5[281] > 6.0


def test_workload_shapes():
    for cid, w in synth.WORKLOADS.items():
        assert w.seed == 0xBA5710 + cid
        assert 1 <= w.K <= w.V and w.n_max <= 256 and w.b <= 32
        t = synth.cost_table(w)
        assert t.shape == (1, w.n_max + 1) and np.all(t > 0)
    w = synth.workload(3)
    p = synth.top1_targets(w)
    assert np.all((p[:, 0] >= 0.3) & (p[:, 0] <= 0.99))
    assert np.allclose(p[:, 1:] / p[:, :-1], 0.9)


def test_plant_rule():
    w = synth.workload(1)
    n_nodes = np.array([5])
    depth = np.zeros((1, w.n_max), np.int32)
    depth[0, :5] = [0, 1, 1, 2, 4]
    tok = np.arange(w.b * w.K, dtype=np.int32).reshape(1, w.b, w.K) + 100
    pl = synth.plant_tokens(w, n_nodes, depth, tok)
    for i, d in enumerate(depth[0, :5]):
        if d < w.b:
            assert pl[0, i] in tok[0, d]
    assert np.all(pl[0, 5:] == -1)
    x = np.zeros((1, w.n_max, w.V), np.float32)
    synth.plant_into(w, x.ctypes.data, pl)
    for i in range(5):
        assert x[0, i, pl[0, i]] == synth.PLANT_VALUE
