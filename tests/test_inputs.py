"""The shared input generator: determinism, slicing and distribution."""
import math

import numpy as np

import lmoe_inputs as gen


def test_counter_based_slices_are_consistent():
    a = gen.normal_f32(0, 3, 0, 1000, 1.0)
    b = gen.normal_f32(0, 3, 371, 200, 1.0)
    np.testing.assert_array_equal(a[371:571], b)
    c = gen.normal_f32(0, 3, 0, 1000, 1.0)
    np.testing.assert_array_equal(a, c)
    assert not np.array_equal(a, gen.normal_f32(0, 4, 0, 1000, 1.0))
    assert not np.array_equal(a, gen.normal_f32(1, 3, 0, 1000, 1.0))


def test_multithreaded_equals_single_slice():
    n = 300_000
    big = gen.normal_f32(0, 5, 10, n, 0.5)
    parts = np.concatenate([gen.normal_f32(0, 5, 10 + i, 50_000, 0.5) for i in range(0, n, 50_000)])
    np.testing.assert_array_equal(big, parts)


def test_normal_moments():
    z = gen.normal_f32(0, 9, 0, 2_000_000, 1.0).astype(np.float64)
    assert abs(z.mean()) < 3e-3 and abs(z.std() - 1) < 3e-3
    assert abs((z ** 4).mean() - 3) < 3e-2          # Gaussian kurtosis
    assert abs((np.abs(z) < 1).mean() - 0.682689) < 2e-3


def test_deterministic_elementary_functions_are_accurate():
    for x in [1e-300, 1e-10, 0.1, 0.5, 0.7071, 0.99999, 1.0, 3.0, 896.0]:
        assert abs(gen.det_log(x) - math.log(x)) <= 4e-16 * max(1, abs(math.log(x)))
    for y in [-700, -30, -1.2, -1e-3, 0.0, 0.5, 2.0, 40.0]:
        assert abs(gen.det_exp(y) - math.exp(y)) <= 4e-15 * math.exp(y)
    for u in np.linspace(0, 1, 97, endpoint=False):
        s, c = gen.det_sincos_turn(float(u))
        assert abs(s - math.sin(2 * math.pi * u)) < 1e-14 and abs(c - math.cos(2 * math.pi * u)) < 1e-14


def test_bf16_is_rounded_fp32():
    f = gen.normal_f32(0, 1, 0, 4096, 1.0)
    b = gen.normal_bf16(0, 1, 0, 4096, 1.0)
    up = (b.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.abs(up - f) <= np.abs(f) * 2.0 ** -8)


def test_zipf_bias_is_log_popularity():
    b = gen.zipf_bias(896, 1.2, 0.18).astype(np.float64)
    r = np.arange(1, 897, dtype=np.float64)
    p = r ** -1.2 / (r ** -1.2).sum()
    np.testing.assert_allclose(b, 0.18 * np.log(p), rtol=1e-6)


def test_small_decode_workloads():
    for name, T in (("decode1", 1), ("decode16", 16)):
        wl = gen.WORKLOADS[name]
        assert (wl.T, wl.d, wl.E, wl.k, wl.I) == (T, 3584, 896, 16, 512)
        assert wl.P <= 4 * wl.E  # 16-token tiles
        # the same tokens as the first T of the 64-token decode batch (one seed, one stream)
        np.testing.assert_array_equal(gen.x_bf16(wl), gen.x_bf16(gen.WORKLOADS["decode"], 0, T))


def test_workload_shapes():
    wl = gen.WORKLOADS["tiny"]
    assert gen.x_bf16(wl).shape == (8, 512)
    assert gen.router_f32(wl).shape == (896, 512)
    assert gen.expert_f32(wl, "gate", 3, 5).shape == (2, 64, 512)
    assert gen.expert_f32(wl, "down", 0, 1).shape == (1, 512, 64)
    np.testing.assert_array_equal(gen.expert_f32(wl, "up", 4, 5)[0], gen.expert_f32(wl, "up", 3, 6)[1])
