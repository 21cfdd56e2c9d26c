"""The seeded input generator: determinism, range restarts and distribution."""
import numpy as np

import synth


def test_counter_based_ranges_agree():
    a = synth.normal_bf16_bits(0, synth.tensor_id("wq", 3), 10_000, 0.02)
    b = synth.normal_bf16_bits(0, synth.tensor_id("wq", 3), 4_000, 0.02, start=6_000)
    assert np.array_equal(a[6_000:], b)
    c = synth.normal_bf16_bits(1, synth.tensor_id("wq", 3), 10_000, 0.02)
    assert not np.array_equal(a, c)


def test_distribution_moments():
    x = synth.normal_f64(0, synth.tensor_id("wg", 0), (1_000_000,), 0.02)
    assert abs(x.mean()) < 1e-4
    assert abs(x.std() - 0.02) < 2e-4
    assert np.max(np.abs(x)) <= 2 * np.sqrt(3) * 0.02 * 1.01
    ids = synth.uniform_i32(0, synth.tensor_id("ids"), 200_000, 1000)
    assert ids.min() == 0 and ids.max() == 999
    assert abs(np.bincount(ids).std() / 200 - 0) < 0.15
