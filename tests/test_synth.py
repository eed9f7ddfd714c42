"""The seeded input generator (CPU only)."""
import numpy as np

import synth


def test_normal_is_deterministic_counter_based_and_standard():
    a = synth.normal(0, "t", (1 << 20,))
    b = synth.normal(0, "t", (1 << 20,))
    assert np.array_equal(a, b)
    assert np.array_equal(synth.normal(0, "t", (1001,)), a[:1001])  # prefix property
    assert not np.array_equal(synth.normal(1, "t", (16,)), a[:16])
    assert not np.array_equal(synth.normal(0, "u", (16,)), a[:16])
    n = a.size
    assert abs(float(a.mean())) < 5 / np.sqrt(n)
    assert abs(float(a.std()) - 1.0) < 5 / np.sqrt(2 * n)
    c = synth.normal(0, "t", (1 << 16,), std=0.02, mean=1.0)
    assert abs(float(c.mean()) - 1.0) < 1e-3 and abs(float(c.std()) - 0.02) < 1e-3


def test_bf16_round_to_nearest_even():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20, 0.0], dtype=np.float32)
    bits = synth.f32_to_bf16_bits(vals)
    # 1 + 2^-8 is a tie between 0x3F80 and 0x3F81 -> even 0x3F80; 1 + 3*2^-8 -> 0x3F82
    assert list(bits) == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81, 0x0000]
    assert np.array_equal(synth.bf16_bits_to_f32(bits)[[0, 3]], np.array([1.0, -2.5], dtype=np.float32))


def test_uniform_int_range():
    t = synth.uniform_int(0, "tok", (100000,), 128256)
    assert t.dtype == np.int32 and t.min() >= 0 and t.max() < 128256
    assert abs(float(t.mean()) - 128255 / 2) < 128256 * 0.01
