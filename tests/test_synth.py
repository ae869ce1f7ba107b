"""The seeded input generator: numpy and C copies agree bit for bit, keys separate streams,
and the values have the stated mean and standard deviation."""
import numpy as np

import synth


def test_numpy_and_c_agree():
    for key in [synth.tensor_key(0, "a"), synth.tensor_key(7, "Wgu", 3), 0]:
        for start, n in [(0, 1000), (123456789, 4097)]:
            np.testing.assert_array_equal(synth.np_u64(key, start, n), synth.host_u64(key, start, n))
            np.testing.assert_array_equal(synth.np_normal_bf16(key, start, n, 0.02),
                                          synth.host_normal(key, start, n, 0.02, "bf16"))
            a = synth.np_normal_f32(key, start, n, 0.05)
            b = synth.host_normal(key, start, n, 0.05, "f32")
            np.testing.assert_array_equal(a.view(np.uint32), b.view(np.uint32))


def test_moments_and_bounds():
    v = synth.host_normal(synth.tensor_key(1, "m"), 0, 1 << 20, 2.0, "f32").astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 2.0) < 0.01
    assert np.abs(v).max() <= 2.0 * 3.4642
    u = synth.np_uniform01(synth.tensor_key(1, "u"), 0, 1 << 16)
    assert 0.0 <= u.min() and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.01


def test_keys_are_distinct():
    keys = {synth.tensor_key(0, c, l, n) for c in ["c2", "c3"] for l in range(40) for n in ["Wr", "Wgu", "Wd"]}
    assert len(keys) == 2 * 40 * 3


def test_bf16_rounding_is_nearest_even():
    f = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], np.float32)
    bits = synth.f32_to_bf16_bits(f)
    np.testing.assert_array_equal(synth.bf16_bits_to_f32(bits), [1.0, 1.0, 1.0 + 2 ** -6, -2.5])


def test_subrange_matches_full_tensor():
    key = synth.tensor_key(3, "slice")
    full = synth.host_normal(key, 0, 10000, 1.0, "bf16")
    np.testing.assert_array_equal(full[4000:7000], synth.host_normal(key, 4000, 3000, 1.0, "bf16"))
