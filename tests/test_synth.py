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


# ---------------------------------------------------------------- FP8 E4M3 codes
E4M3_FIXED = [(448.0, 0x7E), (-448.0, 0xFE), (500.0, 0x7E), (1.0, 0x38), (0.5, 0x30), (2.0 ** -6, 0x08),
              (2.0 ** -9, 0x01), (0.0, 0x00), (1.0625, 0x38), (1.1875, 0x3A), (1.5 * 2.0 ** -9, 0x02),
              (2.5 * 2.0 ** -9, 0x02), (240.0, 0x77), (-3.0, 0xC4), (7.5 * 2.0 ** -9, 0x08)]


def test_e4m3_fixed_values_numpy_and_c():
    """Values worked from the format (bias 7, 3 mantissa bits, max 448, subnormals m*2^-9):
    exact points, ties to the even mantissa in the normal and the subnormal range, saturation."""
    f = np.array([v for v, _ in E4M3_FIXED], np.float32)
    want = np.array([c for _, c in E4M3_FIXED], np.uint8)
    np.testing.assert_array_equal(synth.f32_to_e4m3(f), want)
    np.testing.assert_array_equal(synth.host_f32_to_e4m3(f), want)


def test_e4m3_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    v = synth.e4m3_to_f32(codes)
    np.testing.assert_array_equal(synth.f32_to_e4m3(v), codes)
    np.testing.assert_array_equal(synth.host_f32_to_e4m3(v), codes)
    assert v[codes == 0x7E][0] == 448.0 and v[codes == 0x01][0] == 2.0 ** -9


def test_e4m3_is_nearest_even_by_brute_force():
    rng = np.random.default_rng(5)
    f = np.concatenate([rng.uniform(-448, 448, 20000), rng.normal(0, 0.02, 5000), rng.normal(0, 64, 5000)])
    f = f.astype(np.float32)
    pos = np.array([c for c in range(0x7F)], np.uint8)
    vals = synth.e4m3_to_f32(pos).astype(np.float64)
    got = synth.f32_to_e4m3(f)
    a = np.abs(f.astype(np.float64))
    d = np.abs(vals[None, :] - a[:, None])
    best = d.min(1)
    for i in range(len(f)):
        cand = np.flatnonzero(d[i] == best[i])
        c = cand[0] if len(cand) == 1 else [x for x in cand if x % 2 == 0][0]
        assert (got[i] & 0x7F) == c and (got[i] >> 7) == (1 if f[i] < 0 else 0), (f[i], got[i], c)
    np.testing.assert_array_equal(synth.host_f32_to_e4m3(f), got)


def test_e4m3_codes_and_row_scales_numpy_equals_c():
    key = synth.tensor_key(9, "e4m3")
    for start, n in [(0, 50000), (123456789, 4097)]:
        np.testing.assert_array_equal(synth.np_e4m3(key, start, n, 64.0), synth.host_normal(key, start, n, 64.0, "e4m3"))
        np.testing.assert_array_equal(synth.np_row_scales(key, start, n), synth.host_row_scales(key, start, n))
    s = synth.np_row_scales(key, 0, 10000)
    assert set(np.unique(s * 2.0 ** 16).astype(int)) <= set(range(16, 32))


def test_correlated_block_inputs():
    """host_h0 with correlation a: unit variance per element and correlation ~a^2 between two
    tokens of one request, ~0 across requests."""
    from synth import workloads as W
    cfg = W.LAYER
    h = W.host_h0(cfg, 2, correlation=0.9).astype(np.float64).reshape(2, cfg.P, cfg.H)
    assert abs(h.std() - 1.0) < 0.02
    same = np.corrcoef(h[0, 0], h[0, 5])[0, 1]
    other = np.corrcoef(h[0, 0], h[1, 0])[0, 1]
    assert abs(same - 0.81) < 0.05 and abs(other) < 0.08
    np.testing.assert_array_equal(W.host_h0(cfg, 2), W.host_h0(cfg, 2, correlation=0.0))
