"""The seeded input generator: determinism, distributions, bf16 rounding (CPU only)."""

import numpy as np

import bm_inputs as gen


def test_splitmix64_reference_values():
    # splitmix64 with state 0: the first outputs of the published generator.
    z = gen.splitmix64(0, np.arange(3, dtype=np.uint64))
    assert [int(v) for v in z] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_streams_are_counter_based():
    a = gen.normal(7, 1000)
    b = gen.normal(7, 400, offset=600)
    assert np.array_equal(a[600:], b)
    assert not np.array_equal(gen.normal(8, 10), a[:10])


def test_distributions():
    u = gen.uniform(3, 200000, -1.0, 1.0)
    assert u.min() >= -1.0 and u.max() < 1.0 and abs(u.mean()) < 0.01
    x = gen.normal(4, 200000, std=0.02)
    assert abs(x.std() - 0.02) < 0.0005 and abs(x.mean()) < 0.0005
    i = gen.integers(5, 100000, -8, 8)
    assert set(np.unique(i)) == set(range(-8, 9))


def test_bf16_round_nearest_even():
    vals = np.array([1.0, 1.00390625, 1.01171875, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, -2.5,
                     np.inf, 3.4e38], dtype=np.float32)
    bits = gen.f32_to_bf16_bits(vals)
    # 1 + 2^-8 is exactly half-way between 1 and 1 + 2^-7: ties go to even (1.0).
    # 1 + 3*2^-9 is 0.75 ulp above 1.0 and rounds up; 3.4e38 overflows to +inf.
    assert [hex(b) for b in bits] == ['0x3f80', '0x3f80', '0x3f82', '0x3f80', '0x3f81', '0xc020',
                                      '0x7f80', '0x7f80']
    back = gen.bf16_bits_to_f32(gen.f32_to_bf16_bits(np.float32([0.15625, -3.0])))
    assert np.array_equal(back, np.float32([0.15625, -3.0]))
    assert gen.f32_to_bf16_bits(np.float32([np.nan]))[0] == gen.BF16_NAN


def test_symmetric_and_padding():
    s = gen.symmetric_f32(33, seed=9)
    assert np.array_equal(s, s.T)
    m = gen.matrix_bf16(4, 5, "uniform", seed=1)
    p = gen.pad_ld(m, 8, gen.BF16_NAN)
    assert p.shape == (4, 8) and np.array_equal(p[:, :5], m) and np.all(p[:, 5:] == gen.BF16_NAN)


def test_e4m3_table_and_rounding():
    v = gen.E4M3_VALUES
    assert len(v) == 127 and v[0] == 0.0 and v[1] == 2.0 ** -9 and v[8] == 2.0 ** -6 and v[-1] == 448.0
    assert np.all(np.diff(v) > 0)
    # integers up to 16 are exact, 17 is a tie between 16 and 18 and goes to the even code (16)
    ints = np.arange(-16, 17, dtype=np.float32)
    assert np.array_equal(gen.e4m3_bits_to_f32(gen.f32_to_e4m3_bits(ints)), ints)
    assert gen.e4m3_bits_to_f32(gen.f32_to_e4m3_bits(np.float32([17.0, 19.0, 1000.0, -1000.0]))).tolist() == \
        [16.0, 20.0, 448.0, -448.0]
    # every code decodes and re-encodes to itself (NaN excepted)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    back = gen.f32_to_e4m3_bits(gen.e4m3_bits_to_f32(codes))
    assert np.array_equal(back[codes != 0x80], codes[codes != 0x80])  # -0 may come back as +0 or -0
    assert np.isnan(gen.e4m3_bits_to_f32(np.uint8([0x7F, 0xFF]))).all()
    # nearest: random values land on a neighbour within half a spacing
    x = gen.normal(5, 20000, std=3.0).astype(np.float32)
    y = gen.e4m3_bits_to_f32(gen.f32_to_e4m3_bits(x)).astype(np.float64)
    idx = np.searchsorted(v, np.abs(x))
    gap = v[np.minimum(idx, 126)] - v[np.maximum(idx - 1, 0)]
    assert np.all(np.abs(np.abs(y) - np.abs(x)) <= gap / 2 + 1e-12)
