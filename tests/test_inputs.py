"""The seeded input generator: determinism, slicing, distribution, bf16 rounding."""
import numpy as np

from mqa_attention_gb300 import inputs as I


def test_deterministic_and_seed_dependent():
    a = I.normal_bf16_bits(7, (3, 5, 64))
    b = I.normal_bf16_bits(7, (3, 5, 64))
    c = I.normal_bf16_bits(8, (3, 5, 64))
    assert a.dtype == np.uint16 and np.array_equal(a, b) and not np.array_equal(a, c)


def test_prefix_consistency_across_chunks():
    """Counter-based: a longer draw starts with the shorter one (also across the
    internal chunk boundary)."""
    n = (1 << 22) + 37
    long = I.normal_bf16_bits(3, (n,))
    short = I.normal_bf16_bits(3, (1001,))
    assert np.array_equal(long[:1001], short)
    odd = I._normals(3, (1 << 22) - 1, 3)
    full = I._normals(3, 0, (1 << 22) + 2)
    assert np.array_equal(odd, full[-3:])


def test_standard_normal_moments():
    x = I.bf16_bits_to_f64(I.normal_bf16_bits(11, (1 << 20,)))
    assert abs(x.mean()) < 5e-3
    assert abs(x.std() - 1.0) < 5e-3
    assert abs((x ** 4).mean() - 3.0) < 0.05


def test_bf16_rounding_is_nearest_even():
    x32 = np.array([1.0, 1.0 + 2 ** -9, 1.0 + 3 * 2 ** -9, -2.0 - 2 ** -8, 3.14159], np.float32)
    got = I.bf16_bits_to_f32(I._f32_to_bf16_bits(x32))
    want = np.array([1.0, 1.0, 1.0 + 2 ** -7, -2.0, 3.140625], np.float32)
    assert np.array_equal(got, want)


def test_seed_convention():
    assert I.seed_for(2, "q") == 2000 and I.seed_for(2, "dout") == 2003
