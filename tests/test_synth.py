"""The seeded input generator: distributions, rounding and canonical packing."""
from fractions import Fraction

import numpy as np

from bit_weight_only_groupwise_gb300 import synth


def test_stream_is_counter_based_and_prefix_consistent():
    a = synth.draws(0, 3, 0, 100)
    b = synth.draws(0, 3, 40, 60)
    assert np.array_equal(a[40:], b)
    x8 = synth.activations(0, 8, 256, outliers=True)
    x3 = synth.activations(0, 3, 256, outliers=True)
    assert np.array_equal(x8[:3], x3)
    assert not np.array_equal(synth.draws(1, 3, 0, 10), synth.draws(0, 3, 0, 10))


def test_code_ranges_are_uniform():
    for bits in (4, 5):
        c = synth.uniform_codes(0, 1, 64, 4096, bits)
        lo, hi = -(1 << (bits - 1)), (1 << (bits - 1)) - 1
        assert c.min() == lo and c.max() == hi
        counts = np.bincount((c.astype(np.int32) - lo).ravel(), minlength=1 << bits)
        expect = c.size / (1 << bits)
        assert np.all(np.abs(counts - expect) < 6 * np.sqrt(expect))


def test_bf16_rounding_is_single_round_to_nearest_even():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(20000) * 20.0,
                        # exact halfway points between neighbouring bf16 values
                        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(2.0 + 2.0 ** -7)])])
    bits = synth.fp64_to_bf16_bits(x)
    vals = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    for xi, vi, bi in zip(x, vals, bits):
        # neighbours of the chosen value must not be closer, ties to even mantissa
        up = (np.uint32(bi + 1) << 16).view(np.float32)
        dn = (np.uint32(bi - 1) << 16).view(np.float32)
        d = abs(Fraction(xi) - Fraction(float(vi)))
        assert d <= abs(Fraction(xi) - Fraction(float(up)))
        assert d <= abs(Fraction(xi) - Fraction(float(dn)))
        if d == abs(Fraction(xi) - Fraction(float(up))) or d == abs(Fraction(xi) - Fraction(float(dn))):
            assert bi % 2 == 0
    assert synth.fp64_to_bf16_bits(np.array([1.0 + 2.0 ** -8]))[0] == 0x3F80
    assert synth.fp64_to_bf16_bits(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 0x3F82


def test_scales_and_outliers():
    s = synth.group_scales(0, 2, 100, 640)
    v = s.view(np.float16).astype(np.float64)
    assert s.shape == (100, 10)
    assert v.min() >= 0.002 and v.max() < 0.1
    ch = synth.outlier_channels(0, 6144)
    assert len(ch) == 61 and len(np.unique(ch)) == 61
    assert len(synth.outlier_channels(0, 5120)) == 51


def test_pack_canonical_layout():
    codes = np.array([[0, 1, 2, 3, 4, 5, 6, 7, -8, -7, -6, -5, -4, -3, -2, -1]], np.int8)
    assert synth.pack_canonical(codes, 4).tolist() == [[0x10, 0x32, 0x54, 0x76, 0x98, 0xBA, 0xDC, 0xFE]]
    c5 = np.zeros((1, 8), np.int8)
    c5[0, 1] = -1
    assert synth.pack_canonical(c5, 5).tolist() == [[0xE0, 0x03, 0, 0, 0]]


def test_column_parallel_oracle_equals_one_call():
    # the parity tests' thread-pool split of the oracle over token columns
    # gives exactly the single-call result (the oracle is column-independent)
    import oracle
    from tests.oracle_columns import gemm_columns, wide_columns
    p = synth.weights(4, 37, 192, 5)
    x = synth.activations(4, 29, 192, outliers=True)
    Y1, A1 = oracle.gemm_parent(p, x)
    Y2, A2 = gemm_columns(p, x, chunk=4)
    assert np.array_equal(Y1, Y2) and np.array_equal(A1, A2)
    assert np.array_equal(wide_columns(200), np.arange(200))
    c = wide_columns(4096)
    assert c[0] == 0 and c[-1] == 4095 and np.all(np.isin(np.arange(0, 4096, 64), c)) and len(c) >= 64
