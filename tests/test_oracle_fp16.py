"""Pins the oracle's binary16 conversion (written from the IEEE-754 format
definition) against numpy's float16 casts, on every half bit pattern and on
random and edge-case binary32 values."""
import numpy as np

import oracle


def test_f16_to_f32_all_patterns():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.f16_bits_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _check(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    ours = oracle.f32_to_f16_bits(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.all(np.isnan(ours[nan].view(np.float16)))
    bad = np.nonzero(ours[~nan] != ref[~nan])[0]
    assert bad.size == 0, (x[~nan][bad[:5]], ours[~nan][bad[:5]], ref[~nan][bad[:5]])


def test_f32_to_f16_random_bit_patterns():
    rng = np.random.Generator(np.random.PCG64(1))
    bits = rng.integers(0, 2**32, size=10_000_000, dtype=np.uint64).astype(np.uint32)
    _check(bits.view(np.float32))


def test_f32_to_f16_half_range_dense():
    # values concentrated where halves live: exponents -26..16
    rng = np.random.Generator(np.random.PCG64(2))
    e = rng.integers(-26, 17, size=2_000_000)
    m = rng.random(2_000_000) + 1.0
    s = np.where(rng.random(2_000_000) < 0.5, -1.0, 1.0)
    _check((s * np.ldexp(m, e)).astype(np.float32))


def test_f32_to_f16_edge_classes():
    two = np.float32(2.0)
    vals = [0.0, -0.0, np.inf, -np.inf, 65504.0, 65519.996, 65520.0, -65520.0, 1e10,
            2.0**-25, 2.0**-25 * (1 + 2.0**-23), 3 * 2.0**-25, 5 * 2.0**-25, 2.0**-24, 2.0**-14,
            2.0**-14 - 2.0**-25, 2.0**-14 - 2.0**-26, 2.0**-15 * 1.5, 2.0**-26,
            1 + 2.0**-11, 1 + 3 * 2.0**-11, 1 + 2.0**-11 + 2.0**-23, 2047.5, 2048.0 + 1.0, 2049.0,
            1.0 / 7.0, 1.0 / 127.0, 7.0 / 7.0]
    x = np.array(vals, dtype=np.float64).astype(np.float32)
    # all neighbours of each edge value
    xb = x.view(np.uint32)
    nb = np.concatenate([xb - 1, xb, xb + 1]).astype(np.uint32).view(np.float32)
    _check(np.concatenate([nb, -nb, np.nextafter(x, two)]))
