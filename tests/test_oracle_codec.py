"""Pins the oracle's Q4_G64, Q4_G32 and q8_0 codecs.

What fixes the codec: 4-bit signed codes, one fp16 scale for each 64-value group, exactly
4.25 bits/value (den_llama.cpp, "What this fork is", quantized KV cache
bullet); the q8_0-style K of the mixed pair (den_llama.cpp, "Build3 (working
engine)" command block); the pages' "q4_0" V, read as the Q4_G64 rule with
32-value groups (Q4_G32, exactly 4.5 bits/value).  Rounding rule: scale = fp16(absmax/qmax), code =
clamp(rne(x/scale)).  Pins: the storage closed form, hand-worked golden rows,
exact rational brute force of the nearest code, the round-trip bound, special
blocks, exact dequantization, and the append semantics."""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
QRANGE = {oracle.Q4_G64: (-8, 7), oracle.Q8_0: (-127, 127), oracle.Q4_G32: (-8, 7)}
QMAX = {oracle.Q4_G64: 7, oracle.Q8_0: 127, oracle.Q4_G32: 7}
CODECS = (oracle.Q4_G64, oracle.Q8_0, oracle.Q4_G32)


def _load_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            out[k] = v
    return out


def _codes(codec, qs, head_dim):
    """Signed codes from the packed bytes (layout as documented in the fixture)."""
    qs = np.asarray(qs, dtype=np.uint8)
    if codec == oracle.Q8_0:
        return qs.view(np.int8).astype(np.int64)
    lo = (qs & 0xF).astype(np.int64)
    hi = (qs >> 4).astype(np.int64)
    c = np.stack([lo, hi], axis=-1).reshape(qs.shape[:-1] + (head_dim,))
    return np.where(c >= 8, c - 16, c)


@pytest.mark.parametrize("name,codec", [("q4g64_two_groups.txt", oracle.Q4_G64),
                                        ("q8_0_two_groups.txt", oracle.Q8_0),
                                        ("q4g32_two_groups.txt", oracle.Q4_G32)])
def test_golden_rows(name, codec):
    g = _load_golden(name)
    x = np.array([float(v) for v in g["x"]], np.float32)
    qs, sc = oracle.quantize(codec, x[None])
    assert qs.tobytes().hex() == g["qs"][0]
    assert ["%04x" % s for s in sc[0]] == g["scales"]
    # dequantization of the golden bytes is scale * code exactly
    xh = oracle.dequantize(codec, qs, sc, x.size)[0]
    d = np.repeat(np.array([int(s, 16) for s in g["scales"]], np.uint16).view(np.float16).astype(np.float64),
                  oracle.GROUP[codec])
    assert np.array_equal(xh.astype(np.float64), d * _codes(codec, qs, x.size)[0])


@pytest.mark.parametrize("codec,bpv", [(oracle.Q4_G64, Fraction(17, 4)), (oracle.Q8_0, Fraction(17, 2)),
                                       (oracle.Q4_G32, Fraction(9, 2))])
@pytest.mark.parametrize("head_dim", [64, 128, 256, 512])
def test_storage_closed_form(codec, bpv, head_dim):
    rows = 37
    x = np.random.Generator(np.random.PCG64(head_dim)).standard_normal((rows, head_dim)).astype(np.float32)
    qs, sc = oracle.quantize(codec, x)
    assert Fraction(8 * (qs.nbytes + sc.nbytes), rows * head_dim) == bpv


def _groups(rng, n, gs):
    """Groups with a wide spread of magnitudes, including fp16-subnormal scales."""
    mag = np.exp(rng.uniform(np.log(1e-9), np.log(3e4), size=(n, 1)))
    x = rng.standard_normal((n, gs)) * mag
    heavy = rng.random(n) < 0.2
    x[heavy] *= np.exp(rng.standard_normal((heavy.sum(), gs)) * 2)
    return x.astype(np.float32)


@pytest.mark.parametrize("codec", CODECS)
def test_brute_force_nearest_code(codec):
    """Each code is the nearest integer in range to x/scale (exact rational
    distance), ties to even, except within 2^-20 of a tie where the fp32
    quotient may legitimately decide differently."""
    gs = oracle.GROUP[codec]
    rng = np.random.Generator(np.random.PCG64(11))
    x = _groups(rng, 6000, gs)
    qs, sc = oracle.quantize(codec, x)
    codes = _codes(codec, qs, gs)
    d = sc.view(np.float16).astype(np.float64)[:, 0]
    lo, hi = QRANGE[codec]
    ks = np.arange(lo, hi + 1, dtype=np.float64)
    xd = x.astype(np.float64)
    zero = d == 0
    assert np.all(codes[zero] == 0)
    xd, codes, dd = xd[~zero], codes[~zero], d[~zero][:, None]
    with np.errstate(invalid="ignore"):               # an infinite scale (planted mistakes) gives nan
        dist = np.abs(xd[:, :, None] - ks[None, None, :] * dd[:, :, None])   # exact in fp64
    best = dist.min(axis=-1, keepdims=True)
    cand = dist == best
    nearest_even = np.where(cand.sum(-1) > 1, np.where(cand & (ks % 2 == 0), ks, np.inf).min(-1),
                            ks[np.argmax(cand, axis=-1)])
    ratio = xd / dd
    near_tie = np.abs(np.abs(ratio - np.floor(ratio)) - 0.5) <= 2.0**-20 * np.maximum(np.abs(ratio), 1)
    mism = (codes != nearest_even) & ~near_tie
    assert not mism.any(), (xd[mism][:4], codes[mism][:4], nearest_even[mism][:4])
    assert (codes == nearest_even).mean() > 0.999


@pytest.mark.parametrize("codec", CODECS)
def test_scale_rule_and_roundtrip_bound(codec):
    gs = oracle.GROUP[codec]
    rng = np.random.Generator(np.random.PCG64(12))
    x = _groups(rng, 6000, gs)
    qs, sc = oracle.quantize(codec, x)
    d16 = sc.view(np.float16)[:, 0]
    amax = np.abs(x).max(axis=1)
    with np.errstate(over="ignore"):
        expect = (amax / np.float32(QMAX[codec])).astype(np.float32).astype(np.float16)   # numpy's own RNE
    expect = np.where(np.isinf(expect), np.float16(65504.0), expect)    # saturated, not infinite
    with np.errstate(over="ignore"):
        assert np.isinf((amax / np.float32(QMAX[codec])).astype(np.float16)).any()  # the case is exercised
    assert np.array_equal(d16.view(np.uint16), expect.view(np.uint16))
    xh = oracle.dequantize(codec, qs, sc, gs).astype(np.float64)
    d = d16.astype(np.float64)[:, None]
    # the bound holds where the scale is a normal half and did not saturate
    normal = (d[:, 0] >= 2.0**-14) & (amax.astype(np.float64) / QMAX[codec] < 65504.0)
    err = np.abs(x.astype(np.float64) - xh)[normal]
    assert np.all(err <= d[normal] / 2 * (1 + 2.0**-20))
    # the group's absmax element lands on +-qmax
    i = np.abs(x).argmax(axis=1)
    c = _codes(codec, qs, gs)[np.arange(len(x)), i]
    sel = normal & (amax > 0)
    assert np.all(np.abs(c[sel]) == QMAX[codec])


@pytest.mark.parametrize("codec", CODECS)
def test_special_blocks(codec):
    gs, qm = oracle.GROUP[codec], QMAX[codec]
    zero = np.zeros((1, 2 * gs), np.float32)
    qs, sc = oracle.quantize(codec, zero)
    assert not qs.any() and not sc.any()
    for c in (1.0, -3.25, 1e-3, 6e4):
        x = np.full((1, gs), c, np.float32)
        qs, sc = oracle.quantize(codec, x)
        assert np.all(_codes(codec, qs, gs) == np.sign(c) * qm)
        assert sc[0, 0] == np.float16(np.float32(abs(c)) / np.float32(qm)).view(np.uint16)
    # a group whose absmax/qmax is below half the smallest subnormal: scale 0, codes 0
    tiny = np.full((1, gs), 1e-9, np.float32)
    qs, sc = oracle.quantize(codec, tiny)
    assert sc[0, 0] == 0 and not qs.any()
    # groups are independent: one outlier group does not change the next one
    x = np.random.Generator(np.random.PCG64(5)).standard_normal((1, 2 * gs)).astype(np.float32)
    q1, s1 = oracle.quantize(codec, x)
    x2 = x.copy()
    x2[0, :gs] *= 1000
    q2, s2 = oracle.quantize(codec, x2)
    rb = oracle.row_bytes(codec, gs)
    assert np.array_equal(q1[0, rb:], q2[0, rb:]) and s1[0, 1] == s2[0, 1]


def test_minus_eight_decodes():
    """Code -8 (nibble 0x8) is never produced by the rule but must decode."""
    qs = np.full((1, 32), 0x88, np.uint8)
    sc = np.array([[np.float16(0.5).view(np.uint16)]], np.uint16)
    assert np.all(oracle.dequantize(oracle.Q4_G64, qs, sc, 64) == -4.0)


def test_dequant_exact_in_fp64():
    rng = np.random.Generator(np.random.PCG64(13))
    for codec in CODECS:
        x = rng.standard_normal((200, 256)).astype(np.float32) * 3
        qs, sc = oracle.quantize(codec, x)
        xh = oracle.dequantize(codec, qs, sc, 256)
        d = np.repeat(sc.view(np.float16).astype(np.float64), oracle.GROUP[codec], axis=1)
        assert np.array_equal(xh.astype(np.float64), d * _codes(codec, qs, 256))


def test_fp16_sources_quantize_like_their_fp32_widening():
    rng = np.random.Generator(np.random.PCG64(14))
    x16 = rng.standard_normal((50, 128)).astype(np.float16)
    a = oracle.quantize(oracle.Q4_G64, x16)
    b = oracle.quantize(oracle.Q4_G64, x16.astype(np.float32))
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_append_positions_and_error_bit():
    rng = np.random.Generator(np.random.PCG64(15))
    S, n_new, Hk, D, cap = 3, 2, 2, 128, 8
    for codec in CODECS:
        cache = oracle.Cache(codec, S, Hk, D, cap)
        src = rng.standard_normal((S, n_new, Hk, D)).astype(np.float32)
        pos0 = np.array([0, 6, 7], np.int32)          # the last one overflows capacity
        err = oracle.quantize_append(cache, src, pos0)
        assert err == 1
        assert not cache.qs[2].any() and not cache.scales[2].any()
        for s in (0, 1):
            for i in range(n_new):
                for h in range(Hk):
                    qs, sc = oracle.quantize(codec, src[s, i, h][None])
                    assert np.array_equal(cache.qs[s, h, pos0[s] + i], qs[0])
                    assert np.array_equal(cache.scales[s, h, pos0[s] + i], sc[0])
        untouched = np.ones((S, Hk, cap), bool)
        for s in (0, 1):
            untouched[s, :, pos0[s]:pos0[s] + n_new] = False
        assert not cache.qs[untouched].any()
        assert oracle.quantize_append(cache, src, np.array([-1, 0, 0], np.int32)) == 1
