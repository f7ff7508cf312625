"""Pins the oracle's NVFP4 codec and its two number formats.

What fixes them: the pages name NVFP4 as a KV cache type (den_llama.cpp,
"What this fork is", quantized KV cache bullet; "build3 (working engine) --
additions" table, NVFP4 KV row) but not its format, which is read as
NVIDIA's published NVFP4: FP4 E2M1 values in blocks of 16, one FP8 E4M3 scale
per block, no per-tensor scale; scale = e4m3(absmax / 6), code = e2m1(x /
scale), both round-to-nearest-even and saturating.  Pins: torch's
float8_e4m3fn conversions (an independent implementation), the published
E2M1 value table (tests/golden/e2m1_values.txt), a rounding written another
way (the quantum of the binade, Python's half-even round()), a hand-worked
golden row, the storage closed form, the round-trip bound and special
blocks."""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
NV = oracle.NVFP4
HAS_F8 = hasattr(torch, "float8_e4m3fn")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            k, *v = line.split()
            out[k] = v
    return out


def _e2m1_table():
    g = _golden("e2m1_values.txt")
    return [float(v) for v in g["values"]]


def _round_to_grid(a, max_exp, mant_bits, min_exp, max_value):
    """Round |a| (a Python float) to the nearest value of a binary format with
    mant_bits fraction bits, binades 2^min_exp .. 2^max_exp, subnormals below
    2^min_exp, ties to even, held at max_value: scale |a| by the quantum of its
    binade, round half to even as an integer, scale back."""
    a = abs(a)
    e = max(min_exp, math.frexp(a)[1] - 1) if a > 0 else min_exp
    e = min(e, max_exp)
    quantum = 2.0 ** (e - mant_bits)
    r = round(a / quantum) * quantum            # exact: a / quantum is exact in binary
    return min(r, max_value)


# ---------------------------------------------------------------- E2M1


def test_e2m1_decode_is_the_published_table():
    t = _e2m1_table()
    assert t == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    got = oracle.e2m1_to_f32(np.arange(16))
    assert list(got[:8]) == t
    assert list(-got[8:]) == t
    assert all(math.copysign(1.0, v) < 0 for v in got[8:])          # code 8 is -0


def _e2m1_reference(x):
    """E2M1 code of fp32 x via the binade quantum (bias 1, 1 fraction bit,
    binades 2^0 .. 2^2, subnormal quantum 0.5, largest 6)."""
    r = _round_to_grid(float(x), 2, 1, 0, 6.0)
    c = _e2m1_table().index(r)
    return c | (8 if math.copysign(1.0, float(x)) < 0 else 0)


def test_e2m1_encode_matches_binade_rounding():
    t = _e2m1_table()
    vals = set()
    for i in range(len(t) - 1):
        mid = (t[i] + t[i + 1]) / 2
        for v in (t[i], mid, t[i + 1]):
            f = np.float32(v)
            vals.update([f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(10))])
    vals.update(np.float32(v) for v in (6.5, 7.0, 7.99, 8.0, 100.0, 1e30, 1e-30, 0.0))
    rng = np.random.default_rng(5)
    vals.update(rng.uniform(0, 8, 2000).astype(np.float32))
    x = np.array(sorted(vals), np.float32)
    x = np.concatenate([x, -x])
    got = oracle.f32_to_e2m1(x)
    ref = np.array([_e2m1_reference(v) for v in x], np.uint8)
    assert np.array_equal(got, ref)


def test_e2m1_ties_and_signed_zero():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.1, -0.25, -0.0, 0.0], np.float32)
    assert list(oracle.f32_to_e2m1(x)) == [0x0, 0x2, 0x2, 0x4, 0x4, 0x6, 0x6, 0x8, 0x8, 0x8, 0x0]


# ---------------------------------------------------------------- E4M3


def _e4m3_positive_values():
    return [float(v) for v in oracle.e4m3_to_f32(np.arange(127))]


@pytest.mark.skipif(not HAS_F8, reason="torch without float8_e4m3fn")
def test_e4m3_decode_matches_torch():
    codes = np.array([c for c in range(256) if c & 0x7F != 0x7F], np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = oracle.e4m3_to_f32(codes)
    assert np.array_equal(got, ref)
    assert np.isnan(oracle.e4m3_to_f32(np.array([0x7F, 0xFF], np.uint8))).all()
    assert got.max() == 448.0


@pytest.mark.skipif(not HAS_F8, reason="torch without float8_e4m3fn")
def test_e4m3_encode_matches_torch_in_range():
    v = _e4m3_positive_values()
    vals = set()
    for i in range(len(v) - 1):
        for a in (v[i], (v[i] + v[i + 1]) / 2, v[i + 1]):
            f = np.float32(a)
            vals.update([f, np.nextafter(f, np.float32(0)), np.nextafter(f, np.float32(1e4))])
    rng = np.random.default_rng(11)
    vals.update((2.0 ** rng.uniform(-12, 8.8, 20000)).astype(np.float32))
    x = np.array(sorted(a for a in vals if a <= 448.0), np.float32)
    x = np.concatenate([x, -x])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(oracle.f32_to_e4m3(x), ref)


def test_e4m3_encode_matches_binade_rounding_and_saturates():
    v = _e4m3_positive_values()
    rng = np.random.default_rng(13)
    x = np.concatenate([(2.0 ** rng.uniform(-12, 10, 5000)).astype(np.float32),
                        np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 0.0], np.float32)])
    for a in x:
        r = _round_to_grid(float(a), 8, 3, -6, 448.0)
        assert oracle.e4m3_to_f32(oracle.f32_to_e4m3(np.array([a], np.float32)))[0] == r
    assert v.index(448.0) == 126


# ---------------------------------------------------------------- NVFP4 codec


def test_golden_row():
    g = _golden("nvfp4_two_blocks.txt")
    x = np.array([float(v) for v in g["x"]], np.float32)
    qs, sc = oracle.quantize(NV, x[None])
    assert sc.dtype == np.uint8
    assert qs.tobytes().hex() == g["qs"][0]
    assert ["%02x" % s for s in sc[0]] == g["scales"]


def test_storage_is_4_5_bits_per_value():
    for d in (64, 128, 256, 512):
        assert (oracle.row_bytes(NV, d) + oracle.scales_per_row(NV, d)) * 8 == 4.5 * d


def _reference_quantize(x):
    """The codec rule with independently pinned pieces: torch's (or the binade)
    E4M3 rounding of the fp32 absmax / 6, then the binade E2M1 rounding of the
    fp32 quotients."""
    x = np.asarray(x, np.float32).reshape(-1, 16)
    codes, scales = [], []
    for blk in x:
        q = np.float32(np.abs(blk).max()) / np.float32(6.0)
        s = _round_to_grid(float(q), 8, 3, -6, 448.0)
        scales.append(_e4m3_positive_values().index(s))
        for v in blk:
            codes.append(0 if s == 0 else _e2m1_reference(np.float32(v) / np.float32(s)))
    return np.array(codes, np.uint8), np.array(scales, np.uint8)


@pytest.mark.parametrize("dist", ["normal", "outliers", "tiny", "mixed"])
def test_quantize_matches_the_rule_written_another_way(dist):
    rng = np.random.default_rng({"normal": 1, "outliers": 2, "tiny": 3, "mixed": 4}[dist])
    x = rng.standard_normal((6, 64)).astype(np.float32)
    if dist == "outliers":
        x *= np.where(rng.random(x.shape) < 0.05, 40.0, 1.0).astype(np.float32)
    elif dist == "tiny":
        x *= np.float32(1e-3)
    elif dist == "mixed":
        x *= (2.0 ** rng.integers(-14, 9, (6, 4, 1))).repeat(16, 2).reshape(6, 64).astype(np.float32)
    qs, sc = oracle.quantize(NV, x)
    codes = np.stack([qs & 0xF, qs >> 4], -1).reshape(-1)
    rc, rs = _reference_quantize(x)
    assert np.array_equal(sc.reshape(-1), rs)
    assert np.array_equal(codes, rc)


def test_roundtrip_bound_and_exact_dequant():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((40, 128)) * np.exp(rng.uniform(-6, 6, (40, 1)))).astype(np.float32)
    qs, sc = oracle.quantize(NV, x)
    xh = oracle.dequantize(NV, qs, sc, 128).astype(np.float64)
    s = np.repeat(oracle.e4m3_to_f32(sc).astype(np.float64), 16, axis=1)
    codes = np.stack([qs & 0xF, qs >> 4], -1).reshape(40, 128)
    assert np.array_equal(xh, s * oracle.e2m1_to_f32(codes).astype(np.float64))    # exact product
    a = np.abs(x.astype(np.float64))
    # within the grid the error is at most half of the widest gap (2 s); past 6 s, |x| - 6 s
    assert np.all(np.abs(x - xh) <= np.maximum(s, a - 6 * s) * (1 + 1e-12))


def test_special_blocks():
    z = np.zeros((1, 16), np.float32)
    qs, sc = oracle.quantize(NV, z)
    assert not qs.any() and not sc.any()
    tiny = np.full((1, 16), 5e-4, np.float32)           # absmax / 6 below half of E4M3's 2^-9: scale 0
    qs, sc = oracle.quantize(NV, tiny * np.where(np.arange(16) % 2, -1, 1).astype(np.float32))
    assert sc[0, 0] == 0 and not qs.any()               # all codes +0 when the scale is 0
    big = np.full((1, 16), 6000.0, np.float32)          # 1000 saturates to 448: x / s = 13.4 -> 6
    qs, sc = oracle.quantize(NV, big)
    assert sc[0, 0] == 0x7E and (qs == 0x77).all()
    const = np.full((1, 16), -3.0, np.float32)          # s = 0.5 exactly: -3 / 0.5 = -6
    qs, sc = oracle.quantize(NV, const)
    assert oracle.e4m3_to_f32(sc)[0, 0] == 0.5 and (qs == 0xFF).all()


def test_append_and_attention_accept_nvfp4():
    rng = np.random.default_rng(9)
    k = oracle.Cache(NV, 1, 1, 64, 64)
    v = oracle.Cache(NV, 1, 1, 64, 64)
    src = rng.standard_normal((1, 5, 1, 64)).astype(np.float32)
    assert oracle.quantize_append(k, src, np.array([3], np.int32)) == 0
    assert oracle.quantize_append(v, src, np.array([3], np.int32)) == 0
    qs, sc = oracle.quantize(NV, src[0, :, 0])
    assert np.array_equal(k.qs[0, 0, 3:8], qs) and np.array_equal(k.scales[0, 0, 3:8], sc)
    q = rng.standard_normal((1, 1, 1, 64)).astype(np.float32)
    o, lse = oracle.decode_attention(k, v, q, np.array([8], np.int32), 0.125)
    kd = oracle.dequantize(NV, k.qs[0, 0, :8], k.scales[0, 0, :8], 64).astype(np.float64)
    vd = oracle.dequantize(NV, v.qs[0, 0, :8], v.scales[0, 0, :8], 64).astype(np.float64)
    z = kd @ q[0, 0, 0].astype(np.float64) * 0.125
    p = np.exp(z - z.max())
    assert np.allclose(o[0, 0, 0], p @ vd / p.sum(), rtol=0, atol=1e-12)
    assert abs(lse[0, 0, 0] - (z.max() + np.log(p.sum()))) < 1e-12
