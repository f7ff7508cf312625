"""Pins the oracle's decode attention: fp64 softmax attention of the new query
tokens over the dequantized cache, grouped-query heads (query head h reads kv
head h // G), causal among the n_q new tokens (den_llama.cpp, "What's in the
fork": the fattn-vec-instance-q4_g64 kernels; "Results": MTP n-max 2, so
1 + 2 query tokens per verify step), plus split-then-merge by log-sum-exp.

Pins: torch's float64 scaled_dot_product_attention on the same dequantized
tensors, an exact-rational brute force on tiny shapes, and invariants."""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import dequant_cache, oracle_caches


def _wl(n_seq=2, H=6, Hk=2, D=128, cached=(5, 37), n_new=1, kc=workloads.Q4_G64, vc=workloads.Q4_G64,
        seed=1, dist="normal"):
    return workloads.custom(n_seq=n_seq, n_heads=H, n_kv_heads=Hk, head_dim=D, cached=cached, n_new=n_new,
                            k_codec=kc, v_codec=vc, src_dtype="f32", q_dtype="f32", dist=dist, seed=seed)


def _torch_reference(wl, kc, vc):
    """SDPA in float64 with kv heads repeated over their query-head group and a
    per-row boolean mask of the visible keys; lse via torch.logsumexp."""
    sp = wl.spec
    K = torch.from_numpy(dequant_cache(kc).astype(np.float64))          # [S][Hk][T][D]
    V = torch.from_numpy(dequant_cache(vc).astype(np.float64))
    Q = torch.from_numpy(wl.q.astype(np.float64))                        # [S][n_q][H][D]
    G = sp.n_heads // sp.n_kv_heads
    outs, lses = [], []
    for s in range(sp.n_seq):
        T = int(wl.kv_len[s])
        k = K[s, :, :T].repeat_interleave(G, dim=0)                      # [H][T][D]
        v = V[s, :, :T].repeat_interleave(G, dim=0)
        q = Q[s].transpose(0, 1)                                         # [H][n_q][D]
        vis = torch.tensor([T - sp.n_q + i + 1 for i in range(sp.n_q)])
        mask = torch.arange(T)[None, :] < vis[:, None]                  # [n_q][T]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=sp.scale)
        z = (q @ k.transpose(-1, -2)) * sp.scale
        lse = torch.logsumexp(z.masked_fill(~mask, -math.inf), dim=-1)
        outs.append(o.transpose(0, 1).numpy())
        lses.append(lse.transpose(0, 1).numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("kc,vc", [(workloads.Q4_G64, workloads.Q4_G64), (workloads.Q8_0, workloads.Q4_G64),
                                   (workloads.Q8_0, workloads.Q4_G32), (workloads.NVFP4, workloads.NVFP4),
                                   (workloads.Q8_0, workloads.NVFP4)])
@pytest.mark.parametrize("n_new", [1, 2, 3])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_matches_torch_sdpa_float64(kc, vc, n_new, D):
    wl = _wl(D=D, n_new=n_new, kc=kc, vc=vc, seed=D + n_new)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    o_ref, lse_ref = _torch_reference(wl, k, v)
    assert np.abs(o - o_ref).max() < 1e-12
    assert np.abs(lse - lse_ref).max() < 1e-12


def test_gqa_head_mapping_is_contiguous():
    """Query head h must read kv head h // G: make the kv heads wildly
    different and compare against per-kv-head single-head attention."""
    wl = _wl(n_seq=1, H=6, Hk=3, D=64, cached=(20,), seed=3)
    k, v = oracle_caches(wl)
    o, _ = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    G = 2
    for h in range(6):
        kh = h // G
        k1 = oracle.Cache(k.codec, 1, 1, 64, k.capacity)
        v1 = oracle.Cache(v.codec, 1, 1, 64, v.capacity)
        k1.qs[0, 0], k1.scales[0, 0] = k.qs[0, kh], k.scales[0, kh]
        v1.qs[0, 0], v1.scales[0, 0] = v.qs[0, kh], v.scales[0, kh]
        o1, _ = oracle.decode_attention(k1, v1, np.ascontiguousarray(wl.q[:, :, h:h + 1]), wl.kv_len, wl.spec.scale)
        assert np.array_equal(o1[0, :, 0], o[0, :, h])


def _fraction_reference(q, K, V, scale):
    """Exact rational dot products, then fp64 exp: the plain definition."""
    zs = []
    for krow in K:
        dot = sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(q, krow)), Fraction(0))
        zs.append(float(dot * Fraction(scale)))
    m = max(zs)
    p = [math.exp(z - m) for z in zs]
    l = math.fsum(p)
    o = [math.fsum(pi * float(V[j][d]) for j, pi in enumerate(p)) / l for d in range(len(V[0]))]
    return np.array(o), m + math.log(l)


@pytest.mark.parametrize("T", [1, 2, 3, 5, 8])
def test_exact_rational_brute_force(T):
    wl = _wl(n_seq=1, H=2, Hk=1, D=64, cached=(T - 1,), seed=10 + T)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    K, V = dequant_cache(k)[0, 0, :T], dequant_cache(v)[0, 0, :T]
    for h in range(2):
        o_ref, lse_ref = _fraction_reference(wl.q[0, 0, h], K, V, wl.spec.scale)
        assert np.abs(o[0, 0, h] - o_ref).max() < 1e-13
        assert abs(lse[0, 0, h] - lse_ref) < 1e-13


def test_equal_scores_give_mean_of_v():
    wl = _wl(n_seq=1, H=2, Hk=1, D=128, cached=(49,), seed=4)
    k, v = oracle_caches(wl)
    q0 = np.zeros_like(wl.q)
    o, lse = oracle.decode_attention(k, v, q0, wl.kv_len, wl.spec.scale)
    Vh = dequant_cache(v)[0, 0, :50].astype(np.float64)
    assert np.abs(o[0, 0, 0] - Vh.mean(axis=0)).max() < 1e-14
    assert abs(lse[0, 0, 0] - math.log(50)) < 1e-14


def test_dominant_key_returns_its_value_row():
    wl = _wl(n_seq=1, H=1, Hk=1, D=128, cached=(63,), seed=5)
    j = 17
    qv = wl.q[0, 0, 0].astype(np.float64)
    wl.k_prefill[0][j, 0] = (40.0 * qv / np.linalg.norm(qv)).astype(np.float32) * math.sqrt(128) / 4
    k, v = oracle_caches(wl)
    o, _ = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    Vh = dequant_cache(v)[0, 0].astype(np.float64)
    assert np.abs(o[0, 0, 0] - Vh[j]).max() < 1e-9


def test_single_visible_key():
    wl = _wl(n_seq=1, H=3, Hk=1, D=64, cached=(0,), n_new=1, seed=6)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    Vh, Kh = dequant_cache(v)[0, 0, 0], dequant_cache(k)[0, 0, 0]
    for h in range(3):
        assert np.array_equal(o[0, 0, h], Vh.astype(np.float64))
        z = float(np.dot(wl.q[0, 0, h].astype(np.float64), Kh.astype(np.float64))) * wl.spec.scale
        assert abs(lse[0, 0, h] - z) < 1e-12


def test_causal_rows_and_empty_rows():
    """With n_q = 3, row i sees kv_len - 3 + i + 1 keys; rows with no key get o = 0, lse = -inf."""
    wl = _wl(n_seq=2, H=2, Hk=1, D=64, cached=(4, 0), n_new=3, seed=7)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    for s in range(2):
        for i in range(3):
            kv = wl.kv_len.copy()
            kv[s] = wl.kv_len[s] - 3 + i + 1
            q1 = np.ascontiguousarray(np.repeat(wl.q[:, i:i + 1], 1, axis=1))
            o1, l1 = oracle.decode_attention(k, v, q1, kv, wl.spec.scale)
            assert np.array_equal(o1[s, 0], o[s, i]) and np.array_equal(l1[s, 0], lse[s, i])
    short = wl.kv_len.copy()
    short[1] = 1                                          # only the last row sees a key
    o2, l2 = oracle.decode_attention(k, v, wl.q, short, wl.spec.scale)
    assert np.all(o2[1, :2] == 0) and np.all(np.isneginf(l2[1, :2])) and np.isfinite(l2[1, 2]).all()


def test_permuting_cache_rows_keeps_output():
    wl = _wl(n_seq=1, H=4, Hk=2, D=128, cached=(99,), seed=8)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    perm = np.random.Generator(np.random.PCG64(0)).permutation(100)
    for c in (k, v):
        c.qs[0, :, :100] = c.qs[0][:, perm]
        c.scales[0, :, :100] = c.scales[0][:, perm]
    o2, lse2 = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    assert np.abs(o - o2).max() < 1e-13 and np.abs(lse - lse2).max() < 1e-13


@pytest.mark.parametrize("n_new", [1, 3])
def test_split_then_merge_equals_unsplit(n_new):
    wl = _wl(n_seq=3, H=6, Hk=2, D=64, cached=(1, 9, 30), n_new=n_new, seed=9)
    k, v = oracle_caches(wl)
    o, lse = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale)
    for n_splits in list(range(1, 36)) + [64]:
        po, pl = oracle.decode_attention_split(k, v, wl.q, wl.kv_len, wl.spec.scale, n_splits)
        om, lm = oracle.merge_splits(po, pl)
        assert np.abs(om - o).max() < 1e-13 and np.abs(lm - lse).max() < 1e-13


def test_merge_closed_forms():
    rng = np.random.Generator(np.random.PCG64(1))
    o1 = rng.standard_normal((1, 4, 32))
    l1 = rng.standard_normal((1, 4))
    om, lm = oracle.merge_splits(o1, l1)                      # one part: identity
    assert np.array_equal(om, o1[0]) and np.array_equal(lm, l1[0])
    om, lm = oracle.merge_splits(np.concatenate([o1, o1]), np.concatenate([l1, l1]))
    assert np.abs(om - o1[0]).max() < 1e-15 and np.abs(lm - (l1[0] + math.log(2))).max() < 1e-14
    o2 = rng.standard_normal((1, 4, 32))                      # exp-weighted mean of two parts
    l2 = l1 + math.log(3.0)                                   # part 2 carries 3x the mass
    om, lm = oracle.merge_splits(np.concatenate([o1, o2]), np.concatenate([l1, l2]))
    assert np.abs(om - (o1[0] + 3 * o2[0]) / 4).max() < 1e-14
    assert np.abs(lm - (l1[0] + math.log(4))).max() < 1e-14
    ninf = np.full((2, 4), -np.inf)                           # all parts empty
    om, lm = oracle.merge_splits(np.zeros((2, 4, 32)), ninf)
    assert not om.any() and np.all(np.isneginf(lm))
    lmix = np.concatenate([l1, np.full((1, 4), -np.inf)])     # an empty part carries no weight
    om, lm = oracle.merge_splits(np.concatenate([o1, np.full((1, 4, 32), 1e300)]), lmix)
    assert np.array_equal(om, o1[0]) and np.array_equal(lm, l1[0])


def test_thread_count_does_not_change_results():
    """The oracle's threads split (sequence, kv head, query row) items; every
    row's arithmetic is the same on any thread, so the results are bitwise
    equal for any thread count."""
    wl = workloads.custom(n_seq=3, n_heads=12, n_kv_heads=2, head_dim=128, cached=(300, 77, 5), n_new=3,
                          src_dtype="f16", q_dtype="f16", seed=31)
    k, v = oracle_caches(wl)
    o1, l1 = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale, n_threads=1)
    for n in (2, 3, 8):
        on, ln = oracle.decode_attention(k, v, wl.q, wl.kv_len, wl.spec.scale, n_threads=n)
        assert np.array_equal(o1, on) and np.array_equal(l1, ln)
