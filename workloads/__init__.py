"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers and lays them out; it holds none of the
codec or attention arithmetic, so that both the CUDA path and the oracle can be
fed the same arrays without sharing any of the method's code.

Workloads 0-4 stand in for the long-context decode and MTP-verify runs of
a 27B hybrid model described on den_llama.cpp ("Results": 32K and 65K serving
with MTP n-max 2; "What this fork is": up to 196K context; "Build3 (working
engine)": the matched Q4_G64 pair and the mixed q8_0-K / Q4_G64-V pair).  No
dataset or model weights are involved: K, V and Q are Gaussian draws with the
shapes below.

Recipe (numpy ``Generator(PCG64)``; base seed 20261202 + workload index;
``SeedSequence.spawn`` gives one independent stream each for K, V, Q, K bias,
V bias, the outlier mask and the sequence lengths):

  0 tiny      S=1, Hq=Hkv=1, D=128, 255 cached + 1 appended token, n_q=1,
              K/V/Q fp32 ~ N(0,1), Q4_G64 K and V, scale 1/sqrt(128).
  1 gqa32k    S=1, Hq=24, Hkv=4, D=256, 32767 cached + 1 appended, n_q=1,
              K/V fp16 ~ N(0,1) with each element x8 with probability 0.01,
              Q fp16 ~ N(0,1); Q4_G64 K and V.
  2 mixed65k  as 1 with 65535 cached + 1 appended, K/V fp16 ~ N(0,1) without
              outliers; K q8_0, V Q4_G64.
  3 long196k  as 1 with 196607 cached + 1 appended; K/V fp16 = N(0, 0.5^2)
              + bias, bias ~ N(0, 2^2) per (kv head, channel), drawn
              separately for K and V.
  4 mtp16     S=16, L_s = round(exp(U(ln 1024, ln 65536))) cached tokens,
              3 appended tokens per sequence (1 + 2 draft), n_q=3 (causal),
              K/V/Q fp16 ~ N(0,1); Q4_G64 K and V.
  5 ship65k   as 2 with K q8_0 / V Q4_G32 (the pages' shipped -ctk q8_0 -ctv q4_0
              pair, q4_0 read as Q4 with 32-value groups); not a benchmark
              workload, it carries that pair through the same tests.
  6 nvfp4_65k as 2 with K and V in NVFP4 (the pages' matched -ctk nvfp4 -ctv
              nvfp4 KV type); likewise a test case.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

Q4_G64 = 1
Q8_0 = 2
Q4_G32 = 3
NVFP4 = 4                 # E2M1 values, one E4M3 scale per 16
BASE_SEED = 20261202
TOKEN_ALIGN = 64          # cache capacity is a multiple of this many tokens


@dataclasses.dataclass
class Spec:
    name: str
    n_seq: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    cached: tuple            # tokens already in the cache, per sequence (None = draw log-uniform)
    n_new: int               # tokens appended (and queried) per step, per sequence
    k_codec: int
    v_codec: int
    src_dtype: str           # 'f32' or 'f16' for K/V sources
    q_dtype: str             # 'f32' or 'f16'
    dist: str                # 'normal', 'outliers', 'bias'
    seed: int
    len_range: Optional[tuple] = None

    @property
    def n_q(self) -> int:
        return self.n_new

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)


def spec(index: int) -> Spec:
    s = BASE_SEED + index
    if index == 0:
        return Spec("tiny", 1, 1, 1, 128, (255,), 1, Q4_G64, Q4_G64, "f32", "f32", "normal", s)
    if index == 1:
        return Spec("gqa32k", 1, 24, 4, 256, (32767,), 1, Q4_G64, Q4_G64, "f16", "f16", "outliers", s)
    if index == 2:
        return Spec("mixed65k", 1, 24, 4, 256, (65535,), 1, Q8_0, Q4_G64, "f16", "f16", "normal", s)
    if index == 3:
        return Spec("long196k", 1, 24, 4, 256, (196607,), 1, Q4_G64, Q4_G64, "f16", "f16", "bias", s)
    if index == 4:
        return Spec("mtp16", 16, 24, 4, 256, None, 3, Q4_G64, Q4_G64, "f16", "f16", "normal", s,
                    len_range=(1024, 65536))
    if index == 5:
        return Spec("ship65k", 1, 24, 4, 256, (65535,), 1, Q8_0, Q4_G32, "f16", "f16", "normal", s)
    if index == 6:
        return Spec("nvfp4_65k", 1, 24, 4, 256, (65535,), 1, NVFP4, NVFP4, "f16", "f16", "normal", s)
    raise ValueError(index)


N_CONFIGS = 7                # 0..4 the benchmark's workloads, 5 the shipped q8_0-K / q4_0-V pair, 6 NVFP4


@dataclasses.dataclass
class Workload:
    spec: Spec
    cached_len: np.ndarray   # int32 [S]: tokens already in the cache (= append position)
    kv_len: np.ndarray       # int32 [S]: keys visible to the last query token
    capacity: int
    k_prefill: list          # per sequence s: [cached_len[s]][Hkv][D]
    v_prefill: list
    k_new: np.ndarray        # [S][n_new][Hkv][D]
    v_new: np.ndarray
    q: np.ndarray            # [S][n_q][Hq][D]

    @property
    def max_kv_len(self) -> int:
        return int(self.kv_len.max())


def _np_dtype(name: str):
    return np.float32 if name == "f32" else np.float16


def _draw_values(rng, mask_rng, shape, dist, bias, dtype):
    if dist == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    elif dist == "outliers":
        x = rng.standard_normal(shape, dtype=np.float32)
        x *= np.where(mask_rng.random(shape, dtype=np.float32) < 0.01, np.float32(8.0), np.float32(1.0))
    elif dist == "bias":
        x = rng.standard_normal(shape, dtype=np.float32) * np.float32(0.5) + bias
    else:
        raise ValueError(dist)
    return x.astype(dtype)


def make(sp: Spec, cached=None) -> Workload:
    """Draw a workload.  ``cached`` overrides the cached lengths (a shorter
    instance of the same recipe, e.g. for tests the oracle must finish fast)."""
    ss = np.random.SeedSequence(sp.seed)
    k_ss, v_ss, q_ss, kb_ss, vb_ss, m_ss, l_ss = ss.spawn(7)
    if cached is None:
        if sp.cached is None:
            lo, hi = sp.len_range
            u = np.random.Generator(np.random.PCG64(l_ss)).uniform(math.log(lo), math.log(hi), sp.n_seq)
            cached = np.rint(np.exp(u)).astype(np.int64)
        else:
            cached = np.array(sp.cached, dtype=np.int64)
    cached = np.asarray(cached, dtype=np.int64).reshape(sp.n_seq)
    kv_len = cached + sp.n_new
    capacity = int(-(-int(kv_len.max()) // TOKEN_ALIGN) * TOKEN_ALIGN)
    S, Hk, D, H = sp.n_seq, sp.n_kv_heads, sp.head_dim, sp.n_heads
    dt = _np_dtype(sp.src_dtype)
    kb = vb = None
    if sp.dist == "bias":
        kb = np.random.Generator(np.random.PCG64(kb_ss)).standard_normal((Hk, D), dtype=np.float32) * 2.0
        vb = np.random.Generator(np.random.PCG64(vb_ss)).standard_normal((Hk, D), dtype=np.float32) * 2.0
    k_rng = np.random.Generator(np.random.PCG64(k_ss))
    v_rng = np.random.Generator(np.random.PCG64(v_ss))
    m_rng = np.random.Generator(np.random.PCG64(m_ss))
    k_pre, v_pre = [], []
    k_new = np.empty((S, sp.n_new, Hk, D), dt)
    v_new = np.empty((S, sp.n_new, Hk, D), dt)
    for s in range(S):          # each sequence: its cached tokens, then the new ones
        c = int(cached[s])
        ka = _draw_values(k_rng, m_rng, (c + sp.n_new, Hk, D), sp.dist, kb, dt)
        va = _draw_values(v_rng, m_rng, (c + sp.n_new, Hk, D), sp.dist, vb, dt)
        k_pre.append(ka[:c])
        v_pre.append(va[:c])
        k_new[s] = ka[c:]
        v_new[s] = va[c:]
    q = np.random.Generator(np.random.PCG64(q_ss)).standard_normal((S, sp.n_q, H, D), dtype=np.float32)
    q = q.astype(_np_dtype(sp.q_dtype))
    return Workload(sp, cached.astype(np.int32), kv_len.astype(np.int32), capacity,
                    k_pre, v_pre, k_new, v_new, q)


def custom(name="custom", n_seq=1, n_heads=1, n_kv_heads=1, head_dim=128, cached=(64,), n_new=1,
           k_codec=Q4_G64, v_codec=Q4_G64, src_dtype="f32", q_dtype="f32", dist="normal", seed=7):
    sp = Spec(name, n_seq, n_heads, n_kv_heads, head_dim, tuple(cached), n_new, k_codec, v_codec,
              src_dtype, q_dtype, dist, BASE_SEED + 1000 + seed)
    return make(sp)


def kv_bytes_per_token(sp: Spec) -> int:
    """Packed K + V bytes of one token over all kv heads (codes + scales)."""
    def row(codec):
        if codec == NVFP4:
            return sp.head_dim // 2 + sp.head_dim // 16
        if codec == Q4_G64:
            return sp.head_dim // 2 + 2 * (sp.head_dim // 64)
        if codec == Q4_G32:
            return sp.head_dim // 2 + 2 * (sp.head_dim // 32)
        return sp.head_dim + 2 * (sp.head_dim // 32)
    return sp.n_kv_heads * (row(sp.k_codec) + row(sp.v_codec))


def rand_partials(n_splits: int, rows: int, head_dim: int, seed: int = 3, empty_frac: float = 0.1):
    """Random split partials for merge tests: o ~ N(0,1), lse ~ N(0, 4^2);
    a fraction of (split, row) entries are empty (lse = -inf, o = 0)."""
    rng = np.random.Generator(np.random.PCG64(BASE_SEED + 5000 + seed))
    o = rng.standard_normal((n_splits, rows, head_dim), dtype=np.float32)
    lse = (rng.standard_normal((n_splits, rows), dtype=np.float32) * 4.0).astype(np.float32)
    empty = rng.random((n_splits, rows)) < empty_frac
    lse[empty] = -np.inf
    o[empty] = 0.0
    return o, lse


def wide_range_rows(n_rows: int, head_dim: int, seed: int = 0, dtype=np.float32) -> np.ndarray:
    """Rows whose 32-value blocks span magnitudes 1e-9..3e4 (fp16-subnormal and
    saturating scales included), for codec edge cases."""
    rng = np.random.Generator(np.random.PCG64(BASE_SEED + 7000 + seed))
    nb = head_dim // 32
    mag = np.exp(rng.uniform(np.log(1e-9), np.log(3e4), size=(n_rows, nb, 1)))
    x = rng.standard_normal((n_rows, nb, 32)) * mag
    heavy = rng.random((n_rows, nb)) < 0.2
    x[heavy] *= np.exp(rng.standard_normal((int(heavy.sum()), 32)) * 2)
    x = x.reshape(n_rows, head_dim)
    if dtype == np.float16:
        x = np.clip(x, -60000, 60000)
    return x.astype(dtype)
