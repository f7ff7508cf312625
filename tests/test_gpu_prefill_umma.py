"""Prompt chunks on the tcgen05 kernel (blocks of 128 query rows per CTA,
Q4_G64 K and V, fp16 queries, head_dim 64/128/256) against the fp64 oracle,
at the decode bar: max-abs 2e-3, rel-L2 1e-2, lse 1e-3.

Rows per kv head >= 64 with those codecs take this kernel (the Q4_G32 pairs
below run the same shapes through the mma.sync kernel); the shapes below
cover one block exactly at its lower bound (64 rows), a ragged single block
(72, 96 rows), one row past a block (132 rows = 128 + 4), several blocks
with a ragged last one (240, 1,536 rows), split counts that leave some
splits empty, ragged batches with sequences shorter than one tile, and rows
that see no key at all."""
import numpy as np
import pytest

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import gpu_caches, run_decode
from helpers import check_close, oracle_caches

pytestmark = pytest.mark.gpu

G64, G32 = kvq.KVQ_CODEC_Q4_G64, kvq.KVQ_CODEC_Q4_G32


def _both(wl):
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    return k, v, ko, vo


@pytest.mark.parametrize("kc,vc", [(G64, G64), (G32, G64), (G64, G32), (G32, G32)])
@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("G,n_new", [(8, 8), (6, 22), (6, 40)])
def test_prompt_chunk_blocks_of_128_rows(kc, vc, D, G, n_new):
    wl = workloads.custom(n_seq=2, n_heads=2 * G, n_kv_heads=2, head_dim=D, cached=(1000 - n_new, 150), n_new=n_new,
                          k_codec=kc, v_codec=vc, src_dtype="f16", q_dtype="f16", seed=kc + 5 * vc + D + 7 * G + n_new)
    k, v, ko, vo = _both(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    for n_splits in (0, 1, 3, 9):
        o, lse, err = run_decode(wl, k, v, n_splits=n_splits)
        assert err == 0
        check_close(o, o_ref, lse, lse_ref)


@pytest.mark.parametrize("D", [128, 256])
def test_outlier_keys_and_values(D):
    """Source values N(0,1) with 1% outliers x8 in K and V."""
    wl = workloads.custom(n_seq=1, n_heads=12, n_kv_heads=2, head_dim=D, cached=(3000,), n_new=24, src_dtype="f16",
                          q_dtype="f16", dist="outliers", seed=300 + D)
    k, v, ko, vo = _both(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    for n_splits in (0, 1, 4):
        o, lse, err = run_decode(wl, k, v, n_splits=n_splits)
        assert err == 0
        check_close(o, o_ref, lse, lse_ref)


def test_ragged_batch():
    """Four sequences, one shorter than a tile and one with fewer cached keys
    than the chunk: rows of the first chunk tokens see very few keys."""
    wl = workloads.custom(n_seq=4, n_heads=12, n_kv_heads=2, head_dim=256, cached=(5, 700, 64, 3000), n_new=12,
                          src_dtype="f16", q_dtype="f16", seed=310)
    k, v, ko, vo = _both(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    for n_splits in (0, 1, 5, 40):
        o, lse, err = run_decode(wl, k, v, n_splits=n_splits)
        assert err == 0
        check_close(o, o_ref, lse, lse_ref)


def test_rows_without_keys():
    """kv_len < n_q: the first rows of sequence 0 see no key -> out = 0, lse = -inf."""
    wl = workloads.custom(n_seq=2, n_heads=6, n_kv_heads=1, head_dim=128, cached=(0, 10), n_new=16, src_dtype="f16",
                          q_dtype="f16", seed=311)
    k, v, ko, vo = _both(wl)
    kv_len = wl.kv_len.copy()
    kv_len[0] = 5                       # tokens 0..10 of sequence 0 see nothing
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, kv_len, wl.spec.scale)
    for n_splits in (1, 3):
        o, lse, err = run_decode(wl, k, v, n_splits=n_splits, kv_len=kv_len)
        assert err == 0
        check_close(o, o_ref, lse, lse_ref)
        assert np.all(o[0, :11] == 0) and np.all(np.isneginf(lse[0, :11]))


def test_long_chunk_many_blocks():
    """A 256-token chunk of 24 query heads over 4 kv heads (1,536 rows per kv
    head = 12 blocks) after 7,936 cached keys, default and explicit splits."""
    wl = workloads.custom(n_seq=1, n_heads=24, n_kv_heads=4, head_dim=256, cached=(7936,), n_new=256,
                          src_dtype="f16", q_dtype="f16", seed=312)
    k, v, ko, vo = _both(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale, n_threads=oracle.max_threads())
    for n_splits in (0, 2):
        o, lse, err = run_decode(wl, k, v, n_splits=n_splits)
        assert err == 0
        check_close(o, o_ref, lse, lse_ref)


def test_fp32_query_chunk_stays_exact():
    """fp32 queries of a prompt chunk take the mma.sync kernel (two fp16 query
    parts); the split count is the one the tcgen05 shape asks for."""
    wl = workloads.custom(n_seq=1, n_heads=12, n_kv_heads=2, head_dim=256, cached=(2000,), n_new=24,
                          src_dtype="f16", q_dtype="f32", dist="outliers", seed=313)
    k, v, ko, vo = _both(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    o, lse, err = run_decode(wl, k, v)
    assert err == 0
    check_close(o, o_ref, lse, lse_ref)
