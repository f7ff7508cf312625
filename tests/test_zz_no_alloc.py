"""kvq_decode_attention_static: decode attention for callers that cannot
allocate device memory where they decode (for example while a CUDA graph is
being captured, or inside an engine that owns all device memory through its
own pool).  Its results must meet the same bar against the fp64 oracle as
kvq_decode_attention's, call after call, and match that entry point's results
with a caller-owned workspace; requests whose split scratch cannot fit the
library's static array are refused, except that the default split count is
lowered until it fits.

This file is collected last on purpose (its name), so that a run stopping at
the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import dev, gpu_caches
from helpers import check_close, oracle_caches

pytestmark = pytest.mark.gpu


def _static_twice(wl, k, v, n_splits):
    S, nq, H, D = wl.q.shape
    q, kv_len = dev(wl.q), dev(wl.kv_len)
    max_kv = int(wl.kv_len.max())
    results = []
    for _ in range(2):                         # the array keeps the last call's contents
        out = torch.full((S, nq, H, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((S, nq, H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_decode_attention_static(k, v, q, nq, H, wl.spec.scale, kv_len, max_kv, n_splits, out, lse, d_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        results.append((out.cpu().numpy(), lse.cpu().numpy()))
    return results


@pytest.mark.parametrize("n_new,n_splits", [(1, 8), (3, 5), (1, 0)])
def test_static_scratch_matches_oracle_and_workspace_entry_point(n_new, n_splits):
    wl = workloads.custom(n_seq=2, n_heads=24, n_kv_heads=4, head_dim=256, cached=(3000, 1200), n_new=n_new,
                          src_dtype="f16", q_dtype="f16", dist="outliers", seed=90 + n_new)
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    S, nq, H, D = wl.q.shape
    max_kv = int(wl.kv_len.max())
    assert kvq.kvq_decode_workspace_bytes(k, v, H, nq, max_kv, n_splits) <= kvq.kvq_static_scratch_bytes()
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    ws_o, ws_lse = kvq.decode(k, v, dev(wl.q), dev(wl.kv_len), max_kv, wl.spec.scale, n_splits=n_splits)
    for o, lse in _static_twice(wl, k, v, n_splits):
        check_close(o, o_ref, lse, lse_ref)                                    # the acceptance bar
        check_close(o, ws_o.cpu().numpy(), lse, ws_lse.cpu().numpy(), atol=1e-6, rtol_l2=1e-6, lse_atol=1e-6)


def test_static_default_splits_lowered_to_fit():
    """A batch whose default split count would need more scratch than the
    static array holds: with n_splits = 0 the count is lowered until it fits,
    and the result still meets the bar."""
    lens = (1500, 1800, 2000, 1700, 1900, 1600, 2000, 1999, 1888, 1777, 1666, 1555, 1444, 1950, 1850, 1750)
    wl = workloads.custom(n_seq=16, n_heads=24, n_kv_heads=4, head_dim=256, cached=lens, n_new=3,
                          src_dtype="f16", q_dtype="f16", seed=97)
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    S, nq, H, D = wl.q.shape
    max_kv = int(wl.kv_len.max())
    assert kvq.kvq_decode_workspace_bytes(k, v, H, nq, max_kv, 0) > kvq.kvq_static_scratch_bytes()
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale, n_threads=oracle.max_threads())
    for o, lse in _static_twice(wl, k, v, 0):
        check_close(o, o_ref, lse, lse_ref)


def test_static_scratch_rejects_oversized_request():
    wl = workloads.custom(n_seq=1, n_heads=24, n_kv_heads=4, head_dim=256, cached=(2047,), n_new=1,
                          src_dtype="f16", q_dtype="f16", seed=95)
    k, v = gpu_caches(wl)
    n_splits = 4096
    need = kvq.kvq_decode_workspace_bytes(k, v, 24, 1, 2048, n_splits)
    assert need > kvq.kvq_static_scratch_bytes()
    out = torch.zeros((1, 1, 24, 256), dtype=torch.float32, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attention_static(k, v, dev(wl.q), 1, 24, wl.spec.scale, dev(wl.kv_len), 2048, n_splits, out)
    assert e.value.status == kvq.KVQ_EWORKSPACE
    assert "static array" in str(e.value)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attention_static(k, v, dev(wl.q), 1, 24, wl.spec.scale, dev(wl.kv_len), 2048, 4097, out)
    assert e.value.status == kvq.KVQ_EINVAL
    torch.cuda.synchronize()
    assert not out.any()                       # nothing was launched
