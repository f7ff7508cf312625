"""kvq_decode_attention_static: decode attention for callers that cannot
allocate device memory where they decode (for example while a CUDA graph is
being captured, or inside an engine that owns all device memory through its
own pool).  It must give the same results as kvq_decode_attention with a
caller-owned workspace, call after call, and refuse requests whose split
scratch would not fit the library's static array.

This file is collected last on purpose (its name), so that a run stopping at
the first failure has already run every other test."""
import numpy as np
import pytest
import torch

import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import dev, gpu_caches
from helpers import check_close

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_new,n_splits", [(1, 8), (3, 5), (1, 0)])
def test_static_scratch_matches_workspace_entry_point_two_calls(n_new, n_splits):
    wl = workloads.custom(n_seq=2, n_heads=24, n_kv_heads=4, head_dim=256, cached=(3000, 1200), n_new=n_new,
                          src_dtype="f16", q_dtype="f16", dist="outliers", seed=90 + n_new)
    k, v = gpu_caches(wl)
    q, kv_len = dev(wl.q), dev(wl.kv_len)
    max_kv = int(wl.kv_len.max())
    S, nq, H, D = wl.q.shape
    assert kvq.kvq_decode_workspace_bytes(k, v, H, nq, max_kv, n_splits) <= kvq.kvq_static_scratch_bytes()
    ref, ref_lse = kvq.decode(k, v, q, kv_len, max_kv, wl.spec.scale, n_splits=n_splits)
    for _ in range(2):                         # the array keeps the last call's contents
        out = torch.full((S, nq, H, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((S, nq, H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_decode_attention_static(k, v, q, nq, H, wl.spec.scale, kv_len, max_kv, n_splits, out, lse, d_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        check_close(out.cpu().numpy(), ref.cpu().numpy(), lse.cpu().numpy(), ref_lse.cpu().numpy())


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
    torch.cuda.synchronize()
    assert not out.any()                       # nothing was launched
