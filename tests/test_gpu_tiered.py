"""Host-tier KV streaming (den_llama.cpp, "Adaptive KV streaming
(contributed)"): the authoritative cache in pinned host memory, the first
tokens resident on the device, the rest streamed in pages through a bounded
device ring; the attention must meet the same bar against the fp64 oracle as
kvq_decode_attention over the whole device cache, and agree with it."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import dev, gpu_caches
from helpers import check_close, oracle_caches

pytestmark = pytest.mark.gpu


def _tiered(wl, k, v, kh, vh, n_res, page, n_slots, repeats=2):
    S, nq, H, D = wl.q.shape
    kv_len = int(wl.kv_len[0])
    kd, vd = (k, v) if n_res > 0 else (None, None)
    ring = kvq.alloc_workspace(kvq.kvq_tiered_ring_bytes(kh, vh, page, n_slots))
    ws = kvq.alloc_workspace(kvq.kvq_tiered_workspace_bytes(kh, vh, kd, vd, H, nq, kv_len, n_res, page))
    q = dev(wl.q)
    results = []
    for _ in range(repeats):                   # the ring and workspace are reused call after call
        out = torch.full((S, nq, H, D), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((S, nq, H), float("nan"), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        kvq.kvq_decode_attention_tiered(kh, vh, kd, vd, n_res, q, nq, H, wl.spec.scale, kv_len, page, n_slots,
                                        ring, out, lse, ws, d_err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        results.append((out.cpu().numpy(), lse.cpu().numpy()))
    return results


@pytest.mark.parametrize("kc,D,q_dtype,dist", [(kvq.KVQ_CODEC_Q4_G64, 256, "f16", "outliers"),
                                               (kvq.KVQ_CODEC_Q8_0, 256, "f16", "outliers"),
                                               (kvq.KVQ_CODEC_Q4_G64, 128, "f32", "outliers"),
                                               (kvq.KVQ_CODEC_Q4_G64, 128, "f32", "normal")])
@pytest.mark.parametrize("n_res,page,n_slots", [(1024, 640, 2), (0, 1024, 3), (5000, 640, 1), (4992, 64, 1),
                                                (3000, 128, 4)])
def test_tiered_matches_oracle_and_device_path(kc, D, q_dtype, dist, n_res, page, n_slots):
    # 5,000 keys, 3 query tokens (MTP verify rows attend causally: the new
    # tokens sit in the last page, or in the resident part when n_res = 5000)
    wl = workloads.custom(n_seq=1, n_heads=24, n_kv_heads=4, head_dim=D, cached=(4997,), n_new=3, k_codec=kc,
                          src_dtype="f16", q_dtype=q_dtype, dist=dist, seed=70 + kc + D)
    k, v = gpu_caches(wl)
    kh, vh = k.to_host(), v.to_host()
    ko, vo = oracle_caches(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    d_out, d_lse = kvq.decode(k, v, dev(wl.q), dev(wl.kv_len), int(wl.kv_len[0]), wl.spec.scale)
    for o, lse in _tiered(wl, k, v, kh, vh, n_res, page, n_slots):
        check_close(o, o_ref, lse, lse_ref)
        # the device path partitions the keys differently (split boundaries, so
        # the running maxima and the fp16 rounding of the weights differ): the
        # two agree within a quarter of the bar
        check_close(o, d_out.cpu().numpy(), lse, d_lse.cpu().numpy(), atol=5e-4, rtol_l2=2.5e-3, lse_atol=2.5e-4)


def test_tiered_long_context_many_pages():
    """65,536 keys with 8,192 resident and the rest in 56 pages of 1,024 through
    a ring of 3 slots."""
    wl = workloads.custom(n_seq=1, n_heads=24, n_kv_heads=4, head_dim=256, cached=(65535,), n_new=1,
                          src_dtype="f16", q_dtype="f16", seed=77)
    k, v = gpu_caches(wl)
    kh, vh = k.to_host(), v.to_host()
    ko, vo = oracle_caches(wl)
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale, n_threads=oracle.max_threads())
    for o, lse in _tiered(wl, k, v, kh, vh, 8192, 1024, 3, repeats=1):
        check_close(o, o_ref, lse, lse_ref)
