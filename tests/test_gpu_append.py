"""Quantize-on-append on the GPU is byte-identical to the oracle (den_llama.cpp,
"build3 (working engine) -- additions": the Q4_G64 quantizer byte-identical to
the CPU reference, the dequantizer bit-identical)."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import dev, gpu_caches, host_planes
from helpers import oracle_caches

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg", range(workloads.N_CONFIGS))
def test_workload_caches_byte_exact(cfg):
    wl = workloads.make(workloads.spec(cfg))
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    for g, o in ((k, ko), (v, vo)):
        qs, sc = host_planes(g)
        for s in range(wl.spec.n_seq):
            n = int(wl.kv_len[s])
            assert np.array_equal(qs[s, :, :n], o.qs[s, :, :n])
            assert np.array_equal(sc[s, :, :n], o.scales[s, :, :n])


@pytest.mark.parametrize("codec", [kvq.KVQ_CODEC_Q4_G64, kvq.KVQ_CODEC_Q8_0, kvq.KVQ_CODEC_Q4_G32,
                                   kvq.KVQ_CODEC_NVFP4])
@pytest.mark.parametrize("D", [64, 128, 256, 512])
@pytest.mark.parametrize("dtype", [np.float32, np.float16])
def test_wide_range_rows_byte_exact(codec, D, dtype):
    S, n_new, Hk, cap = 3, 5, 2, 64
    x = workloads.wide_range_rows(S * n_new * Hk, D, seed=D + codec, dtype=dtype).reshape(S, n_new, Hk, D)
    pos0 = np.array([0, 17, 60], np.int32)          # 60 + 5 > 64: the last one is skipped and flagged
    c = kvq.KVCache(codec, S, Hk, D, cap)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_quantize_append(c, None, dev(x), None, n_new, dev(pos0), err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.KVQ_ERR_APPEND_POS
    oc = oracle.Cache(codec, S, Hk, D, cap)
    assert oracle.quantize_append(oc, x, pos0) == 1
    qs, sc = host_planes(c)
    assert np.array_equal(qs, oc.qs) and np.array_equal(sc, oc.scales)
    # dequantization on the GPU is bit-identical to scale * code
    out = torch.empty((S, Hk, cap, D), dtype=torch.float32, device="cuda")
    kvq.kvq_dequantize(c, out)
    ref = oracle.dequantize(codec, oc.qs, oc.scales, D)
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_append_k_only_and_v_only():
    wl = workloads.custom(n_seq=2, n_heads=2, n_kv_heads=2, head_dim=128, cached=(3, 9), n_new=2, src_dtype="f16")
    k = kvq.KVCache(kvq.KVQ_CODEC_Q4_G64, 2, 2, 128, wl.capacity)
    v = kvq.KVCache(kvq.KVQ_CODEC_Q8_0, 2, 2, 128, wl.capacity)
    pos = dev(wl.cached_len)
    kvq.kvq_quantize_append(k, None, dev(wl.k_new), None, 2, pos)
    kvq.kvq_quantize_append(None, v, None, dev(wl.v_new), 2, pos)
    torch.cuda.synchronize()
    ko = oracle.Cache(oracle.Q4_G64, 2, 2, 128, wl.capacity)
    vo = oracle.Cache(oracle.Q8_0, 2, 2, 128, wl.capacity)
    oracle.quantize_append(ko, wl.k_new, wl.cached_len)
    oracle.quantize_append(vo, wl.v_new, wl.cached_len)
    for g, o in ((k, ko), (v, vo)):
        qs, sc = host_planes(g)
        assert np.array_equal(qs, o.qs) and np.array_equal(sc, o.scales)


def test_negative_position_is_flagged():
    c = kvq.KVCache(kvq.KVQ_CODEC_Q4_G64, 1, 1, 64, 64)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = torch.ones((1, 1, 1, 64), dtype=torch.float32, device="cuda")
    kvq.kvq_quantize_append(c, None, x, None, 1, torch.tensor([-1], dtype=torch.int32, device="cuda"), err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.KVQ_ERR_APPEND_POS and not c.qs.any()
