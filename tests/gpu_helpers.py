"""GPU-side test helpers: build device caches through the library's append entry point."""
import numpy as np
import torch

import quantized_kv_cache_q4_gb300 as kvq
import workloads


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_caches(wl: workloads.Workload, append=True):
    """Quantize the cached tokens of every sequence (one append call per
    sequence, positions 0..L-1) and then the new tokens at their positions."""
    sp = wl.spec
    k = kvq.KVCache(sp.k_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    v = kvq.KVCache(sp.v_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    zero = torch.zeros(1, dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for s in range(sp.n_seq):
        L = int(wl.cached_len[s])
        if L == 0:
            continue
        kvq.kvq_quantize_append(k.seq_view(s), v.seq_view(s), dev(wl.k_prefill[s][None]),
                                dev(wl.v_prefill[s][None]), L, zero, err)
    if append:
        kvq.kvq_quantize_append(k, v, dev(wl.k_new), dev(wl.v_new), sp.n_new, dev(wl.cached_len), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return k, v


def host_planes(c: kvq.KVCache):
    """The planes as the oracle holds them: codes uint8, scales uint16 fp16 bit
    patterns (uint8 E4M3 bytes for NVFP4)."""
    if c.scales.dtype == torch.uint8:
        return c.qs.cpu().numpy(), c.scales.cpu().numpy()
    return c.qs.cpu().numpy(), c.scales.cpu().view(torch.int16).numpy().view(np.uint16)


def run_decode(wl, k, v, n_splits=0, kv_len=None, max_kv_len=None, q=None):
    sp = wl.spec
    kv_len = wl.kv_len if kv_len is None else kv_len
    max_kv_len = int(np.max(kv_len)) if max_kv_len is None else max_kv_len
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = kvq.decode(k, v, dev(wl.q if q is None else q), dev(np.asarray(kv_len, np.int32)), max(1, max_kv_len),
                          softmax_scale=sp.scale, n_splits=n_splits, d_err=err)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), int(err.item())
