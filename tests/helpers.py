"""Test-side helpers: build oracle caches from a seeded workload and compare results."""
import numpy as np

import oracle
import workloads


def oracle_caches(wl: workloads.Workload, append=True):
    """Quantize the cached tokens (and, if ``append``, the new tokens at their
    append positions) into oracle caches."""
    sp = wl.spec
    k = oracle.Cache(sp.k_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    v = oracle.Cache(sp.v_codec, sp.n_seq, sp.n_kv_heads, sp.head_dim, wl.capacity)
    for s in range(sp.n_seq):
        L = int(wl.cached_len[s])
        if L == 0:
            continue
        for cache, src in ((k, wl.k_prefill), (v, wl.v_prefill)):
            qs, sc = oracle.quantize(cache.codec, np.ascontiguousarray(src[s].transpose(1, 0, 2)))
            cache.qs[s, :, :L] = qs
            cache.scales[s, :, :L] = sc
    if append:
        assert oracle.quantize_append(k, wl.k_new, wl.cached_len) == 0
        assert oracle.quantize_append(v, wl.v_new, wl.cached_len) == 0
    return k, v


def dequant_cache(cache: oracle.Cache) -> np.ndarray:
    return oracle.dequantize(cache.codec, cache.qs, cache.scales, cache.head_dim)


def check_close(o_gpu, o_ref, lse_gpu=None, lse_ref=None, atol=2e-3, rtol_l2=1e-2, lse_atol=1e-3):
    """Acceptance bar: max |o - o_ref| <= atol and ||o - o_ref||_2 / ||o_ref||_2 <= rtol_l2;
    lse within lse_atol where finite and -inf exactly where the reference is."""
    o_gpu = np.asarray(o_gpu, np.float64)
    o_ref = np.asarray(o_ref, np.float64)
    assert o_gpu.shape == o_ref.shape
    assert np.all(np.isfinite(o_gpu))
    err = np.abs(o_gpu - o_ref)
    maxabs = float(err.max()) if err.size else 0.0
    nref = float(np.linalg.norm(o_ref))
    rel = float(np.linalg.norm(o_gpu - o_ref) / nref) if nref > 0 else float(np.linalg.norm(o_gpu))
    assert maxabs <= atol, f"max-abs {maxabs:.3e} > {atol}"
    assert rel <= rtol_l2, f"rel-L2 {rel:.3e} > {rtol_l2}"
    if lse_gpu is not None:
        lg = np.asarray(lse_gpu, np.float64)
        lr = np.asarray(lse_ref, np.float64)
        fin = np.isfinite(lr)
        assert np.array_equal(np.isfinite(lg), fin)
        if fin.any():
            assert np.abs(lg[fin] - lr[fin]).max() <= lse_atol
    return maxabs, rel
