"""The decode kernel for up to 8 query rows per kv head (12 warps per SM, each
streaming its own run of 16-token blocks) against the fp64 oracle, on the
cases its softmax bookkeeping has to survive.

That kernel raises its running reference maximum lazily: only when a block's
maximum passes it by more than 2^8, so p = 2^(s - m) may reach 2^8 -- unless a
V scale of the block is 256 or more, where P' = p * scale would overflow fp16
and the reference follows every new maximum exactly.

Bar: the acceptance bar of test_gpu_decode (max-abs 2e-3, relative L2 1e-2,
lse 1e-3); an output whose V was multiplied by c is compared divided by c
(attention is linear in V, the lse does not depend on it)."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import gpu_caches, run_decode
from helpers import check_close, oracle_caches

pytestmark = pytest.mark.gpu


def _run(wl, n_splits=0):
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    o, lse, err = run_decode(wl, k, v, n_splits=n_splits)
    assert err == 0
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale, n_threads=oracle.max_threads())
    return o, lse, o_ref, lse_ref


@pytest.mark.parametrize("factor", [300.0, 2000.0])
@pytest.mark.parametrize("kc", [workloads.Q4_G64, workloads.Q8_0])
def test_large_v_scales(factor, kc):
    """V values of a few hundred to ~10,000 (V scales up to ~1,500): P' stays
    finite and the result meets the bar relative to the V factor."""
    wl = workloads.custom(n_seq=1, n_heads=24, n_kv_heads=4, head_dim=256, cached=(12000,), n_new=1, k_codec=kc,
                          src_dtype="f16", q_dtype="f16", dist="normal", seed=300 + int(factor) + kc)
    f16 = np.float16
    wl.v_prefill = [(x.astype(np.float32) * factor).astype(f16) for x in wl.v_prefill]
    wl.v_new = (wl.v_new.astype(np.float32) * factor).astype(f16)
    assert np.isfinite(wl.v_prefill[0]).all() and np.abs(wl.v_prefill[0]).max() < 60000
    o, lse, o_ref, lse_ref = _run(wl)
    assert np.isfinite(o).all()
    check_close(o / factor, o_ref / factor, lse, lse_ref)


@pytest.mark.parametrize("n_splits", [0, 4])
def test_scores_climbing_along_the_sequence(n_splits):
    """Keys drift towards the queries along the sequence, so the row maxima keep
    growing (by ~45 in log2 units over the run): the lazy reference is raised
    over and over and the accumulators rescaled each time."""
    wl = workloads.custom(n_seq=2, n_heads=24, n_kv_heads=4, head_dim=256, cached=(9000, 5000), n_new=1,
                          src_dtype="f16", q_dtype="f16", seed=310 + n_splits)
    f16 = np.float16
    for s in range(2):
        L = wl.k_prefill[s].shape[0]
        drift = np.linspace(0.0, 2.0, L + 1, dtype=np.float32)
        wl.k_prefill[s] = (wl.k_prefill[s].astype(np.float32) + drift[:L, None, None]).astype(f16)
        wl.k_new[s] = (wl.k_new[s].astype(np.float32) + drift[L]).astype(f16)
    wl.q = (wl.q.astype(np.float32) + 1.0).astype(f16)
    o, lse, o_ref, lse_ref = _run(wl, n_splits)
    # the scores span a wide range, as intended
    assert float(np.max(lse_ref)) > 20.0
    check_close(o, o_ref, lse, lse_ref)
