"""Failure detection on the GPU without a fault: a bounded device wait that
runs out reports KVQ_ERR_TIMEOUT through the caller's error word, and the
context stays usable afterwards."""
import numpy as np
import pytest
import torch

import oracle
import quantized_kv_cache_q4_gb300 as kvq
import workloads
from gpu_helpers import gpu_caches, run_decode
from helpers import check_close, oracle_caches

pytestmark = pytest.mark.gpu


def test_bounded_wait_gives_up_and_reports():
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    kvq.kvq_selftest_bounded_wait(err)
    torch.cuda.synchronize()
    assert int(err.item()) == kvq.KVQ_ERR_TIMEOUT
    # the same context still decodes correctly
    wl = workloads.make(workloads.spec(0))
    k, v = gpu_caches(wl)
    ko, vo = oracle_caches(wl)
    o, lse, e = run_decode(wl, k, v)
    assert e == 0
    o_ref, lse_ref = oracle.decode_attention(ko, vo, wl.q, wl.kv_len, wl.spec.scale)
    check_close(o, o_ref, lse, lse_ref)


def test_selftest_rejects_null_error_word():
    with pytest.raises(kvq.KvqError):
        kvq.kvq_selftest_bounded_wait(None)
