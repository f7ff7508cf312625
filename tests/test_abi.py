"""The C-ABI library loads, exports every entry point include/kvq.h declares,
and rejects bad arguments on the host before launching anything (these calls
never reach a kernel, so they run without a GPU)."""
import ctypes
import os
import re

import pytest

import quantized_kv_cache_q4_gb300 as kvq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "kvq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq_[a-z_0-9]+)\s*\(", src)))


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "kvq_decode_attention" in names and "kvq_quantize_append" in names and "kvq_merge_splits" in names
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(kvq.EXPORTED)


def test_row_sizes():
    assert kvq.kvq_row_bytes(kvq.KVQ_CODEC_Q4_G64, 256) == 128
    assert kvq.kvq_scales_per_row(kvq.KVQ_CODEC_Q4_G64, 256) == 4
    assert kvq.kvq_row_bytes(kvq.KVQ_CODEC_Q8_0, 256) == 256
    assert kvq.kvq_scales_per_row(kvq.KVQ_CODEC_Q8_0, 256) == 8
    assert kvq.kvq_row_bytes(kvq.KVQ_CODEC_Q4_G32, 256) == 128
    assert kvq.kvq_scales_per_row(kvq.KVQ_CODEC_Q4_G32, 256) == 8
    assert kvq.kvq_row_bytes(kvq.KVQ_CODEC_NVFP4, 256) == 128
    assert kvq.kvq_scales_per_row(kvq.KVQ_CODEC_NVFP4, 256) == 16
    assert kvq.kvq_row_bytes(99, 256) == 0
    assert [kvq.kvq_scale_bytes(c) for c in (1, 2, 3, 4, 99)] == [2, 2, 2, 1, 0]
    # 4.25, 8.5, 4.5 and 4.5 bits per value
    for codec, bits in ((kvq.KVQ_CODEC_Q4_G64, 4.25), (kvq.KVQ_CODEC_Q8_0, 8.5), (kvq.KVQ_CODEC_Q4_G32, 4.5),
                        (kvq.KVQ_CODEC_NVFP4, 4.5)):
        for d in (64, 128, 256, 512):
            sb = kvq.kvq_scale_bytes(codec)
            assert (kvq.kvq_row_bytes(codec, d) + sb * kvq.kvq_scales_per_row(codec, d)) * 8 == bits * d


def _fake_cache(**kw):
    c = dict(codec=kvq.KVQ_CODEC_Q4_G64, n_seq=1, n_kv_heads=4, head_dim=256, capacity=1024, qs=4096, scales=8192)
    c.update(kw)
    return kvq.kvq_cache(c["codec"], c["n_seq"], c["n_kv_heads"], c["head_dim"], c["capacity"], c["qs"], c["scales"])


def _append(k, v, ksrc=4096, vsrc=4096, dtype=kvq.KVQ_F16, n_new=1, pos=4096):
    lib = kvq._lib
    return lib.kvq_quantize_append(ctypes.byref(k) if k else None, ctypes.byref(v) if v else None,
                                   ksrc if k else None, vsrc if v else None, dtype, n_new, pos, None, None)


@pytest.mark.parametrize("bad,status", [
    (dict(codec=5), kvq.KVQ_EINVAL), (dict(codec=0), kvq.KVQ_EINVAL), (dict(head_dim=96), kvq.KVQ_EINVAL), (dict(head_dim=1024), kvq.KVQ_EINVAL),
    (dict(capacity=100), kvq.KVQ_EINVAL), (dict(capacity=0), kvq.KVQ_EINVAL), (dict(n_seq=0), kvq.KVQ_EINVAL),
    (dict(qs=0), kvq.KVQ_EINVAL), (dict(qs=4097), kvq.KVQ_EINVAL), (dict(scales=8200), kvq.KVQ_EINVAL),
    (dict(head_dim=192), kvq.KVQ_EUNSUPPORTED)])
def test_append_rejects_bad_cache(bad, status):
    assert _append(_fake_cache(**bad), None) == status
    assert kvq.kvq_last_error()


def test_append_rejects_bad_arguments():
    k, v = _fake_cache(), _fake_cache()
    assert _append(None, None) == kvq.KVQ_EINVAL
    assert _append(k, v, dtype=7) == kvq.KVQ_EINVAL
    assert _append(k, v, n_new=-1) == kvq.KVQ_EINVAL
    assert _append(k, v, pos=None) == kvq.KVQ_EINVAL
    assert _append(k, v, ksrc=4100) == kvq.KVQ_EINVAL
    assert _append(k, _fake_cache(n_kv_heads=2)) == kvq.KVQ_EINVAL
    assert _append(k, v, n_new=0) == kvq.KVQ_OK          # nothing to do, nothing launched


def _decode(k, v, q=4096, q_dtype=kvq.KVQ_F16, n_q=1, n_heads=24, scale=0.0625, kv_len=4096, max_kv_len=512,
            n_splits=1, out=4096, ws=None, ws_bytes=0):
    return kvq._lib.kvq_decode_attention(ctypes.byref(k), ctypes.byref(v), q, q_dtype, n_q, n_heads, scale, kv_len,
                                         max_kv_len, n_splits, out, None, ws, ws_bytes, None, None)


def test_decode_rejects_bad_arguments():
    k, v = _fake_cache(), _fake_cache()
    assert _decode(k, _fake_cache(capacity=2048)) == kvq.KVQ_EINVAL
    assert _decode(k, v, q=None) == kvq.KVQ_EINVAL
    assert _decode(k, v, q_dtype=5) == kvq.KVQ_EINVAL
    assert _decode(k, v, n_q=0) == kvq.KVQ_EINVAL
    assert _decode(k, v, n_heads=22) == kvq.KVQ_EINVAL                 # not a multiple of 4 kv heads
    assert _decode(k, v, scale=float("inf")) == kvq.KVQ_EINVAL
    assert _decode(k, v, kv_len=None) == kvq.KVQ_EINVAL
    assert _decode(k, v, max_kv_len=0) == kvq.KVQ_EINVAL
    assert _decode(k, v, max_kv_len=1025) == kvq.KVQ_EINVAL            # beyond capacity
    assert _decode(k, v, n_splits=-1) == kvq.KVQ_EINVAL
    assert _decode(k, v, n_splits=5000) == kvq.KVQ_EINVAL
    assert _decode(k, v, out=None) == kvq.KVQ_EINVAL
    assert _decode(k, v, n_splits=8) == kvq.KVQ_EWORKSPACE             # splits need a workspace
    need = kvq.kvq_decode_workspace_bytes(k, v, 24, 1, 512, 8)
    assert _decode(k, v, n_splits=8, ws=1 << 20, ws_bytes=need - 1) == kvq.KVQ_EWORKSPACE
    assert _decode(k, v, n_splits=8, ws=(1 << 20) + 16, ws_bytes=need) == kvq.KVQ_EINVAL   # misaligned


def test_workspace_sizes():
    k, v = _fake_cache(capacity=32768), _fake_cache(capacity=32768)
    assert kvq.kvq_decode_workspace_bytes(k, v, 24, 1, 32768, 1) == 0
    rows = 1 * 1 * 24
    n = kvq.kvq_decode_workspace_bytes(k, v, 24, 1, 32768, 64)
    assert n >= 64 * rows * 257 * 4 and n % 256 == 0
    kb, vb = _fake_cache(n_seq=16, capacity=65600), _fake_cache(n_seq=16, capacity=65600)
    assert kvq.kvq_decode_workspace_bytes(kb, vb, 24, 3, 65539, 16) >= 16 * 16 * 3 * 24 * 257 * 4
    d = kvq.kvq_decode_default_splits(k, v, 24, 1, 32768)
    assert 1 <= d <= 4096
    assert kvq.kvq_decode_workspace_bytes(k, v, 24, 1, 32768) >= d * rows * 257 * 4
    assert kvq.kvq_decode_default_splits(k, v, 24, 1, 100) == 1        # short context: no split
    # invalid arguments: one split, no workspace
    assert kvq.kvq_decode_default_splits(k, v, 22, 1, 32768) == 1      # 22 heads over 4 kv heads
    assert kvq.kvq_decode_workspace_bytes(k, v, 24, 0, 32768) == 0


@pytest.mark.parametrize("n_seq,L,n_q", [(1, 32768, 1), (1, 65536, 1), (1, 196608, 1), (1, 1000, 3),
                                         (16, 65536, 3), (1, 32768, 512)])
def test_default_splits_leave_no_split_empty(n_seq, L, n_q):
    """Splits are whole 64-token tiles; the default count is one that every
    split of the longest sequence gets a tile of."""
    k, v = _fake_cache(n_seq=n_seq, capacity=-(-L // 64) * 64), _fake_cache(n_seq=n_seq, capacity=-(-L // 64) * 64)
    s = kvq.kvq_decode_default_splits(k, v, 24, n_q, L)
    tiles = -(-L // 64)
    per_split = -(-tiles // s)
    assert 1 <= s <= tiles and -(-tiles // per_split) == s


def test_merge_rejects_bad_arguments():
    lib = kvq._lib
    assert lib.kvq_merge_splits(4096, 4096, 0, 4, 256, 4096, None, None) == kvq.KVQ_EINVAL
    assert lib.kvq_merge_splits(4096, 4096, 5000, 4, 256, 4096, None, None) == kvq.KVQ_EINVAL
    assert lib.kvq_merge_splits(4096, 4096, 2, -1, 256, 4096, None, None) == kvq.KVQ_EINVAL
    assert lib.kvq_merge_splits(4096, 4096, 2, 4, 6, 4096, None, None) == kvq.KVQ_EINVAL
    assert lib.kvq_merge_splits(None, 4096, 2, 4, 256, 4096, None, None) == kvq.KVQ_EINVAL
    assert lib.kvq_merge_splits(4096, 4096, 2, 0, 256, 4096, None, None) == kvq.KVQ_OK


def test_status_strings():
    for s in range(5):
        assert kvq.kvq_status_string(s)
    assert kvq.kvq_status_string(99) == "unknown status"


def _tiered(k, v, kd=None, vd=None, n_res=0, q=4096, n_q=1, n_heads=24, kv_len=1000, page=256, slots=2,
            ring=1 << 20, ring_bytes=1 << 30, out=4096, ws=1 << 20, ws_bytes=1 << 30):
    ref = lambda c: ctypes.byref(c) if c is not None else None   # noqa: E731
    return kvq._lib.kvq_decode_attention_tiered(ref(k), ref(v), ref(kd), ref(vd), n_res, q, kvq.KVQ_F16, n_q,
                                                n_heads, 0.0625, kv_len, page, slots, ring, ring_bytes, out, None,
                                                ws, ws_bytes, None, None)


def test_tiered_rejects_bad_arguments():
    k, v = _fake_cache(), _fake_cache()
    assert _tiered(_fake_cache(n_seq=2), _fake_cache(n_seq=2)) == kvq.KVQ_EUNSUPPORTED   # one sequence only
    assert _tiered(k, _fake_cache(head_dim=128)) == kvq.KVQ_EINVAL
    assert _tiered(k, v, n_heads=22) == kvq.KVQ_EINVAL
    assert _tiered(k, v, n_q=0) == kvq.KVQ_EINVAL
    assert _tiered(k, v, kv_len=0) == kvq.KVQ_EINVAL
    assert _tiered(k, v, kv_len=1025) == kvq.KVQ_EINVAL                 # beyond the host capacity
    assert _tiered(k, v, page=100) == kvq.KVQ_EINVAL                    # not a multiple of 64
    assert _tiered(k, v, slots=0) == kvq.KVQ_EINVAL
    assert _tiered(k, v, n_res=10) == kvq.KVQ_EINVAL                    # resident part without device caches
    assert _tiered(k, v, n_res=1001) == kvq.KVQ_EINVAL                  # more resident keys than keys
    assert _tiered(k, v, kd=_fake_cache(codec=kvq.KVQ_CODEC_Q8_0), vd=_fake_cache(), n_res=10) == kvq.KVQ_EINVAL
    assert _tiered(k, v, kd=_fake_cache(capacity=64), vd=_fake_cache(capacity=64), n_res=100) == kvq.KVQ_EINVAL
    assert _tiered(k, v, q=None) == kvq.KVQ_EINVAL
    assert _tiered(k, v, out=None) == kvq.KVQ_EINVAL
    need = kvq.kvq_tiered_ring_bytes(k, v, 256, 2)
    assert _tiered(k, v, ring_bytes=need - 1) == kvq.KVQ_EWORKSPACE
    assert _tiered(k, v, ring=None) == kvq.KVQ_EWORKSPACE
    assert _tiered(k, v, ring=(1 << 20) + 16) == kvq.KVQ_EINVAL          # misaligned
    assert _tiered(k, v, ws_bytes=64) == kvq.KVQ_EWORKSPACE
    assert _tiered(k, v, ws=(1 << 20) + 16) == kvq.KVQ_EINVAL
    assert kvq.kvq_last_error()


def test_tiered_sizes():
    k, v = _fake_cache(), _fake_cache(codec=kvq.KVQ_CODEC_Q8_0)
    # a slot holds every kv head's page of each plane, each plane 256-byte aligned
    rows = 4 * 256
    slot = rows * 128 + rows * 8 + rows * 256 + rows * 16
    assert kvq.kvq_tiered_ring_bytes(k, v, 256, 3) == 3 * slot
    assert kvq.kvq_tiered_ring_bytes(k, v, 0, 3) == 0
    # per-part partials (resident part + ceil(900 / 256) = 4 pages) and split scratch
    ws = kvq.kvq_tiered_workspace_bytes(k, v, None, None, 24, 3, 1000, 100, 256)
    assert ws >= 5 * 3 * 24 * (256 + 1) * 4
    assert kvq.kvq_tiered_workspace_bytes(k, v, None, None, 22, 3, 1000, 100, 256) == 0
