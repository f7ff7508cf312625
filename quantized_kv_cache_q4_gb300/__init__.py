"""Python binding of libkvq.so: quantized KV cache append and decode attention
for GB300 (sm_103a).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  The functions carry the
names of the C entry points in ``include/kvq.h``; they raise ``KvqError`` for
any status other than KVQ_OK.  If the compiled library is missing the import
of this package fails -- there is no other implementation to fall back on.
"""
from __future__ import annotations

import ctypes
import os

import torch

KVQ_OK, KVQ_EINVAL, KVQ_EUNSUPPORTED, KVQ_EWORKSPACE, KVQ_ECUDA = range(5)
KVQ_CODEC_Q4_G64 = 1
KVQ_CODEC_Q8_0 = 2
KVQ_CODEC_Q4_G32 = 3
KVQ_CODEC_NVFP4 = 4
KVQ_F32, KVQ_F16 = 0, 1
KVQ_ERR_APPEND_POS, KVQ_ERR_KV_LEN, KVQ_ERR_TIMEOUT = 1, 2, 4
KVQ_CAPACITY_ALIGN = 64

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")


class KvqError(RuntimeError):
    def __init__(self, status: int, detail: str):
        super().__init__(f"kvq status {status}: {detail}")
        self.status = status


class kvq_cache(ctypes.Structure):
    _fields_ = [("codec", ctypes.c_int32), ("n_seq", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("qs", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with quantized_kv_cache_q4_gb300.build.build() "
                          "(nvcc, sm_103a); there is no fallback implementation")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    C = ctypes.POINTER(kvq_cache)
    sig = {
        "kvq_row_bytes": (I32, [I32, I32]),
        "kvq_scales_per_row": (I32, [I32, I32]),
        "kvq_scale_bytes": (I32, [I32]),
        "kvq_selftest_bounded_wait": (I32, [P, P]),
        "kvq_quantize_append": (I32, [C, C, P, P, I32, I32, P, P, P]),
        "kvq_decode_default_splits": (I32, [C, C, I32, I32, I32]),
        "kvq_decode_workspace_bytes": (SZ, [C, C, I32, I32, I32, I32]),
        "kvq_decode_attention": (I32, [C, C, P, I32, I32, I32, F, P, I32, I32, P, P, P, SZ, P, P]),
        "kvq_merge_splits": (I32, [P, P, I32, I32, I32, P, P, P]),
        "kvq_dequantize": (I32, [C, P, P]),
        "kvq_static_scratch_bytes": (SZ, []),
        "kvq_decode_attention_static": (I32, [C, C, P, I32, I32, I32, F, P, I32, I32, P, P, P, P]),
        "kvq_tiered_ring_bytes": (SZ, [C, C, I32, I32]),
        "kvq_tiered_workspace_bytes": (SZ, [C, C, C, C, I32, I32, I32, I32, I32]),
        "kvq_decode_attention_tiered": (I32, [C, C, C, C, I32, P, I32, I32, I32, F, I32, I32, I32, P, SZ, P, P, P,
                                              SZ, P, P]),
        "kvq_status_string": (ctypes.c_char_p, [I32]),
        "kvq_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()
EXPORTED = ("kvq_row_bytes", "kvq_scales_per_row", "kvq_scale_bytes", "kvq_quantize_append", "kvq_decode_default_splits",
            "kvq_decode_workspace_bytes", "kvq_decode_attention", "kvq_merge_splits", "kvq_dequantize",
            "kvq_status_string", "kvq_last_error", "kvq_static_scratch_bytes", "kvq_decode_attention_static",
            "kvq_selftest_bounded_wait", "kvq_tiered_ring_bytes", "kvq_tiered_workspace_bytes",
            "kvq_decode_attention_tiered")


def _check(status: int):
    if status != KVQ_OK:
        raise KvqError(status, _lib.kvq_last_error().decode() or _lib.kvq_status_string(status).decode())


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def kvq_row_bytes(codec: int, head_dim: int) -> int:
    return int(_lib.kvq_row_bytes(codec, head_dim))


def kvq_scales_per_row(codec: int, head_dim: int) -> int:
    return int(_lib.kvq_scales_per_row(codec, head_dim))


def kvq_scale_bytes(codec: int) -> int:
    return int(_lib.kvq_scale_bytes(codec))


def kvq_selftest_bounded_wait(d_err, stream=None):
    """Run the library's bounded device wait on a barrier nothing completes: after
    about 1 s KVQ_ERR_TIMEOUT is OR-ed into d_err (see include/kvq.h)."""
    _check(_lib.kvq_selftest_bounded_wait(_ptr(d_err), _stream(stream)))


class KVCache:
    """One layer's K or V cache in device memory: a qs uint8 plane and a scales
    plane (fp16; uint8 E4M3 for NVFP4), [n_seq][n_kv_heads][capacity][...]
    (layout as in include/kvq.h)."""

    def __init__(self, codec, n_seq, n_kv_heads, head_dim, capacity, device="cuda", qs=None, scales=None):
        self.codec, self.n_seq, self.n_kv_heads = int(codec), int(n_seq), int(n_kv_heads)
        self.head_dim, self.capacity = int(head_dim), int(capacity)
        rb, ns = kvq_row_bytes(codec, head_dim), kvq_scales_per_row(codec, head_dim)
        shape = (self.n_seq, self.n_kv_heads, self.capacity)
        self.qs = qs if qs is not None else torch.zeros(shape + (rb,), dtype=torch.uint8, device=device)
        sdt = torch.uint8 if kvq_scale_bytes(codec) == 1 else torch.float16
        self.scales = scales if scales is not None else torch.zeros(shape + (ns,), dtype=sdt, device=device)
        self._c = kvq_cache(self.codec, self.n_seq, self.n_kv_heads, self.head_dim, self.capacity,
                            self.qs.data_ptr(), self.scales.data_ptr())

    @property
    def c(self):
        return ctypes.byref(self._c)

    def nbytes(self) -> int:
        return self.qs.numel() + self.scales.numel() * self.scales.element_size()

    def seq_view(self, s: int) -> "KVCache":
        """The planes of sequence s alone, as a one-sequence cache (shares memory)."""
        return KVCache(self.codec, 1, self.n_kv_heads, self.head_dim, self.capacity,
                       qs=self.qs[s:s + 1], scales=self.scales[s:s + 1])

    def to_host(self) -> "KVCache":
        """A copy whose planes are in pinned host memory (the host tier of a
        streamed cache; the structure's pointers are host addresses)."""
        return KVCache(self.codec, self.n_seq, self.n_kv_heads, self.head_dim, self.capacity,
                       qs=self.qs.cpu().pin_memory(), scales=self.scales.cpu().pin_memory())

    def clone(self) -> "KVCache":
        return KVCache(self.codec, self.n_seq, self.n_kv_heads, self.head_dim, self.capacity,
                       qs=self.qs.clone(), scales=self.scales.clone())


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return KVQ_F16
    if t.dtype == torch.float32:
        return KVQ_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def kvq_quantize_append(k: KVCache | None, v: KVCache | None, k_src, v_src, n_new: int, d_pos0,
                        d_err=None, stream=None, src_dtype: int | None = None):
    """Quantize k_src / v_src ([n_seq][n_new][n_kv_heads][head_dim]) into the caches
    at positions d_pos0[s] + i.  Tensors or raw device pointers are accepted."""
    if src_dtype is None:
        src_dtype = _dtype_code(k_src if k_src is not None else v_src)
    _check(_lib.kvq_quantize_append(k.c if k is not None else None, v.c if v is not None else None,
                                    _ptr(k_src), _ptr(v_src), src_dtype, int(n_new), _ptr(d_pos0),
                                    _ptr(d_err), _stream(stream)))


def _cref(c):
    """A KVCache or a bare kvq_cache structure, as the C pointer argument."""
    return c.c if isinstance(c, KVCache) else ctypes.byref(c)


def _cref_opt(c):
    return None if c is None else _cref(c)


def kvq_decode_default_splits(k, v, n_heads: int, n_q: int, max_kv_len: int) -> int:
    return int(_lib.kvq_decode_default_splits(_cref(k), _cref(v), int(n_heads), int(n_q), int(max_kv_len)))


def kvq_decode_workspace_bytes(k, v, n_heads: int, n_q: int, max_kv_len: int, n_splits: int = 0) -> int:
    return int(_lib.kvq_decode_workspace_bytes(_cref(k), _cref(v), int(n_heads), int(n_q), int(max_kv_len),
                                               int(n_splits)))


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor | None:
    """A 256-byte aligned device buffer of at least nbytes (torch allocations are)."""
    if nbytes == 0:
        return None
    return torch.empty(nbytes, dtype=torch.uint8, device=device)


def kvq_decode_attention(k: KVCache, v: KVCache, q, n_q: int, n_heads: int, softmax_scale: float, d_kv_len,
                         max_kv_len: int, n_splits: int, out, out_lse=None, workspace=None, workspace_bytes=None,
                         d_err=None, stream=None, q_dtype: int | None = None):
    if q_dtype is None:
        q_dtype = _dtype_code(q)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    _check(_lib.kvq_decode_attention(k.c, v.c, _ptr(q), q_dtype, int(n_q), int(n_heads), float(softmax_scale),
                                     _ptr(d_kv_len), int(max_kv_len), int(n_splits), _ptr(out), _ptr(out_lse),
                                     _ptr(workspace), int(workspace_bytes), _ptr(d_err), _stream(stream)))


def kvq_static_scratch_bytes() -> int:
    return int(_lib.kvq_static_scratch_bytes())


def kvq_decode_attention_static(k: KVCache, v: KVCache, q, n_q: int, n_heads: int, softmax_scale: float, d_kv_len,
                                max_kv_len: int, n_splits: int, out, out_lse=None, d_err=None, stream=None,
                                q_dtype: int | None = None):
    """kvq_decode_attention without a workspace: the library's own static
    device scratch is used and nothing is allocated (see include/kvq.h)."""
    if q_dtype is None:
        q_dtype = _dtype_code(q)
    _check(_lib.kvq_decode_attention_static(k.c, v.c, _ptr(q), q_dtype, int(n_q), int(n_heads),
                                            float(softmax_scale), _ptr(d_kv_len), int(max_kv_len), int(n_splits),
                                            _ptr(out), _ptr(out_lse), _ptr(d_err), _stream(stream)))


def kvq_tiered_ring_bytes(k_host, v_host, page_tokens: int, n_slots: int) -> int:
    return int(_lib.kvq_tiered_ring_bytes(_cref(k_host), _cref(v_host), int(page_tokens), int(n_slots)))


def kvq_tiered_workspace_bytes(k_host, v_host, k_dev, v_dev, n_heads: int, n_q: int, kv_len: int, n_resident: int,
                               page_tokens: int) -> int:
    return int(_lib.kvq_tiered_workspace_bytes(_cref(k_host), _cref(v_host), _cref_opt(k_dev), _cref_opt(v_dev),
                                               int(n_heads), int(n_q), int(kv_len), int(n_resident),
                                               int(page_tokens)))


def kvq_decode_attention_tiered(k_host: KVCache, v_host: KVCache, k_dev: KVCache | None, v_dev: KVCache | None,
                                n_resident: int, q, n_q: int, n_heads: int, softmax_scale: float, kv_len: int,
                                page_tokens: int, n_slots: int, ring, out, out_lse=None, workspace=None,
                                ring_bytes=None, workspace_bytes=None, d_err=None, stream=None,
                                q_dtype: int | None = None):
    """Decode attention for one sequence whose cache planes are in pinned host
    memory (k_host, v_host); the first n_resident tokens are read from the
    device caches k_dev, v_dev, the rest streamed in pages of page_tokens
    through the device ring (see include/kvq.h)."""
    if q_dtype is None:
        q_dtype = _dtype_code(q)
    if ring_bytes is None:
        ring_bytes = ring.numel() * ring.element_size() if isinstance(ring, torch.Tensor) else 0
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if isinstance(workspace, torch.Tensor) else 0
    _check(_lib.kvq_decode_attention_tiered(k_host.c, v_host.c, _cref_opt(k_dev), _cref_opt(v_dev), int(n_resident),
                                            _ptr(q), q_dtype, int(n_q), int(n_heads), float(softmax_scale),
                                            int(kv_len), int(page_tokens), int(n_slots), _ptr(ring), int(ring_bytes),
                                            _ptr(out), _ptr(out_lse), _ptr(workspace), int(workspace_bytes),
                                            _ptr(d_err), _stream(stream)))


def kvq_merge_splits(part_o, part_lse, n_splits: int, rows: int, head_dim: int, out, out_lse=None, stream=None):
    _check(_lib.kvq_merge_splits(_ptr(part_o), _ptr(part_lse), int(n_splits), int(rows), int(head_dim),
                                 _ptr(out), _ptr(out_lse), _stream(stream)))


def kvq_dequantize(c: KVCache, out, stream=None):
    _check(_lib.kvq_dequantize(c.c, _ptr(out), _stream(stream)))


def kvq_status_string(status: int) -> str:
    return _lib.kvq_status_string(status).decode()


def kvq_last_error() -> str:
    return _lib.kvq_last_error().decode()


def decode(k: KVCache, v: KVCache, q: torch.Tensor, d_kv_len: torch.Tensor, max_kv_len: int, softmax_scale=None,
           n_splits: int = 0, d_err=None, stream=None):
    """Convenience wrapper: allocates out/out_lse/workspace with torch and calls
    kvq_decode_attention.  Returns (out, out_lse)."""
    n_seq, n_q, n_heads, D = q.shape
    if softmax_scale is None:
        softmax_scale = D ** -0.5
    out = torch.empty((n_seq, n_q, n_heads, D), dtype=torch.float32, device=q.device)
    lse = torch.empty((n_seq, n_q, n_heads), dtype=torch.float32, device=q.device)
    ws = alloc_workspace(kvq_decode_workspace_bytes(k, v, n_heads, n_q, max_kv_len, n_splits), q.device)
    kvq_decode_attention(k, v, q, n_q, n_heads, softmax_scale, d_kv_len, max_kv_len, n_splits, out, lse, ws,
                         d_err=d_err, stream=stream)
    return out, lse
