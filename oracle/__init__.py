"""CPU oracle for the quantized KV cache decode path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The CUDA
library never calls it, and it shares no code with the CUDA library: the C
source next to this file states the codec and the attention from their
definitions (den_llama.cpp, "What this fork is" and the "build3 (working
engine) -- additions" table for Q4_G64 and the NVFP4 KV type; the mixed
"-ctk q8_0 -ctv q4_g64" pair of the "Build3 (working engine)" command block).

Every function takes and returns numpy arrays.  Parity status: every function
here is pinned by ``tests/test_oracle_*.py`` (closed forms, a hand-worked
golden block, numpy's float16 and torch's float8_e4m3fn conversions, torch's
float64 attention, exact rational brute force, invariants).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_G64 = 1
Q8_0 = 2
Q4_G32 = 3                  # the pages' "q4_0", read as Q4_G64 with 32-value groups
NVFP4 = 4                   # E2M1 values, one E4M3 scale per 16 (NVIDIA's NVFP4, no tensor scale)
GROUP = {Q4_G64: 64, Q8_0: 32, Q4_G32: 32, NVFP4: 16}
FOUR_BIT = (Q4_G64, Q4_G32)                 # integer 4-bit codes
NIBBLE = (Q4_G64, Q4_G32, NVFP4)            # two codes per byte
SCALE_DTYPE = {Q4_G64: np.uint16, Q8_0: np.uint16, Q4_G32: np.uint16, NVFP4: np.uint8}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kvq_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (C11, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _declare(lib):
    P, I, I64, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.orc_f32_to_f16.argtypes = [ctypes.c_float]
    lib.orc_f32_to_f16.restype = ctypes.c_uint16
    lib.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
    lib.orc_f16_to_f32.restype = ctypes.c_float
    lib.orc_f32_to_f16_array.argtypes = [P, I64, P]
    lib.orc_f16_to_f32_array.argtypes = [P, I64, P]
    lib.orc_f32_to_e4m3_array.argtypes = [P, I64, P]
    lib.orc_f32_to_e2m1_array.argtypes = [P, I64, P]
    lib.orc_e4m3_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_to_f32.restype = ctypes.c_float
    lib.orc_e2m1_to_f32.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_to_f32.restype = ctypes.c_float
    lib.orc_quantize.argtypes = [I, P, I64, I, P, P]
    lib.orc_dequantize.argtypes = [I, P, P, I64, I, P]
    lib.orc_quantize_append.argtypes = [I, P, I, I, I, I, I, P, P, P]
    lib.orc_quantize_append.restype = I
    lib.orc_decode_attention.argtypes = [I, P, P, I, P, P, I, I, I, I, P, I, I, P, D, P, P, I]
    lib.orc_decode_attention_split.argtypes = [I, P, P, I, P, P, I, I, I, I, P, I, I, P, D, I, P, P]
    lib.orc_merge_splits.argtypes = [P, P, I, I64, I, P, P]
    lib.orc_omp_max_threads.restype = I
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
        return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Test hook: route every function of this module through another build of
    the oracle source (the planted-mistake tests compile mutants with it)."""
    global _lib
    old = _load()
    _lib = _declare(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = old


def compile_source(src_text: str, out_path: str) -> str:
    """Compile C source text with the oracle's flags into a shared library."""
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
                    "-fno-fast-math", "-o", out_path, c_path, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def row_bytes(codec: int, head_dim: int) -> int:
    return head_dim // 2 if codec in NIBBLE else head_dim


def scales_per_row(codec: int, head_dim: int) -> int:
    return head_dim // GROUP[codec]


def f32_to_f16_bits(x) -> np.ndarray:
    """fp32 -> fp16 bit patterns, round to nearest even (element by element)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib.orc_f32_to_f16_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_bits_to_f32(h) -> np.ndarray:
    lib = _load()
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    lib.orc_f16_to_f32_array(_ptr(h), h.size, _ptr(out))
    return out


def f32_to_e4m3(x) -> np.ndarray:
    """fp32 -> E4M3 bytes, round to nearest even, saturating at 448."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.orc_f32_to_e4m3_array(_ptr(x), x.size, _ptr(out))
    return out


def f32_to_e2m1(x) -> np.ndarray:
    """fp32 -> E2M1 codes (low nibble), round to nearest even, saturating at 6."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.orc_f32_to_e2m1_array(_ptr(x), x.size, _ptr(out))
    return out


def e4m3_to_f32(b) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_e4m3_to_f32(int(v)) for v in np.ravel(b)], np.float32).reshape(np.shape(b))


def e2m1_to_f32(n) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_e2m1_to_f32(int(v)) for v in np.ravel(n)], np.float32).reshape(np.shape(n))


def _as_f32_rows(x: np.ndarray) -> np.ndarray:
    """Widen fp16/fp32 inputs to fp32 (exact)."""
    if x.dtype == np.float16:
        x = x.astype(np.float32)
    return np.ascontiguousarray(x, dtype=np.float32)


def quantize(codec: int, x: np.ndarray):
    """Quantize rows x[..., head_dim] -> (qs uint8 [..., row_bytes], scales: fp16 bit
    patterns as uint16, or E4M3 bytes as uint8 for NVFP4)."""
    lib = _load()
    x = _as_f32_rows(x)
    D = x.shape[-1]
    n = int(np.prod(x.shape[:-1])) if x.ndim > 1 else 1
    qs = np.zeros(x.shape[:-1] + (row_bytes(codec, D),), dtype=np.uint8)
    sc = np.zeros(x.shape[:-1] + (scales_per_row(codec, D),), dtype=SCALE_DTYPE[codec])
    lib.orc_quantize(codec, _ptr(x), n, D, _ptr(qs), _ptr(sc))
    return qs, sc


def dequantize(codec: int, qs: np.ndarray, sc: np.ndarray, head_dim: int) -> np.ndarray:
    lib = _load()
    qs = np.ascontiguousarray(qs, dtype=np.uint8)
    sc = np.ascontiguousarray(sc, dtype=SCALE_DTYPE[codec])
    n = qs.size // row_bytes(codec, head_dim)
    out = np.empty(qs.shape[:-1] + (head_dim,), dtype=np.float32)
    lib.orc_dequantize(codec, _ptr(qs), _ptr(sc), n, head_dim, _ptr(out))
    return out


class Cache:
    """One layer's K or V cache as numpy planes [n_seq][n_kv_heads][capacity][...]."""

    def __init__(self, codec: int, n_seq: int, n_kv_heads: int, head_dim: int, capacity: int):
        self.codec, self.n_seq, self.n_kv_heads = codec, n_seq, n_kv_heads
        self.head_dim, self.capacity = head_dim, capacity
        self.qs = np.zeros((n_seq, n_kv_heads, capacity, row_bytes(codec, head_dim)), np.uint8)
        self.scales = np.zeros((n_seq, n_kv_heads, capacity, scales_per_row(codec, head_dim)), SCALE_DTYPE[codec])


def quantize_append(cache: Cache, src: np.ndarray, pos0: np.ndarray) -> int:
    """Quantize src [n_seq][n_new][n_kv_heads][head_dim] into cache at pos0[s] + i.
    Returns the error bits (bit 0: a sequence's positions were out of range)."""
    lib = _load()
    src = _as_f32_rows(src)
    pos0 = np.ascontiguousarray(pos0, dtype=np.int32)
    n_seq, n_new, hk, D = src.shape
    assert (n_seq, hk, D) == (cache.n_seq, cache.n_kv_heads, cache.head_dim)
    return lib.orc_quantize_append(cache.codec, _ptr(src), n_seq, n_new, hk, D, cache.capacity,
                                   _ptr(pos0), _ptr(cache.qs), _ptr(cache.scales))


def decode_attention(k: Cache, v: Cache, q: np.ndarray, kv_len: np.ndarray, scale: float,
                     n_threads: int = 1):
    """fp64 attention of q [n_seq][n_q][n_heads][head_dim] over the dequantized
    caches.  Returns (o float64 [n_seq][n_q][n_heads][head_dim], lse float64)."""
    lib = _load()
    q = _as_f32_rows(q)
    kv_len = np.ascontiguousarray(kv_len, dtype=np.int32)
    S, n_q, H, D = q.shape
    out = np.zeros((S, n_q, H, D), np.float64)
    lse = np.zeros((S, n_q, H), np.float64)
    lib.orc_decode_attention(k.codec, _ptr(k.qs), _ptr(k.scales), v.codec, _ptr(v.qs), _ptr(v.scales),
                             S, k.n_kv_heads, D, k.capacity, _ptr(q), n_q, H, _ptr(kv_len),
                             float(scale), _ptr(out), _ptr(lse), int(n_threads))
    return out, lse


def decode_attention_split(k: Cache, v: Cache, q: np.ndarray, kv_len: np.ndarray, scale: float,
                           n_splits: int):
    lib = _load()
    q = _as_f32_rows(q)
    kv_len = np.ascontiguousarray(kv_len, dtype=np.int32)
    S, n_q, H, D = q.shape
    po = np.zeros((n_splits, S, n_q, H, D), np.float64)
    pl = np.zeros((n_splits, S, n_q, H), np.float64)
    lib.orc_decode_attention_split(k.codec, _ptr(k.qs), _ptr(k.scales), v.codec, _ptr(v.qs),
                                   _ptr(v.scales), S, k.n_kv_heads, D, k.capacity, _ptr(q), n_q, H,
                                   _ptr(kv_len), float(scale), n_splits, _ptr(po), _ptr(pl))
    return po, pl


def merge_splits(part_o: np.ndarray, part_lse: np.ndarray):
    """LSE merge of part_o [n_splits][rows...][head_dim], part_lse [n_splits][rows...]."""
    lib = _load()
    po = np.ascontiguousarray(part_o, dtype=np.float64)
    pl = np.ascontiguousarray(part_lse, dtype=np.float64)
    n_splits, D = po.shape[0], po.shape[-1]
    rows = int(np.prod(po.shape[1:-1]))
    out = np.zeros(po.shape[1:], np.float64)
    lse = np.zeros(pl.shape[1:], np.float64)
    lib.orc_merge_splits(_ptr(po), _ptr(pl), n_splits, rows, D, _ptr(out), _ptr(lse))
    return out, lse


def max_threads() -> int:
    return int(_load().orc_omp_max_threads())
