"""CPU oracle for the FP8 KV-cache write and paged attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package.  The product path (the CUDA library and its Python
binding) never calls it.  The arithmetic lives in ``oracle.c`` (plain C, float64
attention, integer-bit e4m3 encoder); this module compiles it with gcc and
marshals numpy arrays through ctypes.  It shares no code with the CUDA library.

Interface values (the same numbers the C-ABI uses, restated here on purpose):
``kv_dtype`` 0 = e4m3, 1 = bf16; ``scale_mode`` 0 = per tensor, 1 = per KV head,
2 = per token and KV head.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

KV_E4M3, KV_BF16 = 0, 1
SCALE_PER_TENSOR, SCALE_PER_HEAD, SCALE_PER_TOKEN_HEAD = 0, 1, 2

CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared",
          "-pthread"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc; no GPU needed)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            L.oracle_e4m3_encode.argtypes = [ctypes.c_float]
            L.oracle_e4m3_encode.restype = ctypes.c_uint8
            L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_decode.restype = f64
            L.oracle_e4m3_encode_array.argtypes = [P, P, i64]
            L.oracle_e4m3_encode_array.restype = None
            L.oracle_e4m3_decode_array.argtypes = [P, P, i64]
            L.oracle_e4m3_decode_array.restype = None
            L.oracle_kv_cache_write.argtypes = [P, P, P, i64, i32, i32, i32, i32, P, P, P, P, P,
                                                P, i64]
            L.oracle_kv_cache_write.restype = i32
            L.oracle_decode_attn.argtypes = [P, P, P, i32, i32, P, P, P, P, P, i32, P, i32, i32,
                                             i32, i32, i64, f64, i32, P, i64, P, i32]
            L.oracle_decode_attn.restype = i32
            L.oracle_prefill_attn.argtypes = [P, P, P, P, i32, i32, P, P, P, P, P, i32, P, i32,
                                              i32, i32, i32, i64, f64, P, i64, P, i32]
            L.oracle_prefill_attn.restype = i32
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def e4m3_encode(x) -> np.ndarray:
    """fp32 values -> e4m3fn codes (RNE, saturate to +-448, NaN kept)."""
    x = _c(np.asarray(x, dtype=np.float32), np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(x), _ptr(out), x.size)
    return out


def e4m3_decode(c) -> np.ndarray:
    """e4m3fn codes -> exact float64 values."""
    c = _c(np.asarray(c, dtype=np.uint8), np.uint8)
    out = np.empty(c.shape, dtype=np.float64)
    lib().oracle_e4m3_decode_array(_ptr(c), _ptr(out), c.size)
    return out


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, *, kv_dtype, scale_mode=0,
                   k_scale=None, v_scale=None, k_scale_cache=None, v_scale_cache=None) -> int:
    """Write bf16 K/V rows (uint16 bit patterns [T][Hkv][D]) into the caches in place.

    k_cache/v_cache: uint8 (e4m3) or uint16 (bf16) arrays [num_blocks][Hkv][16][D];
    scale caches: float32 [num_blocks][Hkv][16] (per-token-head only).  Returns the
    oracle status (0, or -6 when a slot points past the cache).
    """
    k = _c(k, np.uint16)
    v = _c(v, np.uint16)
    T, Hkv, D = k.shape
    slots = _c(slot_mapping, np.int64)
    for a in (k_cache, v_cache, k_scale_cache, v_scale_cache):
        if a is not None and not a.flags.c_contiguous:
            raise ValueError("cache arrays must be C-contiguous (written in place)")
    ks = _c(k_scale, np.float32)
    vs = _c(v_scale, np.float32)
    return lib().oracle_kv_cache_write(_ptr(k), _ptr(v), _ptr(slots), T, Hkv, D, kv_dtype,
                                       scale_mode, _ptr(ks), _ptr(vs), _ptr(k_cache),
                                       _ptr(v_cache), _ptr(k_scale_cache), _ptr(v_scale_cache),
                                       k_cache.shape[0])


def _units(units, n_a, Hq):
    if units is None:
        a, h = np.meshgrid(np.arange(n_a), np.arange(Hq), indexing="ij")
        units = np.stack([a.ravel(), h.ravel()], axis=1)
    return _c(np.asarray(units).reshape(-1, 2), np.int32)


def decode_attn(q, k_cache, v_cache, block_table, context_lens, *, kv_dtype, scale_mode=0,
                k_scale=None, v_scale=None, k_scale_cache=None, v_scale_cache=None,
                softmax_scale=None, window=0, units=None, nthreads=1):
    """float64 decode attention.  q: uint16 bf16 bits [B][Hq][D].

    units: optional (seq, hq) pairs; default all B*Hq in order.  Returns
    (status, out[n_units][D] float64).
    """
    q = _c(q, np.uint16)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    u = _units(units, B, Hq)
    out = np.zeros((u.shape[0], D), dtype=np.float64)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    st = lib().oracle_decode_attn(
        _ptr(q), _ptr(np.ascontiguousarray(k_cache)), _ptr(np.ascontiguousarray(v_cache)),
        kv_dtype, scale_mode, _ptr(_c(k_scale, np.float32)), _ptr(_c(v_scale, np.float32)),
        _ptr(_c(k_scale_cache, np.float32)), _ptr(_c(v_scale_cache, np.float32)), _ptr(bt),
        bt.shape[1], _ptr(cl), B, Hq, Hkv, D, k_cache.shape[0], float(softmax_scale),
        int(window), _ptr(u), u.shape[0], _ptr(out), int(nthreads))
    return st, out


def prefill_attn(q, cu_seqlens_q, k_cache, v_cache, block_table, context_lens, *, kv_dtype,
                 scale_mode=0, k_scale=None, v_scale=None, k_scale_cache=None,
                 v_scale_cache=None, softmax_scale=None, units=None, nthreads=1):
    """float64 causal chunked-prefill attention.  q: uint16 bf16 bits [Tq][Hq][D].

    units: optional (token, hq) pairs; default all Tq*Hq in order.  Returns
    (status, out[n_units][D] float64).
    """
    q = _c(q, np.uint16)
    Tq, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    cu = _c(cu_seqlens_q, np.int32)
    bt = _c(block_table, np.int32)
    cl = _c(context_lens, np.int32)
    u = _units(units, Tq, Hq)
    out = np.zeros((u.shape[0], D), dtype=np.float64)
    if softmax_scale is None:
        softmax_scale = 1.0 / np.sqrt(D)
    st = lib().oracle_prefill_attn(
        _ptr(q), _ptr(cu), _ptr(np.ascontiguousarray(k_cache)),
        _ptr(np.ascontiguousarray(v_cache)), kv_dtype, scale_mode,
        _ptr(_c(k_scale, np.float32)), _ptr(_c(v_scale, np.float32)),
        _ptr(_c(k_scale_cache, np.float32)), _ptr(_c(v_scale_cache, np.float32)), _ptr(bt),
        bt.shape[1], _ptr(cl), cu.shape[0] - 1, Hq, Hkv, D, k_cache.shape[0],
        float(softmax_scale), _ptr(u), u.shape[0], _ptr(out), int(nthreads))
    return st, out
