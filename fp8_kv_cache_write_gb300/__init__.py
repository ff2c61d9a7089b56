"""fp8_kv_cache_write_gb300 -- Python binding of libfp8kv (FP8 paged KV cache and
attention over it, hand-written CUDA for GB300 / sm_103a).

This module only marshals arguments: it checks dtypes/devices, allocates outputs
and workspaces with torch when the caller does not pass them, and calls the C
ABI declared in include/fp8kv.h with raw device pointers and the current CUDA
stream.  Every step of the computation runs in the library's kernels; there is
no CPU fallback, and every call raises if libfp8kv.so is missing.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8kv.so")

PAGE_SIZE = 16
KV_E4M3, KV_BF16 = 0, 1
SCALE_PER_TENSOR, SCALE_PER_HEAD, SCALE_PER_TOKEN_HEAD = 0, 1, 2
OUT_F32, OUT_BF16 = 0, 1
# decode flags (include/fp8kv.h): what may run before the preceding kernel ends
DECODE_EARLY_SETUP, DECODE_EARLY_PAGES = 1, 2
# prefill flags: two-level accumulation, operand precision of the e4m3 path
PREFILL_TWO_LEVEL, PREFILL_SPLIT_ALWAYS, PREFILL_SPLIT_NEVER = 1, 2, 4

STATUS = {0: "FP8KV_OK", -1: "FP8KV_ERR_INVALID", -2: "FP8KV_ERR_UNSUPPORTED",
          -3: "FP8KV_ERR_WORKSPACE", -4: "FP8KV_ERR_CUDA", -5: "FP8KV_ERR_TIMEOUT",
          -6: "FP8KV_ERR_BAD_INDEX"}

EXPORTS = ("fp8kv_kv_cache_write", "fp8kv_decode_plan", "fp8kv_paged_decode_attn",
           "fp8kv_decode_step", "fp8kv_paged_decode_attn_noalloc", "fp8kv_prefill_attn",
           "fp8kv_prefill_attn_ws", "fp8kv_prefill_workspace_bytes", "fp8kv_quantize_e4m3",
           "fp8kv_resolve_scales", "fp8kv_status_string", "fp8kv_last_warning")
NOALLOC_DECODE_SCRATCH_BYTES = 8 << 20

_lib = None


class Fp8kvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status_string(status)})")


def build(force: bool = False) -> str:
    """Compile libfp8kv.so in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def lib() -> ctypes.CDLL:
    """The loaded C library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libfp8kv.so not found at {LIB_PATH}: build it first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        u32 = ctypes.c_uint
        L.fp8kv_kv_cache_write.argtypes = [P, P, P, i64, i32, i32, P, P, i64, i32, i32, P, P, P,
                                           P, P, P]
        L.fp8kv_kv_cache_write.restype = i32
        L.fp8kv_decode_plan.argtypes = [i32, i32, i32, i32, i32, i32, i32,
                                        ctypes.POINTER(i32), ctypes.POINTER(sz)]
        L.fp8kv_decode_plan.restype = i32
        L.fp8kv_paged_decode_attn.argtypes = [P, P, P, i32, i32, P, P, P, P, P, i32, P, i32, i32,
                                              i32, i32, i64, f32, i32, i32, P, sz, P, i32, u32, P,
                                              P]
        L.fp8kv_paged_decode_attn.restype = i32
        L.fp8kv_decode_step.argtypes = [P, P, P, P, P, i32, i32, P, P, P, P, P, i32, P, i32, i32,
                                        i32, i32, i64, f32, i32, i32, P, sz, P, i32, u32, P, P]
        L.fp8kv_decode_step.restype = i32
        L.fp8kv_paged_decode_attn_noalloc.argtypes = [P, P, P, i32, i32, P, P, P, P, P, i32, P,
                                                      i32, i32, i32, i32, i64, f32, i32, i32, P,
                                                      i32, P, P]
        L.fp8kv_paged_decode_attn_noalloc.restype = i32
        L.fp8kv_prefill_attn.argtypes = [P, P, i32, P, P, i32, i32, P, P, P, P, f32, f32, P, i32, P,
                                         i32, i32, i32, i32, i64, f32, i32, P, i32, P, P]
        L.fp8kv_prefill_attn.restype = i32
        L.fp8kv_prefill_attn_ws.argtypes = [P, P, i32, P, P, i32, i32, P, P, P, P, f32, f32, P,
                                            i32, P, i32, i32, i32, i32, i64, f32, i32, P, sz, P,
                                            i32, P, P]
        L.fp8kv_prefill_attn_ws.restype = i32
        L.fp8kv_prefill_workspace_bytes.argtypes = [i32, ctypes.POINTER(sz)]
        L.fp8kv_prefill_workspace_bytes.restype = i32
        L.fp8kv_quantize_e4m3.argtypes = [P, f32, P, i64, P]
        L.fp8kv_quantize_e4m3.restype = i32
        FP = ctypes.POINTER(f32)
        L.fp8kv_resolve_scales.argtypes = [i32, i32, i32, FP, FP, f32, f32, FP, FP, FP, FP]
        L.fp8kv_resolve_scales.restype = i32
        L.fp8kv_status_string.argtypes = [i32]
        L.fp8kv_status_string.restype = ctypes.c_char_p
        L.fp8kv_last_warning.argtypes = []
        L.fp8kv_last_warning.restype = ctypes.c_char_p
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fp8kv_status_string(int(status)).decode()


def last_warning() -> str:
    return lib().fp8kv_last_warning().decode()


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype=None, device=True, contiguous=True, pinned_ok=False):
    """dtype / contiguity / placement check.  pinned_ok: pinned host memory is
    accepted too (the kernels read or write it directly over the host link)."""
    if t is None:
        return
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if device and not t.is_cuda and not (pinned_ok and t.is_pinned()):
        raise ValueError(f"{name}: expected a CUDA tensor" +
                         (" or pinned host memory" if pinned_ok else ""))
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name}: expected a contiguous tensor")


def _raise(st, what):
    if st != 0:
        raise Fp8kvError(st, what)


def kv_cache_write(k, v, slot_mapping, k_cache, v_cache, *, kv_dtype, scale_mode=SCALE_PER_TENSOR,
                   k_scale=None, v_scale=None, k_scale_cache=None, v_scale_cache=None,
                   err_flag=None, stream=None) -> None:
    """Store bf16 K/V rows [T][Hkv][D] at slot_mapping into the paged cache
    (uint8 e4m3 or bf16 [num_blocks][Hkv][16][D]); see fp8kv_kv_cache_write."""
    _check(k, "k", torch.bfloat16, pinned_ok=True)
    _check(v, "v", torch.bfloat16, pinned_ok=True)
    _check(slot_mapping, "slot_mapping", torch.int64, pinned_ok=True)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(t, n, torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale), ("k_scale_cache", k_scale_cache),
                 ("v_scale_cache", v_scale_cache)):
        _check(t, n, torch.float32)
    _check(err_flag, "err_flag", torch.int32)
    T, Hkv, D = k.shape
    st = lib().fp8kv_kv_cache_write(
        _ptr(k), _ptr(v), _ptr(slot_mapping), T, Hkv, D, _ptr(k_cache), _ptr(v_cache),
        k_cache.shape[0], kv_dtype, scale_mode, _ptr(k_scale), _ptr(v_scale),
        _ptr(k_scale_cache), _ptr(v_scale_cache), _ptr(err_flag), _stream(stream))
    _raise(st, "kv_cache_write")


def decode_plan(B, Hq, Hkv, D, max_blocks_per_seq, window=0, num_splits=0):
    """(num_splits, workspace_bytes) that paged_decode_attn will use."""
    s = ctypes.c_int(0)
    w = ctypes.c_size_t(0)
    st = lib().fp8kv_decode_plan(B, Hq, Hkv, D, max_blocks_per_seq, window, num_splits,
                                 ctypes.byref(s), ctypes.byref(w))
    _raise(st, "decode_plan")
    return s.value, w.value


def paged_decode_attn(q, k_cache, v_cache, block_table, context_lens, *, kv_dtype,
                      scale_mode=SCALE_PER_TENSOR, k_scale=None, v_scale=None,
                      k_scale_cache=None, v_scale_cache=None, softmax_scale=None, window=0,
                      num_splits=0, workspace=None, out=None, out_dtype=OUT_F32, flags=0,
                      err_flag=None, stream=None):
    """Decode attention of q [B][Hq][D] (bf16) over the paged cache; returns out
    [B][Hq][D] (fp32 or bf16).  flags: 0 or DECODE_EARLY_SETUP / DECODE_EARLY_PAGES.
    See fp8kv_paged_decode_attn."""
    _check(q, "q", torch.bfloat16, pinned_ok=True)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(t, n, torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16)
    _check(block_table, "block_table", torch.int32)
    _check(context_lens, "context_lens", torch.int32, pinned_ok=True)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale), ("k_scale_cache", k_scale_cache),
                 ("v_scale_cache", v_scale_cache)):
        _check(t, n, torch.float32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    mbs = block_table.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    splits, ws_bytes = decode_plan(B, Hq, Hkv, D, mbs, window, num_splits)
    if ws_bytes > 0 and (workspace is None or workspace.numel() * workspace.element_size()
                         < ws_bytes):
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=k_cache.device)
    if out is None:
        out = torch.empty(B, Hq, D, device=k_cache.device,
                          dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16)
    _check(out, "out", torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
           pinned_ok=True)
    st = lib().fp8kv_paged_decode_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dtype, scale_mode, _ptr(k_scale),
        _ptr(v_scale), _ptr(k_scale_cache), _ptr(v_scale_cache), _ptr(block_table), mbs,
        _ptr(context_lens), B, Hq, Hkv, D, k_cache.shape[0], float(softmax_scale), int(window),
        int(num_splits), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(out),
        out_dtype, int(flags), _ptr(err_flag), _stream(stream))
    _raise(st, "paged_decode_attn")
    return out


def decode_step(q, k_new, v_new, k_cache, v_cache, block_table, context_lens, *, kv_dtype,
                scale_mode=SCALE_PER_TENSOR, k_scale=None, v_scale=None, k_scale_cache=None,
                v_scale_cache=None, softmax_scale=None, window=0, num_splits=0, workspace=None,
                out=None, out_dtype=OUT_F32, flags=0, err_flag=None, stream=None):
    """One decode step in one call: stores the new token k_new / v_new [B][Hkv][D]
    (bf16) of every sequence at position context_lens[b] - 1 of its page table
    (quantized as kv_cache_write does), then attends q [B][Hq][D] over all its
    keys.  Returns out [B][Hq][D].  See fp8kv_decode_step."""
    _check(q, "q", torch.bfloat16, pinned_ok=True)
    _check(k_new, "k_new", torch.bfloat16, pinned_ok=True)
    _check(v_new, "v_new", torch.bfloat16, pinned_ok=True)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(t, n, torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16)
    _check(block_table, "block_table", torch.int32)
    _check(context_lens, "context_lens", torch.int32, pinned_ok=True)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale), ("k_scale_cache", k_scale_cache),
                 ("v_scale_cache", v_scale_cache)):
        _check(t, n, torch.float32)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if tuple(k_new.shape) != (B, Hkv, D) or tuple(v_new.shape) != (B, Hkv, D):
        raise ValueError(f"k_new / v_new: expected shape {(B, Hkv, D)}")
    mbs = block_table.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    splits, ws_bytes = decode_plan(B, Hq, Hkv, D, mbs, window, num_splits)
    if ws_bytes > 0 and (workspace is None or workspace.numel() * workspace.element_size()
                         < ws_bytes):
        workspace = torch.empty(ws_bytes // 4, dtype=torch.float32, device=k_cache.device)
    if out is None:
        out = torch.empty(B, Hq, D, device=k_cache.device,
                          dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16)
    _check(out, "out", torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
           pinned_ok=True)
    st = lib().fp8kv_decode_step(
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), kv_dtype, scale_mode,
        _ptr(k_scale), _ptr(v_scale), _ptr(k_scale_cache), _ptr(v_scale_cache),
        _ptr(block_table), mbs, _ptr(context_lens), B, Hq, Hkv, D, k_cache.shape[0],
        float(softmax_scale), int(window), int(num_splits), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(out),
        out_dtype, int(flags), _ptr(err_flag), _stream(stream))
    _raise(st, "decode_step")
    return out


def paged_decode_attn_noalloc(q, k_cache, v_cache, block_table, context_lens, *, kv_dtype,
                              scale_mode=SCALE_PER_TENSOR, k_scale=None, v_scale=None,
                              k_scale_cache=None, v_scale_cache=None, softmax_scale=None,
                              window=0, num_splits=0, out, out_dtype=OUT_F32, err_flag=None,
                              stream=None):
    """paged_decode_attn without a workspace, for callers that cannot allocate
    device memory: the split partials live in the library's static device array
    (NOALLOC_DECODE_SCRATCH_BYTES per GPU).  `out` must be passed.  Calls that
    overlap on the GPU race on that array; the first call on a device should
    come before any stream capture."""
    _check(q, "q", torch.bfloat16, pinned_ok=True)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(t, n, torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16)
    _check(block_table, "block_table", torch.int32)
    _check(context_lens, "context_lens", torch.int32, pinned_ok=True)
    _check(out, "out", torch.float32 if out_dtype == OUT_F32 else torch.bfloat16,
           pinned_ok=True)
    B, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    mbs = block_table.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    st = lib().fp8kv_paged_decode_attn_noalloc(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), kv_dtype, scale_mode, _ptr(k_scale),
        _ptr(v_scale), _ptr(k_scale_cache), _ptr(v_scale_cache), _ptr(block_table), mbs,
        _ptr(context_lens), B, Hq, Hkv, D, k_cache.shape[0], float(softmax_scale), int(window),
        int(num_splits), _ptr(out), out_dtype, _ptr(err_flag), _stream(stream))
    if st == -3:
        if num_splits == 0:
            raise Fp8kvError(st, f"paged_decode_attn_noalloc: one split slot per (sequence, KV "
                                 f"head) already needs B*Hq*(D+2)*4 = {B * Hq * (D + 2) * 4} "
                                 f"bytes, more than the static array's "
                                 f"{NOALLOC_DECODE_SCRATCH_BYTES}; use paged_decode_attn with "
                                 f"a workspace")
        _, need = decode_plan(B, Hq, Hkv, D, mbs, window, num_splits)
        raise Fp8kvError(st, f"paged_decode_attn_noalloc: the split plan needs {need} bytes of "
                             f"scratch but the static array holds "
                             f"{NOALLOC_DECODE_SCRATCH_BYTES}; pass fewer num_splits (or 0) or "
                             f"use paged_decode_attn with a workspace")
    _raise(st, "paged_decode_attn_noalloc")
    return out


def prefill_workspace_bytes(D):
    """Bytes of the workspace fp8kv_prefill_attn_ws takes at head_dim D."""
    n = ctypes.c_size_t(0)
    _raise(lib().fp8kv_prefill_workspace_bytes(int(D), ctypes.byref(n)), "prefill_workspace_bytes")
    return n.value


# zero-filled prefill workspaces, one per (device, stream, D): the kernel leaves
# its counters zero after each call, and calls on one stream never overlap
_prefill_ws = {}


def prefill_workspace(device, stream, D):
    """The cached zero-initialised workspace prefill_attn uses on `stream` (a
    torch stream; None: the current one)."""
    key = (torch.device(device).index, _stream(stream).value or 0, int(D))
    ws = _prefill_ws.get(key)
    if ws is None:
        ws = torch.zeros(prefill_workspace_bytes(D), dtype=torch.uint8, device=device)
        _prefill_ws[key] = ws
    return ws


def prefill_attn(q, cu_seqlens_q, max_seqlen_q, k_cache, v_cache, block_table, context_lens,
                 *, kv_dtype=KV_E4M3, scale_mode=SCALE_PER_TENSOR, k_scale=None, v_scale=None,
                 k_scale_cache=None, v_scale_cache=None, q_scale=1.0, prob_scale=1.0,
                 softmax_scale=None, two_level=False, split="auto", out=None, out_dtype=OUT_F32,
                 err_flag=None, stream=None, workspace="auto"):
    """Chunked causal FP8 prefill of q [Tq][Hq][D] (bf16) over the paged cache;
    returns out [Tq][Hq][D].  split: "auto" (split e4m3 operands for blocks of
    rows under 8192 keys), "always" or "never".  workspace: "auto" (a cached
    zeroed workspace per device and stream, so that launches with more query
    tiles than SMs run balanced over persistent CTAs), a zeroed uint8 tensor of
    prefill_workspace_bytes(D), or None (one CTA per query tile).  See
    fp8kv_prefill_attn and fp8kv_prefill_attn_ws."""
    if split not in ("auto", "always", "never"):
        raise ValueError("split: 'auto', 'always' or 'never'")
    flags = (PREFILL_TWO_LEVEL if two_level else 0) | {
        "auto": 0, "always": PREFILL_SPLIT_ALWAYS, "never": PREFILL_SPLIT_NEVER}[split]
    _check(q, "q", torch.bfloat16)
    _check(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache)):
        _check(t, n, torch.uint8 if kv_dtype == KV_E4M3 else torch.bfloat16)
    _check(block_table, "block_table", torch.int32)
    _check(context_lens, "context_lens", torch.int32)
    for n, t in (("k_scale", k_scale), ("v_scale", v_scale), ("k_scale_cache", k_scale_cache),
                 ("v_scale_cache", v_scale_cache)):
        _check(t, n, torch.float32)
    Tq, Hq, D = q.shape
    Hkv = k_cache.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty(Tq, Hq, D, device=q.device,
                          dtype=torch.float32 if out_dtype == OUT_F32 else torch.bfloat16)
    _check(out, "out", torch.float32 if out_dtype == OUT_F32 else torch.bfloat16)
    if isinstance(workspace, str):
        if workspace != "auto":
            raise ValueError("workspace: 'auto', a uint8 tensor or None")
        workspace = prefill_workspace(q.device, stream, D)
    _check(workspace, "workspace", torch.uint8)
    st = lib().fp8kv_prefill_attn_ws(
        _ptr(q), _ptr(cu_seqlens_q), int(max_seqlen_q), _ptr(k_cache), _ptr(v_cache), kv_dtype,
        scale_mode, _ptr(k_scale), _ptr(v_scale), _ptr(k_scale_cache), _ptr(v_scale_cache),
        float(q_scale), float(prob_scale),
        _ptr(block_table), block_table.shape[1], _ptr(context_lens), cu_seqlens_q.numel() - 1,
        Hq, Hkv, D, k_cache.shape[0], float(softmax_scale), flags, _ptr(workspace),
        workspace.numel() if workspace is not None else 0, _ptr(out),
        out_dtype, _ptr(err_flag), _stream(stream))
    _raise(st, "prefill_attn")
    return out


def quantize_e4m3(x, scale=1.0, out=None, stream=None):
    """e4m3 codes (uint8) of fp32 x / scale, computed on the GPU."""
    _check(x, "x", torch.float32)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _check(out, "out", torch.uint8)
    st = lib().fp8kv_quantize_e4m3(_ptr(x), float(scale), _ptr(out), x.numel(), _stream(stream))
    _raise(st, "quantize_e4m3")
    return out


def _floats(x):
    if x is None:
        return []
    if isinstance(x, torch.Tensor):
        return [float(e) for e in x.detach().cpu().reshape(-1).tolist()]
    if isinstance(x, (int, float)):
        return [float(x)]
    return [float(e) for e in x]


def resolve_scales(kv_dtype, scale_mode, k_loaded=None, v_loaded=None, q_loaded=-1.0,
                   prob_loaded=-1.0):
    """Scales to use from what a checkpoint loader found; -1.0 (any negative
    value) means "not loaded".  k_loaded / v_loaded: one float (per-tensor) or a
    sequence of Hkv floats (per-head); unused for per-token-head and bf16 caches.
    Returns (k_scales, v_scales, q_scale, prob_scale) with k/v as lists (None
    where the mode has no per-tensor scale).  Host-only (no GPU needed); the
    rules are those of fp8kv_resolve_scales in include/fp8kv.h."""
    per_tensor_like = kv_dtype == KV_E4M3 and scale_mode in (SCALE_PER_TENSOR, SCALE_PER_HEAD)
    if per_tensor_like:
        ks, vs = _floats(k_loaded), _floats(v_loaded)
        if len(ks) != len(vs):
            raise ValueError("k_loaded and v_loaded differ in length")
    else:
        ks = vs = []
    n = len(ks)
    FA = ctypes.c_float * max(n, 1)
    kin, vin, kout, vout = FA(*ks), FA(*vs), FA(), FA()
    q, pr = ctypes.c_float(), ctypes.c_float()
    st = lib().fp8kv_resolve_scales(kv_dtype, scale_mode, n, kin, vin, float(q_loaded),
                                    float(prob_loaded), kout, vout, ctypes.byref(q),
                                    ctypes.byref(pr))
    _raise(st, "resolve_scales")
    if not per_tensor_like:
        return None, None, q.value, pr.value
    return list(kout[:n]), list(vout[:n]), q.value, pr.value
