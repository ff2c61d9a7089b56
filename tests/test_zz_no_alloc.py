"""The allocation-free decode entry point against the regular one.

fp8kv_paged_decode_attn_noalloc exists for callers that cannot allocate device
memory: a host program or plugin handed only its input and output tensors by
the framework that owns the GPU's memory pool, or a serving loop that cannot
afford the device synchronization of cudaMalloc / cudaFree.  It keeps the split
partials in a static device array inside the library instead of a workspace.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test already.  It must pass on its own in a fresh
process as well as after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._parity import gpu_decode, gpu_fill

pytestmark = pytest.mark.gpu

RTOL = ATOL = 2e-5          # the split-count invariance tolerance of the decode tests


def _p(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _noalloc_call(w, cache, out, num_splits=0):
    """One call of the C entry point with no workspace argument."""
    q, bt, cl = w.q.cuda(), w.block_table.cuda(), w.context_lens.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = fk.lib().fp8kv_paged_decode_attn_noalloc(
        _p(q), _p(cache["k"]), _p(cache["v"]), cache["kv_dtype"], cache["mode"],
        _p(cache["k_scale"]), _p(cache["v_scale"]), _p(cache["ks"]), _p(cache["vs"]), _p(bt),
        bt.shape[1], _p(cl), w.B, w.Hq, w.Hkv, w.D, w.num_blocks, w.softmax_scale, w.window,
        num_splits, _p(out), fk.OUT_F32, _p(err), ctypes.c_void_p(torch.cuda.current_stream()
                                                                   .cuda_stream))
    torch.cuda.synchronize()
    assert st == 0, fk.status_string(st)
    assert int(err.item()) == 0
    return out


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    # Two different problems back to back: the second call reuses the static
    # array that still holds the first call's partials.
    w1 = synth.decode_workload(31, [2000, 33, 900], 32, 8, 128, fk.SCALE_PER_TOKEN_HEAD,
                               outlier_frac=0.01)
    w2 = synth.decode_workload(32, [5000, 1, 17, 4096], 16, 2, 64, fk.SCALE_PER_HEAD)
    c1, c2 = gpu_fill(w1, fk.KV_E4M3), gpu_fill(w2, fk.KV_E4M3)
    want1 = gpu_decode(w1, c1).cpu().numpy()
    want2 = gpu_decode(w2, c2).cpu().numpy()
    s1, _ = fk.decode_plan(w1.B, w1.Hq, w1.Hkv, w1.D, w1.block_table.shape[1])
    s2, _ = fk.decode_plan(w2.B, w2.Hq, w2.Hkv, w2.D, w2.block_table.shape[1])
    assert s1 > 1 and s2 > 1            # both calls use the split scratch
    out1 = torch.full((w1.B, w1.Hq, w1.D), float("nan"), device="cuda")
    out2 = torch.full((w2.B, w2.Hq, w2.D), float("nan"), device="cuda")
    got1 = _noalloc_call(w1, c1, out1).cpu().numpy()
    got2 = _noalloc_call(w2, c2, out2).cpu().numpy()
    np.testing.assert_allclose(got1, want1, rtol=RTOL, atol=ATOL)
    np.testing.assert_allclose(got2, want2, rtol=RTOL, atol=ATOL)


def test_noalloc_rejects_plans_larger_than_the_static_array():
    # 64 sequences x 64 heads x 64 splits x (256 + 2) floats is far above the
    # array; the call returns FP8KV_ERR_WORKSPACE before touching any pointer.
    s, need = fk.decode_plan(64, 64, 8, 256, 4096, 0, 64)
    assert need > fk.NOALLOC_DECODE_SCRATCH_BYTES
    N = ctypes.c_void_p(0)
    st = fk.lib().fp8kv_paged_decode_attn_noalloc(N, N, N, 0, 0, N, N, N, N, N, 4096, N, 64, 64,
                                                  8, 256, 1000, 0.06, 0, 64, N, 0, N, N)
    assert st == -3
    # the binding reports the same rejection with the sizes involved
    one = torch.ones(1, device="cuda")
    with pytest.raises(fk.Fp8kvError, match="static array"):
        fk.paged_decode_attn_noalloc(
            torch.zeros(64, 64, 256, dtype=torch.bfloat16, device="cuda"),
            torch.zeros(1000, 8, 16, 256, dtype=torch.uint8, device="cuda"),
            torch.zeros(1000, 8, 16, 256, dtype=torch.uint8, device="cuda"),
            torch.zeros(64, 4096, dtype=torch.int32, device="cuda"),
            torch.zeros(64, dtype=torch.int32, device="cuda"), kv_dtype=0, scale_mode=0,
            k_scale=one, v_scale=one, num_splits=64,
            out=torch.empty(64, 64, 256, device="cuda"))


def test_noalloc_automatic_plan_is_lowered_to_fit_the_array():
    # 32 sequences x 64 query heads at head_dim 128: the regular automatic plan
    # (one wave of CTAs) needs more partial slots than the static array holds,
    # so the entry point uses fewer CTAs instead of rejecting the call.
    w = synth.decode_workload(33, [1900 + 7 * i for i in range(32)], 64, 8, 128,
                              fk.SCALE_PER_TOKEN_HEAD)
    _, need = fk.decode_plan(w.B, w.Hq, w.Hkv, w.D, w.block_table.shape[1])
    assert need > fk.NOALLOC_DECODE_SCRATCH_BYTES
    c = gpu_fill(w, fk.KV_E4M3)
    want = gpu_decode(w, c).cpu().numpy()
    out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
    for _ in range(2):
        got = _noalloc_call(w, c, out).cpu().numpy()
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)


def test_noalloc_rejects_a_batch_whose_unit_slots_alone_exceed_the_array():
    # B * Hq * (D + 2) * 4 bytes (one slot per sequence and query head) above the
    # array: no CTA count fits; the binding names the term and the alternative.
    B, Hq, Hkv, D = 256, 64, 8, 128
    assert B * Hq * (D + 2) * 4 > fk.NOALLOC_DECODE_SCRATCH_BYTES
    one = torch.ones(1, device="cuda")
    with pytest.raises(fk.Fp8kvError, match="workspace"):
        fk.paged_decode_attn_noalloc(
            torch.zeros(B, Hq, D, dtype=torch.bfloat16, device="cuda"),
            torch.zeros(64, Hkv, 16, D, dtype=torch.uint8, device="cuda"),
            torch.zeros(64, Hkv, 16, D, dtype=torch.uint8, device="cuda"),
            torch.zeros(B, 4, dtype=torch.int32, device="cuda"),
            torch.zeros(B, dtype=torch.int32, device="cuda"), kv_dtype=0, scale_mode=0,
            k_scale=one, v_scale=one, out=torch.empty(B, Hq, D, device="cuda"))


def test_noalloc_sliding_window_uses_no_scratch():
    # a sliding window of at most 16 visible pages takes one CTA per unit that
    # combines in shared memory: no scratch, and no limit from the unit slots
    w = synth.hybrid_layer(layer=0)
    c = gpu_fill(w, fk.KV_BF16)
    want = gpu_decode(w, c).cpu().numpy()
    out = torch.full((w.B, w.Hq, w.D), float("nan"), device="cuda")
    for _ in range(2):
        got = _noalloc_call(w, c, out).cpu().numpy()
        np.testing.assert_allclose(got, want, rtol=RTOL, atol=ATOL)

