"""GPU parity of the fused decode step (fp8kv_decode_step): the kernel stores
every sequence's new token at position ctx - 1 and attends over all keys in the
same launch ("[vLLM] KV Cache Quantization": per-token-head scales computed when
the kernel stores the cache; "vLLM FP8 KV-Cache 및 Attention 양자화 업데이트":
attention over the FP8 cache).

The cache after the call must equal the oracle's writer byte for byte, the
output must match the float64 oracle within 4e-3 and the unfused path
(kv_cache_write then paged_decode_attn) to fp32 rounding."""
import numpy as np
import pytest
import torch

import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._parity import (DECODE_TOL, assert_same_cache, device_cache, gpu_decode, gpu_fill,
                           gpu_write, oracle_cache, oracle_decode)

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 511, 1300]


def _step(w, cache, err=None, pinned=False, **kw):
    q, kn, vn = w.q, w.k_new, w.v_new
    if pinned:
        q, kn, vn = q.pin_memory(), kn.pin_memory(), vn.pin_memory()
    else:
        q, kn, vn = q.cuda(), kn.cuda(), vn.cuda()
    return fk.decode_step(q, kn, vn, cache["k"], cache["v"], w.block_table.cuda(),
                          w.context_lens.cuda(), kv_dtype=cache["kv_dtype"],
                          scale_mode=cache["mode"], k_scale=cache["k_scale"],
                          v_scale=cache["v_scale"], k_scale_cache=cache["ks"],
                          v_scale_cache=cache["vs"], window=w.window, err_flag=err, **kw)


def _history_only(w, kv_dtype, fill=None, err=None):
    cache = device_cache(w, kv_dtype)
    if fill is not None:
        for key in ("k", "v"):
            cache[key].view(torch.uint8).fill_(fill)
    gpu_write(w, cache, w.k_hist, w.v_hist, w.hist_slots, err)
    return cache


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv_dtype,mode", [(0, 0), (0, 1), (0, 2), (1, 0)])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 16])
def test_step_parity(D, kv_dtype, mode, G):
    # 8 sequences x 4 KV heads: G = 2 and 4 pack adjacent KV heads into one unit
    # (rows of at most 128 bytes), whose new tokens the same warp stores
    w = synth.decode_workload(300 + D + G, RAGGED, 4 * G, 4, D, mode, outlier_frac=0.01)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc = _history_only(w, kv_dtype, err=err)
    out = _step(w, gc, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc = oracle_cache(w, kv_dtype)
    assert_same_cache(gc, oc)                       # the new tokens, bit for bit
    ref = oracle_decode(w, oc)
    e = float(np.abs(out.cpu().numpy().reshape(-1, D) - ref).max())
    assert e <= DECODE_TOL, e
    unfused = gpu_decode(w, gpu_fill(w, kv_dtype))
    np.testing.assert_allclose(out.cpu().numpy(), unfused.cpu().numpy(), rtol=0, atol=2e-6)


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_step_window(kv_dtype):
    w = synth.decode_workload(41, [5, 128, 129, 700], 8, 2, 128, 2 if kv_dtype == 0 else 0,
                              window=128)
    gc = _history_only(w, kv_dtype)
    out = _step(w, gc)
    oc = oracle_cache(w, kv_dtype)
    assert_same_cache(gc, oc)
    e = float(np.abs(out.cpu().numpy().reshape(-1, 128) - oracle_decode(w, oc)).max())
    assert e <= DECODE_TOL, e


@pytest.mark.parametrize("kv_dtype,mode", [(0, 2), (0, 0), (1, 0)])
def test_stale_bytes_in_the_new_slot_are_replaced(kv_dtype, mode):
    # every byte of the cache starts as 0xFF (an e4m3 / bf16 NaN); the page copy
    # the kernel streams may predate its own store, so the staged row must be
    # the new token, not the NaN it replaced
    w = synth.decode_workload(43, [1, 16, 17, 333], 32, 8, 128, mode)
    gc = _history_only(w, kv_dtype, fill=0xFF)
    out = _step(w, gc)
    assert torch.isfinite(out).all()
    oc = oracle_cache(w, kv_dtype)
    e = float(np.abs(out.cpu().numpy().reshape(-1, 128) - oracle_decode(w, oc)).max())
    assert e <= DECODE_TOL, e


def test_llama8b_step_sampled():
    w = synth.llama8b()
    gc = _history_only(w, 0)
    out = _step(w, gc)
    oc_units = [(s, h) for s in range(w.B) for h in (0, 13, 31)]
    oc = oracle_cache(w, 0)
    assert_same_cache(gc, oc)
    ref = oracle_decode(w, oc, units=oc_units)
    got = out.cpu().numpy().reshape(-1, w.D)
    got = np.stack([got[s * w.Hq + h] for s, h in oc_units])
    assert float(np.abs(got - ref).max()) <= DECODE_TOL


def test_pinned_host_inputs():
    w = synth.decode_workload(44, [900, 31], 32, 8, 128, 2)
    gc = _history_only(w, 0)
    out = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32).pin_memory()
    _step(w, gc, pinned=True, out=out)
    torch.cuda.synchronize()
    oc = oracle_cache(w, 0)
    assert_same_cache(gc, oc)
    assert float(np.abs(out.numpy().reshape(-1, 128) - oracle_decode(w, oc)).max()) <= DECODE_TOL


def test_bad_block_id_for_the_new_token():
    w = synth.decode_workload(45, [40, 20], 8, 2, 128, 2)
    gc = _history_only(w, 0)
    bt = w.block_table.clone()
    bt[1, (20 - 1) // 16] = w.num_blocks + 5          # the new token's page
    w.block_table = bt
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = _step(w, gc, err)
    torch.cuda.synchronize()
    assert int(err.item()) == -6                      # FP8KV_ERR_BAD_INDEX
    assert torch.isfinite(out).all()


def test_graph_replays_match_eager():
    w = synth.decode_workload(46, [3000, 70, 1500, 16], 32, 8, 128, 2)
    gc = _history_only(w, 0)
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    bt, cl = w.block_table.cuda(), w.context_lens.cuda()
    _, ws_bytes = fk.decode_plan(w.B, w.Hq, w.Hkv, w.D, bt.shape[1])
    ws = torch.empty(ws_bytes // 4, dtype=torch.float32, device="cuda")
    out = torch.empty(w.B, w.Hq, w.D, device="cuda")

    def call():
        fk.decode_step(q, kn, vn, gc["k"], gc["v"], bt, cl, kv_dtype=0, scale_mode=2,
                       k_scale_cache=gc["ks"], v_scale_cache=gc["vs"], workspace=ws, out=out)

    call()
    torch.cuda.synchronize()
    eager = out.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                call()
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)


@pytest.mark.parametrize("kv_dtype,mode", [(0, 2), (1, 0)])
def test_step_batch_beyond_32(kv_dtype, mode):
    # 40 sequences: the set-up and the merge scan the batch 32 at a time
    g = torch.Generator().manual_seed(47)
    lens = torch.randint(1, 1200, (40,), generator=g).tolist()
    lens[5], lens[32], lens[39] = 0, 1, 16
    w = synth.decode_workload(47, lens, 16, 2, 128, mode)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc = _history_only(w, kv_dtype, err=err)
    out = _step(w, gc, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc = oracle_cache(w, kv_dtype)
    assert_same_cache(gc, oc)
    e = float(np.abs(out.cpu().numpy().reshape(-1, w.D) - oracle_decode(w, oc)).max())
    assert e <= DECODE_TOL, e
