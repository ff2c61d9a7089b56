"""GPU parity of paged decode attention (split-K + split_merge) against the
float64 oracle: max-abs error <= 4e-3 on fp32 output, inputs N(0,1).

Covers every head size, cache dtype and scale mode on ragged contexts (0, 1,
15, 16, 17, ... tokens), the sliding window, invariance to the split count and
to the page permutation, the Llama-3.1-8B-shaped workload (contexts 18k-22k,
per-token-head scales, x20 outlier channels) at full size on sampled rows, the
131k-token needle and the hybrid model's layers.  Attention runs over the FP8
cache directly ("vLLM FP8 KV-Cache 및 Attention 양자화 업데이트", opening paragraph).
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._helpers import bits16
from tests._parity import (DECODE_TOL, assert_same_cache, gpu_decode, gpu_fill, oracle_cache,
                           oracle_decode)

pytestmark = pytest.mark.gpu

RAGGED = [0, 1, 15, 16, 17, 100, 511, 1300]


def _check(w, kv_dtype, units=None, **kw):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc = gpu_fill(w, kv_dtype, err)
    oc = oracle_cache(w, kv_dtype)
    assert_same_cache(gc, oc)
    out = gpu_decode(w, gc, err_flag=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ref = oracle_decode(w, oc, units=units)
    got = out.float().cpu().numpy().reshape(-1, w.D)
    if units is not None:
        got = np.stack([got[s * w.Hq + h] for s, h in units])
    e = float(np.abs(got - ref).max())
    return e, got, ref


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv_dtype,mode", [(0, 0), (0, 1), (0, 2), (1, 0)])
@pytest.mark.parametrize("G", [1, 2, 4, 8, 12, 16])
def test_decode_ragged_parity(D, kv_dtype, mode, G):
    # 8 sequences x 4 KV heads: with G = 2 or 4 and rows of at most 128 bytes
    # adjacent KV heads form one unit (their tiles copied together, their query
    # heads sharing the 8 MMA columns); per-head scales then differ between the
    # columns of a unit
    w = synth.decode_workload(100 + D + G, RAGGED, 4 * G, 4, D, mode, outlier_frac=0.01)
    e, _, _ = _check(w, kv_dtype)
    assert e <= DECODE_TOL, e


@pytest.mark.parametrize("kv_dtype,mode", [(0, 1), (0, 2), (1, 0)])
@pytest.mark.parametrize("ctx,Hkv", [([2000, 17, 600] * 4, 3), ([2000, 17, 600], 2)])
def test_four_query_heads_without_packing(kv_dtype, mode, ctx, Hkv):
    # G = 4 but an odd KV head count, or fewer than 32 (sequence, KV head)
    # pairs: one KV head per unit
    w = synth.decode_workload(41, ctx, 4 * Hkv, Hkv, 128, mode, outlier_frac=0.01)
    e, _, _ = _check(w, kv_dtype)
    assert e <= DECODE_TOL, e


@pytest.mark.parametrize("G", [8, 16])
@pytest.mark.parametrize("splits", [1, 3, 0])
def test_gqa_groups_beyond_eight_heads(G, splits):
    # more than 8 query heads per KV head: two 8-head MMA groups share every
    # K and V page; long, split contexts and per-token-head scales
    w = synth.decode_workload(70 + G, [3000, 77, 1500], 2 * G, 2, 128, 2, outlier_frac=0.01)
    e, _, _ = _check(w, 0, num_splits=splits)
    assert e <= DECODE_TOL, e


@pytest.mark.parametrize("splits", [1, 2, 7, 0])
def test_split_count_invariance(splits):
    w = synth.decode_workload(7, [2000, 33, 900, 1500], 32, 8, 128, 2, outlier_frac=0.01)
    gc = gpu_fill(w, 0)
    ref = gpu_decode(w, gc, num_splits=1).cpu().numpy()
    got = gpu_decode(w, gc, num_splits=splits).cpu().numpy()
    # a different split count only regroups fp32 sums
    np.testing.assert_allclose(got, ref, rtol=2e-5, atol=2e-5)
    oc = oracle_cache(w, 0)
    assert np.abs(got.reshape(-1, 128) - oracle_decode(w, oc)).max() <= DECODE_TOL


def test_page_permutation_invariance():
    w = synth.decode_workload(8, [700, 1234], 16, 4, 128, 2)
    gc = gpu_fill(w, 0)
    base = gpu_decode(w, gc).cpu().numpy()
    # move every page to a new block: permute the cache and the table together
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(1))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_blocks)
    gc2 = dict(gc)
    for key in ("k", "v", "ks", "vs"):
        gc2[key] = torch.empty_like(gc[key])
        gc2[key][perm.cuda()] = gc[key]
    bt = w.block_table.clone()
    ok = bt >= 0
    bt[ok] = perm[bt[ok].long()].to(torch.int32)
    w2 = synth.decode_workload(8, [700, 1234], 16, 4, 128, 2)
    w2.block_table = bt
    got = gpu_decode(w2, gc2).cpu().numpy()
    assert np.array_equal(got, base)


@pytest.mark.parametrize("window", [1, 17, 128, 5000])
@pytest.mark.parametrize("kv_dtype", [0, 1])
@pytest.mark.parametrize("Hq,Hkv", [(16, 2), (32, 8)])
def test_window(window, kv_dtype, Hq, Hkv):
    w = synth.decode_workload(9, [0, 5, 130, 1000, 4000], Hq, Hkv, 64, 2, window=window)
    e, _, _ = _check(w, kv_dtype)
    assert e <= DECODE_TOL, e
    if window >= 4000:     # a window covering the context is full attention
        gc = gpu_fill(w, kv_dtype)
        full = gpu_decode(w, gc, num_splits=1).cpu()
        w.window = 0
        assert torch.allclose(gpu_decode(w, gc, num_splits=1).cpu(), full, atol=1e-6)


def test_bf16_output():
    w = synth.decode_workload(10, [300, 2048], 32, 8, 128, 2)
    gc = gpu_fill(w, 0)
    oc = oracle_cache(w, 0)
    got = gpu_decode(w, gc, out_dtype=fk.OUT_BF16)
    assert got.dtype == torch.bfloat16
    ref = oracle_decode(w, oc)
    # bf16 rounding of the output adds up to half an ulp of |o|
    bound = DECODE_TOL + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(got.float().cpu().numpy().reshape(ref.shape) - ref) <= bound)


def test_tiny_config_full_size():
    # 1 sequence, context 1024, 32/8 heads, D 128, per-tensor scale 1.0
    e, _, _ = _check(synth.tiny(), 0)
    assert e <= DECODE_TOL, e


def test_llama8b_full_size_sampled():
    # 8 sequences, contexts 18k-22k, per-token-head scales, outlier channels;
    # the oracle checks 2 query heads of every KV head of every sequence.
    w = synth.llama8b()
    units = [(s, h) for s in range(w.B) for h in range(0, w.Hq, 2)][::4]
    e, _, _ = _check(w, 0, units=units)
    assert e <= DECODE_TOL, e
    e16, _, _ = _check(w, 1, units=units[:8])
    assert e16 <= DECODE_TOL, e16


def test_needle_131k_retrieved():
    # 131072 keys, one aligned to query head hq* with logit +12; per-KV-head
    # scales.  The needle's weight is e^12 / (e^12 + sum of the rest) ~ 0.43.
    w = synth.needle()
    hq = w.extra["needle_hq"]
    units = [(0, hq)] + [(0, h) for h in range(0, w.Hq, 9)]
    e, got, ref = _check(w, 0, units=units)
    assert e <= DECODE_TOL, e
    vn = w.v_hist[w.extra["needle_pos"], w.extra["needle_h"]].float().numpy()
    proj = float(got[0] @ vn / (vn @ vn))
    assert 0.3 < proj < 0.6, proj      # the needle's value dominates the output


@pytest.mark.parametrize("layer", [0, 1])
def test_hybrid_layers(layer):
    # gpt-oss-20b-like: even layers sliding-window 128 on a bf16 cache, odd
    # layers full attention on the e4m3 cache with per-token-head scales.
    w = synth.hybrid_layer(layer=layer, B=6, ctx_lo=1024, ctx_hi=8192)
    kv = w.extra["kv_dtype"]
    e, _, _ = _check(w, kv)
    assert e <= DECODE_TOL, e


def test_bad_block_id_sets_error_flag():
    w = synth.decode_workload(12, [200, 300], 8, 2, 128, 0)
    gc = gpu_fill(w, 0)
    bt = w.block_table.clone()
    bt[1, 3] = w.num_blocks + 5
    w.block_table = bt
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = gpu_decode(w, gc, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -6
    assert torch.isfinite(out).all()


def test_workspace_too_small_is_rejected():
    w = synth.decode_workload(13, [5000], 8, 2, 128, 0)
    gc = gpu_fill(w, 0)
    s, need = fk.decode_plan(1, 8, 2, 128, w.block_table.shape[1], 0, 4)
    assert s > 1
    ws = torch.empty(need // 4 - 1, dtype=torch.float32, device="cuda")
    q, bt, cl = w.q.cuda(), w.block_table.cuda(), w.context_lens.cuda()
    out = torch.empty(1, 8, 128, device="cuda")
    lib = fk.lib()
    import ctypes
    P = lambda t: ctypes.c_void_p(0 if t is None else t.data_ptr())
    st = lib.fp8kv_paged_decode_attn(P(q), P(gc["k"]), P(gc["v"]), 0, 0, P(gc["k_scale"]),
                                     P(gc["v_scale"]), None, None, P(bt), bt.shape[1], P(cl), 1,
                                     8, 2, 128, w.num_blocks, 0.08, 0, 4, P(ws),
                                     ws.numel() * 4, P(out), 0, 0, None, None)
    assert st == -3


@pytest.mark.parametrize("kv_dtype,mode", [(0, 2), (0, 0), (1, 0)])
def test_unwritten_slots_holding_nan_do_not_leak(kv_dtype, mode):
    # Cache bytes and scales of slots no token was written to may hold anything,
    # NaN included; masked positions must contribute exactly nothing.
    w = synth.decode_workload(14, [1, 17, 33, 250], 16, 2, 64, mode)
    clean = gpu_fill(w, kv_dtype)
    dirty = {k: (v.clone() if torch.is_tensor(v) else v) for k, v in clean.items()}
    # e4m3 code 0x7F is NaN; the bf16 cache gets a bf16 NaN
    nan_k = torch.full_like(dirty["k"], 0x7F) if kv_dtype == 0 else \
        torch.full_like(dirty["k"], float("nan"))
    written = torch.zeros(w.num_blocks * 16, dtype=torch.bool)
    written[torch.cat([w.hist_slots, w.new_slots])] = True
    mask = (~written).view(w.num_blocks, 16).cuda()
    for key in ("k", "v"):
        t = dirty[key].permute(0, 2, 1, 3)          # [blk][16][Hkv][D] view
        t[mask] = nan_k.permute(0, 2, 1, 3)[mask]
    for key in ("ks", "vs"):
        t = dirty[key].permute(0, 2, 1)
        t[mask] = float("nan")
    a = gpu_decode(w, clean).cpu()
    b = gpu_decode(w, dirty).cpu()
    assert torch.isfinite(b).all()
    assert torch.equal(a, b)



def test_graph_replays_match_eager_calls():
    # The decode (split kernel + split_merge, both programmatically serialized)
    # captured in a CUDA graph and replayed with new queries gives the bits of an
    # eager call on its own workspace, and agrees with the oracle.
    w = synth.decode_workload(15, [3000, 5000, 1, 0, 7000], 32, 8, 128, 2)
    gc = gpu_fill(w, 0)
    oc = oracle_cache(w, 0)
    mbs = w.block_table.shape[1]
    _, need = fk.decode_plan(w.B, w.Hq, w.Hkv, w.D, mbs, 0)
    ws = torch.empty(need // 4, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt, cl = w.block_table.cuda(), w.context_lens.cuda()
    qbuf = w.q.cuda().clone()
    out = torch.empty(w.B, w.Hq, w.D, device="cuda")

    def call():
        fk.paged_decode_attn(qbuf, gc["k"], gc["v"], bt, cl, kv_dtype=0, scale_mode=2,
                             k_scale_cache=gc["ks"], v_scale_cache=gc["vs"], workspace=ws,
                             out=out, err_flag=err)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    ref = oracle_decode(w, oc)
    assert float(np.abs(out.cpu().numpy().reshape(-1, w.D) - ref).max()) <= DECODE_TOL
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        call()
    g = torch.Generator().manual_seed(16)
    for _ in range(3):
        qbuf.copy_(torch.randn(w.B, w.Hq, w.D, generator=g).to(torch.bfloat16).cuda())
        graph.replay()
        torch.cuda.synchronize()
        got = out.clone()
        fresh = fk.paged_decode_attn(qbuf, gc["k"], gc["v"], bt, cl, kv_dtype=0, scale_mode=2,
                                     k_scale_cache=gc["ks"], v_scale_cache=gc["vs"])
        torch.cuda.synchronize()
        assert torch.equal(got, fresh)
        assert int(err.item()) == 0


def _large_batch_lens(seed, B, hi=1500):
    """Ragged context lengths for more than 32 sequences: the set-up scans the
    batch 32 sequences at a time, so empty, single-token and page-exact
    sequences are placed past the first block too."""
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(0, hi, (B,), generator=g).tolist()
    lens[3], lens[32], lens[-1] = 0, 1, 16
    if B > 40:
        lens[40] = 0
    return lens


@pytest.mark.parametrize("B", [33, 70])
@pytest.mark.parametrize("kv_dtype,mode", [(0, 2), (1, 0)])
def test_decode_batches_beyond_32(B, kv_dtype, mode):
    w = synth.decode_workload(60 + B, _large_batch_lens(60 + B, B), 8, 2, 64, mode,
                              outlier_frac=0.01)
    e, _, _ = _check(w, kv_dtype)
    assert e <= DECODE_TOL, e


def test_window_batch_beyond_32():
    w = synth.decode_workload(61, _large_batch_lens(61, 45), 8, 2, 64, 0, window=128)
    e, _, _ = _check(w, 1)
    assert e <= DECODE_TOL, e
