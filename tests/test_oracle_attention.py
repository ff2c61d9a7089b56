"""Pins for the oracle's float64 attention over the paged cache.

Each case has an answer fixed by mathematics rather than by re-running the
oracle's formula: two keys whose logits differ by ln 3 (weights exactly 1/4 and
3/4), a needle among equal-logit keys (weight e^L / (e^L + n - 1)), constant
values (the output is that value), per-page constant values with equal logits
(the output is the mean page index), GQA head grouping, the sliding window and
the causal prefix of chunked prefill.  The cache layout is [block][kv head]
[16][D] with a page table, page size 16 as in the paged tests of "vLLM
Qwen3.8-Flash-Next: QSA Indexer 캐시를 위한 FP8 지원" (section "코드 분석").
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests._helpers import bf16_from_float, bf16_value, bits16

PAGE = 16
C = {1.0: 0x38, 2.0: 0x40, -2.0: 0xC0, 4.0: 0x48, 0.5: 0x30, 8.0: 0x50, 3.0: 0x44,
     -1.0: 0xB8}


def _cache(nb, Hkv, D, dtype=np.uint8):
    return np.zeros((nb, Hkv, PAGE, D), dtype=dtype)


def test_encoder_points_used_below():
    vals = np.array(list(C.keys()), np.float32)
    assert list(oracle.e4m3_encode(vals)) == list(C.values())


@pytest.mark.parametrize("sign,w1", [(1.0, 0.75), (-1.0, 0.25)])
def test_two_keys_weights_quarter_three_quarters(sign, w1):
    D, nb = 2, 4
    kc, vc = _cache(nb, 1, D), _cache(nb, 1, D)
    bt = np.array([[3]], np.int32)                 # the sequence lives in block 3
    kc[3, 0, 1] = [C[2.0], 0]                       # k1 = (2, 0) * 0.5 = (1, 0)
    vc[3, 0, 0] = [C[1.0], C[-2.0]]                 # v0 = (1, -2) * 0.25
    vc[3, 0, 1] = [C[4.0], C[0.5]]                  # v1 = (4, 0.5) * 0.25
    q = bf16_from_float([[[sign, 0.0]]])
    st, out = oracle.decode_attn(q, kc, vc, bt, [2], kv_dtype=0, scale_mode=0,
                                 k_scale=np.array([0.5], np.float32),
                                 v_scale=np.array([0.25], np.float32),
                                 softmax_scale=math.log(3.0))
    assert st == 0
    w0 = 1 - w1
    want = w0 * np.array([0.25, -0.5]) + w1 * np.array([1.0, 0.125])
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-15)


def test_two_keys_per_token_scales_and_bf16_cache_agree():
    D = 2
    # per-token-head scales: token 1's key code 8 with scale 1/8 gives k1 = (1, 0)
    kc, vc = _cache(1, 1, D), _cache(1, 1, D)
    kc[0, 0, 1] = [C[8.0], 0]
    vc[0, 0, 0] = [C[1.0], C[-1.0]]
    vc[0, 0, 1] = [C[3.0], C[1.0]]
    ksc = np.zeros((1, 1, PAGE), np.float32)
    vsc = np.zeros((1, 1, PAGE), np.float32)
    ksc[0, 0, :2] = [4.0, 0.125]
    vsc[0, 0, :2] = [2.0, 0.5]                      # v0 = (2, -2), v1 = (1.5, 0.5)
    q = bf16_from_float([[[1.0, 0.0]]])
    st, out = oracle.decode_attn(q, kc, vc, np.array([[0]], np.int32), [2], kv_dtype=0,
                                 scale_mode=2, k_scale_cache=ksc, v_scale_cache=vsc,
                                 softmax_scale=math.log(3.0))
    assert st == 0
    want = 0.25 * np.array([2.0, -2.0]) + 0.75 * np.array([1.5, 0.5])
    np.testing.assert_allclose(out[0], want, rtol=0, atol=1e-15)
    # the same keys and values stored as bf16
    kb, vb = _cache(1, 1, D, np.uint16), _cache(1, 1, D, np.uint16)
    kb[0, 0, :2] = bf16_from_float([[0.0, 0.0], [1.0, 0.0]])
    vb[0, 0, :2] = bf16_from_float([[2.0, -2.0], [1.5, 0.5]])
    st, outb = oracle.decode_attn(q, kb, vb, np.array([[0]], np.int32), [2], kv_dtype=1,
                                  softmax_scale=math.log(3.0))
    assert st == 0
    np.testing.assert_allclose(outb[0], want, rtol=0, atol=1e-15)


@pytest.mark.parametrize("n", [1, 17, 1000])
def test_needle_weight_closed_form(n):
    # all keys zero except the needle at position n // 2 whose logit is 8 * 1.5 = 12
    D = 2
    nblk = (n + PAGE - 1) // PAGE
    kc, vc = _cache(nblk, 1, D), _cache(nblk, 1, D)
    bt = np.random.default_rng(n).permutation(nblk).astype(np.int32)[None]
    p = n // 2
    blk = bt[0, p // PAGE]
    kc[blk, 0, p % PAGE] = [C[8.0], 0]
    vc[blk, 0, p % PAGE] = [C[3.0], C[-1.0]]
    q = bf16_from_float([[[1.0, 0.0]]])
    st, out = oracle.decode_attn(q, kc, vc, bt, [n], kv_dtype=0, scale_mode=0,
                                 k_scale=np.array([1.5], np.float32),
                                 v_scale=np.array([1.0], np.float32), softmax_scale=1.0)
    assert st == 0
    w = math.exp(12.0) / (math.exp(12.0) + (n - 1))
    np.testing.assert_allclose(out[0], w * np.array([3.0, -1.0]), rtol=1e-14, atol=0)


def test_constant_values_return_the_value():
    D, nb, ctx = 64, 10, 150
    g = np.random.default_rng(1)
    kc = g.integers(0, 0x7E, size=(nb, 2, PAGE, D), dtype=np.uint8)
    kc |= (g.integers(0, 2, size=kc.shape, dtype=np.uint8) << 7)
    vc = _cache(nb, 2, D)
    vc[:, 0] = C[3.0]
    vc[:, 1] = C[-2.0]
    bt = g.permutation(nb).astype(np.int32)[None]
    q = bits16(torch.randn(1, 4, D).to(torch.bfloat16))
    st, out = oracle.decode_attn(q, kc, vc, bt, [ctx], kv_dtype=0, scale_mode=1,
                                 k_scale=np.array([0.01, 0.02], np.float32),
                                 v_scale=np.array([0.5, 2.0], np.float32))
    assert st == 0
    np.testing.assert_allclose(out[:2], 1.5, rtol=1e-14)
    np.testing.assert_allclose(out[2:], -4.0, rtol=1e-14)


def test_gqa_grouping_is_contiguous():
    # Hq = 6, Hkv = 3: query heads 0,1 -> kv 0; 2,3 -> kv 1; 4,5 -> kv 2
    D, ctx = 16, 20
    kc, vc = _cache(2, 3, D), _cache(2, 3, D)
    for h, val in enumerate([1.0, 2.0, 4.0]):
        vc[:, h] = C[val]
    q = bits16(torch.randn(1, 6, D).to(torch.bfloat16))
    st, out = oracle.decode_attn(q, kc, vc, np.array([[1, 0]], np.int32), [ctx], kv_dtype=0,
                                 scale_mode=0, k_scale=np.ones(1, np.float32),
                                 v_scale=np.ones(1, np.float32))
    assert st == 0
    np.testing.assert_allclose(out[:, 0], [1, 1, 2, 2, 4, 4], rtol=1e-15)


@pytest.mark.parametrize("ctx", [1, 15, 16, 17, 200])
def test_equal_logits_average_the_pages(ctx):
    # zero keys (equal logits); each page holds its logical index as value
    D = 8
    nblk = (ctx + PAGE - 1) // PAGE
    kc, vc = _cache(nblk + 3, 1, D), _cache(nblk + 3, 1, D)
    bt = np.random.default_rng(ctx).permutation(nblk + 3)[:nblk].astype(np.int32)[None]
    codes = oracle.e4m3_encode(np.arange(nblk, dtype=np.float32))
    for p in range(nblk):
        vc[bt[0, p], 0] = codes[p]
    q = bits16(torch.randn(1, 1, D).to(torch.bfloat16))
    st, out = oracle.decode_attn(q, kc, vc, bt, [ctx], kv_dtype=0, scale_mode=0,
                                 k_scale=np.ones(1, np.float32), v_scale=np.ones(1, np.float32))
    assert st == 0
    want = sum(t // PAGE for t in range(ctx)) / ctx
    np.testing.assert_allclose(out[0], want, rtol=1e-14)


def _random_case(seed, B=3, Hq=4, Hkv=2, D=32, ctxs=(1, 40, 77), kv_dtype=0, scale_mode=2):
    g = torch.Generator().manual_seed(seed)
    nblk = [(c + PAGE - 1) // PAGE for c in ctxs]
    nb = sum(nblk) + 2
    perm = torch.randperm(nb, generator=g).numpy().astype(np.int32)
    bt = np.full((B, max(nblk)), -1, np.int32)
    at = 0
    for s, n in enumerate(nblk):
        bt[s, :n] = perm[at:at + n]
        at += n
    if kv_dtype == 0:
        kc = torch.randint(0, 256, (nb, Hkv, PAGE, D), generator=g, dtype=torch.uint8).numpy()
        vc = torch.randint(0, 256, (nb, Hkv, PAGE, D), generator=g, dtype=torch.uint8).numpy()
        kc[(kc & 0x7F) == 0x7F] = 0x11                       # no NaN codes in a valid cache
        vc[(vc & 0x7F) == 0x7F] = 0x22
        kc, vc = kc.copy(), vc.copy()
    else:
        kc = bits16(torch.randn(nb, Hkv, PAGE, D, generator=g).to(torch.bfloat16)).copy()
        vc = bits16(torch.randn(nb, Hkv, PAGE, D, generator=g).to(torch.bfloat16)).copy()
    ksc = (torch.rand(nb, Hkv, PAGE, generator=g) * 0.01).numpy()
    vsc = (torch.rand(nb, Hkv, PAGE, generator=g) * 0.02).numpy()
    q = bits16(torch.randn(B, Hq, D, generator=g).to(torch.bfloat16))
    return q, kc, vc, bt, np.array(ctxs, np.int32), ksc, vsc


def _dense_keys(cache, bt, ctx, s, h, kv_dtype, scale):
    """Gather one sequence's dequantized keys/values with numpy fancy indexing."""
    t = np.arange(ctx)
    blk, off = bt[s, t // PAGE], t % PAGE
    raw = cache[blk, h, off]
    if kv_dtype == 0:
        return oracle.e4m3_decode(raw) * scale[blk, h, off][:, None].astype(np.float64)
    return bf16_value(raw)


@pytest.mark.parametrize("kv_dtype", [0, 1])
def test_agrees_with_dense_library_softmax(kv_dtype):
    # An independent path: dense gather + numpy matmul + scipy softmax.
    scipy_special = pytest.importorskip("scipy.special")
    q, kc, vc, bt, ctx, ksc, vsc = _random_case(5, kv_dtype=kv_dtype)
    st, out = oracle.decode_attn(q, kc, vc, bt, ctx, kv_dtype=kv_dtype, scale_mode=2,
                                 k_scale_cache=ksc, v_scale_cache=vsc)
    assert st == 0
    B, Hq, D = q.shape
    G = Hq // kc.shape[1]
    qv = bf16_value(q)
    for s in range(B):
        for hq in range(Hq):
            K = _dense_keys(kc, bt, ctx[s], s, hq // G, kv_dtype, ksc)
            V = _dense_keys(vc, bt, ctx[s], s, hq // G, kv_dtype, vsc)
            w = scipy_special.softmax(K @ qv[s, hq] / math.sqrt(D))
            np.testing.assert_allclose(out[s * Hq + hq], w @ V, rtol=1e-12, atol=1e-14)


def test_window_keeps_the_last_keys():
    q, kc, vc, bt, ctx, ksc, vsc = _random_case(6)
    kw = dict(kv_dtype=0, scale_mode=2, k_scale_cache=ksc, v_scale_cache=vsc)
    _, full = oracle.decode_attn(q, kc, vc, bt, ctx, **kw)
    _, wide = oracle.decode_attn(q, kc, vc, bt, ctx, window=int(ctx.max()), **kw)
    np.testing.assert_array_equal(full, wide)
    _, one = oracle.decode_attn(q, kc, vc, bt, ctx, window=1, **kw)
    B, Hq, _ = q.shape
    G = Hq // kc.shape[1]
    for s in range(B):
        for hq in range(Hq):
            V = _dense_keys(vc, bt, ctx[s], s, hq // G, 0, vsc)
            np.testing.assert_allclose(one[s * Hq + hq], V[-1], rtol=1e-15)
    # window w equals full attention over a sequence cut to its last w tokens
    _, w5 = oracle.decode_attn(q, kc, vc, bt, ctx, window=5, **kw)
    s = 2
    u = [(s, hq) for hq in range(Hq)]
    # shift the page table so that position ctx-5 becomes position 0: use the
    # dense path on the last 5 keys
    for hq in range(Hq):
        K = _dense_keys(kc, bt, ctx[s], s, hq // G, 0, ksc)[-5:]
        V = _dense_keys(vc, bt, ctx[s], s, hq // G, 0, vsc)[-5:]
        z = K @ bf16_value(q)[s, hq] / math.sqrt(q.shape[2])
        w = np.exp(z - z.max())
        np.testing.assert_allclose(w5[s * Hq + hq], (w / w.sum()) @ V, rtol=1e-12, atol=1e-15)
    assert len(u) == Hq


def test_empty_context_gives_zeros_and_units_select_rows():
    q, kc, vc, bt, ctx, ksc, vsc = _random_case(7)
    ctx0 = ctx.copy()
    ctx0[1] = 0
    kw = dict(kv_dtype=0, scale_mode=2, k_scale_cache=ksc, v_scale_cache=vsc)
    st, out = oracle.decode_attn(q, kc, vc, bt, ctx0, **kw)
    assert st == 0
    Hq = q.shape[1]
    assert np.all(out[Hq:2 * Hq] == 0)
    units = np.array([[2, 3], [0, 1]])
    _, sub = oracle.decode_attn(q, kc, vc, bt, ctx0, units=units, **kw)
    np.testing.assert_array_equal(sub[0], out[2 * Hq + 3])
    np.testing.assert_array_equal(sub[1], out[1])
    # threads do not change the result
    _, thr = oracle.decode_attn(q, kc, vc, bt, ctx0, nthreads=4, **kw)
    np.testing.assert_array_equal(thr, out)


def test_bad_block_id_is_reported():
    q, kc, vc, bt, ctx, ksc, vsc = _random_case(8)
    bt = bt.copy()
    bt[2, 0] = kc.shape[0]
    st, _ = oracle.decode_attn(q, kc, vc, bt, ctx, kv_dtype=0, scale_mode=2,
                               k_scale_cache=ksc, v_scale_cache=vsc)
    assert st == -6


def test_prefill_causal_prefix_means():
    # zero keys: row i averages the values at positions 0 .. ctx - n + i
    D, Hkv, Hq = 8, 1, 2
    ctxs, chunks = [40, 23], [9, 23]
    nblk = [(c + PAGE - 1) // PAGE for c in ctxs]
    nb = sum(nblk)
    bt = np.full((2, max(nblk)), -1, np.int32)
    perm = np.random.default_rng(3).permutation(nb).astype(np.int32)
    bt[0, :nblk[0]], bt[1, :nblk[1]] = perm[:nblk[0]], perm[nblk[0]:]
    kc = _cache(nb, Hkv, D)
    vals = np.random.default_rng(4).integers(-8, 9, size=(2, max(ctxs))).astype(np.float32)
    vc = _cache(nb, Hkv, D)
    for s in range(2):
        for t in range(ctxs[s]):
            vc[bt[s, t // PAGE], 0, t % PAGE] = oracle.e4m3_encode(vals[s, t:t + 1])[0]
    cu = np.array([0, 9, 32], np.int32)
    q = bits16(torch.randn(32, Hq, D).to(torch.bfloat16))
    st, out = oracle.prefill_attn(q, cu, kc, vc, bt, np.array(ctxs, np.int32), kv_dtype=0,
                                  scale_mode=0, k_scale=np.ones(1, np.float32),
                                  v_scale=np.ones(1, np.float32))
    assert st == 0
    out = out.reshape(32, Hq, D)
    for s in range(2):
        for i in range(chunks[s]):
            pos = ctxs[s] - chunks[s] + i
            want = vals[s, :pos + 1].astype(np.float64).mean()
            np.testing.assert_allclose(out[cu[s] + i], want, rtol=1e-13, atol=1e-15)


def test_prefill_last_row_equals_decode():
    q, kc, vc, bt, ctx, ksc, vsc = _random_case(9, ctxs=(33, 70, 5))
    kw = dict(kv_dtype=0, scale_mode=2, k_scale_cache=ksc, v_scale_cache=vsc)
    # chunk lengths 4, 1, 5: the last query of each sequence sits at ctx - 1
    chunks = [4, 1, 5]
    cu = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    B, Hq, D = q.shape
    qp = np.zeros((cu[-1], Hq, D), np.uint16)
    for s in range(B):
        qp[cu[s + 1] - 1] = q[s]
    st, pre = oracle.prefill_attn(qp, cu, kc, vc, bt, ctx, **kw)
    assert st == 0
    _, dec = oracle.decode_attn(q, kc, vc, bt, ctx, **kw)
    pre = pre.reshape(cu[-1], Hq, D)
    for s in range(B):
        np.testing.assert_array_equal(pre[cu[s + 1] - 1], dec.reshape(B, Hq, D)[s])
