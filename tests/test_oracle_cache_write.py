"""Pins for the oracle's KV-cache write, against properties the method fixes.

Per-token-head mode ("[vLLM] KV Cache Quantization: KV 캐시 FP8/INT8 양자화",
section "Per-Token-Head vs Per-Tensor 양자화": the kernel computes one scale per
token and head when it stores the cache) with scale = amax / 448:
  - the row's largest |x| lands on the top code (+-448, code 0x7E/0xFE);
  - 448 * scale reproduces amax to within fp32 rounding;
  - every code dequantizes to within half an e4m3 quantum of x / scale;
  - an all-zero row stores scale 0 and codes 0.
Per-tensor mode with the uncalibrated default 1.0 ("vLLM FP8 KV-Cache 및 Attention
양자화 업데이트", section "정확도 및 검증") stores exactly the encoder's code of x.
Per-KV-head scales ("커널 및 퓨전 최적화": one scale per KV head) use head h's scale.
The slot of token t is block * 16 + offset; negative slots are skipped.
"""
import numpy as np
import pytest
import torch

import oracle
from tests._helpers import bf16_value, bits16

PAGE = 16


def _rows(T, Hkv, D, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(T, Hkv, D, generator=g) * scale).to(torch.bfloat16)


def _empty(num_blocks, Hkv, D, dtype=np.uint8, fill=0x5A):
    a = np.empty((num_blocks, Hkv, PAGE, D), dtype=dtype)
    a.fill(fill)
    return a


def _half_quantum(y):
    """Half the e4m3 quantum at magnitude |y| (<= 448)."""
    ay = np.abs(y)
    e = np.floor(np.log2(np.maximum(ay, 2.0 ** -6)))
    return 2.0 ** (e - 4)


def test_per_token_head_scale_properties():
    T, Hkv, D, nb = 40, 4, 128, 8
    k, v = _rows(T, Hkv, D, 1), _rows(T, Hkv, D, 2, scale=3.0)
    slots = np.random.default_rng(0).permutation(nb * PAGE)[:T].astype(np.int64)
    kc, vc = _empty(nb, Hkv, D), _empty(nb, Hkv, D)
    ksc = np.full((nb, Hkv, PAGE), -7.0, np.float32)
    vsc = np.full((nb, Hkv, PAGE), -7.0, np.float32)
    st = oracle.kv_cache_write(bits16(k), bits16(v), slots, kc, vc, kv_dtype=0, scale_mode=2,
                               k_scale_cache=ksc, v_scale_cache=vsc)
    assert st == 0
    for x, cache, sc in ((k, kc, ksc), (v, vc, vsc)):
        xv = bf16_value(bits16(x))
        for t in range(T):
            blk, off = divmod(int(slots[t]), PAGE)
            for h in range(Hkv):
                row = xv[t, h]
                codes = cache[blk, h, off]
                s = float(sc[blk, h, off])
                amax = np.abs(row).max()
                # top code at the largest element
                i = int(np.argmax(np.abs(row)))
                assert codes[i] == (0xFE if row[i] < 0 else 0x7E)
                assert np.all((codes & 0x7F) <= 0x7E)
                # 448 * scale reproduces amax (one fp32 rounding of amax/448)
                assert abs(448.0 * s - amax) <= amax * 2.0 ** -23
                # each code is the nearest grid point of x / scale
                y = row / s
                dq = oracle.e4m3_decode(codes)
                # (slack: x / scale itself is rounded once to fp32 before encoding)
                assert np.all(np.abs(dq - y) <= _half_quantum(y) + np.abs(y) * 2.0 ** -23)


def test_zero_row_stores_zero_scale_and_codes():
    k = torch.zeros(1, 2, 64, dtype=torch.bfloat16)
    v = _rows(1, 2, 64, 3)
    kc, vc = _empty(1, 2, 64), _empty(1, 2, 64)
    ksc = np.full((1, 2, PAGE), -1.0, np.float32)
    vsc = np.full((1, 2, PAGE), -1.0, np.float32)
    assert oracle.kv_cache_write(bits16(k), bits16(v), np.array([5]), kc, vc, kv_dtype=0,
                                 scale_mode=2, k_scale_cache=ksc, v_scale_cache=vsc) == 0
    assert np.all(ksc[0, :, 5] == 0.0) and np.all(kc[0, :, 5] == 0)
    assert np.all(vsc[0, :, 5] > 0)


def test_per_tensor_unit_scale_is_plain_encode():
    T, Hkv, D = 33, 2, 64
    k, v = _rows(T, Hkv, D, 4, 50.0), _rows(T, Hkv, D, 5, 0.01)
    slots = np.arange(T, dtype=np.int64) + 3
    kc, vc = _empty(3, Hkv, D), _empty(3, Hkv, D)
    one = np.ones(1, np.float32)
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots, kc, vc, kv_dtype=0, scale_mode=0,
                                 k_scale=one, v_scale=one) == 0
    for x, cache in ((k, kc), (v, vc)):
        want = oracle.e4m3_encode(bf16_value(bits16(x)).astype(np.float32))
        for t in range(T):
            blk, off = divmod(int(slots[t]), PAGE)
            assert np.array_equal(cache[blk, :, off], want[t])


def test_per_head_scales_pick_the_head():
    T, Hkv, D = 16, 4, 32
    k = _rows(T, Hkv, D, 6)
    sk = np.array([2.0 ** -3, 2.0 ** -1, 2.0, 2.0 ** 3], np.float32)   # exact powers of two
    kc, vc = _empty(1, Hkv, D), _empty(1, Hkv, D)
    assert oracle.kv_cache_write(bits16(k), bits16(k), np.arange(T), kc, vc, kv_dtype=0,
                                 scale_mode=1, k_scale=sk, v_scale=sk[::-1].copy()) == 0
    xv = bf16_value(bits16(k))
    for h in range(Hkv):
        # x / 2^j is exact, so the code is the encoder's code of the scaled value
        want = oracle.e4m3_encode((xv[:, h] / sk[h]).astype(np.float32))
        assert np.array_equal(kc[0, h], want)
        want_v = oracle.e4m3_encode((xv[:, h] / sk[::-1][h]).astype(np.float32))
        assert np.array_equal(vc[0, h], want_v)


def test_slots_land_on_block_and_offset_and_negatives_skip():
    T, Hkv, D, nb = 6, 2, 16, 4
    # token t holds the constant value t + 1 in every channel
    x = torch.arange(1, T + 1, dtype=torch.float32).view(T, 1, 1).expand(T, Hkv, D)
    x = x.contiguous().to(torch.bfloat16)
    slots = np.array([17, -1, 63, 0, -5, 32], np.int64)
    kc, vc = _empty(nb, Hkv, D, np.uint16, 0x7FC1), _empty(nb, Hkv, D, np.uint16, 0x7FC1)
    before = kc.copy()
    assert oracle.kv_cache_write(bits16(x), bits16(x), slots, kc, vc, kv_dtype=1) == 0
    vals = bf16_value(kc)
    touched = np.zeros(kc.shape[:3], bool)
    for t, s in enumerate(slots):
        if s < 0:
            continue
        blk, off = divmod(int(s), PAGE)
        assert np.all(vals[blk, :, off] == t + 1)
        touched[blk, :, off] = True
    assert np.array_equal(kc[~touched], before[~touched])
    assert np.array_equal(kc, vc)


def test_bf16_copy_is_bit_exact():
    k = _rows(20, 3, 128, 7)
    kc, vc = _empty(2, 3, 128, np.uint16), _empty(2, 3, 128, np.uint16)
    assert oracle.kv_cache_write(bits16(k), bits16(k), np.arange(20) + 7, kc, vc,
                                 kv_dtype=1) == 0
    flat = kc.transpose(0, 2, 1, 3).reshape(-1, 3, 128)
    assert np.array_equal(flat[7:27], bits16(k))


def test_slot_past_cache_is_reported():
    k = _rows(2, 1, 16, 8)
    kc, vc = _empty(1, 1, 16), _empty(1, 1, 16)
    one = np.ones(1, np.float32)
    assert oracle.kv_cache_write(bits16(k), bits16(k), np.array([3, 16]), kc, vc, kv_dtype=0,
                                 scale_mode=0, k_scale=one, v_scale=one) == -6


@pytest.mark.parametrize("D", [64, 128, 256])
def test_outlier_channels_keep_small_values_resolvable(D):
    # A x20 outlier channel raises the per-token-head scale; the remaining
    # channels still round to their nearest grid point (no saturation, no flush
    # of values above 2^-10 * scale).
    k = _rows(8, 1, D, 9)
    k[:, 0, 3] = (k[:, 0, 3].float() * 20).to(torch.bfloat16)
    kc, vc = _empty(1, 1, D), _empty(1, 1, D)
    ksc = np.zeros((1, 1, PAGE), np.float32)
    assert oracle.kv_cache_write(bits16(k), bits16(k), np.arange(8), kc, vc, kv_dtype=0,
                                 scale_mode=2, k_scale_cache=ksc, v_scale_cache=ksc.copy()) == 0
    xv = bf16_value(bits16(k))[:, 0]
    dq = oracle.e4m3_decode(kc[0, 0, :8]) * ksc[0, 0, :8, None]
    y = xv / ksc[0, 0, :8, None]
    bound = (_half_quantum(y) + np.abs(y) * 2.0 ** -23) * ksc[0, 0, :8, None]
    assert np.all(np.abs(dq - xv) <= bound * (1 + 1e-12))


def _torch_e4m3(y):
    """e4m3fn codes by torch's own cast (round to nearest even); valid for |y| <= 464,
    where torch and satfinite agree."""
    t = torch.from_numpy(np.ascontiguousarray(y, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_per_token_head_is_the_ieee_quotient():
    # "Per-Token-Head vs Per-Tensor 양자화": scale = amax / 448 and code = e4m3 of
    # x / scale.  Both are single IEEE fp32 divisions (numpy's float32 '/' is one),
    # so the stored scale and every code must equal them bit for bit.  Rows with
    # x20 outlier channels make scales far from powers of two, where x * fp32(1/s)
    # and fp32(amax * fp32(1/448)) differ from the quotients: the test requires
    # that such values occur, so an oracle that multiplies by a reciprocal fails.
    T, Hkv, D, nb = 256, 4, 128, 64
    g = torch.Generator().manual_seed(77)
    k = torch.randn(T, Hkv, D, generator=g)
    v = torch.randn(T, Hkv, D, generator=g) * 3.0
    idx = torch.randperm(Hkv * D, generator=g)[: int(np.ceil(0.01 * Hkv * D))]
    for x in (k, v):
        for i in idx.tolist():
            h, c = divmod(i, D)
            x[:, h, c] *= 20.0
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    slots = np.random.default_rng(5).permutation(nb * PAGE)[:T].astype(np.int64)
    kc, vc = _empty(nb, Hkv, D), _empty(nb, Hkv, D)
    ksc = np.full((nb, Hkv, PAGE), -7.0, np.float32)
    vsc = np.full((nb, Hkv, PAGE), -7.0, np.float32)
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots, kc, vc, kv_dtype=0, scale_mode=2,
                                 k_scale_cache=ksc, v_scale_cache=vsc) == 0
    recip_scale_differs = recip_code_differs = 0
    for x, cache, sc in ((k, kc, ksc), (v, vc, vsc)):
        xf = bf16_value(bits16(x)).astype(np.float32)        # exact: bf16 -> fp32
        blk, off = np.divmod(slots, PAGE)
        got_s = sc[blk, :, off]                              # [T][Hkv]
        got_c = cache[blk, :, off]                           # [T][Hkv][D]
        amax = np.abs(xf).max(axis=2)
        want_s = amax / np.float32(448.0)
        assert want_s.dtype == np.float32
        assert np.array_equal(got_s.view(np.uint32), want_s.view(np.uint32))
        recip_scale_differs += int(np.count_nonzero(
            (amax * (np.float32(1.0) / np.float32(448.0))).view(np.uint32)
            != want_s.view(np.uint32)))
        y = xf / want_s[:, :, None]                          # IEEE fp32 quotients
        assert y.dtype == np.float32 and np.abs(y).max() <= 464.0
        want_c = _torch_e4m3(y)
        assert np.array_equal(got_c, want_c)
        assert np.array_equal(got_c, oracle.e4m3_encode(y))
        y_recip = xf * (np.float32(1.0) / want_s)[:, :, None]
        recip_code_differs += int(np.count_nonzero(_torch_e4m3(y_recip) != want_c))
    assert recip_scale_differs > 0
    assert recip_code_differs > 0
