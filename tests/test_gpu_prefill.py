"""GPU parity of the FP8 chunked prefill (tcgen05) against the float64 oracle.

The kernel rounds Q and the softmax weights to e4m3 for the FP8 tensor-core
contractions ("vLLM FP8 KV-Cache 및 Attention 양자화 업데이트": attention in FP8,
"정확도를 위한 2단계 누적": the two-level switch); the oracle keeps them exact.
The bar is max-abs 1e-2 on fp32 output at every context length, two-level
accumulation on and off.  Blocks of query rows under 8192 keys take split
operands (two e4m3 terms each for Q and P); longer rows take single e4m3
operands, whose rounding error averages out over the keys.
"""
import numpy as np
import pytest
import torch

import oracle
import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._helpers import bits16

pytestmark = pytest.mark.gpu

PREFILL_TOL = 1e-2


def _caches(w, scale_mode=0):
    """The cache written by the library and by the oracle (compared bit for bit);
    per-token-head mode also returns both sides' scale caches."""
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.uint8, device="cuda")
    vc = torch.zeros_like(kc)
    ksc = torch.zeros(nb, Hkv, 16, dtype=torch.float32, device="cuda")
    vsc = torch.zeros_like(ksc)
    ks, vs = w.k_scale.cuda(), w.v_scale.cuda()
    fk.kv_cache_write(w.k_all.cuda(), w.v_all.cuda(), w.all_slots.cuda(), kc, vc, kv_dtype=0,
                      scale_mode=scale_mode, k_scale=ks, v_scale=vs, k_scale_cache=ksc,
                      v_scale_cache=vsc)
    okc = np.zeros((nb, Hkv, 16, D), np.uint8)
    ovc = np.zeros_like(okc)
    oks = np.zeros((nb, Hkv, 16), np.float32)
    ovs = np.zeros_like(oks)
    assert oracle.kv_cache_write(bits16(w.k_all), bits16(w.v_all), w.all_slots.numpy(), okc, ovc,
                                 kv_dtype=0, scale_mode=scale_mode, k_scale=w.k_scale.numpy(),
                                 v_scale=w.v_scale.numpy(), k_scale_cache=oks,
                                 v_scale_cache=ovs) == 0
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    if scale_mode == 2:
        assert np.array_equal(ksc.cpu().numpy().view(np.uint32), oks.view(np.uint32))
        return (kc, vc, ks, vs, ksc, vsc), (okc, ovc, oks, ovs)
    return (kc, vc, ks, vs, None, None), (okc, ovc, None, None)


def _gpu(w, dev_c, scale_mode=0, two_level=False, **kw):
    kc, vc, ks, vs, ksc, vsc = dev_c
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fk.prefill_attn(w.q.cuda(), w.cu_seqlens_q.cuda(), w.max_seqlen_q, kc, vc,
                          w.block_table.cuda(), w.context_lens.cuda(), kv_dtype=0,
                          scale_mode=scale_mode, k_scale=ks, v_scale=vs, k_scale_cache=ksc,
                          v_scale_cache=vsc, two_level=two_level, err_flag=err, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    return out


def _oracle(w, host_c, units, scale_mode=0):
    okc, ovc, oks, ovs = host_c
    st, ref = oracle.prefill_attn(bits16(w.q), w.cu_seqlens_q.numpy(), okc, ovc,
                                  w.block_table.numpy(), w.context_lens.numpy(), kv_dtype=0,
                                  scale_mode=scale_mode, k_scale=w.k_scale.numpy(),
                                  v_scale=w.v_scale.numpy(), k_scale_cache=oks,
                                  v_scale_cache=ovs, units=units, nthreads=16)
    assert st == 0
    return ref


def _rows(w, every=1):
    Tq, Hq = w.q.shape[0], w.Hq
    return [(t, h) for t in range(0, Tq, every) for h in range(Hq)]


def _n_keys(w, t):
    cu = w.cu_seqlens_q.numpy()
    b = int(np.searchsorted(cu, t, side="right") - 1)
    nq = cu[b + 1] - cu[b]
    return int(w.context_lens[b]) - nq + (t - cu[b]) + 1


def _max_err(w, out, ref, units):
    got = np.stack([out[t, h] for t, h in units])
    return float(np.abs(got - ref).max())


@pytest.mark.parametrize("two_level", [False, True])
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 8, 1), (128, 8, 2), (128, 4, 4), (256, 16, 1)])
def test_prefill_parity_long_context(two_level, D, Hq, Hkv):
    w = synth.prefill(seed=300 + D + Hq, ctx=(4100, 6001), chunk=(123, 300), Hq=Hq, Hkv=Hkv,
                      D=D)
    dev_c, host_c = _caches(w)
    out = _gpu(w, dev_c, two_level=two_level).cpu().numpy()
    units = _rows(w, 5)
    ref = _oracle(w, host_c, units)
    got = np.stack([out[t, h] for t, h in units])
    err = float(np.abs(got - ref).max())
    assert err <= PREFILL_TOL, err


@pytest.mark.parametrize("two_level", [False, True])
def test_prefill_parity_short_context(two_level):
    w = synth.prefill(seed=305, ctx=(700, 1301, 17), chunk=(123, 300, 17), Hq=8, Hkv=2, D=128)
    dev_c, host_c = _caches(w)
    out = _gpu(w, dev_c, two_level=two_level).cpu().numpy()
    units = _rows(w, 2)
    ref = _oracle(w, host_c, units)
    err = _max_err(w, out, ref, units)
    assert err <= PREFILL_TOL, err


@pytest.mark.parametrize("two_level", [False, True])
def test_prefill_single_operands_on_long_rows(two_level):
    # every row sees >= 8192 keys: single e4m3 operands (the automatic choice)
    w = synth.prefill(seed=307, ctx=(9000, 12500), chunk=(300, 200), Hq=8, Hkv=2, D=128)
    dev_c, host_c = _caches(w)
    auto = _gpu(w, dev_c, two_level=two_level)
    never = _gpu(w, dev_c, two_level=two_level, split="never")
    assert torch.equal(auto, never)
    units = _rows(w, 3)
    ref = _oracle(w, host_c, units)
    err = _max_err(w, auto.cpu().numpy(), ref, units)
    assert err <= PREFILL_TOL, err
    # split operands on the same rows: within the bar and closer to the oracle
    always = _gpu(w, dev_c, two_level=two_level, split="always").cpu().numpy()
    err_split = _max_err(w, always, ref, units)
    assert err_split <= PREFILL_TOL and err_split < err, (err_split, err)


def test_prefill_q_and_prob_scales():
    # single operands with q_scale 1/2 and prob_scale 2: Q and the weights are
    # stored as e4m3(q / q_scale) and e4m3(p / prob_scale); the scales cancel in
    # the result, which still matches the oracle
    w = synth.prefill(seed=308, ctx=(9000,), chunk=(256,), Hq=8, Hkv=1, D=256)
    dev_c, host_c = _caches(w)
    plain = _gpu(w, dev_c, split="never")
    scaled = _gpu(w, dev_c, split="never", q_scale=0.5, prob_scale=2.0)
    units = _rows(w, 4)
    ref = _oracle(w, host_c, units)
    err = _max_err(w, scaled.cpu().numpy(), ref, units)
    assert err <= PREFILL_TOL, err
    assert float((scaled - plain).abs().max()) <= PREFILL_TOL


@pytest.mark.parametrize("two_level", [False, True])
@pytest.mark.parametrize("scale_mode", [0, 2])
@pytest.mark.parametrize("Hq,Hkv", [(8, 1), (64, 8)])
def test_prefill_head_dim_64(two_level, scale_mode, Hq, Hkv):
    # head_dim 64 ("커널 및 퓨전 최적화": prefill tiling for head_dim 64): 64-byte
    # e4m3 rows; rows under 8192 keys take split operands, the 9000-key sequence
    # single ones
    w = synth.prefill(seed=410 + Hq + scale_mode, ctx=(700, 9000, 33), chunk=(123, 160, 33),
                      Hq=Hq, Hkv=Hkv, D=64)
    dev_c, host_c = _caches(w, scale_mode=scale_mode)
    out = _gpu(w, dev_c, scale_mode=scale_mode, two_level=two_level).cpu().numpy()
    units = _rows(w, 3) if Hq == 8 else [(t, h) for t, h in _rows(w, 3) if h % 7 == 0]
    ref = _oracle(w, host_c, units, scale_mode=scale_mode)
    err = _max_err(w, out, ref, units)
    assert err <= PREFILL_TOL, err


def test_prefill_with_prequantized_q_isolates_p_rounding():
    # Single operands.  Feed the oracle the e4m3-rounded queries (its own
    # encoder, q_scale 1): the exact attention of those queries differs from
    # the kernel only by the rounding of P, ~1e-3 standard deviation at 5 000 keys.
    w = synth.prefill(seed=306, ctx=(5000,), chunk=(200,), Hq=8, Hkv=1, D=256)
    dev_c, host_c = _caches(w)
    out = _gpu(w, dev_c, split="never").cpu().numpy()
    qv = w.q.float().numpy()
    q8 = oracle.e4m3_decode(oracle.e4m3_encode(qv)).astype(np.float32)
    wq = synth.prefill(seed=306, ctx=(5000,), chunk=(200,), Hq=8, Hkv=1, D=256)
    wq.q = torch.from_numpy(q8).to(torch.bfloat16)        # e4m3 values are exact in bf16
    assert torch.equal(wq.q.float(), torch.from_numpy(q8))
    units = _rows(w, 4)
    ref_q8 = _oracle(wq, host_c, units)
    ref = _oracle(w, host_c, units)
    got = np.stack([out[t, h] for t, h in units])
    e_q8, e_raw = float(np.abs(got - ref_q8).max()), float(np.abs(got - ref).max())
    assert e_q8 <= 6e-3, (e_q8, e_raw)
    assert e_q8 <= e_raw


def test_two_level_on_and_off_agree():
    w = synth.prefill(seed=310, ctx=(3000,), chunk=(256,), Hq=8, Hkv=1, D=256)
    dev_c, _ = _caches(w)
    off = _gpu(w, dev_c, two_level=False)
    on = _gpu(w, dev_c, two_level=True)
    assert torch.isfinite(off).all() and torch.isfinite(on).all()
    # both sum the same e4m3 products in fp32, in a different order
    assert float((off - on).abs().max()) <= 1e-4


def test_prefill_per_head_scales():
    w = synth.prefill(seed=320, ctx=(5000,), chunk=(200,), Hq=8, Hkv=2, D=128)
    w.k_scale = synth.per_head_calibration(w.k_all)
    w.v_scale = synth.per_head_calibration(w.v_all)
    dev_c, host_c = _caches(w, scale_mode=1)
    out = _gpu(w, dev_c, scale_mode=1).cpu().numpy()
    units = _rows(w, 4)
    ref = _oracle(w, host_c, units, scale_mode=1)
    got = np.stack([out[t, h] for t, h in units])
    assert float(np.abs(got - ref).max()) <= PREFILL_TOL


def _with_outliers(w, seed, frac=0.01, factor=20.0):
    """1 % of the (KV head, channel) pairs of every token scaled x20 in K and V (the
    outlier channels per-token-head scales are for), plus 5 % of the tokens'
    values x8 so that the V scales of a tile differ by up to 8x."""
    g = torch.Generator().manual_seed(seed)
    Hkv, D = w.Hkv, w.D
    n = max(1, int(np.ceil(frac * Hkv * D)))
    idx = torch.randperm(Hkv * D, generator=g)[:n]
    for t in (w.k_all, w.v_all):
        for i in idx.tolist():
            h, c = divmod(i, D)
            t[:, h, c] = (t[:, h, c].float() * factor).to(torch.bfloat16)
    loud = torch.randperm(w.v_all.shape[0], generator=g)[: w.v_all.shape[0] // 20]
    w.v_all[loud] = (w.v_all[loud].float() * 8.0).to(torch.bfloat16)
    return w


def _loud_values(w, seed, frac=0.05, factor=8.0):
    """5 % of the tokens' values x8: their per-token-head V scales are 8x the
    others', so the running V-scale bound grows and most weights sit 8x under it."""
    g = torch.Generator().manual_seed(seed)
    loud = torch.randperm(w.v_all.shape[0], generator=g)[: int(w.v_all.shape[0] * frac)]
    w.v_all[loud] = (w.v_all[loud].float() * factor).to(torch.bfloat16)
    return w


@pytest.mark.parametrize("two_level", [False, True])
@pytest.mark.parametrize("D,Hq,Hkv", [(256, 8, 1), (128, 8, 2)])
def test_prefill_per_token_head_long_context(two_level, D, Hq, Hkv):
    # The error model above with the values' rms in place of 1 (the loud tokens
    # raise it to ~2): rounding P to e4m3 is the only approximation, per row.
    w = _loud_values(synth.prefill(seed=360 + D, ctx=(4100, 6001), chunk=(123, 300), Hq=Hq,
                                   Hkv=Hkv, D=D), 361 + D)
    dev_c, host_c = _caches(w, scale_mode=2)
    out = _gpu(w, dev_c, scale_mode=2, two_level=two_level).cpu().numpy()
    units = _rows(w, 5)
    ref = _oracle(w, host_c, units, scale_mode=2)
    err = _max_err(w, out, ref, units)
    assert err <= PREFILL_TOL, err


@pytest.mark.parametrize("two_level", [False, True])
def test_prefill_per_token_head_short_context(two_level):
    w = synth.prefill(seed=370, ctx=(700, 1301, 17), chunk=(123, 300, 17), Hq=8, Hkv=2, D=128)
    dev_c, host_c = _caches(w, scale_mode=2)
    out = _gpu(w, dev_c, scale_mode=2, two_level=two_level).cpu().numpy()
    units = _rows(w, 2)
    ref = _oracle(w, host_c, units, scale_mode=2)
    err = _max_err(w, out, ref, units)
    assert err <= PREFILL_TOL, err


@pytest.mark.parametrize("two_level", [False, True])
def test_prefill_per_token_head_outliers(two_level):
    # x20 (head, channel) pairs in K and V plus x8 loud value tokens: the values
    # reach ~500 and the logits spread ~3x wider than N(0,1) data.  Errors scale
    # with the values, so each output channel is compared in units of that
    # channel's value rms (1 for the N(0,1) data the 1e-2 bar is stated for).
    w = _with_outliers(synth.prefill(seed=375, ctx=(700, 3001, 17), chunk=(123, 300, 17), Hq=8,
                                     Hkv=1, D=256), 376)
    dev_c, host_c = _caches(w, scale_mode=2)
    out = _gpu(w, dev_c, scale_mode=2, two_level=two_level).cpu().numpy()
    units = _rows(w, 2)
    ref = _oracle(w, host_c, units, scale_mode=2)
    got = np.stack([out[t, h] for t, h in units])
    okc, ovc, oks, ovs = host_c
    vdq = oracle.e4m3_decode(ovc).astype(np.float64) * ovs[..., None]   # [nb][Hkv][16][D]
    used = np.zeros(ovc.shape[:3], bool)
    slots = w.all_slots.numpy()
    used[slots // 16, :, slots % 16] = True
    rms = np.sqrt((vdq[used] ** 2).mean(axis=0))                          # [D]
    rel = float((np.abs(got - ref) / rms[None, :]).max())
    print(f"per-token-head outliers two_level={two_level}: max-abs "
          f"{float(np.abs(got - ref).max()):.4f}, max in value-rms units {rel:.5f}")
    assert rel <= PREFILL_TOL, rel


@pytest.mark.parametrize("scale_mode", [0, 2])
def test_prefill_error_by_key_count(scale_mode):
    # N(0,1) data: the largest error in each band of key counts, automatic operand
    # choice against single operands forced (printed as a table; run with -s)
    ctx = (16, 64, 256, 1024, 4096, 8190, 12000)
    chunk = (16, 64, 200, 300, 300, 300, 300)
    w = synth.prefill(seed=395 + scale_mode, ctx=ctx, chunk=chunk, Hq=8, Hkv=1, D=128)
    dev_c, host_c = _caches(w, scale_mode=scale_mode)
    units = _rows(w, 3)
    ref = _oracle(w, host_c, units, scale_mode=scale_mode)
    keys = np.array([_n_keys(w, t) for t, _ in units])
    bands = [(1, 16), (17, 64), (65, 256), (257, 1024), (1025, 4096), (4097, 8191),
             (8192, 12000)]
    rows = {}
    for split in ("auto", "never", "always"):
        out = _gpu(w, dev_c, scale_mode=scale_mode, split=split).cpu().numpy()
        got = np.stack([out[t, h] for t, h in units])
        e = np.abs(got - ref).max(axis=1)
        rows[split] = [float(e[(keys >= lo) & (keys <= hi)].max()) for lo, hi in bands]
    print(f"\nmax-abs error by keys per row (scale_mode {scale_mode}, D 128, N(0,1)):")
    print("keys        " + " ".join(f"{lo:>5}-{hi:<5}" for lo, hi in bands))
    for split, r in rows.items():
        print(f"{split:<11} " + " ".join(f"{x:11.2e}" for x in r))
    assert max(rows["auto"]) <= PREFILL_TOL
    assert max(rows["always"]) <= PREFILL_TOL


def test_prefill_per_token_head_two_level_agree():
    w = _with_outliers(synth.prefill(seed=380, ctx=(3000,), chunk=(256,), Hq=8, Hkv=1, D=256),
                       381)
    dev_c, _ = _caches(w, scale_mode=2)
    off = _gpu(w, dev_c, scale_mode=2, two_level=False)
    on = _gpu(w, dev_c, scale_mode=2, two_level=True)
    assert torch.isfinite(off).all() and torch.isfinite(on).all()
    scale = max(1.0, float(off.abs().max()))
    assert float((off - on).abs().max()) <= 1e-4 * scale


def test_prefill_per_token_head_stale_scales_do_not_leak():
    # scale slots past ctx on the last page hold NaN / inf: never read for a
    # logit, never in the V-scale bound
    w = synth.prefill(seed=390, ctx=(1000,), chunk=(40,), Hq=8, Hkv=1, D=256)
    dev_c, _ = _caches(w, scale_mode=2)
    clean = _gpu(w, dev_c, scale_mode=2).clone()
    kc, vc, ks, vs, ksc, vsc = dev_c
    last_blk = int(w.block_table[0, (1000 - 1) // 16])
    ksc[last_blk, :, 1000 % 16:] = float("nan")
    vsc[last_blk, :, 1000 % 16:] = float("inf")
    kc[last_blk, :, 1000 % 16:] = 0x7F
    vc[last_blk, :, 1000 % 16:] = 0x7F
    dirty = _gpu(w, dev_c, scale_mode=2)
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)


def test_prefill_config5_full_size_sampled():
    # 4096 new queries at positions 28672..32767 of a 32768-token e4m3 cache,
    # 8 query heads / 1 KV head, head_dim 256, per-tensor 1.0, both switch settings
    w = synth.prefill()
    dev_c, host_c = _caches(w)
    units = [(t, h) for t in list(range(0, 4096, 97)) + [4095] for h in range(8)]
    ref = _oracle(w, host_c, units)
    for two_level in (False, True):
        out = _gpu(w, dev_c, two_level=two_level).cpu().numpy()
        got = np.stack([out[t, h] for t, h in units])
        err = float(np.abs(got - ref).max())
        assert err <= PREFILL_TOL, (two_level, err)


def test_prefill_after_full_prefix_sampled():
    # the other reading of the chunked-prefill workload: 4096 new queries after a
    # complete 32768-token prefix (positions 32768..36863 of a 36864-token cache)
    w = synth.prefill(seed=1015, ctx=(36864,), chunk=(4096,))
    dev_c, host_c = _caches(w)
    units = [(t, h) for t in list(range(0, 4096, 257)) + [4095] for h in range(8)]
    ref = _oracle(w, host_c, units)
    out = _gpu(w, dev_c).cpu().numpy()
    got = np.stack([out[t, h] for t, h in units])
    assert float(np.abs(got - ref).max()) <= PREFILL_TOL


def test_unwritten_tail_slots_do_not_leak():
    # the last page of the sequence holds NaN codes past ctx
    w = synth.prefill(seed=330, ctx=(1000,), chunk=(40,), Hq=8, Hkv=1, D=256)
    dev_c, _ = _caches(w)
    clean = _gpu(w, dev_c).clone()
    kc, vc, ks, vs, _, _ = dev_c
    last_blk = int(w.block_table[0, (1000 - 1) // 16])
    kc[last_blk, :, 1000 % 16:] = 0x7F
    vc[last_blk, :, 1000 % 16:] = 0x7F
    dirty = _gpu(w, (kc, vc, ks, vs, None, None))
    assert torch.isfinite(dirty).all()
    assert torch.equal(clean, dirty)


def test_uncalibrated_scales_warn():
    w = synth.prefill(seed=340, ctx=(300,), chunk=(20,), Hq=8, Hkv=1, D=128)
    dev_c, _ = _caches(w)
    _gpu(w, dev_c)
    assert "uncalibrated" in fk.last_warning()
    _gpu(w, dev_c, q_scale=0.5, prob_scale=0.25)
    assert fk.last_warning() == ""


def test_bf16_output_close_to_fp32():
    w = synth.prefill(seed=350, ctx=(600,), chunk=(64,), Hq=8, Hkv=1, D=256)
    dev_c, _ = _caches(w)
    a = _gpu(w, dev_c)
    b = _gpu(w, dev_c, out_dtype=fk.OUT_BF16).float()
    assert float((a - b).abs().max()) <= 2 ** -8 * max(1.0, float(a.abs().max()))


def _bf16_caches(w):
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    fk.kv_cache_write(w.k_all.cuda(), w.v_all.cuda(), w.all_slots.cuda(), kc, vc, kv_dtype=1)
    okc = np.zeros((nb, Hkv, 16, D), np.uint16)
    ovc = np.zeros_like(okc)
    assert oracle.kv_cache_write(bits16(w.k_all), bits16(w.v_all), w.all_slots.numpy(), okc, ovc,
                                 kv_dtype=1) == 0
    return kc, vc, okc, ovc


@pytest.mark.parametrize("two_level", [False, True])
@pytest.mark.parametrize("D,Hq,Hkv,ctx,chunk", [(256, 8, 1, (4100, 700), (123, 300)),
                                                 (128, 8, 2, (5000, 33), (200, 33)),
                                                 (64, 64, 8, (3000, 17), (150, 17))])
def test_bf16_twin_parity(two_level, D, Hq, Hkv, ctx, chunk):
    # The bf16 twin keeps Q in bf16 and rounds P to bf16 (8 mantissa bits), so it
    # meets the 1e-2 bar at every context length.
    w = synth.prefill(seed=360 + D, ctx=ctx, chunk=chunk, Hq=Hq, Hkv=Hkv, D=D)
    kc, vc, okc, ovc = _bf16_caches(w)
    err_flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fk.prefill_attn(w.q.cuda(), w.cu_seqlens_q.cuda(), w.max_seqlen_q, kc, vc,
                          w.block_table.cuda(), w.context_lens.cuda(), kv_dtype=1,
                          two_level=two_level, err_flag=err_flag).cpu().numpy()
    torch.cuda.synchronize()
    assert int(err_flag.item()) == 0
    units = _rows(w, 3)
    st, ref = oracle.prefill_attn(bits16(w.q), w.cu_seqlens_q.numpy(), okc, ovc,
                                  w.block_table.numpy(), w.context_lens.numpy(), kv_dtype=1,
                                  units=units, nthreads=16)
    assert st == 0
    got = np.stack([out[t, h] for t, h in units])
    err = float(np.abs(got - ref).max())
    assert err <= PREFILL_TOL, err
    assert fk.last_warning() == ""
