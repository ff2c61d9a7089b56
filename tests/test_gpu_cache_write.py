"""GPU parity of kv_cache_write and the e4m3 encoder: bit-exact against the oracle.

Cache codes and stored per-token-head scales must equal the oracle's byte for
byte (scale = fp32(amax / 448), code = e4m3_rn_satfinite(fp32(x / scale)); "[vLLM]
KV Cache Quantization: KV 캐시 FP8/INT8 양자화", section "Per-Token-Head vs Per-Tensor
양자화").  The encoder is also swept over every fp32 bit pattern.
"""
import concurrent.futures as cf

import numpy as np
import pytest
import torch

import oracle
import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._helpers import bits16
from tests._parity import assert_same_cache, gpu_fill, oracle_cache

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("kv_dtype,mode", [(0, 0), (0, 1), (0, 2), (1, 0)])
def test_cache_write_bit_exact(D, kv_dtype, mode):
    w = synth.decode_workload(11 + D, [1, 15, 16, 17, 300, 1000], 8, 4, D, mode,
                              outlier_frac=0.01, spare_blocks=5)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc = gpu_fill(w, kv_dtype, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_same_cache(gc, oracle_cache(w, kv_dtype))


def test_llama_shaped_bulk_fill_bit_exact():
    # Llama-3.1-8B-shaped cache fill: 8 KV heads, D 128, outlier channels x20.
    w = synth.llama8b(seed=21, B=2, ctx_lo=3000, ctx_hi=5000)
    assert_same_cache(gpu_fill(w, 0), oracle_cache(w, 0))


def test_zero_rows_negative_slots_and_untouched_bytes():
    T, Hkv, D, nb = 40, 2, 128, 6
    g = torch.Generator().manual_seed(3)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    k[5] = 0                                              # all-zero rows: scale 0, codes 0
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[::7] = -1                                       # padding tokens are skipped
    kc = torch.full((nb, Hkv, 16, D), 0x5A, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ks = torch.full((nb, Hkv, 16), -3.0, device="cuda")
    vs = ks.clone()
    fk.kv_cache_write(k.cuda(), v.cuda(), slots.cuda(), kc, vc, kv_dtype=0, scale_mode=2,
                      k_scale_cache=ks, v_scale_cache=vs)
    okc = np.full((nb, Hkv, 16, D), 0x5A, np.uint8)
    ovc = okc.copy()
    oks = np.full((nb, Hkv, 16), -3.0, np.float32)
    ovs = oks.copy()
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots.numpy(), okc, ovc, kv_dtype=0,
                                 scale_mode=2, k_scale_cache=oks, v_scale_cache=ovs) == 0
    assert np.array_equal(kc.cpu().numpy(), okc) and np.array_equal(vc.cpu().numpy(), ovc)
    assert np.array_equal(ks.cpu().numpy(), oks) and np.array_equal(vs.cpu().numpy(), ovs)
    blk, off = divmod(int(slots[5]), 16)
    if int(slots[5]) >= 0:
        assert np.all(okc[blk, :, off] == 0) and np.all(oks[blk, :, off] == 0)


def test_slot_outside_cache_sets_error_and_skips():
    T, Hkv, D, nb = 4, 1, 64, 2
    k = torch.randn(T, Hkv, D).to(torch.bfloat16).cuda()
    slots = torch.tensor([0, 32, 5, 1 << 40], dtype=torch.int64, device="cuda")
    kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    one = torch.ones(1, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fk.kv_cache_write(k, k, slots, kc, vc, kv_dtype=0, scale_mode=0, k_scale=one, v_scale=one,
                      err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == -6
    want = oracle.e4m3_encode(k.float().cpu().numpy())
    assert np.array_equal(kc[0, 0, 0].cpu().numpy(), want[0, 0])
    assert np.array_equal(kc[0, 0, 5].cpu().numpy(), want[2, 0])


def _oracle_encode_parallel(x: np.ndarray, workers=16) -> np.ndarray:
    out = np.empty(x.shape, np.uint8)
    n = x.size
    step = (n + workers - 1) // workers

    def run(i):
        lo, hi = i * step, min(n, (i + 1) * step)
        out[lo:hi] = oracle.e4m3_encode(x[lo:hi])

    with cf.ThreadPoolExecutor(workers) as ex:
        list(ex.map(run, range(workers)))
    return out


def test_encoder_matches_oracle_on_every_fp32_pattern():
    # All 2^32 fp32 bit patterns through the device encoder (scale 1), against
    # the oracle's integer-arithmetic encoder.  NaN inputs stay NaN codes on both
    # sides (the sign of a NaN code is not compared).
    chunk = 1 << 28
    for start in range(0, 1 << 32, chunk):
        bits = torch.arange(start, start + chunk, dtype=torch.int64, device="cuda")
        bits = torch.where(bits >= 1 << 31, bits - (1 << 32), bits).to(torch.int32)
        x = bits.view(torch.float32)
        got = fk.quantize_e4m3(x, 1.0).cpu().numpy()
        xh = x.cpu().numpy()
        want = _oracle_encode_parallel(xh)
        nan = np.isnan(xh)
        assert np.array_equal(got[~nan], want[~nan]), f"chunk at {start:#x}"
        assert np.all((got[nan] & 0x7F) == 0x7F)
        del bits, x


@pytest.mark.parametrize("scale", [0.37, 1.0 / 448, 3.0e-3, 17.5])
def test_encoder_with_scales_matches_oracle(scale):
    g = torch.Generator().manual_seed(5)
    x = torch.randn(1 << 20, generator=g) * 10
    got = fk.quantize_e4m3(x.cuda(), scale).cpu().numpy()
    q = (x.numpy().astype(np.float32) / np.float32(scale)).astype(np.float32)
    assert np.array_equal(got, oracle.e4m3_encode(q))


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("Hkv", [3, 8])
@pytest.mark.parametrize("kv_dtype,mode", [(0, 0), (0, 1), (0, 2), (1, 0)])
def test_bulk_write_bit_exact(D, Hkv, kv_dtype, mode):
    # Bulk writes (T * Hkv >= 8192 rows, device inputs) go through the
    # shared-memory staged kernel: chunked rows, ragged last chunk, a head count
    # that is not a power of two, padding slots, all-zero rows, a x20 outlier
    # channel and bytes outside the written slots left untouched.
    T = 3000 if Hkv == 3 else 1100
    nb = T // 16 + 9
    g = torch.Generator().manual_seed(40 + D + Hkv + 7 * mode + 11 * kv_dtype)
    k = torch.randn(T, Hkv, D, generator=g)
    v = torch.randn(T, Hkv, D, generator=g)
    k[:, 0, 5] *= 20
    v[:, Hkv - 1, D - 1] *= 20
    k[17] = 0
    v[T - 2, 0] = 0
    k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    slots[3::97] = -1
    dt = torch.uint8 if kv_dtype == 0 else torch.bfloat16
    kc = torch.full((nb, Hkv, 16, D), 0x5A, dtype=torch.uint8, device="cuda").view(dt) \
        if kv_dtype == 0 else torch.full((nb, Hkv, 16, D), 7.0, dtype=dt, device="cuda")
    vc = kc.clone()
    ks = torch.full((nb, Hkv, 16), -3.0, device="cuda")
    vs = ks.clone()
    ksc = vsc = None
    if kv_dtype == 0 and mode == 0:
        ksc, vsc = torch.tensor([0.37]), torch.tensor([3.0e-3])
    elif kv_dtype == 0 and mode == 1:
        ksc = torch.rand(Hkv, generator=g) * 0.05 + 1e-3
        vsc = torch.rand(Hkv, generator=g) * 0.05 + 1e-3
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fk.kv_cache_write(k.cuda(), v.cuda(), slots.cuda(), kc, vc, kv_dtype=kv_dtype, scale_mode=mode,
                      k_scale=None if ksc is None else ksc.cuda(),
                      v_scale=None if vsc is None else vsc.cuda(),
                      k_scale_cache=ks, v_scale_cache=vs, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    if kv_dtype == 0:
        okc = np.full((nb, Hkv, 16, D), 0x5A, np.uint8)
    else:
        okc = np.full((nb, Hkv, 16, D), bits16(torch.tensor([7.0]).to(torch.bfloat16))[0],
                      np.uint16)
    ovc = okc.copy()
    oks = np.full((nb, Hkv, 16), -3.0, np.float32)
    ovs = oks.copy()
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots.numpy(), okc, ovc,
                                 kv_dtype=kv_dtype, scale_mode=mode,
                                 k_scale=None if ksc is None else ksc.numpy(),
                                 v_scale=None if vsc is None else vsc.numpy(),
                                 k_scale_cache=oks, v_scale_cache=ovs) == 0
    view = (lambda t: t.cpu().numpy()) if kv_dtype == 0 else \
        (lambda t: t.view(torch.int16).cpu().numpy().view(np.uint16))
    assert np.array_equal(view(kc), okc), "K cache bytes differ"
    assert np.array_equal(view(vc), ovc), "V cache bytes differ"
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))


def test_encoder_every_bf16_value_under_many_scales():
    # Every finite bf16 value divided by 256 scales spread over the whole fp32
    # range (tiny, subnormal, huge, negative, amax/448-shaped), through the
    # writer's quantizer, against the oracle's encoder of numpy's IEEE fp32
    # quotient.  NaN quotients are left out (their sign is not compared).
    allbf = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    allbf = allbf[np.isfinite(allbf)]
    rng = np.random.default_rng(9)
    scales = np.concatenate([
        np.float32([1.0, 448.0, 1.0 / 448, -0.37, 2.0 ** -149, 2.0 ** -130, 2.0 ** -127,
                    2.0 ** 126, 3 * 2.0 ** 125, np.finfo(np.float32).max, 1e-30, 3.0e38]),
        (np.abs(rng.standard_normal(180)) * 10.0 ** rng.uniform(-44, 38, 180)).astype(np.float32),
        ((rng.integers(1, 0x7f80, 64, dtype=np.uint32) << 16).view(np.float32)
         / np.float32(448)).astype(np.float32)])
    xd = torch.from_numpy(allbf).cuda()
    for s in scales:
        s = np.float32(s)
        if not np.isfinite(s) or s == 0:
            continue
        got = fk.quantize_e4m3(xd, float(s)).cpu().numpy()
        with np.errstate(all="ignore"):
            q = (allbf / s).astype(np.float32)
        keep = ~np.isnan(q)
        want = oracle.e4m3_encode(q)
        assert np.array_equal(got[keep], want[keep]), f"scale {s!r}"


def test_bulk_write_from_pinned_host_memory():
    # A bulk write whose K / V live in pinned host memory takes the plain-load
    # kernel (read over the host link) and must give the same bytes as from
    # device memory and as the oracle.
    T, Hkv, D = 4096, 8, 128
    nb = T // 16 + 3
    g = torch.Generator().manual_seed(77)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    slots = torch.randperm(nb * 16, generator=g)[:T].to(torch.int64)
    outs = []
    for kin, vin in ((k.pin_memory(), v.pin_memory()), (k.cuda(), v.cuda())):
        kc = torch.zeros(nb, Hkv, 16, D, dtype=torch.uint8, device="cuda")
        vc = torch.zeros_like(kc)
        ks = torch.zeros(nb, Hkv, 16, device="cuda")
        vs = torch.zeros_like(ks)
        fk.kv_cache_write(kin, vin, slots.cuda(), kc, vc, kv_dtype=0, scale_mode=2,
                          k_scale_cache=ks, v_scale_cache=vs)
        torch.cuda.synchronize()
        outs.append([t.cpu().numpy() for t in (kc, vc, ks, vs)])
    okc = np.zeros((nb, Hkv, 16, D), np.uint8)
    ovc = okc.copy()
    oks = np.zeros((nb, Hkv, 16), np.float32)
    ovs = oks.copy()
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots.numpy(), okc, ovc, kv_dtype=0,
                                 scale_mode=2, k_scale_cache=oks, v_scale_cache=ovs) == 0
    for got in outs:
        assert np.array_equal(got[0], okc) and np.array_equal(got[1], ovc)
        assert np.array_equal(got[2].view(np.uint32), oks.view(np.uint32))
        assert np.array_equal(got[3].view(np.uint32), ovs.view(np.uint32))


@pytest.mark.parametrize("path", ["staged", "direct"])
@pytest.mark.parametrize("D", [64, 256])
def test_scale_of_every_bf16_row_maximum(path, D):
    # Per-token-head scales: every finite non-negative bf16 value (0, subnormals,
    # up to the largest) is the max |x| of some K row, plus one row whose maximum
    # is +inf and rows holding NaN (which the maximum ignores).  Stored scales
    # must be fp32(amax / 448) bit for bit and the codes the oracle's, through
    # the staged kernel (one bulk call) and the plain-load kernel (calls of
    # fewer than 8192 rows).
    amax = (np.arange(0x7f80, dtype=np.uint32) << 16).view(np.float32)
    rng = np.random.default_rng(D)
    n = amax.size
    x = amax[:, None].astype(np.float64) * rng.uniform(-1.0, 1.0, (n, D))
    col = rng.integers(0, D, n)
    x[np.arange(n), col] = amax * np.where(rng.random(n) < 0.5, -1.0, 1.0)
    extra = rng.standard_normal((3, D))
    extra[0, 7] = np.inf                         # infinite maximum: scale +inf
    extra[1, 9] = np.nan                         # NaN ignored by the maximum
    extra[2, ::5] = np.nan
    x = np.concatenate([x, extra])
    T = x.shape[0]
    k = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).reshape(T, 1, D)
    v = k.flip(0).contiguous()
    nb = (T + 15) // 16
    slots = torch.randperm(nb * 16, generator=torch.Generator().manual_seed(D))[:T].to(torch.int64)
    kc = torch.zeros((nb, 1, 16, D), dtype=torch.uint8, device="cuda")
    vc = kc.clone()
    ks = torch.zeros((nb, 1, 16), device="cuda")
    vs = ks.clone()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    step = T if path == "staged" else 8000
    for a in range(0, T, step):
        fk.kv_cache_write(k[a:a + step].cuda(), v[a:a + step].cuda(), slots[a:a + step].cuda(),
                          kc, vc, kv_dtype=0, scale_mode=2, k_scale_cache=ks, v_scale_cache=vs,
                          err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    okc = np.zeros((nb, 1, 16, D), np.uint8)
    ovc = okc.copy()
    oks = np.zeros((nb, 1, 16), np.float32)
    ovs = oks.copy()
    assert oracle.kv_cache_write(bits16(k), bits16(v), slots.numpy(), okc, ovc, kv_dtype=0,
                                 scale_mode=2, k_scale_cache=oks, v_scale_cache=ovs) == 0
    assert np.array_equal(ks.cpu().numpy().view(np.uint32), oks.view(np.uint32))
    assert np.array_equal(vs.cpu().numpy().view(np.uint32), ovs.view(np.uint32))
    for got, want in ((kc.cpu().numpy(), okc), (vc.cpu().numpy(), ovc)):
        nan = (want & 0x7F) == 0x7F              # NaN codes: the sign is not compared
        assert np.array_equal(got[~nan], want[~nan])
        assert np.all((got[nan] & 0x7F) == 0x7F)
