"""GPU parity of the balanced (persistent) FP8 prefill against the float64 oracle.

With a workspace (fp8kv_prefill_attn_ws, the binding's default) a launch with
more query tiles than SMs runs one CTA per SM, each on an equal share of all
(query tile, key tile) work; query tiles cut between CTAs are finished by
merging fp32 partials (O, running max, running sum), as the split decode
merges its partials.  The bar is the one of
every prefill test: max-abs 1e-2 on fp32 output.  The workloads below have more
than 152 query tiles, mix rows under and over 8192 keys (split and single e4m3
operands in one launch) and ragged chunk lengths.
"""
import numpy as np
import pytest
import torch

import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests.test_gpu_prefill import (PREFILL_TOL, _bf16_caches, _caches, _max_err, _oracle,
                                    _rows, _with_outliers)
from tests._helpers import bits16

import oracle

pytestmark = pytest.mark.gpu


def _sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _q_tiles(w):
    tpt = 128 // (w.Hq // w.Hkv)
    cu = w.cu_seqlens_q.numpy()
    return int(sum((cu[b + 1] - cu[b] + tpt - 1) // tpt for b in range(len(cu) - 1))) * w.Hkv


def _run(w, dev_c, workspace, scale_mode=0, two_level=False, kv_dtype=0, **kw):
    kc, vc, ks, vs, ksc, vsc = dev_c
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = fk.prefill_attn(w.q.cuda(), w.cu_seqlens_q.cuda(), w.max_seqlen_q, kc, vc,
                          w.block_table.cuda(), w.context_lens.cuda(), kv_dtype=kv_dtype,
                          scale_mode=scale_mode, k_scale=ks, v_scale=vs, k_scale_cache=ksc,
                          v_scale_cache=vsc, two_level=two_level, err_flag=err,
                          workspace=workspace, **kw)
    torch.cuda.synchronize()
    assert int(err.item()) == 0, int(err.item())
    return out


def _workspace(D):
    return torch.zeros(fk.prefill_workspace_bytes(D), dtype=torch.uint8, device="cuda")


def _counters_zero(ws):
    n = _sm_count()
    return int(ws[: 4 * n].view(torch.int32).abs().sum()) == 0


# (D, Hq, Hkv, ctx, chunk): > 152 query tiles, rows under and over 8192 keys
_SHAPES = [
    (128, 16, 4, (2300, 4100, 9000, 700), (600, 900, 700, 300)),
    (256, 8, 1, (2300, 4100, 9000, 700), (600, 900, 700, 300)),
    (64, 64, 8, (3000, 9000, 33), (700, 500, 33)),
]


@pytest.mark.parametrize("two_level", [False, True])
@pytest.mark.parametrize("scale_mode", [0, 2])
@pytest.mark.parametrize("D,Hq,Hkv,ctx,chunk", _SHAPES)
def test_balanced_prefill_parity(two_level, scale_mode, D, Hq, Hkv, ctx, chunk):
    w = synth.prefill(seed=500 + D + scale_mode, ctx=ctx, chunk=chunk, Hq=Hq, Hkv=Hkv, D=D)
    assert _q_tiles(w) > _sm_count()
    dev_c, host_c = _caches(w, scale_mode=scale_mode)
    ws = _workspace(D)
    out = _run(w, dev_c, ws, scale_mode=scale_mode, two_level=two_level)
    assert _counters_zero(ws)
    units = _rows(w, 7) if Hq <= 16 else [(t, h) for t, h in _rows(w, 5) if h % 9 == 0]
    ref = _oracle(w, host_c, units, scale_mode=scale_mode)
    err = _max_err(w, out.cpu().numpy(), ref, units)
    assert err <= PREFILL_TOL, err
    # one CTA per query tile on the same inputs: the same bar
    grid = _run(w, dev_c, None, scale_mode=scale_mode, two_level=two_level)
    assert float((out - grid).abs().max()) <= PREFILL_TOL


def test_balanced_prefill_is_deterministic():
    # the split of the work and the merge order are fixed: repeated calls give
    # the same bits, and the counters are back to zero after each
    D, Hq, Hkv, ctx, chunk = _SHAPES[1]
    w = synth.prefill(seed=520, ctx=ctx, chunk=chunk, Hq=Hq, Hkv=Hkv, D=D)
    dev_c, _ = _caches(w)
    ws = _workspace(D)
    a = _run(w, dev_c, ws).clone()
    assert _counters_zero(ws)
    b = _run(w, dev_c, ws)
    assert _counters_zero(ws)
    assert torch.equal(a, b)


@pytest.mark.parametrize("split", ["auto", "always"])
def test_balanced_prefill_outliers_per_token_head(split):
    # x20 outlier channels and x8 loud value tokens, per-token-head scales, errors
    # in units of each channel's value rms.  Cutting query tiles into pieces must
    # not cost accuracy: per sequence, the balanced launch stays within the error
    # of one CTA per query tile.  (On this data neither meets 1e-2 everywhere:
    # rows of >= 8192 keys under the automatic choice take single e4m3 weights,
    # whose range loses the many small weights of heavy-tailed rows, ~0.3;
    # split operands reach ~1.5e-2.  Measured in the design notes.)
    w = _with_outliers(synth.prefill(seed=530, ctx=(2300, 4100, 9000), chunk=(900, 1100, 700),
                                     Hq=8, Hkv=1, D=256), 531)
    assert _q_tiles(w) > _sm_count()
    dev_c, host_c = _caches(w, scale_mode=2)
    units = _rows(w, 9)
    ref = _oracle(w, host_c, units, scale_mode=2)
    okc, ovc, oks, ovs = host_c
    vdq = oracle.e4m3_decode(ovc).astype(np.float64) * ovs[..., None]
    used = np.zeros(ovc.shape[:3], bool)
    slots = w.all_slots.numpy()
    used[slots // 16, :, slots % 16] = True
    rms = np.sqrt((vdq[used] ** 2).mean(axis=0))
    cu = w.cu_seqlens_q.numpy()
    seq = np.array([int(np.searchsorted(cu, t, side="right") - 1) for t, _ in units])

    def per_seq(ws):
        out = _run(w, dev_c, ws, scale_mode=2, split=split).cpu().numpy()
        got = np.stack([out[t, h] for t, h in units])
        rel = np.abs(got - ref) / rms[None, :]
        return [float(rel[seq == b].max()) for b in range(3)]

    balanced, grid = per_seq(_workspace(256)), per_seq(None)
    print(f"outliers, split={split}: balanced {balanced}, one CTA per tile {grid}")
    for e_b, e_g in zip(balanced, grid):
        assert e_b <= 1.5 * e_g + 1e-3, (balanced, grid)


@pytest.mark.parametrize("two_level", [False, True])
def test_balanced_prefill_bf16_twin_and_bf16_out(two_level):
    D, Hq, Hkv, ctx, chunk = _SHAPES[0]
    w = synth.prefill(seed=540, ctx=ctx, chunk=chunk, Hq=Hq, Hkv=Hkv, D=D)
    kc, vc, okc, ovc = _bf16_caches(w)
    dev_c = (kc, vc, None, None, None, None)
    out = _run(w, dev_c, _workspace(D), kv_dtype=1, two_level=two_level)
    units = _rows(w, 7)
    st, ref = oracle.prefill_attn(bits16(w.q), w.cu_seqlens_q.numpy(), okc, ovc,
                                  w.block_table.numpy(), w.context_lens.numpy(), kv_dtype=1,
                                  units=units, nthreads=16)
    assert st == 0
    err = _max_err(w, out.cpu().numpy(), ref, units)
    assert err <= PREFILL_TOL, err
    half = _run(w, dev_c, _workspace(D), kv_dtype=1, two_level=two_level,
                out_dtype=fk.OUT_BF16).float()
    assert float((half - out).abs().max()) <= 2 ** -8 * max(1.0, float(out.abs().max()))


def test_balanced_prefill_workspace_checks():
    D, Hq, Hkv, ctx, chunk = _SHAPES[1]
    w = synth.prefill(seed=550, ctx=ctx, chunk=chunk, Hq=Hq, Hkv=Hkv, D=D)
    dev_c, _ = _caches(w)
    small = torch.zeros(fk.prefill_workspace_bytes(D) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(fk.Fp8kvError) as e:
        _run(w, dev_c, small)
    assert e.value.status == -3                       # FP8KV_ERR_WORKSPACE
    # a launch with fewer query tiles than SMs ignores the workspace
    w2 = synth.prefill(seed=551, ctx=(3000,), chunk=(200,), Hq=8, Hkv=1, D=256)
    assert _q_tiles(w2) <= _sm_count()
    dev_c2, _ = _caches(w2)
    assert torch.equal(_run(w2, dev_c2, small), _run(w2, dev_c2, None))


def test_balanced_prefill_tile_cut_into_many_pieces():
    # one 60 000-key query tile beside 7 sequences of 25 short query tiles each
    # (the balanced launch takes at most 8 sequences): the long tile's key
    # tiles spread over ~60 CTAs, whose partials the last of them merges
    ctx = (60000,) + (400,) * 7
    chunk = (16,) + (400,) * 7
    w = synth.prefill(seed=560, ctx=ctx, chunk=chunk, Hq=8, Hkv=1, D=128)
    assert _q_tiles(w) > _sm_count()
    dev_c, host_c = _caches(w)
    ws = _workspace(128)
    out = _run(w, dev_c, ws)
    assert _counters_zero(ws)
    units = [(t, h) for t in range(16) for h in range(8)] + \
            [(t, h) for t in range(16, w.q.shape[0], 37) for h in (0, 5)]
    ref = _oracle(w, host_c, units)
    err = _max_err(w, out.cpu().numpy(), ref, units)
    assert err <= PREFILL_TOL, err
    grid = _run(w, dev_c, None)
    assert float((out - grid).abs().max()) <= PREFILL_TOL
