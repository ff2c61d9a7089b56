"""Host-side scale resolution (no GPU): the rules of [KVQ] "BaseKVCacheMethod"
(-1.0 = not loaded), "Per-Token-Head vs Per-Tensor 양자화", "Q/Prob 스케일과
FP8 Attention" and "스케일 통합 로직" (page "[vLLM] KV Cache Quantization: KV 캐시
FP8/INT8 양자화"), each case written out from the page's text."""
import math

import pytest

import fp8_kv_cache_write_gb300 as fk

E4, BF = fk.KV_E4M3, fk.KV_BF16
PT, PH, PTH = fk.SCALE_PER_TENSOR, fk.SCALE_PER_HEAD, fk.SCALE_PER_TOKEN_HEAD

pytestmark = pytest.mark.skipif(not __import__("os").path.exists(fk.LIB_PATH),
                                reason="libfp8kv.so not built")


def test_both_loaded_are_used_as_loaded():
    k, v, q, p = fk.resolve_scales(E4, PT, 0.5, 0.25, q_loaded=0.125, prob_loaded=0.0625)
    assert (k, v, q, p) == ([0.5], [0.25], 0.125, 0.0625)
    assert fk.last_warning() == ""


def test_nothing_loaded_defaults_to_one_and_warns():
    k, v, q, p = fk.resolve_scales(E4, PT, -1.0, -1.0)
    assert (k, v, q, p) == ([1.0], [1.0], 1.0, 1.0)
    assert "uncalibrated" in fk.last_warning()


def test_q_alone_uncalibrated_still_warns():
    fk.resolve_scales(E4, PT, 0.5, 0.5, q_loaded=-1.0, prob_loaded=0.25)
    assert "uncalibrated" in fk.last_warning()
    fk.resolve_scales(E4, PT, 0.5, 0.5, q_loaded=0.3, prob_loaded=-1.0)
    assert "uncalibrated" in fk.last_warning()


@pytest.mark.parametrize("kl,vl,want", [(0.3, -1.0, 0.3), (0.3, 0.0, 0.3), (0.75, -2.0, 0.75)])
def test_single_kv_scale_serves_both(kl, vl, want):
    k, v, _, _ = fk.resolve_scales(E4, PT, kl, vl, q_loaded=1.5, prob_loaded=1.5)
    assert k == [pytest.approx(want)] and v == k


@pytest.mark.parametrize("kl,vl", [(-1.0, 0.5), (0.0, -1.0), (0.0, 0.5), (0.0, 0.0)])
def test_single_scale_needs_a_positive_k(kl, vl):
    with pytest.raises(fk.Fp8kvError) as e:
        fk.resolve_scales(E4, PT, kl, vl)
    assert e.value.status == -1


def test_per_head_elementwise():
    k, v, _, _ = fk.resolve_scales(E4, PH, [0.5, -1.0, 0.25, 2.0], [0.125, -1.0, -1.0, 0.0],
                                   q_loaded=0.5, prob_loaded=0.5)
    assert k == [0.5, 1.0, 0.25, 2.0]
    assert v == [0.125, 1.0, 0.25, 2.0]


def test_per_head_one_bad_head_rejects_the_call():
    with pytest.raises(fk.Fp8kvError):
        fk.resolve_scales(E4, PH, [0.5, -1.0], [0.5, 0.5])


@pytest.mark.parametrize("dtype,mode", [(E4, PTH), (BF, PT), (BF, PH), (BF, PTH)])
def test_no_per_tensor_scale_to_resolve(dtype, mode):
    k, v, q, p = fk.resolve_scales(dtype, mode, 0.5, 0.5, q_loaded=0.25, prob_loaded=0.25)
    assert (k, v, q, p) == (None, None, 1.0, 1.0)
    assert fk.last_warning() == ""


def test_invalid_inputs():
    for args in [(E4, PT, math.nan, 0.5), (E4, PT, 0.5, math.nan), (E4, 7, 0.5, 0.5),
                 (5, PT, 0.5, 0.5), (E4, PT, [0.5, 0.5], [0.5, 0.5])]:
        with pytest.raises(fk.Fp8kvError):
            fk.resolve_scales(*args)
    with pytest.raises(fk.Fp8kvError):
        fk.resolve_scales(E4, PT, 0.5, 0.5, q_loaded=math.nan)
    with pytest.raises(ValueError):
        fk.resolve_scales(E4, PH, [0.5, 0.5], [0.5])
