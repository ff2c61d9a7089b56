"""The argument behind the cache writer's fast encoder, checked on the CPU.

The writer must store e4m3_rn_satfinite(fp32(x / s)) ("[vLLM] KV Cache
Quantization: KV 캐시 FP8/INT8 양자화", section "Per-Token-Head vs Per-Tensor
양자화").  Instead of dividing every value it multiplies x by two reciprocals,
r (1 - 2^-19) and r (1 + 2^-19), where r is within 2 ulps of 1 / s, and keeps
the code when both products encode alike (rounding to e4m3 is monotone, so the
IEEE quotient, which lies between them, has that code too); other pairs are
divided.  This restates that rule with numpy fp32 arithmetic (IEEE round to
nearest) and the oracle's encoder, with r perturbed to the ends of its error
bound, and checks it against the oracle's code of numpy's IEEE quotient.  The
GPU tests check the kernel itself; this pins the reasoning it relies on.
"""
import numpy as np

import oracle

enc = oracle.e4m3_encode


def _bracket_codes(x, s, rel):
    """Codes at both ends of the bracket with a reciprocal of relative error `rel`."""
    with np.errstate(all="ignore"):
        r = np.float32(np.float64(np.float32(1.0) / s) * (1.0 + rel))
        r_lo = np.float32(r * np.float32(1.0 - 2.0 ** -19))
        r_hi = np.float32(r * np.float32(1.0 + 2.0 ** -19))
        return enc((x * r_lo).astype(np.float32)), enc((x * r_hi).astype(np.float32))


def _check(x, scales, rel):
    accepted = 0
    for s in scales:
        s = np.float32(s)
        e = (int(s.view(np.uint32)) >> 23) & 0xFF
        if not 1 <= e <= 252:                     # the writer divides outside [2^-126, 2^126)
            continue
        lo, hi = _bracket_codes(x, s, rel)
        with np.errstate(all="ignore"):
            q = (x / s).astype(np.float32)
        want = enc(q)
        keep = (lo == hi) & ~np.isnan(q)
        assert np.array_equal(lo[keep], want[keep]), f"scale {s!r}, reciprocal error {rel}"
        accepted += int(keep.sum())
    return accepted


def test_bracket_codes_equal_quotient_codes_for_every_bf16_value():
    x = (np.arange(1 << 16, dtype=np.uint32) << 16).view(np.float32)
    x = x[np.isfinite(x)]
    rng = np.random.default_rng(12)
    scales = [1.0, 448.0, 1.0 / 448, -0.37, 2.0 ** -126, 2.0 ** 125.9, 1e-30, 3e37]
    scales += list((np.abs(rng.standard_normal(120)) * 10.0 ** rng.uniform(-37.5, 37.5, 120)))
    # per-token-head scales: fp32(amax / 448) of bf16 maxima
    am = (rng.integers(1, 0x7F80, 60, dtype=np.uint32) << 16).view(np.float32)
    scales += list((am / np.float32(448)).astype(np.float32))
    for rel in (-2.0 ** -21, 0.0, 2.0 ** -21):
        assert _check(x, scales, rel) > 0.9 * x.size * len(scales) * 0.5


def test_bracket_on_normal_rows_rarely_needs_the_divide():
    # bf16 N(0,1) rows with per-token-head scales: the multiply settles ~99 % of
    # the values; the rest sit within a step of an e4m3 rounding midpoint
    rng = np.random.default_rng(13)
    x = rng.standard_normal((400, 128)).astype(np.float32)
    x = (x.view(np.uint32) & 0xFFFF0000).view(np.float32)
    s = (np.abs(x).max(1) / np.float32(448)).astype(np.float32)
    total = settled = 0
    for i in range(x.shape[0]):
        lo, hi = _bracket_codes(x[i], s[i], 0.0)
        with np.errstate(all="ignore"):
            want = enc((x[i] / s[i]).astype(np.float32))
        same = lo == hi
        assert np.array_equal(lo[same], want[same])
        total += x.shape[1]
        settled += int(same.sum())
    assert settled / total > 0.98
