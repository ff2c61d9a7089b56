"""Pins for the oracle's e4m3fn codec, against facts other than the oracle itself.

- printed points: the 2^-9 grid step at denormal magnitudes and the sign-magnitude
  code order stated with the assert_fp8_within_one_ulp helper ("vLLM
  Qwen3.8-Flash-Next: QSA Indexer 캐시를 위한 FP8 지원", section "코드 분석"), and the
  format's closed-form largest finite value 448 (tests/golden/e4m3_points.txt);
- closed forms: every code decodes to (1 + m/8) 2^(e-7) or m 2^-9;
- properties: all 256 codes round-trip, code order is value order within a sign,
  every midpoint between neighbours rounds to the even code and its neighbours
  round away from it;
- a library routine: torch's float8_e4m3fn cast rounds to nearest even and
  agrees wherever it does not overflow (|x| <= 464; above that torch yields NaN
  where the satfinite encoder saturates to 448).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_points.txt")


def _parse_value(tok: str) -> float:
    if tok.startswith("0x") and len(tok) == 10:
        return float(np.array([int(tok, 16)], dtype=np.uint32).view(np.float32)[0])
    return float(tok)


def test_golden_points():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            rows.append((_parse_value(parts[0]), int(parts[1], 16), " ".join(parts[2:])))
    assert len(rows) >= 20
    x = np.array([r[0] for r in rows], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    for (v, want, why), g in zip(rows, got):
        assert g == want, f"{v!r}: got {g:#04x}, want {want:#04x} ({why})"


def test_decode_closed_form():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert math.isnan(got[c])
            continue
        mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        assert got[c] == (-mag if s else mag), hex(c)
    assert got[0x7E] == 448.0 and got[0xFE] == -448.0
    assert got[0x01] == 2.0 ** -9


def test_all_codes_round_trip():
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    back = oracle.e4m3_encode(vals.astype(np.float32))
    finite = ~np.isnan(vals)
    assert np.array_equal(back[finite], codes[finite])
    assert np.array_equal(np.sort(back[~finite]), np.array([0x7F, 0xFF], dtype=np.uint8))
    assert finite.sum() == 254


def test_code_order_is_value_order():
    pos = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(pos) > 0)
    neg = oracle.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(neg, -pos)


def test_denormal_grid_step():
    # Codes 0..16 (subnormals and the first binade) sit 2^-9 apart.
    v = oracle.e4m3_decode(np.arange(17, dtype=np.uint8))
    assert np.all(np.diff(v) == 2.0 ** -9)


def test_midpoints_round_to_even():
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2        # exact in fp32
        even = c if c % 2 == 0 else c + 1
        below = np.nextafter(mid, np.float32(-np.inf))
        above = np.nextafter(mid, np.float32(np.inf))
        got = oracle.e4m3_encode(np.array([mid, below, above, -mid, -below, -above],
                                          dtype=np.float32))
        assert list(got) == [even, c, c + 1, 0x80 | even, 0x80 | c, 0x80 | (c + 1)], hex(c)


def test_saturation():
    x = np.array([448, 448.0001, 455, 463.99, 464, 479, 480, 1e6, 3.4e38, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(x) == 0x7E)
    assert np.all(oracle.e4m3_encode(-x) == 0xFE)


def _torch_cast(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_all_bf16_inputs_match_torch_cast():
    x = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    x = x[~np.isnan(x) & (np.abs(x) < 464)]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_cast(x))


@pytest.mark.parametrize("start", [0, 1, 2])
def test_fp32_sweep_matches_torch_cast(start):
    # Every 37th fp32 bit pattern from a rotating start: ~1.2e8 values over the
    # three cases, restricted to the magnitudes where torch's cast cannot overflow.
    bits = np.arange(start, 2 ** 32, 37, dtype=np.uint64)[::3].astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x) & (np.abs(x) < 464)]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_cast(x))


def test_torch_overflow_band_is_the_only_difference():
    # 464 itself is a tie that rounds down to 448 on both sides; above it torch
    # rounds to the (absent) 480 and returns NaN.
    x = np.linspace(464, 479.9, 4001, dtype=np.float32)[1:]
    assert np.all(oracle.e4m3_encode(x) == 0x7E)
    assert oracle.e4m3_encode(np.array([464], np.float32))[0] == _torch_cast(
        np.array([464], np.float32))[0] == 0x7E
    assert np.all(np.isnan(torch.from_numpy(x).to(torch.float8_e4m3fn).float().numpy()))


def test_nan_keeps_sign():
    x = np.array([np.nan, -np.nan], dtype=np.float32)
    got = oracle.e4m3_encode(x)
    assert got[0] & 0x7F == 0x7F and got[1] & 0x7F == 0x7F
