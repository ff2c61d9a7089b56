"""The C-ABI library loads, exports every symbol include/fp8kv.h declares, and
rejects invalid host arguments before touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import fp8_kv_cache_write_gb300 as fk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8kv.h")


@pytest.fixture(scope="module")
def lib():
    fk.build()
    return fk.lib()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8kv_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_exports():
    assert _declared_functions() == sorted(fk.EXPORTS)


def test_binding_constants_match_the_header():
    text = open(os.path.join(os.path.dirname(__file__), "..", "include", "fp8kv.h")).read()
    def define(name):
        m = re.search(r"#define\s+" + name + r"\s+\((\d+)u << (\d+)\)", text)
        return int(m.group(1)) << int(m.group(2))
    assert define("FP8KV_NOALLOC_DECODE_SCRATCH_BYTES") == fk.NOALLOC_DECODE_SCRATCH_BYTES
    def flag(name):
        return int(re.search(r"#define\s+" + name + r"\s+(\d+)u", text).group(1))
    assert flag("FP8KV_DECODE_EARLY_SETUP") == fk.DECODE_EARLY_SETUP
    assert flag("FP8KV_DECODE_EARLY_PAGES") == fk.DECODE_EARLY_PAGES
    for name in ("TWO_LEVEL", "SPLIT_ALWAYS", "SPLIT_NEVER"):
        m = re.search(r"#define\s+FP8KV_PREFILL_" + name + r"\s+(\d+)", text)
        assert int(m.group(1)) == getattr(fk, "PREFILL_" + name)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert fk.status_string(code) not in ("", "unknown status")
    assert fk.status_string(17) == "unknown status"
    assert fk.last_warning() == ""


def test_decode_plan_is_consistent(lib):
    # num_splits = CTAs of the balanced partition (4 worker warps each); one
    # workspace slot per warp plus one per unit, of the unit's query heads x
    # (D + 2) floats.  A unit packs two adjacent KV heads (hpt = 2) when each has
    # 2 or 4 query heads, Hkv is even, an e4m3 row is at most 128 bytes and the
    # batch holds at least 32 (sequence, KV head) pairs.
    for B, Hq, Hkv, D, mbs, win in [(8, 32, 8, 128, 1375, 0), (1, 64, 8, 128, 8192, 0),
                                    (32, 64, 8, 64, 2048, 128), (1, 32, 8, 128, 64, 0),
                                    (4, 16, 8, 64, 100, 0), (2, 12, 3, 128, 50, 0),
                                    (8, 32, 8, 256, 100, 0)]:
        s, ws = fk.decode_plan(B, Hq, Hkv, D, mbs, win)
        G = Hq // Hkv
        hpt = 2 if G in (2, 4) and Hkv % 2 == 0 and D <= 128 and B * Hkv >= 32 else 1
        if win and (win + 15) // 16 + 1 <= 16 and G * hpt <= 8:
            # a short sliding window: one CTA per unit, no workspace
            assert (s, ws) == (B * Hkv // hpt, 16)
            continue
        assert 1 <= s <= 1024
        assert ws == (4 * s * hpt + B * Hkv) * G * (D + 2) * 4
        for req in (1, 2, 7):
            s2, _ = fk.decode_plan(B, Hq, Hkv, D, mbs, win, req)
            assert 1 <= s2 <= min(1024, req * B * Hkv)
    # a window bounds the visible pages: 128 keys touch at most 9 pages per unit
    s, _ = fk.decode_plan(1, 8, 8, 64, 4096, 128, 1000)
    assert s <= 9 * 8
    # ... and then the automatic plan gives every (seq, KV head) unit one CTA
    s, _ = fk.decode_plan(32, 64, 8, 64, 2048, 128)
    assert s == 32 * 8
    # small work: at least 16 tiles per CTA
    s, _ = fk.decode_plan(1, 32, 8, 128, 64, 0)
    assert s <= (8 * 64 + 15) // 16


def _null():
    return ctypes.c_void_p(0)


def test_write_rejects_bad_arguments_without_a_gpu(lib):
    N = _null()
    call = lambda **kw: lib.fp8kv_kv_cache_write(
        kw.get("k", N), kw.get("v", N), kw.get("slots", N), kw.get("T", 4), kw.get("Hkv", 2),
        kw.get("D", 128), kw.get("kc", N), kw.get("vc", N), 10, kw.get("dtype", 0),
        kw.get("mode", 0), N, N, N, N, N, N)
    assert call() == -1            # null pointers
    assert call(D=96) == -2
    assert call(dtype=5) == -1
    assert call(mode=3) == -1
    assert call(T=-1) == -1
    assert call(T=0) == 0          # nothing to do, nothing launched


def test_decode_rejects_bad_arguments_without_a_gpu(lib):
    N = _null()

    def call(B=2, Hq=8, Hkv=2, D=128, dtype=0, mode=0, out_dtype=0, window=0, splits=0,
             flags=0):
        return lib.fp8kv_paged_decode_attn(N, N, N, dtype, mode, N, N, N, N, N, 4, N, B, Hq, Hkv,
                                           D, 10, 0.1, window, splits, N, 0, N, out_dtype, flags,
                                           N, N)

    assert call() == -1            # null pointers
    assert call(Hq=9) == -1        # Hq % Hkv
    assert call(Hq=34, Hkv=2) == -2   # group of 17 query heads (16 at most)
    assert call(D=80) == -2
    assert call(dtype=2) == -1
    assert call(mode=7) == -1
    assert call(out_dtype=3) == -1
    assert call(window=-1) == -1
    assert call(flags=4) == -1     # unknown flag bit
    assert call(B=0) == 0
    assert call(B=0, flags=fk.DECODE_EARLY_SETUP | fk.DECODE_EARLY_PAGES) == 0


def test_quantize_rejects_bad_arguments_without_a_gpu(lib):
    assert lib.fp8kv_quantize_e4m3(_null(), 1.0, _null(), 5, _null()) == -1
    assert lib.fp8kv_quantize_e4m3(_null(), 1.0, _null(), 0, _null()) == 0
    assert lib.fp8kv_quantize_e4m3(_null(), 1.0, _null(), -1, _null()) == -1


def test_prefill_rejects_bad_arguments_without_a_gpu(lib):
    N = _null()

    def call(B=1, Hq=8, Hkv=1, D=256, dtype=0, mode=0, q_scale=1.0, prob_scale=1.0,
             two_level=0, out_dtype=0, max_q=128):
        return lib.fp8kv_prefill_attn(N, N, max_q, N, N, dtype, mode, N, N, N, N, q_scale,
                                      prob_scale, N, 4, N, B, Hq, Hkv, D, 10, 0.0625, two_level,
                                      N, out_dtype, N, N)

    assert call() == -1                 # null pointers
    assert call(Hq=9, Hkv=2) == -1      # Hq % Hkv
    assert call(Hq=9) == -2             # a group of 9 does not tile 128 MMA rows
    assert call(D=80) == -2             # prefill tiles: D 64, 128 or 256
    assert call(dtype=2) == -1
    assert call(mode=3) == -1
    assert call(out_dtype=2) == -1
    assert call(two_level=8) == -1      # unknown flag bit
    assert call(two_level=6) == -1      # split always and never
    assert call(q_scale=0.0) == -1
    assert call(prob_scale=-1.0) == -1
    assert call(max_q=-1) == -1
    assert call(B=0) == 0               # nothing to do, nothing launched
    assert call(max_q=0) == 0


def test_prefill_with_workspace_rejects_bad_arguments_without_a_gpu(lib):
    # fp8kv_prefill_attn_ws checks its arguments as fp8kv_prefill_attn does, before
    # any workspace or device question
    N = _null()

    def call(B=1, Hq=8, Hkv=1, D=256, dtype=0, flags=0, max_q=128, ws_bytes=0):
        return lib.fp8kv_prefill_attn_ws(N, N, max_q, N, N, dtype, 0, N, N, N, N, 1.0, 1.0, N, 4,
                                         N, B, Hq, Hkv, D, 10, 0.0625, flags, N, ws_bytes, N, 0,
                                         N, N)

    assert call() == -1                 # null pointers
    assert call(Hq=9) == -2
    assert call(D=80) == -2
    assert call(dtype=2) == -1
    assert call(flags=8) == -1
    assert call(flags=6) == -1
    assert call(max_q=-1) == -1
    assert call(B=0) == 0
    assert call(max_q=0, ws_bytes=1 << 20) == 0


def test_prefill_workspace_bytes_without_a_gpu(lib):
    n = ctypes.c_size_t(0)
    assert lib.fp8kv_prefill_workspace_bytes(80, ctypes.byref(n)) == -2
    assert lib.fp8kv_prefill_workspace_bytes(256, None) == -1
    st = lib.fp8kv_prefill_workspace_bytes(256, ctypes.byref(n))
    # no device here: FP8KV_ERR_CUDA; with one, two partial slots of
    # 128 x (D + 2) floats per SM after the 256-byte-padded counters
    assert st in (0, -4), st
    if st == 0:
        slot = 128 * (256 + 2) * 4
        sms = [k for k in range(1, 1025)
               if n.value == (k * 4 + 255) // 256 * 256 + 2 * k * slot]
        assert sms, n.value
