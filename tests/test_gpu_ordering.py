"""Ordering of the decode calls against the preceding kernel of their stream.

The decode kernels launch with programmatic stream serialization: they may be
resident while the kernel before them finishes.  With flags 0 (the default)
they must read nothing before that kernel has completed, so any kernel may
produce any of their inputs.  Two producers are tested, each launched directly
before the decode call with every input already on the device (no copy between
the launches):
  - the library's own cache writer storing a whole history, then decode_step;
  - a kernel that lets its dependents start at once and writes the context
    lengths only after a delay, then paged_decode_attn (split over many warps, so
    split_merge reads the lengths too).
Outputs are compared with the float64 oracle at the decode tolerance.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch

import fp8_kv_cache_write_gb300 as fk
from fp8_kv_cache_write_gb300 import synth
from tests._parity import DECODE_TOL, device_cache, gpu_write, oracle_cache, oracle_decode

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def helper(tmp_path_factory):
    """tests/pdl_helper.cu built for sm_103a (test-only kernel)."""
    out = str(tmp_path_factory.mktemp("pdl") / "libpdl_helper.so")
    nvcc = "/usr/local/cuda/bin/nvcc" if os.path.exists("/usr/local/cuda/bin/nvcc") else "nvcc"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O2", "-shared",
                    "-Xcompiler", "-fPIC", os.path.join(HERE, "pdl_helper.cu"), "-o", out],
                   check=True)
    L = ctypes.CDLL(out)
    L.pdl_delayed_copy.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                   ctypes.c_ulonglong, ctypes.c_void_p]
    L.pdl_delayed_copy.restype = ctypes.c_int
    return L


def _sampled_units(w, n_seq_heads=24, seed=0):
    rng = np.random.default_rng(seed)
    return sorted({(int(rng.integers(w.B)), int(rng.integers(w.Hq))) for _ in range(n_seq_heads)})


@pytest.mark.parametrize("kv_dtype", [fk.KV_E4M3, fk.KV_BF16])
def test_cache_write_then_decode_step_back_to_back(kv_dtype):
    # a long bulk write of the history (staged path), then the fused step that
    # stores the new tokens and attends over every key; the cache starts as
    # 0xFF bytes (NaN codes), so a page streamed before the writer finished
    # would show up in the output
    w = synth.llama8b(seed=71, B=8, ctx_lo=6000, ctx_hi=9000)
    cache = device_cache(w, kv_dtype)
    for key in ("k", "v"):
        cache[key].view(torch.uint8).fill_(0xFF)
    kh, vh, hs = w.k_hist.cuda(), w.v_hist.cuda(), w.hist_slots.cuda()
    q, kn, vn = w.q.cuda(), w.k_new.cuda(), w.v_new.cuda()
    bt, cl = w.block_table.cuda(), w.context_lens.cuda()
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.empty(w.B, w.Hq, w.D, device="cuda")
    torch.cuda.synchronize()
    fk.kv_cache_write(kh, vh, hs, cache["k"], cache["v"], kv_dtype=cache["kv_dtype"],
                      scale_mode=cache["mode"], k_scale=cache["k_scale"],
                      v_scale=cache["v_scale"], k_scale_cache=cache["ks"],
                      v_scale_cache=cache["vs"], err_flag=err)
    fk.decode_step(q, kn, vn, cache["k"], cache["v"], bt, cl, kv_dtype=cache["kv_dtype"],
                   scale_mode=cache["mode"], k_scale=cache["k_scale"], v_scale=cache["v_scale"],
                   k_scale_cache=cache["ks"], v_scale_cache=cache["vs"], out=out, err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    oc = oracle_cache(w, kv_dtype)
    # every written slot holds the oracle's bytes (the others keep the 0xFF fill)
    slots = torch.cat([w.hist_slots, w.new_slots]).numpy()
    blk, off = slots // 16, slots % 16
    for key in ("k", "v"):
        g = cache[key].view(torch.uint8).cpu().numpy()
        o = oc[key].view(np.uint8)
        assert np.array_equal(g[blk, :, off], o[blk, :, off]), key
    if cache["mode"] == fk.SCALE_PER_TOKEN_HEAD and kv_dtype == fk.KV_E4M3:
        for key in ("ks", "vs"):
            g = cache[key].cpu().numpy().view(np.uint32)
            assert np.array_equal(g[blk, :, off], oc[key].view(np.uint32)[blk, :, off]), key
    got = out.cpu().numpy().reshape(-1, w.D)
    assert np.isfinite(got).all()
    units = _sampled_units(w)
    ref = oracle_decode(w, oc, units=units, nthreads=16)
    e = float(np.abs(np.stack([got[b * w.Hq + h] for b, h in units]) - ref).max())
    assert e <= DECODE_TOL, e


@pytest.mark.parametrize("num_splits", [0, 3])
def test_context_lens_written_by_the_preceding_kernel(helper, num_splits):
    # the cache holds every token; context_lens first say 40 for every sequence,
    # and the preceding kernel replaces them with the real lengths 50 us after
    # it let the decode kernels start
    w = synth.decode_workload(72, [3000, 17, 2500, 4097, 1, 800], 32, 8, 128,
                              fk.SCALE_PER_TOKEN_HEAD, outlier_frac=0.01)
    cache = device_cache(w, fk.KV_E4M3)
    gpu_write(w, cache, w.k_hist, w.v_hist, w.hist_slots)
    gpu_write(w, cache, w.k_new, w.v_new, w.new_slots)
    real = w.context_lens.cuda()
    cl = torch.full_like(real, 40)
    q, bt = w.q.cuda(), w.block_table.cuda()
    out = torch.empty(w.B, w.Hq, w.D, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()
    assert helper.pdl_delayed_copy(cl.data_ptr(), real.data_ptr(), w.B, 50_000,
                                   stream.cuda_stream) == 0
    fk.paged_decode_attn(q, cache["k"], cache["v"], bt, cl, kv_dtype=fk.KV_E4M3,
                         scale_mode=cache["mode"], k_scale_cache=cache["ks"],
                         v_scale_cache=cache["vs"], num_splits=num_splits, out=out,
                         err_flag=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert torch.equal(cl, real)
    oc = oracle_cache(w, fk.KV_E4M3)
    ref = oracle_decode(w, oc, nthreads=16)
    e = float(np.abs(out.cpu().numpy().reshape(-1, w.D) - ref).max())
    assert e <= DECODE_TOL, e
