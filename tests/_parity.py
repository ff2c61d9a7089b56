"""Shared setup for the GPU parity tests: fill a paged cache from a synthetic
workload twice -- once with the CUDA library, once with the oracle from the
same bf16 inputs -- and run decode attention on both.  Nothing here computes
part of the method; it moves tensors between the two implementations."""
import numpy as np
import torch

import oracle
import fp8_kv_cache_write_gb300 as fk
from tests._helpers import bits16

DECODE_TOL = 4e-3          # max-abs, fp32 output vs float64 oracle


def device_cache(w, kv_dtype, dev="cuda"):
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    dt = torch.uint8 if kv_dtype == fk.KV_E4M3 else torch.bfloat16
    kc = torch.zeros(nb, Hkv, 16, D, dtype=dt, device=dev)
    vc = kc.clone()
    ksc = torch.zeros(nb, Hkv, 16, dtype=torch.float32, device=dev)
    return {"k": kc, "v": vc, "ks": ksc, "vs": ksc.clone(), "kv_dtype": kv_dtype,
            "mode": w.scale_mode if kv_dtype == fk.KV_E4M3 else 0,
            "k_scale": None if w.k_scale is None else w.k_scale.to(dev),
            "v_scale": None if w.v_scale is None else w.v_scale.to(dev)}


def gpu_write(w, cache, k, v, slots, err=None):
    fk.kv_cache_write(k.cuda(), v.cuda(), slots.cuda(), cache["k"], cache["v"],
                      kv_dtype=cache["kv_dtype"], scale_mode=cache["mode"],
                      k_scale=cache["k_scale"], v_scale=cache["v_scale"],
                      k_scale_cache=cache["ks"], v_scale_cache=cache["vs"], err_flag=err)


def gpu_fill(w, kv_dtype, err=None):
    cache = device_cache(w, kv_dtype)
    gpu_write(w, cache, w.k_hist, w.v_hist, w.hist_slots, err)
    gpu_write(w, cache, w.k_new, w.v_new, w.new_slots, err)
    return cache


def oracle_cache(w, kv_dtype):
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    dt = np.uint8 if kv_dtype == 0 else np.uint16
    c = {"k": np.zeros((nb, Hkv, 16, D), dt), "v": np.zeros((nb, Hkv, 16, D), dt),
         "ks": np.zeros((nb, Hkv, 16), np.float32), "vs": np.zeros((nb, Hkv, 16), np.float32),
         "kv_dtype": kv_dtype, "mode": w.scale_mode if kv_dtype == 0 else 0,
         "k_scale": None if w.k_scale is None else w.k_scale.numpy(),
         "v_scale": None if w.v_scale is None else w.v_scale.numpy()}
    for k, v, s in ((w.k_hist, w.v_hist, w.hist_slots), (w.k_new, w.v_new, w.new_slots)):
        st = oracle.kv_cache_write(bits16(k), bits16(v), s.cpu().numpy(), c["k"], c["v"],
                                   kv_dtype=kv_dtype, scale_mode=c["mode"],
                                   k_scale=c["k_scale"], v_scale=c["v_scale"],
                                   k_scale_cache=c["ks"], v_scale_cache=c["vs"])
        assert st == 0
    return c


def assert_same_cache(gc, oc):
    gk = gc["k"].view(torch.uint8).cpu().numpy() if gc["kv_dtype"] == 0 else \
        gc["k"].view(torch.int16).cpu().numpy().view(np.uint16)
    gv = gc["v"].view(torch.uint8).cpu().numpy() if gc["kv_dtype"] == 0 else \
        gc["v"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(gk, oc["k"]), "K cache bytes differ"
    assert np.array_equal(gv, oc["v"]), "V cache bytes differ"
    if gc["mode"] == 2 and gc["kv_dtype"] == 0:
        assert np.array_equal(gc["ks"].cpu().numpy().view(np.uint32), oc["ks"].view(np.uint32))
        assert np.array_equal(gc["vs"].cpu().numpy().view(np.uint32), oc["vs"].view(np.uint32))


def gpu_decode(w, cache, **kw):
    return fk.paged_decode_attn(
        w.q.cuda(), cache["k"], cache["v"], w.block_table.cuda(), w.context_lens.cuda(),
        kv_dtype=cache["kv_dtype"], scale_mode=cache["mode"], k_scale=cache["k_scale"],
        v_scale=cache["v_scale"], k_scale_cache=cache["ks"], v_scale_cache=cache["vs"],
        window=w.window, **kw)


def oracle_decode(w, oc, units=None, nthreads=8):
    st, out = oracle.decode_attn(bits16(w.q), oc["k"], oc["v"], w.block_table.numpy(),
                                 w.context_lens.numpy(), kv_dtype=oc["kv_dtype"],
                                 scale_mode=oc["mode"], k_scale=oc["k_scale"],
                                 v_scale=oc["v_scale"], k_scale_cache=oc["ks"],
                                 v_scale_cache=oc["vs"], window=w.window, units=units,
                                 nthreads=nthreads)
    assert st == 0
    return out
