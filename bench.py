"""Benchmark of the FP8 paged-decode hot path on GB300.

One step = the decode step of one attention layer of the Llama-3.1-8B-shaped
workload under load: 8 sequences, contexts uniform in [18000, 22000], 32 query /
8 KV heads, head_dim 128, page 16 with a shuffled page table, per-token-head
e4m3 scales, 1% of (head, channel) pairs scaled x20.  Each step stores the 8 new
tokens into the cache and attends over all keys in one decode_step call (the
attention kernel stores the new tokens itself, + split_merge); the same work as
kv_cache_write followed by paged_decode_attn, which is timed beside it.  The same
step on a bf16 cache is the in-run comparison.

value = algorithmic HBM bytes of a step / step time (GB/s), with the cache
resident in HBM; e2e = the same bytes over a step that also copies its inputs
(q, new K/V, slots, lengths) from pinned host memory and reads the output back.
Caches rotate over 4 copies (each > L2), so no step reads a previous step's data
from L2.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank benchmarks its own GPU on its own batch (weak scaling,
no data-path collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "FP8 paged-decode attn HBM GB/s (% of GB300 peak) & tokens/s vs bf16 KV"
WORKLOAD = ("llama8b-decode: B=8, ctx~U[18000,22000], 32 Q / 8 KV heads, head_dim 128, page 16, "
            "shuffled block_table, e4m3 per-token-head scales, 1% channels x20")
ROTATIONS = 4
FALLBACK_HBM_GBS = 6800.0


# ----------------------------------------------------------------- helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(x: float, group=None) -> float:
    """Max over ranks (identity without a process group)."""
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def reduce_sum(x: float, group=None) -> float:
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(bytes_per_step: float, tokens_per_step: float, seconds: float, steps: int):
    """Whole-job throughput: units of all ranks / the slowest rank's time."""
    t = reduce_max(seconds)
    total_bytes = reduce_sum(bytes_per_step * steps)
    total_tokens = reduce_sum(tokens_per_step * steps)
    return total_bytes / t / 1e9, total_tokens / t, t


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash():
    """Hash of the decode kernel's source with comments and blank lines removed
    (a comment edit leaves the profiled kernel, and so its counters, unchanged);
    the prefill's parameter block of internal.h is not part of it."""
    h = hashlib.sha256()
    for name in ("decode.cu", "common.cuh", "internal.h"):
        with open(os.path.join(ROOT, "fp8_kv_cache_write_gb300", "csrc", name)) as f:
            text = re.sub(r"/\*.*?\*/", "", f.read(), flags=re.S)
        text = re.sub(r"struct PrefillParams \{.*?\};", "", text, flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def profiled_traffic():
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "paged_decode_llama8b.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") == kernel_source_hash():
            return float(d["dram_bytes_per_launch_full_size"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            sel = str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", sel], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- workload
def step_bytes(w, kv_elem_bytes: int, per_token_scales: bool):
    """Algorithmic HBM bytes of one decode step: every visible key and value
    byte once (+ per-token-head scales), q in, out (fp32) out, page-table
    entries, and the cache write of the new tokens."""
    ctx = w.context_lens.to(torch.int64)
    n_tok = int(ctx.sum())
    pages = int(((ctx + 15) // 16).sum())
    kv = n_tok * w.Hkv * (2 * w.D * kv_elem_bytes + (8 if per_token_scales else 0))
    q = w.B * w.Hq * w.D * 2
    out = w.B * w.Hq * w.D * 4
    bt = pages * 4
    write = w.B * w.Hkv * (2 * w.D * 2 + 2 * w.D * kv_elem_bytes + (8 if per_token_scales else 0))
    return kv + q + out + bt, write


def visible_kv_bytes(w, kv_elem_bytes: int, per_token_scales: bool):
    """Key and value bytes (+ per-token-head scales) that one decode call over
    `w` must read: the last `w.window` keys of each sequence when the layer has a
    sliding window, else all of them."""
    ctx = w.context_lens.to(torch.int64)
    if getattr(w, "window", 0):
        ctx = torch.clamp(ctx, max=int(w.window))
    return int(ctx.sum()) * w.Hkv * (2 * w.D * kv_elem_bytes + (8 if per_token_scales else 0))


def build_caches(w, kv_dtype, dev, rotations):
    import fp8_kv_cache_write_gb300 as fk
    dt = torch.uint8 if kv_dtype == fk.KV_E4M3 else torch.bfloat16
    k_hist, v_hist, hs = w.k_hist.to(dev), w.v_hist.to(dev), w.hist_slots.to(dev)
    caches = []
    for _ in range(rotations):
        kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=dt, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.num_blocks, w.Hkv, 16, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        fk.kv_cache_write(k_hist, v_hist, hs, kc, vc, kv_dtype=kv_dtype,
                          scale_mode=w.scale_mode if kv_dtype == fk.KV_E4M3 else 0,
                          k_scale_cache=ks, v_scale_cache=vs)
        caches.append((kc, vc, ks, vs))
    del k_hist, v_hist
    torch.cuda.synchronize(dev)
    return caches


def _graph(fn, n, stream):
    """Capture n calls fn(i) into one CUDA graph on `stream`."""
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n):
            fn(i)
    return g


def _replay_steps(graphs, K, stream):
    """Replay graphs covering exactly K steps: (full graph of n, remainder graph)."""
    full, n, rem = graphs
    for _ in range(K // n):
        full.replay()
    if rem is not None:
        rem.replay()


def _capture_steps(fn, K, n, stream):
    full = _graph(fn, n, stream)
    rem = _graph(fn, K % n, stream) if K % n else None
    return full, n, rem


def run_ours(args, dev, w, world, rank):
    """Times K steps of the fp8 path and of the bf16 twin (CUDA graphs of
    `per_graph` steps replayed back to back), the decode call alone, and the
    end-to-end step with host copies."""
    import fp8_kv_cache_write_gb300 as fk

    cap = torch.cuda.Stream(dev)
    q, kn, vn = w.q.to(dev), w.k_new.to(dev), w.v_new.to(dev)
    slots, bt, cl = w.new_slots.to(dev), w.block_table.to(dev), w.context_lens.to(dev)
    mbs = bt.shape[1]
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    dec_bytes, results, launches_per_step = {}, {}, {}
    K = args.steps
    per_graph = args.rotations * 8
    dtypes = [(fk.KV_E4M3, "fp8"), (fk.KV_BF16, "bf16")]
    if args.only:
        dtypes = [d for d in dtypes if d[1] == args.only]

    for kv_dtype, name in dtypes:
        mode = fk.SCALE_PER_TOKEN_HEAD if kv_dtype == fk.KV_E4M3 else 0
        caches = build_caches(w, kv_dtype, dev, args.rotations)
        splits, ws_bytes = fk.decode_plan(w.B, w.Hq, w.Hkv, w.D, mbs, 0, args.splits)
        ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)
        out = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32, device=dev)
        launches_per_step[name] = 2          # decode (stores the new tokens), split_merge
        d_b, w_b = step_bytes(w, 1 if kv_dtype == fk.KV_E4M3 else 2, kv_dtype == fk.KV_E4M3)
        dec_bytes[name] = d_b

        def write(i, k_in=kn, v_in=vn, s_in=slots):
            kc, vc, ks, vs = caches[i % args.rotations]
            fk.kv_cache_write(k_in, v_in, s_in, kc, vc, kv_dtype=kv_dtype, scale_mode=mode,
                              k_scale_cache=ks, v_scale_cache=vs, err_flag=err)

        def decode(i, q_in=q, cl_in=cl):
            kc, vc, ks, vs = caches[i % args.rotations]
            fk.paged_decode_attn(q_in, kc, vc, bt, cl_in, kv_dtype=kv_dtype, scale_mode=mode,
                                 k_scale_cache=ks, v_scale_cache=vs, workspace=ws, out=out,
                                 num_splits=args.splits, flags=args.decode_flags, err_flag=err)

        def split_step(i):
            write(i)
            decode(i)

        def step(i, q_in=q, k_in=kn, v_in=vn, cl_in=cl, out_t=out, flags=args.decode_flags):
            kc, vc, ks, vs = caches[i % args.rotations]
            fk.decode_step(q_in, k_in, v_in, kc, vc, bt, cl_in, kv_dtype=kv_dtype,
                           scale_mode=mode, k_scale_cache=ks, v_scale_cache=vs, workspace=ws,
                           out=out_t, num_splits=args.splits, flags=flags, err_flag=err)

        def step_wait_first(i):
            step(i, flags=0)

        with torch.cuda.stream(cap):
            for i in range(args.warmup):             # eager warm-up (also first-call setup)
                split_step(i)
                step(i)
        torch.cuda.synchronize(dev)
        graphs = _capture_steps(step, K, per_graph, cap)
        sgraph = _capture_steps(split_step, K, per_graph, cap)
        dgraph = _capture_steps(decode, K, per_graph, cap)
        wgraph = _capture_steps(step_wait_first, K, per_graph, cap)
        for _ in range(max(1, args.warmup // per_graph)):
            graphs[0].replay()
            sgraph[0].replay()
            dgraph[0].replay()
            wgraph[0].replay()
        torch.cuda.synchronize(dev)

        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        sampler = ClockSampler(dev.index) if name == "fp8" else None
        barrier()
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(cap):
            t0.record(cap)
            _replay_steps(graphs, K, cap)
            t1.record(cap)
        torch.cuda.synchronize(dev)
        barrier()
        clocks = sampler.stop() if sampler else None
        secs = t0.elapsed_time(t1) / 1e3

        # the decode call alone (split kernel + split_merge), same caches, and the
        # unfused step (kv_cache_write, then paged_decode_attn)
        with torch.cuda.stream(cap):
            t0.record(cap)
            _replay_steps(dgraph, K, cap)
            t1.record(cap)
        torch.cuda.synchronize(dev)
        dec_ms = t0.elapsed_time(t1) / K
        with torch.cuda.stream(cap):
            t0.record(cap)
            _replay_steps(sgraph, K, cap)
            t1.record(cap)
        torch.cuda.synchronize(dev)
        split_ms = t0.elapsed_time(t1) / K
        with torch.cuda.stream(cap):
            t0.record(cap)
            _replay_steps(wgraph, K, cap)
            t1.record(cap)
        torch.cuda.synchronize(dev)
        wait_first_ms = t0.elapsed_time(t1) / K
        gbs, tok_s, tmax = aggregate(d_b + w_b, w.B, secs, K)
        results[name] = {"gbs": gbs, "tokens_per_s": tok_s, "ms_per_step": tmax / K * 1e3,
                         "decode_ms": dec_ms, "split_step_ms": split_ms,
                         "wait_first_step_ms": wait_first_ms, "num_splits": splits,
                         "clocks": clocks, "secs": tmax}
        if int(err.item()) != 0:
            raise RuntimeError(f"device error flag {int(err.item())} during the {name} run")

        if name == "fp8" and not args.no_e2e:
            # end to end through the public API: every step copies its inputs from
            # pinned host memory and reads the output back (captured as graph nodes)
            # the step's inputs (q, new K/V, slots, lengths) live in pinned host memory
            # and the output goes to pinned host memory: the write and decode kernels
            # read and write them directly over the host link (no staging copies)
            hq, hk, hv = w.q.pin_memory(), w.k_new.pin_memory(), w.v_new.pin_memory()
            hc = w.context_lens.pin_memory()
            hout = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32).pin_memory()
            h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, hc))
            d2h = hout.numel() * hout.element_size()

            def e2e_step(i):
                step(i, q_in=hq, k_in=hk, v_in=hv, cl_in=hc, out_t=hout)

            with torch.cuda.stream(cap):
                for i in range(3):
                    e2e_step(i)
            torch.cuda.synchronize(dev)
            egraphs = _capture_steps(e2e_step, K, per_graph, cap)
            egraphs[0].replay()
            torch.cuda.synchronize(dev)
            barrier()
            with torch.cuda.stream(cap):
                t0.record(cap)
                _replay_steps(egraphs, K, cap)
                t1.record(cap)
            torch.cuda.synchronize(dev)
            barrier()
            e_secs = t0.elapsed_time(t1) / 1e3
            e_gbs, e_tok, _ = aggregate(d_b + w_b, w.B, e_secs, K)
            results["e2e"] = {"value": e_gbs, "unit": "GB/s", "tokens_per_s": e_tok,
                              "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                              "how": "each step: decode_step reading q, new K/V and lengths "
                                     "from pinned host memory and writing the output to pinned "
                                     "host memory (kernel loads/stores over the host link); steps "
                                     "replayed as CUDA graphs"}
            del egraphs
        del graphs, sgraph, dgraph, wgraph, caches
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
    return results, dec_bytes, launches_per_step


class OracleBaseline:
    """The oracle as it stands, timed on the host cores.  Its cache is written
    once by the oracle's own cache write from the same bf16 inputs; each run
    times decode attention for all query heads of the first `n_seq` sequences,
    contexts optionally cut to the first n_tok tokens."""

    def __init__(self, w, nthreads=None):
        import numpy as np

        import oracle
        self.np, self.oracle, self.w = np, oracle, w
        self.cores = nthreads or len(os.sched_getaffinity(0))
        self.bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)
        nb, Hkv, D = w.num_blocks, w.Hkv, w.D
        self.kc = np.zeros((nb, Hkv, 16, D), np.uint8)
        self.vc = np.zeros_like(self.kc)
        self.ks = np.zeros((nb, Hkv, 16), np.float32)
        self.vs = np.zeros_like(self.ks)
        for k, v, sl in ((w.k_hist, w.v_hist, w.hist_slots), (w.k_new, w.v_new, w.new_slots)):
            st = oracle.kv_cache_write(self.bits(k), self.bits(v), sl.numpy(), self.kc, self.vc,
                                       kv_dtype=0, scale_mode=2, k_scale_cache=self.ks,
                                       v_scale_cache=self.vs)
            assert st == 0
        self.q = self.bits(w.q)
        self.bt = w.block_table.numpy()

    def run(self, n_seq=None, n_tok=None, min_seconds=0.0):
        """Returns (GB/s, tokens/s, seconds, sample text); repeats the pass until
        min_seconds of wall time have been spent."""
        np, w = self.np, self.w
        seqs = list(range(w.B if n_seq is None else min(w.B, n_seq)))
        units = [(sq, h) for sq in seqs for h in range(w.Hq)]
        ctx = w.context_lens.numpy().copy()
        if n_tok is not None:
            ctx = np.minimum(ctx, n_tok)
        passes, secs = 0, 0.0
        while passes == 0 or secs < min_seconds:
            t = time.perf_counter()
            st, _ = self.oracle.decode_attn(self.q, self.kc, self.vc, self.bt, ctx, kv_dtype=0,
                                            scale_mode=2, k_scale_cache=self.ks,
                                            v_scale_cache=self.vs, units=units,
                                            nthreads=self.cores)
            secs += time.perf_counter() - t
            assert st == 0
            passes += 1
        n = int(ctx[seqs].sum())
        bytes_ = n * w.Hkv * (2 * w.D + 8) * passes
        sample = (f"{passes} pass(es) over {len(seqs)} of {w.B} sequences x all {w.Hq} query "
                  f"heads, {n} context tokens" + (f" (contexts cut to {n_tok})" if n_tok else ""))
        return bytes_ / secs / 1e9, len(seqs) * passes / secs, secs, sample


def run_reference(args, w, world, rank):
    """The oracle timed on the host cores, K steps of a bounded sample each."""
    if rank != 0:
        return None
    ob = OracleBaseline(w)
    budget = 120.0                                  # seconds for warmup + steps
    per_step = budget / max(1, args.steps + args.warmup)
    _, _, s_cal, _ = ob.run(n_seq=1, n_tok=512)     # calibration: 1 sequence, 512 tokens
    n_tok = int(max(16, min(int(w.context_lens.min()), per_step / (s_cal / 512))))
    for _ in range(args.warmup):
        ob.run(n_seq=1, n_tok=n_tok)
    tot_s, tot_b = 0.0, 0.0
    sample = ""
    for _ in range(args.steps):
        gbs, tps, secs, sample = ob.run(n_seq=1, n_tok=n_tok)
        tot_s += secs
        tot_b += gbs * secs * 1e9
    value = tot_b / tot_s / 1e9
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tot_s / max(1, args.steps) * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "parallelism": "host cores"},
            "cpu_baseline": {"kind": "oracle", "cores": ob.cores, "value": value, "unit": "GB/s",
                             "sample": sample + " per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}



# ----------------------------------------------------------------- extras
def _time_graph(fn, n_calls, stream, warmup=3):
    """Mean ms of fn(i) over n_calls calls captured in one CUDA graph (after
    eager warm-up calls), replayed twice; events on the capture stream."""
    with torch.cuda.stream(stream):
        for i in range(warmup):
            fn(i)
    torch.cuda.synchronize()
    g = _graph(fn, n_calls, stream)
    g.replay()
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        g.replay()
        g.replay()
        t1.record(stream)
    torch.cuda.synchronize()
    return t0.elapsed_time(t1) / (2 * n_calls)


# launch-overlap flags of the decode calls the extras time (--decode-flags): the
# kernel before each call is the previous call's split_merge, which writes only
# `out`, so page streaming may start before it ends
_DECODE_FLAGS = 0
# the oracle timed beside the extras (off with --no-cpu-baseline)
_CPU_BASELINE = True


def _decode_caller(fk, w, kv_dtype, mode, caches, dev, window=0):
    q, bt, cl = w.q.to(dev), w.block_table.to(dev), w.context_lens.to(dev)
    _, ws_bytes = fk.decode_plan(w.B, w.Hq, w.Hkv, w.D, bt.shape[1], window)
    ws = torch.empty(max(ws_bytes // 4, 1), dtype=torch.float32, device=dev)
    out = torch.empty(w.B, w.Hq, w.D, dtype=torch.float32, device=dev)
    ksc = w.k_scale.to(dev) if w.k_scale is not None else None
    vsc = w.v_scale.to(dev) if w.v_scale is not None else None

    def decode(i):
        kc, vc, ks, vs = caches[i % len(caches)]
        fk.paged_decode_attn(q, kc, vc, bt, cl, kv_dtype=kv_dtype, scale_mode=mode,
                             k_scale=ksc, v_scale=vsc, k_scale_cache=ks, v_scale_cache=vs,
                             window=window, workspace=ws, out=out, flags=_DECODE_FLAGS)
    return decode


def _caches_for(fk, w, kv_dtype, mode, dev, copies):
    dt = torch.uint8 if kv_dtype == fk.KV_E4M3 else torch.bfloat16
    k_hist, v_hist, hs = w.k_hist.to(dev), w.v_hist.to(dev), w.hist_slots.to(dev)
    k_new, v_new, ns = w.k_new.to(dev), w.v_new.to(dev), w.new_slots.to(dev)
    ksc = w.k_scale.to(dev) if w.k_scale is not None else None
    vsc = w.v_scale.to(dev) if w.v_scale is not None else None
    out = []
    for _ in range(copies):
        kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=dt, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.num_blocks, w.Hkv, 16, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        for k_in, v_in, s_in in ((k_hist, v_hist, hs), (k_new, v_new, ns)):
            fk.kv_cache_write(k_in, v_in, s_in, kc, vc, kv_dtype=kv_dtype, scale_mode=mode,
                              k_scale=ksc, v_scale=vsc, k_scale_cache=ks, v_scale_cache=vs)
        out.append((kc, vc, ks, vs))
    torch.cuda.synchronize()
    return out


def _copies_for(bytes_per_copy):
    """Cache copies to rotate over so that consecutive calls never find the
    previous call's data in the 129 MB L2."""
    return max(2, math.ceil(260e6 / max(bytes_per_copy, 1)))


def _oracle_decode_baseline(w, kv_dtype, mode, seconds=6.0, max_units=None):
    """The oracle (float64, every host core) on a bounded sample of a decode
    workload's (sequence, query head) units, extrapolated to the whole call.
    Its cache is written by the oracle's own writer from the same bf16 inputs."""
    import numpy as np

    import oracle
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    dt = np.uint8 if kv_dtype == 0 else np.uint16
    kc, vc = np.zeros((nb, Hkv, 16, D), dt), np.zeros((nb, Hkv, 16, D), dt)
    ks, vs = np.zeros((nb, Hkv, 16), np.float32), np.zeros((nb, Hkv, 16), np.float32)
    k_s = None if w.k_scale is None else w.k_scale.cpu().numpy()
    v_s = None if w.v_scale is None else w.v_scale.cpu().numpy()
    for k, v, sl in ((w.k_hist, w.v_hist, w.hist_slots), (w.k_new, w.v_new, w.new_slots)):
        assert oracle.kv_cache_write(bits(k), bits(v), sl.cpu().numpy(), kc, vc,
                                     kv_dtype=kv_dtype, scale_mode=mode, k_scale=k_s,
                                     v_scale=v_s, k_scale_cache=ks, v_scale_cache=vs) == 0
    cores = len(os.sched_getaffinity(0))
    ctx = w.context_lens.cpu().numpy()
    vis = np.minimum(ctx, w.window) if w.window > 0 else ctx
    all_units = [(b, h) for b in range(w.B) for h in range(w.Hq)]
    rng = np.random.default_rng(0)
    order = rng.permutation(len(all_units))
    units, passes, secs = [], 0, 0.0
    n = 4 if max_units is None else max_units
    while True:                         # grow the sample until it takes ~1/4 of the budget
        units = [all_units[i] for i in order[:n]]
        t = time.perf_counter()
        st, _ = oracle.decode_attn(bits(w.q), kc, vc, w.block_table.cpu().numpy(), ctx,
                                   kv_dtype=kv_dtype, scale_mode=mode, k_scale=k_s,
                                   v_scale=v_s, k_scale_cache=ks, v_scale_cache=vs,
                                   window=w.window, units=units, nthreads=cores)
        dt_s = time.perf_counter() - t
        assert st == 0
        if dt_s > seconds / 4 or n >= len(all_units) or max_units is not None:
            break
        n = min(len(all_units), n * 4)
    secs, passes = dt_s, 1
    while secs < seconds and passes < 64:
        t = time.perf_counter()
        oracle.decode_attn(bits(w.q), kc, vc, w.block_table.cpu().numpy(), ctx,
                           kv_dtype=kv_dtype, scale_mode=mode, k_scale=k_s, v_scale=v_s,
                           k_scale_cache=ks, v_scale_cache=vs, window=w.window, units=units,
                           nthreads=cores)
        secs += time.perf_counter() - t
        passes += 1
    keys_sample = sum(int(vis[b]) for b, _ in units)
    keys_all = sum(int(vis[b]) for b, _ in all_units)
    call_s = secs / passes * keys_all / max(keys_sample, 1)
    return {"kind": "oracle", "cores": cores, "ms_per_call": call_s * 1e3,
            "tokens_per_s": w.B / call_s,
            "sample": f"{len(units)} of {len(all_units)} (sequence, query head) units, "
                      f"{passes} pass(es), {secs:.1f} s; extrapolated by visible keys"}


def run_extras(args, dev):
    """The other workloads: decode time against context length (fp8 vs bf16),
    the 131k needle, the 24-layer hybrid model, chunked FP8 prefill and the
    bulk cache write.  One JSON line each."""
    import fp8_kv_cache_write_gb300 as fk
    from fp8_kv_cache_write_gb300 import synth
    stream = torch.cuda.Stream(dev)
    emit = lambda d: print(json.dumps(d), flush=True)
    E4, BF = fk.KV_E4M3, fk.KV_BF16

    want = lambda name: args.extras in ("all", name)

    # (1) inter-token latency against context, decode only, 32/8 heads, D=128:
    # B=8 at 2k..32k, and the single-request sweep B=1 at 1k..128k with fp8
    # per-token-head, fp8 per-tensor and bf16, fitted as t = a + b * ctx
    for ctx in (2048, 4096, 8192, 16384, 32768) if want("itl") else ():
        w = synth.decode_workload(2000 + ctx, [ctx] * 8, 32, 8, 128, 2, device=dev)
        row = {"extra": "itl_vs_context", "B": 8, "context": ctx}
        for kv, name in ((E4, "fp8"), (BF, "bf16")):
            mode = 2 if kv == E4 else 0
            d_b, _ = step_bytes(w, 1 if kv == E4 else 2, kv == E4)
            caches = _caches_for(fk, w, kv, mode, dev, _copies_for(d_b))
            ms = _time_graph(_decode_caller(fk, w, kv, mode, caches, dev), 64, stream)
            row[name + "_us"] = ms * 1e3
            row[name + "_gbs"] = d_b / ms / 1e6
            del caches
            torch.cuda.empty_cache()
        row["fp8_speedup"] = row["bf16_us"] / row["fp8_us"]
        emit(row)
        del w
    if want("itl"):
        variants = (("fp8_per_token_head", E4, 2), ("fp8_per_tensor", E4, 0), ("bf16", BF, 0))
        pts = {name: [] for name, _, _ in variants}
        for ctx in (1024, 2048, 4096, 8192, 16384, 32768, 65536, 131072):
            row = {"extra": "itl_single_request", "B": 1, "context": ctx}
            for name, kv, mode in variants:
                w = synth.decode_workload(3000 + ctx, [ctx], 32, 8, 128, mode, device=dev)
                d_b, _ = step_bytes(w, 1 if kv == E4 else 2, mode == 2)
                caches = _caches_for(fk, w, kv, mode, dev, _copies_for(d_b))
                ms = _time_graph(_decode_caller(fk, w, kv, mode, caches, dev), 64, stream)
                row[name + "_us"] = ms * 1e3
                pts[name].append((ctx, ms * 1e3))
                del caches, w
                torch.cuda.empty_cache()
            emit(row)
        fit = {"extra": "itl_single_request_fit", "B": 1, "model": "t_us = a + b * ctx"}
        for name, _, _ in variants:
            x = [c for c, _ in pts[name]]
            y = [t for _, t in pts[name]]
            n, mx, my = len(x), sum(x) / len(x), sum(y) / len(y)
            b = sum((xi - mx) * (yi - my) for xi, yi in zip(x, y)) / sum((xi - mx) ** 2 for xi in x)
            fit[name] = {"a_us": my - b * mx, "b_us_per_token": b}
        bb = fit["bf16"]["b_us_per_token"]
        for name in ("fp8_per_token_head", "fp8_per_tensor"):
            f = fit[name]
            f["slope_vs_bf16"] = f["b_us_per_token"] / bb
            db = bb - f["b_us_per_token"]
            f["break_even_ctx"] = (f["a_us"] - fit["bf16"]["a_us"]) / db if db > 0 else None
        emit(fit)

    # (2)-(6) the tiny decode, the 131072-token needle, the hybrid model, prefill,
    # the bulk write
    if want("tiny"):
        _extra_tiny(fk, synth, dev, stream, emit)
    if want("needle"):
        _extra_needle(fk, synth, dev, stream, emit)
    if want("hybrid"):
        _extra_hybrid(fk, synth, dev, stream, emit)
    if want("prefill"):
        _extra_prefill(fk, synth, dev, stream, emit)
    if want("write"):
        _extra_write(fk, dev, stream, emit)


def _extra_tiny(fk, synth, dev, stream, emit):
    # 1 sequence, context 1024, 32/8 heads, D 128, per-tensor scale 1.0: a decode
    # call is launch- and latency-bound (2 MiB of e4m3 KV)
    E4, BF = fk.KV_E4M3, fk.KV_BF16
    w = synth.tiny()
    row = {"extra": "tiny_decode", "B": 1, "context": 1024}
    for kv, name in ((E4, "fp8"), (BF, "bf16")):
        d_b, _ = step_bytes(w, 1 if kv == E4 else 2, False)
        caches = _caches_for(fk, w, kv, 0, dev, _copies_for(d_b))
        ms = _time_graph(_decode_caller(fk, w, kv, 0, caches, dev), 64, stream)
        row[name + "_us"] = ms * 1e3
        del caches
    if _CPU_BASELINE:
        row["cpu_baseline"] = _oracle_decode_baseline(w, 0, 0, seconds=3.0)
    emit(row)


def _extra_needle(fk, synth, dev, stream, emit):
    # 131072-token needle: B=1, 64/8 heads, per-KV-head scales
    E4, BF = fk.KV_E4M3, fk.KV_BF16
    w = synth.needle(device=dev)
    row = {"extra": "needle_131k", "B": 1, "context": 131072}
    for kv, name in ((E4, "fp8"), (BF, "bf16")):
        mode = 1 if kv == E4 else 0
        d_b, _ = step_bytes(w, 1 if kv == E4 else 2, False)
        caches = _caches_for(fk, w, kv, mode, dev, _copies_for(d_b))
        ms = _time_graph(_decode_caller(fk, w, kv, mode, caches, dev), 32, stream)
        row[name + "_us"], row[name + "_gbs"] = ms * 1e3, d_b / ms / 1e6
        del caches
        torch.cuda.empty_cache()
    row["fp8_speedup"] = row["bf16_us"] / row["fp8_us"]
    if _CPU_BASELINE:
        row["cpu_baseline"] = _oracle_decode_baseline(w, 0, 1)
    emit(row)


def _extra_hybrid(fk, synth, dev, stream, emit):
    # hybrid model, 24 layers alternating sliding-window-128 / full attention:
    #     one step = the decode of all 24 layers (each layer type rotates over
    #     its own cache copies); tokens/s = B / step time
    E4, BF = fk.KV_E4M3, fk.KV_BF16
    wl = {0: synth.hybrid_layer(layer=0, device=dev), 1: synth.hybrid_layer(layer=1, device=dev)}
    for variant, dtypes in (("all_bf16", (BF, BF)), ("all_fp8", (E4, E4)),
                            ("window_bf16_full_fp8", (BF, E4))):
        calls = []
        for lt in (0, 1):
            w, kv = wl[lt], dtypes[lt]
            mode = 2 if kv == E4 else 0
            d_b, _ = step_bytes(w, 1 if kv == E4 else 2, kv == E4)
            caches = _caches_for(fk, w, kv, mode, dev, 2 if lt == 0 else _copies_for(d_b))
            calls.append(_decode_caller(fk, w, kv, mode, caches, dev, window=w.window))

        def step(i):
            for layer in range(24):
                calls[layer % 2](i * 12 + layer // 2)
        ms = _time_graph(step, 8, stream)
        per_type = [_time_graph(calls[lt], 24, stream) * 1e3 for lt in (0, 1)]
        kv_b = [visible_kv_bytes(wl[lt], 1 if dtypes[lt] == E4 else 2, dtypes[lt] == E4)
                for lt in (0, 1)]
        step_b = 12 * (kv_b[0] + kv_b[1])
        hbm = measured_peaks()[0]
        line = {"extra": "hybrid_24_layers", "variant": variant, "B": 32,
                "ms_per_step": ms, "tokens_per_s": 32 / (ms / 1e3),
                "window_layer_us": per_type[0], "full_layer_us": per_type[1],
                "algorithmic_bytes_per_step": step_b,
                "step_gbs": step_b / (ms / 1e3) / 1e9,
                "step_frac_of_hbm": step_b / (ms / 1e3) / 1e9 / hbm,
                "full_layer_bytes": kv_b[1],
                "full_layer_gbs": kv_b[1] / per_type[1] / 1e3,
                "full_layer_frac_of_hbm": kv_b[1] / per_type[1] / 1e3 / hbm,
                "window_layer_bytes": kv_b[0]}
        if variant == "window_bf16_full_fp8" and _CPU_BASELINE:
            # the oracle on one layer of each type, 12 of each per step
            cb = [_oracle_decode_baseline(wl[lt], dtypes[lt] if lt == 0 else 0,
                                          0 if lt == 0 else 2, seconds=4.0) for lt in (0, 1)]
            step_ms = 12 * (cb[0]["ms_per_call"] + cb[1]["ms_per_call"])
            line["cpu_baseline"] = {"kind": "oracle", "cores": cb[1]["cores"],
                                    "ms_per_step": step_ms, "tokens_per_s": 32 / (step_ms / 1e3),
                                    "sample": "window layer: " + cb[0]["sample"] +
                                              "; full layer: " + cb[1]["sample"]}
        emit(line)
        del calls
        torch.cuda.empty_cache()


def _fp8_mm_peak(dev, n=8192, reps=10):
    """Dense e4m3 GEMM throughput of the library GEMM (torch._scaled_mm, bf16 out):
    the measured fp8 tensor peak that the prefill's fraction is taken against."""
    try:
        g = torch.Generator(device=dev).manual_seed(3)
        a = torch.randn(n, n, generator=g, device=dev).to(torch.float8_e4m3fn)
        b = torch.randn(n, n, generator=g, device=dev).to(torch.float8_e4m3fn).t()
        one = torch.ones((), dtype=torch.float32, device=dev)
        for _ in range(3):
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        best = float("inf")
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(reps):
            t0.record()
            torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
            t1.record()
            torch.cuda.synchronize(dev)
            best = min(best, t0.elapsed_time(t1))
        return 2.0 * n ** 3 / (best / 1e3) / 1e12
    except Exception as e:                      # no fp8 GEMM in this torch build
        return {"unavailable": str(e).splitlines()[0][:120]}


def _oracle_prefill_baseline(w, rows=16, seconds=6.0):
    """The oracle on `rows` query rows spread over the chunk (all query heads),
    extrapolated to the whole chunk by (query, key) pairs."""
    import numpy as np

    import oracle
    bits = lambda t: t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    nb, Hkv, D = w.num_blocks, w.Hkv, w.D
    kc, vc = np.zeros((nb, Hkv, 16, D), np.uint8), np.zeros((nb, Hkv, 16, D), np.uint8)
    one = np.ones(1, np.float32)
    assert oracle.kv_cache_write(bits(w.k_all), bits(w.v_all), w.all_slots.cpu().numpy(), kc, vc,
                                 kv_dtype=0, scale_mode=0, k_scale=one, v_scale=one) == 0
    nq = int(w.cu_seqlens_q[1])
    c0 = int(w.context_lens[0]) - nq
    toks = [int(t) for t in np.linspace(0, nq - 1, rows)]
    units = [(t, h) for t in toks for h in range(w.Hq)]
    cores = len(os.sched_getaffinity(0))
    secs, passes = 0.0, 0
    while passes == 0 or (secs < seconds and passes < 16):
        t = time.perf_counter()
        st, _ = oracle.prefill_attn(bits(w.q), w.cu_seqlens_q.cpu().numpy(), kc, vc,
                                    w.block_table.cpu().numpy(), w.context_lens.cpu().numpy(),
                                    kv_dtype=0, scale_mode=0, k_scale=one, v_scale=one,
                                    units=units, nthreads=cores)
        secs += time.perf_counter() - t
        passes += 1
        assert st == 0
    pairs_sample = sum(c0 + t + 1 for t in toks)
    pairs_all = sum(c0 + i + 1 for i in range(nq))
    call_s = secs / passes * pairs_all / pairs_sample
    return {"kind": "oracle", "cores": cores, "ms_per_call": call_s * 1e3,
            "tflops": 4.0 * D * w.Hq * pairs_all / call_s / 1e12,
            "sample": f"{rows} of {nq} query rows x {w.Hq} heads, {passes} pass(es), "
                      f"{secs:.1f} s; extrapolated by (query, key) pairs"}


def _extra_prefill(fk, synth, dev, stream, emit):
    # chunked prefill: 4096 new queries over 32768 cached tokens, 8/1 heads, D=256
    E4, BF = fk.KV_E4M3, fk.KV_BF16
    peak = _fp8_mm_peak(dev)
    emit({"extra": "fp8_dense_gemm_peak", "how": "torch._scaled_mm e4m3 8192^3, bf16 out, "
                                                  "best of 10", "tflops": peak})
    w = synth.prefill(device=dev)
    q, cu = w.q.to(dev), w.cu_seqlens_q.to(dev)
    bt, cl = w.block_table.to(dev), w.context_lens.to(dev)
    one = torch.ones(1, dtype=torch.float32, device=dev)
    out = torch.empty(q.shape[0], w.Hq, w.D, dtype=torch.float32, device=dev)
    c0 = int(w.context_lens[0]) - int(w.cu_seqlens_q[1])
    pairs = sum(c0 + i + 1 for i in range(int(w.cu_seqlens_q[1])))
    flops = 4.0 * w.D * w.Hq * pairs
    for kv, name in ((E4, "fp8"), (BF, "bf16")):
        dt = torch.uint8 if kv == E4 else torch.bfloat16
        kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=dt, device=dev)
        vc = torch.zeros_like(kc)
        fk.kv_cache_write(w.k_all.to(dev), w.v_all.to(dev), w.all_slots.to(dev), kc, vc,
                          kv_dtype=kv, scale_mode=0, k_scale=one, v_scale=one)
        # split operands ("always") cost two MMAs per contraction; "auto" takes
        # single operands here (every row sees >= 28673 keys)
        variants = [(False, "auto"), (True, "auto")] + (
            [(False, "always"), (True, "always")] if kv == E4 else [])
        for two, split in variants:
            fn = lambda i, kc=kc, vc=vc, kv=kv, two=two, split=split: fk.prefill_attn(
                q, cu, w.max_seqlen_q, kc, vc, bt, cl, kv_dtype=kv, k_scale=one, v_scale=one,
                two_level=two, split=split, out=out)
            ms = _time_graph(fn, 10, stream)
            line = {"extra": "prefill_chunk4096_ctx32768_d256", "kv": name, "two_level": two,
                    "split": split, "ms": ms, "tflops": flops / ms / 1e9}
            if kv == E4 and isinstance(peak, float):
                line["frac_of_fp8_peak"] = flops / ms / 1e9 / peak
            if kv == E4 and not two and split == "auto" and _CPU_BASELINE:
                line["cpu_baseline"] = _oracle_prefill_baseline(w)
            emit(line)
            if kv == E4 and split == "auto":
                # the same call with one CTA per query tile (no workspace): what the
                # balanced persistent launch gains
                fn = lambda i, kc=kc, vc=vc, two=two: fk.prefill_attn(
                    q, cu, w.max_seqlen_q, kc, vc, bt, cl, kv_dtype=E4, k_scale=one,
                    v_scale=one, two_level=two, out=out, workspace=None)
                ms1 = _time_graph(fn, 10, stream)
                emit({"extra": "prefill_chunk4096_ctx32768_d256", "kv": name, "two_level": two,
                      "split": split, "launch": "one CTA per query tile", "ms": ms1,
                      "tflops": flops / ms1 / 1e9})
        del kc, vc
        torch.cuda.empty_cache()
    # the same chunk over a per-token-head e4m3 cache (scales computed at write time)
    kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    ksc = torch.zeros(w.num_blocks, w.Hkv, 16, dtype=torch.float32, device=dev)
    vsc = torch.zeros_like(ksc)
    fk.kv_cache_write(w.k_all.to(dev), w.v_all.to(dev), w.all_slots.to(dev), kc, vc, kv_dtype=E4,
                      scale_mode=fk.SCALE_PER_TOKEN_HEAD, k_scale_cache=ksc, v_scale_cache=vsc)
    for two, split in ((False, "auto"), (True, "auto"), (False, "always")):
        fn = lambda i, two=two, split=split: fk.prefill_attn(
            q, cu, w.max_seqlen_q, kc, vc, bt, cl, kv_dtype=E4,
            scale_mode=fk.SCALE_PER_TOKEN_HEAD, k_scale_cache=ksc, v_scale_cache=vsc,
            two_level=two, split=split, out=out)
        ms = _time_graph(fn, 10, stream)
        emit({"extra": "prefill_chunk4096_ctx32768_d256", "kv": "fp8 per-token-head",
              "two_level": two, "split": split, "ms": ms, "tflops": flops / ms / 1e9})
    del kc, vc, ksc, vsc
    torch.cuda.empty_cache()
    # the other geometry: the 4096-query chunk after a complete 32768-token prefix
    w2 = synth.prefill(seed=1015, ctx=(36864,), chunk=(4096,), device=dev)
    q2, cu2 = w2.q.to(dev), w2.cu_seqlens_q.to(dev)
    bt2, cl2 = w2.block_table.to(dev), w2.context_lens.to(dev)
    c2 = int(w2.context_lens[0]) - int(w2.cu_seqlens_q[1])
    flops2 = 4.0 * w2.D * w2.Hq * sum(c2 + i + 1 for i in range(int(w2.cu_seqlens_q[1])))
    kc = torch.zeros(w2.num_blocks, w2.Hkv, 16, w2.D, dtype=torch.uint8, device=dev)
    vc = torch.zeros_like(kc)
    fk.kv_cache_write(w2.k_all.to(dev), w2.v_all.to(dev), w2.all_slots.to(dev), kc, vc,
                      kv_dtype=E4, scale_mode=0, k_scale=one, v_scale=one)
    fn = lambda i: fk.prefill_attn(q2, cu2, w2.max_seqlen_q, kc, vc, bt2, cl2, kv_dtype=E4,
                                   k_scale=one, v_scale=one, two_level=False, out=out)
    ms = _time_graph(fn, 10, stream)
    emit({"extra": "prefill_chunk4096_after_prefix32768_d256", "kv": "fp8", "two_level": False,
          "ms": ms, "tflops": flops2 / ms / 1e9})
    del kc, vc
    torch.cuda.empty_cache()


def _extra_write(fk, dev, stream, emit):
    # bulk cache write, 8 KV heads x 128, per-token-head e4m3: 32768 tokens, and the
    # whole 158367-token history of the Llama-3.1-8B-shaped decode workload
    E4 = fk.KV_E4M3
    H, D = 8, 128
    for T in (32768, 158367):
        gen = torch.Generator(device=dev).manual_seed(6)
        sets = []
        for _ in range(2):
            k = torch.randn(T, H, D, generator=gen, device=dev).to(torch.bfloat16)
            v = torch.randn(T, H, D, generator=gen, device=dev).to(torch.bfloat16)
            sets.append((k, v))
        # prefill-style slots: 16 consecutive tokens per page, pages in shuffled order
        npages = (T + 15) // 16
        nb = npages + 16
        pages = torch.randperm(nb, generator=gen, device=dev)[:npages].to(torch.int64)
        slots = (pages[:, None] * 16 + torch.arange(16, device=dev)).reshape(-1)[:T].contiguous()
        kc = torch.zeros(nb, H, 16, D, dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros(nb, H, 16, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        fn = lambda i: fk.kv_cache_write(sets[i % 2][0], sets[i % 2][1], slots, kc, vc,
                                         kv_dtype=E4, scale_mode=2, k_scale_cache=ks,
                                         v_scale_cache=vs)
        ms = _time_graph(fn, 20, stream)
        nbytes = T * H * (2 * D * 2 + 2 * D + 8) + T * 8
        emit({"extra": "bulk_cache_write", "tokens": T, "Hkv": H, "D": D, "us": ms * 1e3,
              "gbs": nbytes / ms / 1e6})
        del sets, kc, vc, ks, vs
        torch.cuda.empty_cache()


def run_profile_case(args):
    """A few eager calls of one kernel on one workload, nothing else on the GPU:
    the target of the ncu captures summarised under profiles/."""
    import fp8_kv_cache_write_gb300 as fk
    from fp8_kv_cache_write_gb300 import synth
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    case = args.profile
    if case in ("hybrid_full", "hybrid_window", "needle"):
        if case == "needle":
            w, kv, mode = synth.needle(device=dev), fk.KV_E4M3, 1
        else:
            w = synth.hybrid_layer(layer=1 if case == "hybrid_full" else 0, device=dev)
            kv = w.extra["kv_dtype"]
            mode = 2 if kv == fk.KV_E4M3 else 0
        caches = _caches_for(fk, w, kv, mode, dev, 1)
        fn = _decode_caller(fk, w, kv, mode, caches, dev, window=w.window)
    elif case in ("prefill", "prefill_pt"):
        w = synth.prefill(device=dev)
        mode = 2 if case == "prefill_pt" else 0
        one = torch.ones(1, dtype=torch.float32, device=dev)
        kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.num_blocks, w.Hkv, 16, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        fk.kv_cache_write(w.k_all.to(dev), w.v_all.to(dev), w.all_slots.to(dev), kc, vc,
                          kv_dtype=fk.KV_E4M3, scale_mode=mode, k_scale=one, v_scale=one,
                          k_scale_cache=ks, v_scale_cache=vs)
        q, cu = w.q.to(dev), w.cu_seqlens_q.to(dev)
        bt, cl = w.block_table.to(dev), w.context_lens.to(dev)
        out = torch.empty(q.shape[0], w.Hq, w.D, dtype=torch.float32, device=dev)
        fn = lambda i: fk.prefill_attn(q, cu, w.max_seqlen_q, kc, vc, bt, cl, kv_dtype=fk.KV_E4M3,
                                       scale_mode=mode, k_scale=one, v_scale=one,
                                       k_scale_cache=ks, v_scale_cache=vs, out=out)
    else:                                           # bulk write, llama8b history
        w = synth.llama8b(device=dev)
        kh, vh, hs = w.k_hist.to(dev), w.v_hist.to(dev), w.hist_slots.to(dev)
        kc = torch.zeros(w.num_blocks, w.Hkv, 16, w.D, dtype=torch.uint8, device=dev)
        vc = torch.zeros_like(kc)
        ks = torch.zeros(w.num_blocks, w.Hkv, 16, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        fn = lambda i: fk.kv_cache_write(kh, vh, hs, kc, vc, kv_dtype=fk.KV_E4M3,
                                         scale_mode=fk.SCALE_PER_TOKEN_HEAD,
                                         k_scale_cache=ks, v_scale_cache=vs)
    for i in range(args.calls):
        fn(i)
    torch.cuda.synchronize(dev)
    print(json.dumps({"profile": case, "calls": args.calls}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--only", choices=["fp8", "bf16"], default=None,
                    help="time one cache dtype only (profiling runs)")
    ap.add_argument("--rotations", type=int, default=ROTATIONS,
                    help="cache copies rotated between steps (each larger than L2)")
    ap.add_argument("--splits", type=int, default=0, help="decode split count (0 = planner)")
    ap.add_argument("--decode-flags", type=int, default=2,
                    help="decode launch-overlap flags (0 = wait for the preceding kernel "
                         "first; 2 = early set-up and page streaming: the step's tables and "
                         "older pages are written before the preceding kernel starts)")
    ap.add_argument("--extras", nargs="?", const="all", default=None,
                    choices=["all", "itl", "tiny", "needle", "hybrid", "prefill", "write"],
                    help="time the other workloads (itl, tiny, needle, hybrid, prefill, write; "
                         "all by default) instead of the headline step; one JSON line each")
    ap.add_argument("--profile", default=None,
                    choices=["hybrid_full", "hybrid_window", "needle", "prefill", "prefill_pt",
                             "write"],
                    help="run --calls eager calls of one workload's kernel (for profiler "
                         "captures; prints no measurement)")
    ap.add_argument("--calls", type=int, default=3)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.profile:
        run_profile_case(args)
        return

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    if args.extras and args.impl == "ours":
        import fp8_kv_cache_write_gb300 as fk
        global _DECODE_FLAGS, _CPU_BASELINE
        _DECODE_FLAGS = args.decode_flags
        _CPU_BASELINE = not args.no_cpu_baseline
        fk.lib()
        dev = torch.device("cuda", local)
        torch.cuda.set_device(dev)
        if rank == 0:
            run_extras(args, dev)
        return

    from fp8_kv_cache_write_gb300 import synth
    w = synth.llama8b(seed=1002 + rank)
    if args.impl == "reference":
        line = run_reference(args, w, world, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return

    import fp8_kv_cache_write_gb300 as fk
    fk.lib()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    res, dec_bytes, lps = run_ours(args, dev, w, world, rank)
    peak, peak_kind = measured_peaks()
    if args.only:                       # profiling / sweep runs: a short line
        r = res[args.only]
        if rank == 0:
            print(json.dumps({"only": args.only, "splits": r["num_splits"],
                              "step_gbs": r["gbs"], "ms_per_step": r["ms_per_step"],
                              "decode_ms": r["decode_ms"], "split_step_ms": r["split_step_ms"],
                              "wait_first_step_ms": r["wait_first_step_ms"],
                              "decode_gbs": dec_bytes[args.only] / r["decode_ms"] / 1e6,
                              "tokens_per_s": r["tokens_per_s"], "clocks": r["clocks"]}),
                  flush=True)
    else:
        fp8, bf16 = res["fp8"], res["bf16"]
        achieved = dec_bytes["fp8"] / (fp8["decode_ms"] / 1e3) / 1e9
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            ob = OracleBaseline(w)
            gbs, tps, secs, sample = ob.run(min_seconds=10.0)   # ~10 s of host work
            cpu = {"value": gbs, "unit": "GB/s", "tokens_per_s": tps, "cores": ob.cores,
                   "kind": "oracle", "sample": sample + f"; {secs:.2f} s wall"}
        if rank == 0:
            line = {
                "metric": METRIC, "value": fp8["gbs"], "unit": "GB/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": fp8["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "e4m3", "data": "synthetic",
                "config": {"workload": WORKLOAD, "global_batch": 8 * world,
                           "parallelism": f"replicas x{world}",
                           "l2": f"{args.rotations} rotating cache copies, each larger than L2",
                           "num_splits": fp8["num_splits"],
                           "decode_flags": args.decode_flags,
                           "timing": "CUDA graphs of whole steps replayed back to back"},
                "wait_first_ms_per_step": fp8["wait_first_step_ms"],
                "pct_of_peak": fp8["gbs"] / peak,
                "tokens_per_s": fp8["tokens_per_s"],
                "bf16_twin": {"value": bf16["gbs"], "unit": "GB/s",
                              "tokens_per_s": bf16["tokens_per_s"],
                              "ms_per_step": bf16["ms_per_step"],
                              "decode_ms": bf16["decode_ms"],
                              "decode_gbs": dec_bytes["bf16"] / bf16["decode_ms"] / 1e6},
                "fp8_vs_bf16_tokens_per_s": fp8["tokens_per_s"] / bf16["tokens_per_s"],
                "roofline": {"bound": "hbm", "kernel": "paged_decode_attn (split + split_merge)",
                             "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                             "unit": "GB/s", "frac": achieved / peak,
                             "traffic": profiled_traffic(),
                             "algorithmic_bytes_per_launch": dec_bytes["fp8"],
                             "decode_ms": fp8["decode_ms"]},
                "cpu_baseline": cpu,
                "e2e": res.get("e2e"),
                "gpu_launches": lps["fp8"] * args.steps,
                "clocks": fp8["clocks"],
            }
            print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
