"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws inputs: bf16 K/V/Q tensors, context lengths, shuffled page
tables and the slot of every token.  It holds none of the method's arithmetic
(no quantization, no attention), so the CUDA path and the oracle can both be fed
from it.  Everything is drawn on the CPU from ``torch.Generator().manual_seed``
unless ``device`` asks for a CUDA generator (benchmark-only sizes, where the
oracle checks sampled outputs on bytes copied back from the device).

Workloads (sizes as named by the FP8 KV-cache pages' benchmarks):
  tiny        1 seq, context 1024, 32 Q / 8 KV heads, D 128, per-tensor scale 1.0
  llama8b     8 seqs, contexts uniform in [18000, 22000], 32/8 heads, D 128,
              per-token-head scales, 1% of (head, channel) pairs scaled x20
  needle      1 seq, context 131072, 64/8 heads, D 128, per-KV-head scales, one
              key aligned to a query so that its scaled logit is +12
  hybrid      32 seqs, contexts log-uniform in [1024, 32768], 64/8 heads, D 64,
              24 layers alternating sliding-window-128 (bf16) / full (fp8)
  prefill     4096 new queries at the end of a 32768-token cache, 8 Q / 1 KV
              head, D 256, per-tensor scale 1.0
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

PAGE = 16


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, gen, device="cpu", std=1.0) -> torch.Tensor:
    """N(0, std^2) drawn in fp32, rounded to bf16."""
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16)


def shuffled_block_table(context_lens, gen, spare_blocks=0):
    """Pages of every sequence drawn from one random permutation of the cache.

    Returns (block_table int32 [B][max_blocks], num_blocks).  Entries past a
    sequence's last page are -1 so that an out-of-range read is detectable.
    """
    pages = [(int(c) + PAGE - 1) // PAGE for c in context_lens]
    num_blocks = sum(pages) + spare_blocks
    perm = torch.randperm(max(num_blocks, 1), generator=gen)[:num_blocks].to(torch.int32)
    max_blocks = max(max(pages) if pages else 0, 1)
    bt = torch.full((len(pages), max_blocks), -1, dtype=torch.int32)
    at = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[at:at + n]
        at += n
    return bt, max(num_blocks, 1)


def slots_for(block_table, seq_positions):
    """Slot (block * 16 + offset) of each (seq, position) pair, int64."""
    out = torch.empty(len(seq_positions), dtype=torch.int64)
    for i, (s, p) in enumerate(seq_positions):
        out[i] = int(block_table[s, p // PAGE]) * PAGE + p % PAGE if p >= 0 else -1
    return out


def history_slots(block_table, context_lens, upto_last=True):
    """Slots of positions 0 .. ctx-2 (or ctx-1) of every sequence, packed in order."""
    parts = []
    for s, c in enumerate(context_lens):
        n = int(c) - (1 if upto_last else 0)
        if n <= 0:
            continue
        pos = torch.arange(n, dtype=torch.int64)
        blk = block_table[s, (pos // PAGE)].to(torch.int64)
        parts.append(blk * PAGE + pos % PAGE)
    return torch.cat(parts) if parts else torch.empty(0, dtype=torch.int64)


@dataclass
class DecodeWorkload:
    """One decode step: the cache is filled with ctx-1 tokens per sequence, then
    each sequence writes its new token at position ctx-1 and its queries attend to
    all ctx tokens (the new one included)."""
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    scale_mode: int                  # 0 tensor, 1 per KV head, 2 per token-head
    context_lens: torch.Tensor       # int32 [B]
    block_table: torch.Tensor        # int32 [B][max_blocks]
    num_blocks: int
    k_hist: torch.Tensor             # bf16 [T_hist][Hkv][D]
    v_hist: torch.Tensor
    hist_slots: torch.Tensor         # int64 [T_hist]
    k_new: torch.Tensor              # bf16 [B][Hkv][D]
    v_new: torch.Tensor
    new_slots: torch.Tensor          # int64 [B]
    q: torch.Tensor                  # bf16 [B][Hq][D]
    k_scale: torch.Tensor = None     # fp32 [1] or [Hkv] (per-tensor / per-head)
    v_scale: torch.Tensor = None
    window: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)


def _decode_common(name, seed, context_lens, Hq, Hkv, D, scale_mode, device="cpu",
                   outlier_frac=0.0, spare_blocks=0):
    g = _gen(seed)
    context_lens = torch.as_tensor(context_lens, dtype=torch.int32)
    B = context_lens.numel()
    bt, nb = shuffled_block_table(context_lens.tolist(), g, spare_blocks)
    hs = history_slots(bt, context_lens.tolist())
    T = hs.numel()
    gd = _gen(seed + 7, device) if device != "cpu" else g
    k_hist = normal_bf16((T, Hkv, D), gd, device)
    v_hist = normal_bf16((T, Hkv, D), gd, device)
    k_new = normal_bf16((B, Hkv, D), gd, device)
    v_new = normal_bf16((B, Hkv, D), gd, device)
    q = normal_bf16((B, Hq, D), gd, device)
    extra = {}
    if outlier_frac > 0:
        n_out = math.ceil(outlier_frac * Hkv * D)
        idx = torch.randperm(Hkv * D, generator=g)[:n_out]
        heads, chans = (idx // D).tolist(), (idx % D).tolist()
        for t in (k_hist, v_hist, k_new, v_new):
            for h, c in zip(heads, chans):
                t[:, h, c] = (t[:, h, c].float() * 20.0).to(torch.bfloat16)
        extra["outliers"] = list(zip(heads, chans))
    new_pos = [(s, int(c) - 1) for s, c in enumerate(context_lens.tolist())]
    ns = slots_for(bt, new_pos)
    w = DecodeWorkload(name, B, Hq, Hkv, D, scale_mode, context_lens, bt, nb, k_hist, v_hist,
                       hs, k_new, v_new, ns, q, extra=extra)
    if scale_mode == 0:
        w.k_scale = torch.ones(1, dtype=torch.float32)
        w.v_scale = torch.ones(1, dtype=torch.float32)
    return w


def tiny(seed=1001, device="cpu") -> DecodeWorkload:
    """1 seq, context 1024, 32/8 heads, D 128, per-tensor scale 1.0."""
    return _decode_common("tiny", seed, [1024], 32, 8, 128, 0, device)


def llama8b(seed=1002, device="cpu", B=8, ctx_lo=18000, ctx_hi=22000) -> DecodeWorkload:
    """Llama-3.1-8B-shaped decode under load: contexts uniform in [18k, 22k],
    per-token-head scales, 1% of (head, channel) pairs scaled x20."""
    g = _gen(seed + 1)
    ctx = torch.randint(ctx_lo, ctx_hi + 1, (B,), generator=g, dtype=torch.int64)
    return _decode_common("llama8b", seed, ctx.tolist(), 32, 8, 128, 2, device,
                          outlier_frac=0.01)


def per_head_calibration(k_all: torch.Tensor) -> torch.Tensor:
    """Calibration stand-in for per-KV-head scales: the largest |value| a head
    holds over all its tokens, divided by e4m3's largest finite value (448),
    so that no code saturates.  (Scales are inputs of the method; calibration
    itself is outside it.)"""
    amax = k_all.float().abs().amax(dim=(0, 2))
    return (amax / 448.0).to(torch.float32).cpu()


def needle(seed=1003, device="cpu", ctx=131072, Hq=64, Hkv=8, D=128,
           logit=12.0) -> DecodeWorkload:
    """One sequence with one key aligned to query head hq* so that
    softmax_scale * q . k = +logit; its value is N(0,1) * 4."""
    w = _decode_common("needle", seed, [ctx], Hq, Hkv, D, 1, device)
    g = _gen(seed + 2)
    G = Hq // Hkv
    pos = int(torch.randint(0, ctx - 1, (1,), generator=g))
    hq = int(torch.randint(0, Hq, (1,), generator=g))
    h = hq // G
    qv = w.q[0, hq].float()
    k_needle = (logit * math.sqrt(D)) * qv / (qv * qv).sum()
    v_needle = torch.randn(D, generator=g, dtype=torch.float32) * 4.0
    # position pos < ctx-1 lives in the history rows; its row index is pos
    w.k_hist[pos, h] = k_needle.to(torch.bfloat16).to(w.k_hist.device)
    w.v_hist[pos, h] = v_needle.to(torch.bfloat16).to(w.v_hist.device)
    k_all = torch.cat([w.k_hist, w.k_new])
    v_all = torch.cat([w.v_hist, w.v_new])
    w.k_scale = per_head_calibration(k_all)
    w.v_scale = per_head_calibration(v_all)
    w.extra.update(needle_pos=pos, needle_hq=hq, needle_h=h)
    return w


def hybrid_context_lens(seed, B=32, lo=1024, hi=32768):
    g = _gen(seed + 1)
    u = torch.rand(B, generator=g, dtype=torch.float64)
    return torch.round(torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))).to(torch.int32)


def hybrid_layer(seed=1004, layer=0, device="cpu", B=32, ctx_lo=1024, ctx_hi=32768,
                 window=128) -> DecodeWorkload:
    """One layer of the gpt-oss-20b-like hybrid model: even layers are
    sliding-window-128 layers (kept bf16), odd layers full-attention layers
    (e4m3, per-token-head scales).  All layers share the context lengths."""
    ctx = hybrid_context_lens(seed, B, ctx_lo, ctx_hi)
    w = _decode_common(f"hybrid.L{layer}", seed + 100 * layer, ctx.tolist(), 64, 8, 64, 2,
                       device)
    w.window = window if layer % 2 == 0 else 0
    w.extra["kv_dtype"] = 1 if layer % 2 == 0 else 0
    return w


@dataclass
class PrefillWorkload:
    name: str
    Hq: int
    Hkv: int
    D: int
    context_lens: torch.Tensor      # int32 [B] (all keys, chunk included)
    cu_seqlens_q: torch.Tensor      # int32 [B+1]
    block_table: torch.Tensor
    num_blocks: int
    k_all: torch.Tensor             # bf16 [sum ctx][Hkv][D], every position of every seq
    v_all: torch.Tensor
    all_slots: torch.Tensor         # int64
    q: torch.Tensor                 # bf16 [Tq][Hq][D]
    k_scale: torch.Tensor
    v_scale: torch.Tensor

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def max_seqlen_q(self) -> int:
        return int((self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).max())


def prefill(seed=1005, device="cpu", ctx=(32768,), chunk=(4096,), Hq=8, Hkv=1,
            D=256) -> PrefillWorkload:
    """Chunked prefill: the last `chunk` positions of each `ctx`-token sequence are
    new queries; the whole sequence (chunk included) is in the cache."""
    g = _gen(seed)
    ctx = torch.as_tensor(ctx, dtype=torch.int32)
    chunk = torch.as_tensor(chunk, dtype=torch.int32)
    bt, nb = shuffled_block_table(ctx.tolist(), g)
    slots = history_slots(bt, ctx.tolist(), upto_last=False)
    gd = _gen(seed + 7, device) if device != "cpu" else g
    k_all = normal_bf16((slots.numel(), Hkv, D), gd, device)
    v_all = normal_bf16((slots.numel(), Hkv, D), gd, device)
    cu = torch.zeros(ctx.numel() + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(chunk, 0)
    q = normal_bf16((int(cu[-1]), Hq, D), gd, device)
    one = torch.ones(1, dtype=torch.float32)
    return PrefillWorkload("prefill", Hq, Hkv, D, ctx, cu, bt, nb, k_all, v_all, slots, q,
                           one, one.clone())


def decode_workload(seed, context_lens, Hq, Hkv, D, scale_mode, outlier_frac=0.0,
                    spare_blocks=0, window=0, name="custom", device="cpu") -> DecodeWorkload:
    """A decode step with explicit context lengths (parity tests' ragged cases).
    Per-tensor / per-head scales default to 1.0 / a per-head calibration."""
    w = _decode_common(name, seed, context_lens, Hq, Hkv, D, scale_mode, device,
                       outlier_frac=outlier_frac, spare_blocks=spare_blocks)
    w.window = window
    if scale_mode == 1:
        w.k_scale = per_head_calibration(torch.cat([w.k_hist, w.k_new]))
        w.v_scale = per_head_calibration(torch.cat([w.v_hist, w.v_new]))
    return w
