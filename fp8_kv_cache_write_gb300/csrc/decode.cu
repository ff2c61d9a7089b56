// decode.cu -- paged_decode_attn + split_merge: one query token per sequence
// attends to its paged e4m3 (or bf16) KV cache.
//
// What it computes ("vLLM FP8 KV-Cache 및 Attention 양자화 업데이트": attention runs
// over the FP8 cache (opening paragraph), per-KV-head scales ("커널 및 퓨전
// 최적화"), sliding-window layers on a bf16 cache ("하이브리드 Attention 및 레이어
// 스킵"); "[vLLM] KV Cache Quantization": per-token-head scales): for query head
// hq of sequence b and KV head h = hq / G,
//     z_t = softmax_scale * q . (s_k(t) * code_k(t)),  o = sum_t softmax(z)_t s_v(t) code_v(t)
// over the visible positions t (all ctx keys, or the last `window`).
//
// Design (GB300):
//   * one wave of CTAs of 4 warps; every warp is an independent worker: the
//     (seq, unit, page) tiles of the whole launch are flattened and each warp
//     takes an equal consecutive share, crossing units where its share does, so
//     any mix of context lengths keeps all SMs equally busy.  A unit is one KV
//     head, or -- with G = 2 or 4 query heads per KV head, an even KV head count
//     and tiles of at most 2 KiB -- two adjacent KV heads, whose query heads
//     share the 8 MMA columns and whose page tiles are adjacent in the cache
//     (one copy request and one softmax serve both).
//     Each warp runs its own ring that streams straight across unit
//     boundaries: lane 0 issues 3-D tiled tensor copies (128-byte swizzle) of the
//     K and V page tiles -- plus the 64-byte per-token scale rows -- onto an
//     mbarrier, S stages ahead (1 KiB tiles: 16-byte copies from every lane);
//     two tiles per iteration.
//   * math on the legacy tensor pipe (mma.sync m16n8k16, fp32 accumulate):
//     S^T = K_page . Q^T with M = 16 page tokens, N = 8 query heads of the
//     unit, K = D; then O^T += V_page^T . P^T with M = D, N = heads, K = the 16
//     tokens (for a unit of two KV heads, each head's P^T keeps only its own
//     columns).  e4m3 codes convert exactly to f16 (one cvt per pair), Q is
//     scaled by a per-head power of two into f16's top binade (exact), and P is
//     split into hi + lo halves so the PV product keeps ~22 bits.
//   * per-token-head scales fold out of the dot products: one multiply per
//     logit (k) and per weight (v).  Per-tensor / per-head scales multiply the
//     logit scale and the final output.
//   * online softmax in base 2 with a lazy max (the running max moves only when
//     a page exceeds it by 2^4 for e4m3, 2^8 for bf16), fp32 everywhere.
//   * the fragment row/column orders are permuted (token pi(g), d-chunk pi(g))
//     so that every 16-byte shared-memory read of the swizzled tiles is free of
//     bank conflicts for D = 128 e4m3; the permutation is undone when writing.
//   * a warp that covers a whole unit writes `out` directly; otherwise it leaves
//     (m, l, unnormalised O) in workspace slot worker + unit and split_merge
//     combines the workers that touched each unit.  (A merge inside this kernel,
//     by the CTA that completes a unit, ran slower: its loads queue behind the
//     other SMs' streaming, while split_merge runs on an idle memory system.)
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fp8kv {

namespace {

constexpr int kWarps = kDecodeWarps;
__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }
constexpr float kMaxInit = -1.0e30f;   // running-max start: finite, below any real logit

template <int D, bool BF16, int NT = 1, int HPT = 1>
struct Cfg {
    static constexpr int kElem = BF16 ? 2 : 1;
    static constexpr int kRowB = D * kElem;           // bytes of one token row
    static constexpr int kTileB = kPage * kRowB;      // bytes of one (page, head) tile
    // HPT = 2 packs two adjacent KV heads (of at most 4 query heads each) into
    // the 8 MMA columns: their tiles of a page are adjacent in the cache, so one
    // copy request moves both, and one softmax serves both.  Tiles of at most
    // 2 KiB only (shared memory).
    static_assert(HPT == 1 || (HPT == 2 && kRowB <= 128 && NT == 1), "head packing");
    // pages per iteration: two when a page tile is small and heads are not
    // packed, so each warp works on two independent tiles between waits
    static constexpr int kPPI = HPT > 1 ? 1 : (kRowB <= 128 ? 2 : 1);
    static constexpr int kTiles = kPPI * HPT;         // (page, head) tiles per tensor per stage
    static constexpr int kStageB = 2 * kTiles * kTileB; // K tiles, then V tiles
    // how a stage is filled: 64-byte rows (1 KiB tiles) by 16-byte copies from
    // every lane (many small requests in flight stream short tiles faster),
    // other rows by one lane's tensor copies
    static constexpr bool kLaneCopies = kRowB == 64;
    // bytes in flight per warp: 16 KiB, 12 KiB for 64-byte rows (4 CTAs per SM)
    static constexpr int kStagesRaw = (kRowB == 64 ? 12288 : 16384) / kStageB;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kSegs = kRowB / 64;          // 64-byte segments of a row
    static constexpr int kKPerSeg = 4 / kElem;        // QK k-steps per segment
    static constexpr int kKSteps = D / 16;
    static constexpr int kMTiles = D / 16;            // PV m-tiles (rows of O^T)
    static constexpr int kVBytes = (D / 8) * kElem;   // V bytes a lane reads per token
    static constexpr int kVWords = kVBytes / 4;
    static constexpr int kBoxes = kRowB >= 128 ? kRowB / 128 : 1;
    static constexpr int kWarpSmem = kStages * kStageB;
    static constexpr int kScaleB = 128;               // k + v scales of one (page, head) tile
    static constexpr int kMaxSeg = 16;                // segments a warp lists per pass
    static constexpr int kSegInts = 7;                // ints of one segment record
    static constexpr int kOffBars = kWarps * kWarpSmem + kWarps * kStages * kTiles * kScaleB;
    static constexpr int kOffSegs = kOffBars + kWarps * kStages * 8;
    static constexpr int kOffShare = kOffSegs + kWarps * kMaxSeg * kSegInts * 4;  // [warp][resume, end]
    static constexpr int kOffCtx = kOffShare + kWarps * 16;    // [warp][32] context lengths
    // CTA units: what each warp left for the CTA's combine (0 nothing, 1 a partial
    // in its ring, 2 its unit's output, written whole)
    static constexpr int kOffFlag = kOffCtx + kWarps * 128;
    // NT = 2 (more than 8 query heads per KV head): each warp's query fragments of
    // both 8-head groups, [group][k-step][lane] (8 bytes each), in shared memory
    static constexpr int kOffQsm = kOffFlag + kWarps * 4;
    static constexpr int kQsmBytes = NT > 1 ? kWarps * NT * kKSteps * 32 * 8 : 0;
    static constexpr int kSmem = 1024 + kOffQsm + kQsmBytes;
    // fused step only, after the above: per warp the new token's K row, V row
    // (as stored in the cache) and its two per-token-head scales
    static constexpr int kOffNew = kOffQsm + kQsmBytes;
    static constexpr int kNewB = (2 * kRowB + 8 + 15) / 16 * 16;
    static constexpr int kSmemFused = kSmem + kWarps * HPT * kNewB;
    static_assert(kSegs * kKPerSeg == kKSteps, "k-step split");
};

// An unsigned type of N bytes (2, 4, 8 or 16) for one lane's share of a row.
template <int N> struct LaneBytes;
template <> struct LaneBytes<2> { using T = uint16_t; };
template <> struct LaneBytes<4> { using T = uint32_t; };
template <> struct LaneBytes<8> { using T = uint2; };
template <> struct LaneBytes<16> { using T = uint4; };

// The fragment permutation: M row g <-> token pi(g) (and pi(g)+8); lane group g
// reads V d-chunk pi(g).  pi = 0 4 1 5 2 6 3 7.
__device__ __forceinline__ int perm8(int g) { return (g >> 1) | ((g & 1) << 2); }

// Byte offset of 16-byte chunk `c` of token row `t` inside a page tile laid out
// by the tensor copy with 128-byte swizzle.  Rows of 64 bytes are copied as
// 128-byte rows holding two tokens; wider rows as 128-byte panels of 16 rows.
template <int ROWB>
__device__ __forceinline__ int chunk_off(int t, int c) {
    if constexpr (ROWB == 64) {
        const int r = t >> 1;
        const int cc = ((t & 1) << 2) | c;
        return r * 128 + ((cc ^ (r & 7)) << 4);
    } else {
        const int panel = c >> 3;
        const int cc = c & 7;
        return panel * 2048 + t * 128 + ((cc ^ (t & 7)) << 4);
    }
}

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Visible page range of a sequence with context length c: positions [lo, ctx)
// live in pages [p_lo, p_hi).  Clamps a context longer than the page table (and
// reports it).
__device__ __forceinline__ void visible_of(const DecodeParams& p, int c, int& lo, int& ctx,
                                           int& p_lo, int& p_hi, bool report_errors) {
    ctx = c;
    if (ctx < 0) ctx = 0;
    if (ctx > p.max_blocks_per_seq * kPage) {
        if (report_errors) report(p.err, FP8KV_ERR_BAD_INDEX);
        ctx = p.max_blocks_per_seq * kPage;
    }
    lo = (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;
    p_lo = lo / kPage;
    p_hi = (ctx + kPage - 1) / kPage;
}

__device__ __forceinline__ void visible(const DecodeParams& p, int b, int& lo, int& ctx, int& p_lo,
                                        int& p_hi, bool report_errors) {
    visible_of(p, p.context_lens[b], lo, ctx, p_lo, p_hi, report_errors);
}

// Visible pages of sequence b (0 when its context is empty).
__device__ __forceinline__ int vis_pages(const DecodeParams& p, int b) {
    int lo, ctx, p_lo, p_hi;
    visible(p, b, lo, ctx, p_lo, p_hi, false);
    return p_hi > p_lo ? p_hi - p_lo : 0;
}

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, int out_bf16, size_t idx, float v) {
    if (out_bf16)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(out)[idx] = v;
}

// The new token of unit (b, h) of a fused decode step: lane l quantizes elements
// [l D/32, (l+1) D/32) of k_new / v_new exactly as kv_cache_write does
// (per-token-head scale fp32(max|x| / 448) over the row, codes
// e4m3_rn_satfinite(fp32(x / s)), a zero scale storing code 0; the bf16 cache
// takes the values as they are), stores them at position ctx - 1 of the
// sequence's page table (row bt_row[(ctx-1)/16] * Hkv + h, offset (ctx-1) % 16)
// and keeps row, row and scales in `area` ([K row][V row][s_k, s_v]) for the
// patch of the staged page.  Kept out of line: it runs once per unit and would
// otherwise raise the register pressure of the streaming loop.
template <int D, bool BF16, bool PER_TOKEN>
__device__ __noinline__ bool store_new_token_row(const int32_t* bt_row, int64_t num_blocks, int Hkv,
                                                 const __nv_bfloat16* k_new,
                                                 const __nv_bfloat16* v_new, uint8_t* k_cache,
                                                 uint8_t* v_cache, float* k_scale_cache,
                                                 float* v_scale_cache, int32_t* err, uint8_t* area,
                                                 int lane, int b, int h, int ctx, float ksc,
                                                 float vsc) {
    using C = Cfg<D, BF16>;
    constexpr int kNE = D / 32;                       // elements per lane
    constexpr int kLB = C::kRowB / 32;                // stored bytes per lane
    using LaneT = typename LaneBytes<kLB>::T;
    const int pos = ctx - 1;
    const int blk = bt_row[pos / kPage];
    const bool ok = blk >= 0 && static_cast<int64_t>(blk) < num_blocks;
    const size_t src = (static_cast<size_t>(b) * Hkv + h) * D + lane * kNE;
    LaneT kst, vst;
    float sk = 1.f, sv = 1.f;
    if constexpr (BF16) {
        kst = *reinterpret_cast<const LaneT*>(k_new + src);
        vst = *reinterpret_cast<const LaneT*>(v_new + src);
    } else {
        using RawT = typename LaneBytes<2 * kNE>::T;
        const RawT kr = *reinterpret_cast<const RawT*>(k_new + src);
        const RawT vr = *reinterpret_cast<const RawT*>(v_new + src);
        uint32_t kw[kNE / 2], vw[kNE / 2];
        memcpy(kw, &kr, 2 * kNE);
        memcpy(vw, &vr, 2 * kNE);
        float kf[kNE], vf[kNE];
#pragma unroll
        for (int i = 0; i < kNE / 2; ++i) {
            kf[2 * i] = bf16_bits_to_float(kw[i] & 0xffffu);
            kf[2 * i + 1] = bf16_bits_to_float(kw[i] >> 16);
            vf[2 * i] = bf16_bits_to_float(vw[i] & 0xffffu);
            vf[2 * i + 1] = bf16_bits_to_float(vw[i] >> 16);
        }
        if constexpr (PER_TOKEN) {
            float ka = 0.f, va = 0.f;
#pragma unroll
            for (int i = 0; i < kNE; ++i) {
                ka = fmaxf(ka, fabsf(kf[i]));
                va = fmaxf(va, fabsf(vf[i]));
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                ka = fmaxf(ka, __shfl_xor_sync(0xffffffffu, ka, off));
                va = fmaxf(va, __shfl_xor_sync(0xffffffffu, va, off));
            }
            sk = amax_over_448(ka);
            sv = amax_over_448(va);
        } else {
            sk = ksc;
            sv = vsc;
        }
        // codes of fp32(x / s): the cache writer's certified multiplies, and its
        // IEEE divides for a pair they cannot certify
        uint16_t kc[kNE / 2], vc[kNE / 2];
        auto encode = [](const float* x, float sc, uint16_t* code) {
            if (sc == 0.0f) {                 // a zero scale stores code 0
#pragma unroll
                for (int i = 0; i < kNE / 2; ++i) code[i] = 0;
                return;
            }
            const uint32_t e = (__float_as_uint(sc) >> 23) & 0xffu;
            const bool fast = e >= 1u && e <= 252u;
            const float r = __fdividef(1.0f, sc);
            const uint64_t rl = pack_f32x2(__fmul_rn(r, 1.0f - 0x1p-19f), __fmul_rn(r, 1.0f - 0x1p-19f));
            const uint64_t rh = pack_f32x2(__fmul_rn(r, 1.0f + 0x1p-19f), __fmul_rn(r, 1.0f + 0x1p-19f));
#pragma unroll
            for (int i = 0; i < kNE / 2; ++i) {
                const uint64_t x2 = pack_f32x2(x[2 * i], x[2 * i + 1]);
                const uint32_t lo = e4m3x2_from_f32x2(mul_f32x2(x2, rl));
                const uint32_t hi = e4m3x2_from_f32x2(mul_f32x2(x2, rh));
                code[i] = fast && lo == hi ? static_cast<uint16_t>(lo)
                                           : e4m3x2_by_divide(x[2 * i], x[2 * i + 1], sc);
            }
        };
        encode(kf, sk, kc);
        encode(vf, sv, vc);
        memcpy(&kst, kc, kLB);
        memcpy(&vst, vc, kLB);
    }
    *reinterpret_cast<LaneT*>(area + lane * kLB) = kst;
    *reinterpret_cast<LaneT*>(area + C::kRowB + lane * kLB) = vst;
    if (lane == 0) {
        reinterpret_cast<float*>(area + 2 * C::kRowB)[0] = sk;
        reinterpret_cast<float*>(area + 2 * C::kRowB)[1] = sv;
    }
    if (ok) {
        const size_t row = (static_cast<size_t>(blk) * Hkv + h) * kPage + pos % kPage;
        *reinterpret_cast<LaneT*>(k_cache + row * C::kRowB + lane * kLB) = kst;
        *reinterpret_cast<LaneT*>(v_cache + row * C::kRowB + lane * kLB) = vst;
        if constexpr (PER_TOKEN) {
            if (lane == 0) {
                k_scale_cache[row] = sk;
                v_scale_cache[row] = sv;
            }
        }
    } else if (lane == 0) {
        report(err, FP8KV_ERR_BAD_INDEX);
    }
    __syncwarp();
    return ok;
}

// CTAs resident per SM: 4 (16 warps, 128 registers at most) for 64-byte rows
// (e4m3 at D 64: short pages, more warps hide their latency), 3 (168 registers)
// for other rows up to 256 bytes with one 8-head group, else 2.
template <int D, bool BF16, int NT>
constexpr int decode_min_ctas() {
    return NT > 1 || D > 128 ? 2 : (D * (BF16 ? 2 : 1) == 64 ? 4 : 3);
}

// CTA units: the CTA's unit (b, h) = (blockIdx.x / Hu, blockIdx.x % Hu); its
// warps left partials (O [Gu][D], m [Gu], l [Gu] at the start of their ring,
// flag 1), or wrote the unit whole (flag 2), or had no pages (flag 0).  Rows
// b Hq + h Gu + col get O = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w; an empty
// unit gets zero rows.  Called by every thread after a CTA barrier.
template <int D, bool BF16>
__device__ __noinline__ void cta_combine(const DecodeParams& p, const uint8_t* smem, int warp_smem,
                                         int off_flag) {
    const volatile int* flag = reinterpret_cast<const volatile int*>(smem + off_flag);
    const int Gu = p.Gu;
    int parts = 0, whole = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        parts += flag[w] == 1;
        whole += flag[w] == 2;
    }
    if (parts == 0 && whole > 0) return;
    const size_t row0 = static_cast<size_t>(blockIdx.x / p.Hu) * p.Hq +
                        static_cast<size_t>(blockIdx.x % p.Hu) * Gu;
    for (int idx = threadIdx.x; idx < Gu * D; idx += blockDim.x) {
        const int col = idx / D, d = idx - col * D;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            if (flag[w] == 1)
                M = fmaxf(M, reinterpret_cast<const float*>(smem + w * warp_smem)[Gu * D + col]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w)
            if (flag[w] == 1) {
                const float* po = reinterpret_cast<const float*>(smem + w * warp_smem);
                const float a = ex2(po[Gu * D + col] - M);
                L += a * po[Gu * D + Gu + col];
                O += a * po[col * D + d];
            }
        store_out<BF16>(p.out, p.out_bf16, (row0 + col) * D + d, L > 0.f ? O / L : 0.f);
    }
}

// FUSED: a decode step -- the kernel also stores every sequence's new token
// (k_new / v_new at position ctx - 1).  NT: 8-head groups per KV head (1 for
// G <= 8, 2 for G <= 16); the groups share every K and V conversion.  HPT: KV
// heads per unit (2: adjacent heads h, h + 1 share the 8 columns, G <= 4 each).
// A unit is (sequence, group of HPT KV heads) with Gu = G * HPT query heads.
// CTA: CTA units (p.cta_units) -- a template parameter, so that the flattened
// partition's instances carry none of its code.
template <int D, bool BF16, bool PER_TOKEN, bool FUSED, int NT, int HPT, bool CTA>
__global__ void __launch_bounds__(kWarps * 32, decode_min_ctas<D, BF16, NT>())
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using C = Cfg<D, BF16, NT, HPT>;
    constexpr int PPI = C::kPPI;
    constexpr int TT = C::kTiles;
    constexpr int kMaxSeg = C::kMaxSeg;
    constexpr int kSegInts = C::kSegInts;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int G = p.G;                      // query heads per KV head
    const int Gu = p.Gu;                    // query heads (columns) per unit
    // the KV head (within the unit) of this lane's accumulator columns 2c, 2c + 1
    // (the same head for both: G is even when heads are packed)
    const int hl_lane = HPT > 1 ? ((2 * c) / G < HPT ? (2 * c) / G : HPT - 1) : 0;
    // PV B-operand masks: column g belongs to KV head g / G of the unit
    uint32_t bmask[HPT];
#pragma unroll
    for (int hl = 0; hl < HPT; ++hl) bmask[hl] = g / G == hl ? ~0u : 0u;
    // split_merge may launch while this runs; CTA units have no merge and trigger
    // at their end (a next decode grid launched now would take SM slots as they
    // free up and spread over several waves)
    if constexpr (!CTA) pdl_trigger();
    // Ordering against the preceding kernel of the stream (programmatic launch):
    // by default the kernel waits for it before reading any global memory.  With
    // FP8KV_DECODE_EARLY_SETUP the set-up below -- shares, segments, page-table
    // rows, which read only context_lens, block_table and the constant scales --
    // overlaps that kernel's tail (the caller guarantees those are complete
    // before it starts); with FP8KV_DECODE_EARLY_PAGES the first cache pages
    // stream before the wait too.  q, k_new, v_new and the workspace are read,
    // and anything is written, only after the wait.
    const bool early_setup = (p.flags & (FP8KV_DECODE_EARLY_SETUP | FP8KV_DECODE_EARLY_PAGES)) != 0;
    const bool early_pages = (p.flags & FP8KV_DECODE_EARLY_PAGES) != 0;

    uint8_t* ring = smem + warp * C::kWarpSmem;
    uint8_t* scl = smem + kWarps * C::kWarpSmem + warp * C::kStages * TT * C::kScaleB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars) + warp * C::kStages;
    int* seg = reinterpret_cast<int*>(smem + C::kOffSegs) + warp * kMaxSeg * kSegInts;
    // segment record i: seg[7i + 0..6] = sequence b, unit head group h (KV heads
    // h HPT .. h HPT + HPT - 1), first page, end page, flags (2: starts the unit,
    // 4: ends it), visible positions [lo, ctx)

    // ---- this warp's equal share [t0, t1) of the launch's W (seq, unit, page)
    //      tiles; every warp is an independent worker (no block-wide barrier but
    //      the one that ends a CTA-units launch)
    if (lane == 0) {                      // ring barriers (their fences overlap the loads below)
        // lane copies: every lane arrives once per stage; TMA: lane 0 only
        for (int s = 0; s < C::kStages; ++s)
            mbar_init(smem_addr(&bars[s]), C::kLaneCopies ? 32 : 1);
        mbar_init_fence();
        if constexpr (!C::kLaneCopies) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&vmap);
        }
    }
    if (!early_setup) pdl_wait();         // the preceding kernel's writes are visible
    // the page table's lines reach L2 while the context lengths are read (the
    // CTAs share the prefetch line by line)
    if (warp == 0) {
        const long long lines =
            (static_cast<long long>(p.B) * p.max_blocks_per_seq * 4 + 127) / 128;
        const uintptr_t base = reinterpret_cast<uintptr_t>(p.block_table) & ~uintptr_t{127};
        for (long long ln = blockIdx.x + static_cast<long long>(gridDim.x) * lane; ln < lines;
             ln += static_cast<long long>(gridDim.x) * 32)
            prefetch_l2(reinterpret_cast<const void*>(base + ln * 128));
    }
    // CTA units (p.cta_units): CTA u takes unit u = (b, h) whole, its 4 warps
    // splitting the unit's pages; they combine in shared memory, no split_merge
    constexpr bool cta_mode = CTA;
    if (cta_mode && static_cast<int>(blockIdx.x) >= p.B * p.Hu) return;   // (the whole CTA)
    // the first 32 context lengths are read once and kept in shared memory
    volatile int* ctx32 = reinterpret_cast<volatile int*>(smem + C::kOffCtx) + 32 * warp;
    long long W = 0;
    long long cu_base = 0;                // CTA units: tile index of sequence cu_b's first tile
    int cu_pages = 0;                     //            and its visible pages
    const int cu_b = static_cast<int>(blockIdx.x) / p.Hu;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int bb = b0 + lane;
        long long w = 0;
        int np = 0;
        if (bb < p.B) {
            const int craw = p.context_lens[bb];
            if (b0 == 0) ctx32[lane] = craw;
            int lo_, ctx_, plo_, phi_;
            visible_of(p, craw, lo_, ctx_, plo_, phi_, blockIdx.x == 0 && warp == 0);
            np = phi_ > plo_ ? phi_ - plo_ : 0;
            w = static_cast<long long>(np) * p.Hu;
        }
        if (cta_mode && cu_b >= b0 && cu_b < b0 + 32) {
            long long incl = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            cu_base = W + __shfl_sync(0xffffffffu, incl - w, cu_b - b0);
            cu_pages = __shfl_sync(0xffffffffu, np, cu_b - b0);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) w += __shfl_xor_sync(0xffffffffu, w, off);
        W += w;
    }
    const long long n_workers = W < static_cast<long long>(gridDim.x) * kWarps
                                    ? W : static_cast<long long>(gridDim.x) * kWarps;
    // worker id, recomputed where needed so it does not hold registers
#define FP8KV_WORKER (static_cast<long long>(blockIdx.x) * kWarps + warp)
    volatile int* cta_flag = reinterpret_cast<volatile int*>(smem + C::kOffFlag);
    if (!cta_mode && FP8KV_WORKER >= n_workers) return;
    // [resume, end) of the share lives in shared memory (kept out of registers)
    volatile long long* share = reinterpret_cast<volatile long long*>(smem + C::kOffShare) + 2 * warp;
    if (cta_mode) {
        if (lane == 0) {
            const int cu_h = static_cast<int>(blockIdx.x) - cu_b * p.Hu;
            const long long t0 = cu_base + static_cast<long long>(cu_h) * cu_pages;
            share[0] = t0 + (static_cast<long long>(warp) * cu_pages) / kWarps;
            share[1] = t0 + (static_cast<long long>(warp + 1) * cu_pages) / kWarps;
            cta_flag[warp] = 0;
        }
    } else if (lane == 0) {
        // floor(w W / n) for w and w + 1 with one 64-bit division: W = q n + r,
        // so w W / n = w q + w r / n, and w r < 2^24 (w, r < 4096)
        const long long q = W / n_workers, r = W - q * n_workers;
        const long long w = FP8KV_WORKER;
        share[0] = w * q + static_cast<long long>(static_cast<unsigned>(w * r) /
                                                  static_cast<unsigned>(n_workers));
        share[1] = (w + 1) * q + static_cast<long long>(static_cast<unsigned>((w + 1) * r) /
                                                        static_cast<unsigned>(n_workers));
    }
    __syncwarp();

    // segments of [resume, t1), at most kMaxSeg per pass, into this warp's list.
    // Lane j holds sequence b0 + j's visible range and tile offset; the sequences
    // the share meets come in order from a ballot.
    auto build_segments = [&]() -> int {
        long long t = share[0];
        const long long t1 = share[1];
        int k = 0;
        long long acc = 0;
        for (int b0 = 0; b0 < p.B && t < t1 && k < kMaxSeg; b0 += 32) {
            const int bb = b0 + lane;
            int lo_ = 0, ctx_ = 0, plo_ = 0, phi_ = 0;
            if (bb < p.B)
                visible_of(p, b0 == 0 ? ctx32[lane] : p.context_lens[bb], lo_, ctx_, plo_, phi_,
                           false);
            const int n = phi_ > plo_ ? phi_ - plo_ : 0;
            const long long w = static_cast<long long>(n) * p.Hu;
            long long incl = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            const long long base = acc + incl - w;
            acc += __shfl_sync(0xffffffffu, incl, 31);
            unsigned hit = __ballot_sync(0xffffffffu, w > 0 && base + w > t && base < t1);
            while (hit != 0u && t < t1 && k < kMaxSeg) {
                const int src = __ffs(hit) - 1;
                hit &= hit - 1u;
                const long long sb = __shfl_sync(0xffffffffu, base, src);
                const int sn = __shfl_sync(0xffffffffu, n, src);
                const int slo = __shfl_sync(0xffffffffu, lo_, src);
                const int sctx = __shfl_sync(0xffffffffu, ctx_, src);
                const int splo = __shfl_sync(0xffffffffu, plo_, src);
                while (t < t1 && t < sb + static_cast<long long>(sn) * p.Hu && k < kMaxSeg) {
                    // t - sb < pages * Hkv < 2^31 (checked on the host)
                    const int hq = static_cast<int>(t - sb) / sn;
                    const long long unit_base = sb + static_cast<long long>(hq) * sn;
                    const long long seg_end = t1 < unit_base + sn ? t1 : unit_base + sn;
                    if (lane == 0) {
                        int* r = seg + kSegInts * k;
                        r[0] = b0 + src;
                        r[1] = hq;
                        r[2] = splo + static_cast<int>(t - unit_base);
                        r[3] = splo + static_cast<int>(seg_end - unit_base);
                        r[4] = (t == unit_base ? 2 : 0) | (seg_end == unit_base + sn ? 4 : 0);
                        r[5] = slo;
                        r[6] = sctx;
                    }
                    t = seg_end;
                    ++k;
                }
            }
        }
        __syncwarp();
        if (lane == 0) share[0] = t;
        __syncwarp();
        return k;
    };

    // ---- query fragments (B operand of S^T = K Q^T): head 8 nt + g of the group,
    //      elements d0..d0+3; in registers for one group, in shared memory for two
    uint32_t qb[NT == 1 ? C::kKSteps : 1][2];
    uint2* qsm = reinterpret_cast<uint2*>(smem + C::kOffQsm) + warp * NT * C::kKSteps * 32;
    float hs[NT][2];                        // log2-domain logit multipliers, heads 2c, 2c+1
    // the per-tensor or per-head scale of KV head hk (1 for the bf16 cache and for
    // per-token-head scales, which apply per token)
    auto const_scale = [&](const float* arr, int hk) -> float {
        if constexpr (!BF16 && !PER_TOKEN)
            return arr[p.scale_mode == FP8KV_SCALE_PER_HEAD ? hk : 0];
        else
            return 1.f;
    };
    auto load_q = [&](int b, int h) {
    if constexpr (NT > 1) __syncwarp();     // the previous segment's fragments are read
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
    const int hl = nt * 8 + g;              // column (query head) within the unit
    const int hq_g = h * Gu + hl;
    const float kconst = hl < Gu ? const_scale(p.k_scale, h * HPT + hl / G) : 1.f;
    float qscale = 0.f;                     // log2-domain logit multiplier of head hl
    {
        const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(b) * p.Hq + hq_g) * D;
        uint2 raw[C::kKSteps];
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            const int s = ks / C::kKPerSeg, jj = ks % C::kKPerSeg;
            const int d0 = s * (64 / C::kElem) + c * (16 / C::kElem) + 4 * jj;
            raw[ks] = hl < Gu ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
        }
        uint2 frag[C::kKSteps];
        if constexpr (BF16) {
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) frag[ks] = raw[ks];
            qscale = p.scale_log2;
        } else {
            float amax = 0.f;
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[ks].x & 0xffffu)));
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[ks].x >> 16)));
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[ks].y & 0xffffu)));
                amax = fmaxf(amax, fabsf(bf16_bits_to_float(raw[ks].y >> 16)));
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            // power-of-two factor putting max|q| into [2^14, 2^15): exact in f16
            int e = 0;
            if (amax > 0.f) {
                frexpf(amax, &e);
                e = 15 - e;
                e = e > 126 ? 126 : (e < -126 ? -126 : e);
            }
            const float f = ldexpf(1.f, e);
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                frag[ks].x = pack_f16x2(bf16_bits_to_float(raw[ks].x & 0xffffu) * f,
                                        bf16_bits_to_float(raw[ks].x >> 16) * f);
                frag[ks].y = pack_f16x2(bf16_bits_to_float(raw[ks].y & 0xffffu) * f,
                                        bf16_bits_to_float(raw[ks].y >> 16) * f);
            }
            qscale = p.scale_log2 * kconst / f;
        }
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            if constexpr (NT == 1) {
                qb[ks][0] = frag[ks].x;
                qb[ks][1] = frag[ks].y;
            } else {
                qsm[(nt * C::kKSteps + ks) * 32 + lane] = frag[ks];
            }
        }
    }
    hs[nt][0] = __shfl_sync(0xffffffffu, qscale, (2 * c) * 4);
    hs[nt][1] = __shfl_sync(0xffffffffu, qscale, (2 * c + 1) * 4);
    }
    if constexpr (NT > 1) __syncwarp();     // the fragments are visible to the warp
    };
    // B fragment of k-step ks for group nt
    auto qfrag = [&](int nt, int ks) -> uint2 {
        if constexpr (NT == 1)
            return make_uint2(qb[ks][0], qb[ks][1]);
        else
            return qsm[(nt * C::kKSteps + ks) * 32 + lane];
    };

    // The PV weights w = p * s_v enter the MMA as hi + lo halves (f16 for the
    // e4m3 cache, bf16 for the bf16 cache).  e4m3 path: w is pre-scaled by 16
    // and the lazy max keeps p <= 16, so hi stays below f16's max and lo is a
    // normal f16 for every w >= 2^-7; both accumulate into the same fp32 O
    // (divided by 16 at the end, exactly).
    constexpr float kWScale = BF16 ? 1.f : 16.f;
    constexpr float kLazy = BF16 ? 8.f : 4.f;          // log2 headroom of the lazy max
    float o[NT][C::kMTiles][4];
    float mst[NT][2], lst[NT][2];           // running max and sum, heads 2c and 2c + 1
    auto reset_state = [&]() {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i)
                o[nt][i][0] = o[nt][i][1] = o[nt][i][2] = o[nt][i][3] = 0.f;
            // running max starts finite so that a fully masked group gives ex2(-inf) = 0
            mst[nt][0] = mst[nt][1] = kMaxInit;
            lst[nt][0] = lst[nt][1] = 0.f;
        }
    };

    // per-thread shared-memory offsets inside a page tile (fixed for the kernel)
    const int tA = perm8(g), tB = tA + 8;
    int koffA[C::kSegs], koffB[C::kSegs];
#pragma unroll
    for (int s = 0; s < C::kSegs; ++s) {
        koffA[s] = chunk_off<C::kRowB>(tA, 4 * s + c);
        koffB[s] = chunk_off<C::kRowB>(tB, 4 * s + c);
    }
    int voff[4][C::kVBytes >= 16 ? C::kVBytes / 16 : 1];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int t = c + 4 * r;
        if constexpr (C::kVBytes == 8) {
            voff[r][0] = chunk_off<C::kRowB>(t, perm8(g) >> 1) + (perm8(g) & 1) * 8;
        } else {
#pragma unroll
            for (int q4 = 0; q4 < C::kVBytes / 16; ++q4)
                voff[r][q4] = chunk_off<C::kRowB>(t, perm8(g) * (C::kVBytes / 16) + q4);
        }
    }


    // Finish the segment in `si`: a whole unit writes `out`; otherwise the warp's
    // (m, l, unnormalised O) goes to workspace slot worker + unit.
    auto finish_segment = [&](int si) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                lst[nt][0] += __shfl_xor_sync(0xffffffffu, lst[nt][0], off);
                lst[nt][1] += __shfl_xor_sync(0xffffffffu, lst[nt][1], off);
            }
        }
        const int ub = seg[kSegInts * si + 0], uh = seg[kSegInts * si + 1];
        const int flags = seg[kSegInts * si + 4];
        const bool whole = flags == 6;           // starts and ends the unit
        const int dbase = perm8(g) * (D / 8);
        const size_t unit = static_cast<size_t>(ub) * p.Hu + uh;
        const size_t slot = static_cast<size_t>(FP8KV_WORKER) + unit;
        // CTA units: a partial goes to this warp's ring (its streaming is over):
        // O [Gu][D], then m [Gu], l [Gu]
        float* cta_o = reinterpret_cast<float*>(ring);
        float* cta_m = cta_o + Gu * D;
        float* cta_l = cta_m + Gu;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int head0 = nt * 8 + 2 * c, head1 = head0 + 1;   // columns of the unit
            // V scale of their KV head (both columns belong to the same one)
            const float vconst =
                (head0 < Gu ? const_scale(p.v_scale, uh * HPT + head0 / G) : 1.f) / kWScale;
            const float l0 = lst[nt][0], l1 = lst[nt][1];
            const float f0 = whole ? (l0 > 0.f ? vconst / l0 : 0.f) : vconst;
            const float f1 = whole ? (l1 > 0.f ? vconst / l1 : 0.f) : vconst;
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i) {
                const int d = dbase + 2 * i;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int head = hh ? head1 : head0;
                    if (head >= Gu) continue;
                    const float f = hh ? f1 : f0;
                    const float va = o[nt][i][hh] * f, vb = o[nt][i][2 + hh] * f;
                    if (whole) {
                        const size_t row = static_cast<size_t>(ub) * p.Hq + uh * Gu + head;
                        store_out<BF16>(p.out, p.out_bf16, row * D + d, va);
                        store_out<BF16>(p.out, p.out_bf16, row * D + d + 1, vb);
                    } else {
                        float* dst = cta_mode ? cta_o + head * D + d : p.ws_o + (slot * Gu + head) * D + d;
                        *reinterpret_cast<float2*>(dst) = make_float2(va, vb);
                    }
                }
            }
            if (!whole && g == 0) {
                float* dm = cta_mode ? cta_m : p.ws_m + slot * Gu;
                float* dl = cta_mode ? cta_l : p.ws_l + slot * Gu;
                if (head0 < Gu) {
                    dm[head0] = mst[nt][0];
                    dl[head0] = l0;
                }
                if (head1 < Gu) {
                    dm[head1] = mst[nt][1];
                    dl[head1] = l1;
                }
            }
        }
        if (cta_mode && lane == 0) cta_flag[warp] = whole ? 2 : 1;
    };

    // ---- FUSED: the new token of unit (b, h) sits at position ctx - 1 on the
    //      unit's last page, which exactly one warp's share holds.  That warp
    //      stores it (store_new_token_row) and keeps it in its shared-memory
    //      area to patch the staged copy of the page, which may have been taken
    //      before the store.
    constexpr int kLB = C::kRowB / 32;                // stored bytes per lane
    using LaneT = typename LaneBytes<kLB>::T;
    // one area per KV head of the unit
    uint8_t* newtok = smem + C::kOffNew + warp * HPT * C::kNewB;
    auto store_new_token = [&](int b, int hk, int hl, int ctx) -> bool {
        return store_new_token_row<D, BF16, PER_TOKEN>(
            p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq, p.num_blocks, p.Hkv,
            p.k_new, p.v_new, p.k_cache, p.v_cache, const_cast<float*>(p.k_scale_cache),
            const_cast<float*>(p.v_scale_cache), p.err, newtok + hl * C::kNewB, lane, b, hk, ctx,
            const_scale(p.k_scale, hk), const_scale(p.v_scale, hk));
    };
    // overwrite token row r of page k of stage st (every KV head of the unit)
    // with the stored new tokens
    auto patch_new_token = [&](uint8_t* stage, int st, int k, int r) {
        const int off = chunk_off<C::kRowB>(r, (lane * kLB) >> 4) + ((lane * kLB) & 15);
#pragma unroll
        for (int hl = 0; hl < HPT; ++hl) {
            const uint8_t* area = newtok + hl * C::kNewB;
            const int tt = k * HPT + hl;
            *reinterpret_cast<LaneT*>(stage + tt * C::kTileB + off) =
                *reinterpret_cast<const LaneT*>(area + lane * kLB);
            *reinterpret_cast<LaneT*>(stage + (TT + tt) * C::kTileB + off) =
                *reinterpret_cast<const LaneT*>(area + C::kRowB + lane * kLB);
            if constexpr (PER_TOKEN) {
                if (lane == 0) {
                    float* sc = reinterpret_cast<float*>(scl + (st * PPI + k) * HPT * C::kScaleB);
                    sc[hl * 16 + r] = reinterpret_cast<const float*>(area + 2 * C::kRowB)[0];
                    sc[(HPT + hl) * 16 + r] = reinterpret_cast<const float*>(area + 2 * C::kRowB)[1];
                }
            }
        }
        // the slot is refilled by TMA later: order these generic writes first
        fence_proxy_async();
        __syncwarp();
    };

    // ---- the warp's page stream: issue side runs kStages groups ahead of the
    //      consume side; both walk the same segments in order
    int jring = 0;                          // groups consumed so far (ring phase)
    bool timed_out = false;
    while (share[0] < share[1] && !timed_out) {
        const int nseg = build_segments();
        // issue cursor: segment is_ (its end page, KV head and page-table row
        // cached in registers), next page ipg; block ids of pages
        // [bt_base, bt_base + 32) in bt_cur, the next 32 in bt_next
        int is_ = 0, ipg = seg[2], ipe = seg[3], ih = seg[1];
        const int32_t* ibt = p.block_table + static_cast<size_t>(seg[0]) * p.max_blocks_per_seq;
        int bt_base = ipg, bt_cur = 0, bt_next = 0;
        auto bt_fetch = [&](int base) -> int {
            const int pg = base + lane;
            return pg < ipe ? ibt[pg] : -1;
        };
        // block ids of the first pages of segment si (a segment switch on the issue
        // side then needs no load it waits for)
        auto seg_fetch = [&](int si) -> int {
            const int pg = seg[kSegInts * si + 2] + lane;
            return pg < seg[kSegInts * si + 3]
                       ? p.block_table[static_cast<size_t>(seg[kSegInts * si]) * p.max_blocks_per_seq + pg]
                       : -1;
        };
        bt_cur = bt_fetch(bt_base);
        bt_next = bt_fetch(bt_base + 32);
        int bt_nseg = nseg > 1 ? seg_fetch(1) : -1;
        uint32_t bad_mask = 0u;
        int issued = 0;
        auto issue_next = [&]() {           // called by all lanes of the warp
            if (ipg >= ipe) {               // next segment
                ++is_;
                ipg = seg[kSegInts * is_ + 2];
                ipe = seg[kSegInts * is_ + 3];
                ih = seg[kSegInts * is_ + 1];
                ibt = p.block_table + static_cast<size_t>(seg[kSegInts * is_]) * p.max_blocks_per_seq;
                bt_base = ipg;
                bt_cur = bt_nseg;
                bt_next = bt_fetch(bt_base + 32);
                bt_nseg = is_ + 1 < nseg ? seg_fetch(is_ + 1) : -1;
            } else if (ipg >= bt_base + 32) {
                bt_base += 32;
                bt_cur = bt_next;
                bt_next = bt_fetch(bt_base + 32);
            }
            const int pe_i = ipe;
            const int h_i = ih;
            const int st = (jring + issued) % C::kStages;
            int blk[PPI];
            bool here[PPI];
            uint32_t tx = 0;
#pragma unroll
            for (int k = 0; k < PPI; ++k) {
                blk[k] = __shfl_sync(0xffffffffu, bt_cur, (ipg - bt_base + k) & 31);
                here[k] = ipg + k < pe_i;
                const bool ok = here[k] && blk[k] >= 0 && static_cast<int64_t>(blk[k]) < p.num_blocks;
                const uint32_t bit = 1u << (st * PPI + k);
                bad_mask = ok ? (bad_mask & ~bit) : (bad_mask | bit);
                if (here[k] && !ok) {
                    if (lane == 0) report(p.err, FP8KV_ERR_BAD_INDEX);
                    blk[k] = 0;              // load an in-range page, masked later
                }
                if (here[k]) tx += HPT * (2 * C::kTileB + (PER_TOKEN ? C::kScaleB : 0));
            }
            if constexpr (C::kLaneCopies) {
                // every lane copies 16-byte pieces lane, lane + 32, ... of each tile
                // (the whole warp keeps many small requests in flight, which streams
                // short tiles faster than one bulk request per tile) into the
                // 128-byte-swizzled layout the math reads; the stage's barrier
                // completes when every lane's copies have landed
                const uint32_t bar = smem_addr(&bars[st]);
                const uint32_t base = smem_addr(ring + st * C::kStageB);
                const uint64_t pol = l2_evict_first();   // pages are read once
#pragma unroll
                for (int k = 0; k < PPI; ++k) {
                    if (!here[k]) continue;
                    // the unit's HPT tiles of the page are adjacent in the cache
                    const size_t z = static_cast<size_t>(blk[k]) * p.Hkv + h_i * HPT;
                    const uint8_t* ksrc = p.k_cache + z * C::kTileB + lane * 16;
                    const uint8_t* vsrc = p.v_cache + z * C::kTileB + lane * 16;
#pragma unroll
                    for (int i = 0; i < HPT * C::kTileB / 512; ++i) {
                        const int o = lane * 16 + i * 512;
                        const int ot = o % C::kTileB;
                        const uint32_t soff = (o / C::kTileB) * C::kTileB +
                                              chunk_off<C::kRowB>(ot / C::kRowB, (ot % C::kRowB) >> 4);
                        cp_async16_hint(base + k * HPT * C::kTileB + soff, ksrc + i * 512, pol);
                        cp_async16_hint(base + (TT + k * HPT) * C::kTileB + soff, vsrc + i * 512, pol);
                    }
                    if constexpr (PER_TOKEN) {
                        // 64 HPT bytes of k scales, then as many of v scales
                        if (lane < 8 * HPT) {
                            const bool kk = lane < 4 * HPT;
                            const float* src = (kk ? p.k_scale_cache : p.v_scale_cache) + z * kPage +
                                               (kk ? lane : lane - 4 * HPT) * 4;
                            cp_async16_hint(smem_addr(scl + (st * PPI + k) * HPT * C::kScaleB) + lane * 16,
                                            src, pol);
                        }
                    }
                }
                cp_async_mbar_arrive(bar);
            } else {
                if (lane == 0) {
                    const uint32_t bar = smem_addr(&bars[st]);
                    const uint32_t base = smem_addr(ring + st * C::kStageB);
                    const uint64_t pol = l2_evict_first();   // pages are read once
                    fence_proxy_async();
                    mbar_arrive_expect_tx(bar, tx);
#pragma unroll
                    for (int k = 0; k < PPI; ++k) {
                        if (!here[k]) continue;
                        // one box holds the unit's HPT adjacent tiles of the page
                        const int z = blk[k] * p.Hkv + h_i * HPT;
#pragma unroll
                        for (int box = 0; box < C::kBoxes; ++box) {
                            tma_load_3d_hint(base + k * HPT * C::kTileB + box * 2048, &kmap,
                                             box * 128, 0, z, bar, pol);
                            tma_load_3d_hint(base + (TT + k * HPT) * C::kTileB + box * 2048, &vmap,
                                             box * 128, 0, z, bar, pol);
                        }
                        if constexpr (PER_TOKEN) {
                            const uint32_t sdst = smem_addr(scl + (st * PPI + k) * HPT * C::kScaleB);
                            bulk_load_hint(sdst, p.k_scale_cache + static_cast<size_t>(z) * kPage,
                                           64 * HPT, bar, pol);
                            bulk_load_hint(sdst + 64 * HPT,
                                           p.v_scale_cache + static_cast<size_t>(z) * kPage, 64 * HPT,
                                           bar, pol);
                        }
                    }
                }
            }
            ipg += PPI;
            ++issued;
        };
        // groups in this pass
        int total_groups = 0;
        for (int si = 0; si < nseg; ++si)
            total_groups += (seg[kSegInts * si + 3] - seg[kSegInts * si + 2] + PPI - 1) / PPI;
        const int pre = total_groups < C::kStages ? total_groups : C::kStages;
        if (!early_pages) pdl_wait();       // the preceding kernel's results are visible
        for (int q = 0; q < pre; ++q) issue_next();
        if (early_pages) pdl_wait();

        int consumed = 0;
        for (int si = 0; si < nseg && !timed_out; ++si) {
            const int b = seg[kSegInts * si + 0];
            const int pb = seg[kSegInts * si + 2], pe = seg[kSegInts * si + 3];
            const int lo = seg[kSegInts * si + 5], ctx = seg[kSegInts * si + 6];
            load_q(b, seg[kSegInts * si + 1]);
            bool new_tok = false;           // this segment holds the unit's new tokens
            if constexpr (FUSED) {
                if ((seg[kSegInts * si + 4] & 4) && ctx >= 1) {
#pragma unroll
                    for (int hl = 0; hl < HPT; ++hl)   // same block for every head: same result
                        new_tok = store_new_token(b, seg[kSegInts * si + 1] * HPT + hl, hl, ctx);
                }
            }
            reset_state();
            for (int cpg = pb; cpg < pe; cpg += PPI) {
                const int j = jring + consumed;
                const int st = j % C::kStages;
                const bool arrived = mbar_wait_bounded(smem_addr(&bars[st]),
                                                       static_cast<uint32_t>((j / C::kStages) & 1));
                if (!__all_sync(0xffffffffu, arrived)) {   // leave together
                    timed_out = true;
                    break;
                }
        const uint8_t* stage = ring + st * C::kStageB;
        const int pos0 = cpg * kPage;

        bool bad[PPI], interior[PPI];
#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            bad[k] = (bad_mask >> (st * PPI + k)) & 1u;
            interior[k] = !bad[k] && pos0 + k * kPage >= lo && pos0 + (k + 1) * kPage <= ctx;
        }
        if constexpr (FUSED) {
            // the unit's last page (pe - 1) holds position ctx - 1
            if (new_tok && cpg + PPI >= pe) {
                const int kn = pe - 1 - cpg;
                bool badn = false;
#pragma unroll
                for (int k = 0; k < PPI; ++k) badn = k == kn ? bad[k] : badn;
                if (!badn)
                    patch_new_token(const_cast<uint8_t*>(stage), st, kn, (ctx - 1) % kPage);
            }
        }

        // ---- S^T = K_tile Q^T for each (page, head) tile (rows: tokens tA, tB; cols:
        //      heads 2c, 2c+1 of each 8-head group; with packed heads every tile
        //      fills all columns, of which the lane keeps its own head's)
        float acc[NT][TT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int k = 0; k < TT; ++k)
                acc[nt][k][0] = acc[nt][k][1] = acc[nt][k][2] = acc[nt][k][3] = 0.f;
#pragma unroll
        for (int s = 0; s < C::kSegs; ++s) {
            uint4 kx[TT], ky[TT];
#pragma unroll
            for (int k = 0; k < TT; ++k) {
                kx[k] = *reinterpret_cast<const uint4*>(stage + k * C::kTileB + koffA[s]);
                ky[k] = *reinterpret_cast<const uint4*>(stage + k * C::kTileB + koffB[s]);
            }
#pragma unroll
            for (int jj = 0; jj < C::kKPerSeg; ++jj) {
                const int ks = s * C::kKPerSeg + jj;
#pragma unroll
                for (int k = 0; k < TT; ++k) {
                    const uint32_t wx[4] = {kx[k].x, kx[k].y, kx[k].z, kx[k].w};
                    const uint32_t wy[4] = {ky[k].x, ky[k].y, ky[k].z, ky[k].w};
                    if constexpr (BF16) {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 qf = qfrag(nt, ks);
                            mma_bf16(acc[nt][k], wx[2 * jj], wy[2 * jj], wx[2 * jj + 1],
                                     wy[2 * jj + 1], qf.x, qf.y);
                        }
                    } else {
                        uint32_t xl, xh, yl, yh;
                        f16x2x2_from_e4m3x4(wx[jj], xl, xh);
                        f16x2x2_from_e4m3x4(wy[jj], yl, yh);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            const uint2 qf = qfrag(nt, ks);
                            mma_f16(acc[nt][k], xl, yl, xh, yh, qf.x, qf.y);
                        }
                    }
                }
            }
        }

        // ---- logits (base 2), masked outside [lo, ctx) on boundary pages
        float z[NT][PPI][4], vs[PPI][2];
        float mx[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mx[nt][0] = mx[nt][1] = neg_inf();
#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            const int posA = pos0 + k * kPage + tA, posB = pos0 + k * kPage + tB;
            const bool vA = interior[k] || (!bad[k] && posA >= lo && posA < ctx);
            const bool vB = interior[k] || (!bad[k] && posB >= lo && posB < ctx);
            float ksA = 1.f, ksB = 1.f;
            vs[k][0] = vs[k][1] = 1.f;
            if constexpr (PER_TOKEN) {
                // the page's scales: [k of head 0..HPT-1][v of head 0..HPT-1] x 16 tokens
                const float* sk = reinterpret_cast<const float*>(scl + (st * PPI + k) * HPT * C::kScaleB) +
                                  hl_lane * 16;
                ksA = sk[tA];
                ksB = sk[tB];
                // scales of masked tokens may be any bits (slots never written,
                // pages not fetched): zero them so that 0 * scale stays 0
                vs[k][0] = vA ? sk[HPT * 16 + tA] : 0.f;
                vs[k][1] = vB ? sk[HPT * 16 + tB] : 0.f;
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // the accumulators of this lane's head's tile
                float a4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    a4[i] = acc[nt][k * HPT][i];
                    if constexpr (HPT > 1) a4[i] = hl_lane == 1 ? acc[nt][k * HPT + 1][i] : a4[i];
                }
                z[nt][k][0] = vA ? a4[0] * hs[nt][0] * ksA : neg_inf();
                z[nt][k][1] = vA ? a4[1] * hs[nt][1] * ksA : neg_inf();
                z[nt][k][2] = vB ? a4[2] * hs[nt][0] * ksB : neg_inf();
                z[nt][k][3] = vB ? a4[3] * hs[nt][1] * ksB : neg_inf();
                mx[nt][0] = fmaxf(mx[nt][0], fmaxf(z[nt][k][0], z[nt][k][2]));
                mx[nt][1] = fmaxf(mx[nt][1], fmaxf(z[nt][k][1], z[nt][k][3]));
            }
        }
        // lazy running max: it moves only when a column's logits exceed it by
        // 2^kLazy.  The running max is the same in the 8 lanes of a column, so one
        // vote on the lanes' own logits tells whether any column needs it; only
        // then are the columns' maxima reduced across lanes
        bool move = false;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            move |= mx[nt][0] > mst[nt][0] + kLazy || mx[nt][1] > mst[nt][1] + kLazy;
        if (__any_sync(0xffffffffu, move)) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx[nt][0] = fmaxf(mx[nt][0], __shfl_xor_sync(0xffffffffu, mx[nt][0], off));
                mx[nt][1] = fmaxf(mx[nt][1], __shfl_xor_sync(0xffffffffu, mx[nt][1], off));
            }
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (mx[nt][hh] > mst[nt][hh] + kLazy) {
                    const float a = ex2(mst[nt][hh] - mx[nt][hh]);
                    lst[nt][hh] *= a;
#pragma unroll
                    for (int i = 0; i < C::kMTiles; ++i) {
                        o[nt][i][hh] *= a;
                        o[nt][i][2 + hh] *= a;
                    }
                    mst[nt][hh] = mx[nt][hh];
                }
            }
        }
        }

#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            // ---- P^T as the B operand of each group: hi + lo halves, transposed by
            //      movmatrix; masked logits are -inf and give weight 0 (the running
            //      max is finite)
            uint32_t bh[NT][2], bl[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float p0 = ex2(z[nt][k][0] - mst[nt][0]), p1 = ex2(z[nt][k][1] - mst[nt][1]);
                const float p2 = ex2(z[nt][k][2] - mst[nt][0]), p3 = ex2(z[nt][k][3] - mst[nt][1]);
                lst[nt][0] += p0 + p2;
                lst[nt][1] += p1 + p3;
                // (clamped: only a per-token V scale above ~256 could reach f16's max)
                const float w0 = fminf(p0 * vs[k][0] * kWScale, 65504.f);
                const float w1 = fminf(p1 * vs[k][0] * kWScale, 65504.f);
                const float w2 = fminf(p2 * vs[k][1] * kWScale, 65504.f);
                const float w3 = fminf(p3 * vs[k][1] * kWScale, 65504.f);
                if constexpr (BF16) {
                    const uint32_t hA = pack_bf16x2(w0, w1), hB = pack_bf16x2(w2, w3);
                    const float2 fA = unpack_bf16x2(hA), fB = unpack_bf16x2(hB);
                    bh[nt][0] = movmatrix_trans(hA);
                    bh[nt][1] = movmatrix_trans(hB);
                    bl[nt][0] = movmatrix_trans(pack_bf16x2(w0 - fA.x, w1 - fA.y));
                    bl[nt][1] = movmatrix_trans(pack_bf16x2(w2 - fB.x, w3 - fB.y));
                } else {
                    const uint32_t hA = pack_f16x2(w0, w1), hB = pack_f16x2(w2, w3);
                    const float2 fA = unpack_f16x2(hA), fB = unpack_f16x2(hB);
                    bh[nt][0] = movmatrix_trans(hA);
                    bh[nt][1] = movmatrix_trans(hB);
                    bl[nt][0] = movmatrix_trans(pack_f16x2(w0 - fA.x, w1 - fA.y));
                    bl[nt][1] = movmatrix_trans(pack_f16x2(w2 - fB.x, w3 - fB.y));
                }
            }

            // ---- per KV head of the unit: its V tile, and P^T restricted to its
            //      columns (the B operand's column is the lane's g)
#pragma unroll
            for (int hl = 0; hl < HPT; ++hl) {
            const uint32_t mb = HPT > 1 ? bmask[hl] : ~0u;
            // ---- V rows of tokens c, c+4, c+8, c+12 (k-slots 2c, 2c+1, 2c+8, 2c+9)
            const uint8_t* vt = stage + (TT + k * HPT + hl) * C::kTileB;
            uint32_t vr[4][C::kVWords];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                if constexpr (C::kVBytes == 8) {
                    const uint2 v2 = *reinterpret_cast<const uint2*>(vt + voff[r][0]);
                    vr[r][0] = v2.x;
                    vr[r][1] = v2.y;
                } else {
#pragma unroll
                    for (int q4 = 0; q4 < C::kVBytes / 16; ++q4) {
                        const uint4 v4 = *reinterpret_cast<const uint4*>(vt + voff[r][q4]);
                        vr[r][4 * q4 + 0] = v4.x;
                        vr[r][4 * q4 + 1] = v4.y;
                        vr[r][4 * q4 + 2] = v4.z;
                        vr[r][4 * q4 + 3] = v4.w;
                    }
                }
            }
            if (!interior[k]) {
                // rows outside [lo, ctx) may hold any bytes (even NaN codes): zero them
#pragma unroll
                for (int r = 0; r < 4; ++r) {
                    const int pos = pos0 + k * kPage + c + 4 * r;
                    if (bad[k] || pos < lo || pos >= ctx) {
#pragma unroll
                        for (int w = 0; w < C::kVWords; ++w) vr[r][w] = 0u;
                    }
                }
            }

            // ---- O^T += V^T P^T  (row g <-> d = perm8(g)*D/8 + 2i, row g+8 <-> d+1)
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i) {
                uint32_t a0, a1, a2, a3;
                if constexpr (BF16) {
                    a0 = __byte_perm(vr[0][i], vr[1][i], 0x5410);
                    a1 = __byte_perm(vr[0][i], vr[1][i], 0x7632);
                    a2 = __byte_perm(vr[2][i], vr[3][i], 0x5410);
                    a3 = __byte_perm(vr[2][i], vr[3][i], 0x7632);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_bf16(o[nt][i], a0, a1, a2, a3, bh[nt][0] & mb, bh[nt][1] & mb);
                        mma_bf16(o[nt][i], a0, a1, a2, a3, bl[nt][0] & mb, bl[nt][1] & mb);
                    }
                } else {
                    const int w = i >> 1;
                    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                    const uint32_t x01 = __byte_perm(vr[0][w], vr[1][w], sel);
                    const uint32_t x23 = __byte_perm(vr[2][w], vr[3][w], sel);
                    f16x2x2_from_e4m3x4(x01, a0, a1);
                    f16x2x2_from_e4m3x4(x23, a2, a3);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_f16(o[nt][i], a0, a1, a2, a3, bh[nt][0] & mb, bh[nt][1] & mb);
                        mma_f16(o[nt][i], a0, a1, a2, a3, bl[nt][0] & mb, bl[nt][1] & mb);
                    }
                }
            }
            }   // heads of the unit
        }

        __syncwarp();
                ++consumed;
                if (issued < total_groups) issue_next();
            }
            if (!timed_out) finish_segment(si);
        }
        if (timed_out) {
            if (lane == 0) report(p.err, FP8KV_ERR_TIMEOUT);
            // let this warp's copies still in flight land (each wait bounded)
            for (int j = consumed; j < issued; ++j)
                (void)mbar_wait_bounded(smem_addr(&bars[(jring + j) % C::kStages]),
                                        static_cast<uint32_t>(((jring + j) / C::kStages) & 1));
        }
        jring += consumed;
    }
    // ---- CTA units: combine the warps' partials of the CTA's unit (out of line,
    //      so that it does not weigh on the streaming loop's registers)
    if constexpr (CTA) {
        pdl_wait();                       // (warps without pages have not waited yet)
        __syncthreads();                  // every warp of the CTA gets here
        cta_combine<D, BF16>(p, smem, C::kWarpSmem, C::kOffFlag);
        pdl_trigger();                    // the next kernel may start: this grid is ending
    }
#undef FP8KV_WORKER
}

// split_merge, one block per query head (b, hq) of unit (b, h = hq / Gu): the
// workers (warps) whose shares touched a unit left partials (m, l, O) in slots
// worker + unit and recorded the first and last of them; combine them as
// O = sum_w 2^(m_w - M) O_w / sum_w 2^(m_w - M) l_w.  A unit one worker covered
// whole was written by that worker; an empty unit gets a zero row.  The block's
// warps (4 to 16, sized by the launch to the parts per unit) take the parts
// round-robin, each lane D/32 columns, all loads of a chunk of parts in flight
// together, and meet in shared memory ([warps][D + 2] floats, dynamic).
template <int D>
__global__ void __launch_bounds__(512) split_merge_kernel(const DecodeParams p) {
    constexpr int kCols = D / 32;
    extern __shared__ float merge_smem[];
    const int nw = blockDim.x >> 5;
    float* sm_o = merge_smem;                   // [nw][D]
    float* sm_m = sm_o + nw * D;                // [nw]
    float* sm_l = sm_m + nw;                    // [nw]
    const int row = blockIdx.x;                 // b * Hq + hq
    const int b = row / p.Hq, hq = row % p.Hq;
    const int Gu = p.Gu, h = hq / Gu, head = hq % Gu;
    const int unit = b * p.Hu + h;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // context_lens are read before the wait only when the caller allows it (the
    // decode kernel lets this one start early; it has waited for its own
    // predecessor, so after this wait everything before it is visible too)
    if ((p.flags & (FP8KV_DECODE_EARLY_SETUP | FP8KV_DECODE_EARLY_PAGES)) == 0) pdl_wait();
    const int nvis = vis_pages(p, b);
    // the workers whose shares meet the unit: the decode kernel split the W
    // tiles of the launch as worker w <- [floor(w W / n), floor((w+1) W / n)),
    // so tile t belongs to worker floor(((t+1) n - 1) / W)
    long long first = 0, last = -1;
    {
        long long W = 0, base = 0;
        int nb = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int bb = b0 + lane;
            const long long w = bb < p.B ? static_cast<long long>(vis_pages(p, bb)) * p.Hu : 0;
            long long incl = w;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const long long v = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += v;
            }
            if (b >= b0 && b < b0 + 32) base = W + __shfl_sync(0xffffffffu, incl - w, b - b0);
            W += __shfl_sync(0xffffffffu, incl, 31);
        }
        nb = nvis;
        const long long workers = static_cast<long long>(p.num_splits) * kWarps;
        const long long n = W < workers ? W : workers;
        if (nb > 0 && n > 0) {
            const long long t0 = base + static_cast<long long>(h) * nb, t1 = t0 + nb;
            first = ((t0 + 1) * n - 1) / W;
            last = (t1 * n - 1) / W;
        }
    }
    pdl_wait();                                 // the decode kernel's partials are visible
    // The next kernel may now start its set-up.  Not earlier: a dependent grid
    // launched while the decode grid still runs takes SM slots as they free up
    // and spreads itself over several waves.
    pdl_trigger();
    if (nvis == 0) {
        for (int d = threadIdx.x; d < D; d += blockDim.x)
            store_out<false>(p.out, p.out_bf16, static_cast<size_t>(row) * D + d, 0.f);
        return;
    }
    // first == last: one worker covered the unit whole and wrote the output
    if (last <= first) return;
    float M = neg_inf(), L = 0.f, acc[kCols];
#pragma unroll
    for (int k = 0; k < kCols; ++k) acc[k] = 0.f;
    constexpr int kChunk = 8;
    for (long long w0 = first + warp; w0 <= last; w0 += nw * kChunk) {
        float mi[kChunk], li[kChunk], oi[kChunk][kCols];
#pragma unroll
        for (int q = 0; q < kChunk; ++q) {
            const long long w = w0 + nw * q;
            const bool ok = w <= last;
            const size_t sl = (static_cast<size_t>(ok ? w : first) + unit) * Gu + head;
            mi[q] = ok ? p.ws_m[sl] : neg_inf();
            li[q] = ok ? p.ws_l[sl] : 0.f;
#pragma unroll
            for (int k = 0; k < kCols; ++k) oi[q][k] = ok ? p.ws_o[sl * D + lane + 32 * k] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < kChunk; ++q) {
            const float Mn = fmaxf(M, mi[q]);
            const float a = (M == neg_inf()) ? 0.f : ex2(M - Mn);
            const float bi = (mi[q] == neg_inf()) ? 0.f : ex2(mi[q] - Mn);
            L = L * a + li[q] * bi;
#pragma unroll
            for (int k = 0; k < kCols; ++k) acc[k] = acc[k] * a + oi[q][k] * bi;
            M = Mn;
        }
    }
    if (lane == 0) {
        sm_m[warp] = M;
        sm_l[warp] = L;
    }
#pragma unroll
    for (int k = 0; k < kCols; ++k) sm_o[warp * D + lane + 32 * k] = acc[k];
    __syncthreads();
    float Mt = neg_inf();
    for (int w = 0; w < nw; ++w) Mt = fmaxf(Mt, sm_m[w]);
    float Lt = 0.f;
    for (int w = 0; w < nw; ++w)
        if (sm_m[w] != neg_inf()) Lt += ex2(sm_m[w] - Mt) * sm_l[w];
    const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float o = 0.f;
        for (int w = 0; w < nw; ++w)
            if (sm_m[w] != neg_inf()) o += ex2(sm_m[w] - Mt) * sm_o[w * D + d];
        store_out<false>(p.out, p.out_bf16, static_cast<size_t>(row) * D + d, o * inv);
    }
}

template <int D, bool BF16, bool PER_TOKEN, bool FUSED, int NT, int HPT, bool CTA>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         cudaStream_t stream) {
    using C = Cfg<D, BF16, NT, HPT>;
    constexpr int kSmemBytes = FUSED ? C::kSmemFused : C::kSmem;
    auto kern = paged_decode_kernel<D, BF16, PER_TOKEN, FUSED, NT, HPT, CTA>;
    // opt in to the large dynamic shared-memory size once per context
    static unsigned long long attr_done[64] = {};
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
    // both kernels may start before their predecessor in the stream ends (they
    // wait for its results in-kernel): launch latency and set-up overlap
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.num_splits);
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, kmap, vmap, p);
    if (e != cudaSuccess || CTA) return e;   // CTA units combine in the kernel
    // merge block: about 4 parts per warp at the launch's mean parts per unit,
    // 4 to 16 warps; at most 8 when there are more merge blocks than SMs (larger
    // blocks then hold SM slots the next decode grid, launched early, is
    // waiting for: 16-warp blocks cost 4 us a step on the Llama-shaped batch)
    const long long units = static_cast<long long>(p.B) * p.Hu;
    const long long mean_parts = (static_cast<long long>(p.num_splits) * kWarps + units - 1) / units + 1;
    const long long cap = static_cast<long long>(p.B) * p.Hq > 152 ? 8 : 16;
    long long mw = (mean_parts + 3) / 4;
    mw = mw < 4 ? 4 : (mw > cap ? cap : mw);
    cudaLaunchConfig_t mcfg = cfg;
    mcfg.gridDim = dim3(p.B * p.Hq);
    mcfg.blockDim = dim3(static_cast<unsigned>(32 * mw));
    mcfg.dynamicSmemBytes = static_cast<size_t>(mw) * (D + 2) * sizeof(float);
    return cudaLaunchKernelEx(&mcfg, split_merge_kernel<D>, p);
}

// packed heads (p.hpt == 2) only where the host allows them: one 8-head group,
// tiles of at most 2 KiB
template <int D, bool BF16, bool PER_TOKEN, bool FUSED, int NT, int HPT>
cudaError_t dispatch_cta(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         cudaStream_t s) {
    if constexpr (NT == 1) {                    // CTA units: one 8-column group
        if (p.cta_units) return launch_split<D, BF16, PER_TOKEN, FUSED, NT, HPT, true>(p, kmap, vmap, s);
    }
    return launch_split<D, BF16, PER_TOKEN, FUSED, NT, HPT, false>(p, kmap, vmap, s);
}

template <int D, bool BF16, bool PER_TOKEN, bool FUSED, int NT>
cudaError_t dispatch_hpt(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         cudaStream_t s) {
    if constexpr (NT == 1 && D * (BF16 ? 2 : 1) <= 128) {
        if (p.hpt == 2) return dispatch_cta<D, BF16, PER_TOKEN, FUSED, NT, 2>(p, kmap, vmap, s);
    }
    return dispatch_cta<D, BF16, PER_TOKEN, FUSED, NT, 1>(p, kmap, vmap, s);
}

template <int D, bool FUSED, int NT>
cudaError_t dispatch_dtype(const DecodeParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int kv_dtype, cudaStream_t s) {
    if (kv_dtype == FP8KV_KV_BF16)
        return dispatch_hpt<D, true, false, FUSED, NT>(p, kmap, vmap, s);
    if (p.scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD)
        return dispatch_hpt<D, false, true, FUSED, NT>(p, kmap, vmap, s);
    return dispatch_hpt<D, false, false, FUSED, NT>(p, kmap, vmap, s);
}

template <int D>
cudaError_t dispatch_fused(const DecodeParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int kv_dtype, bool fused, cudaStream_t s) {
    if (p.G > 8)
        return fused ? dispatch_dtype<D, true, 2>(p, kmap, vmap, kv_dtype, s)
                     : dispatch_dtype<D, false, 2>(p, kmap, vmap, kv_dtype, s);
    return fused ? dispatch_dtype<D, true, 1>(p, kmap, vmap, kv_dtype, s)
                 : dispatch_dtype<D, false, 1>(p, kmap, vmap, kv_dtype, s);
}

template <int D, bool BF16, int NT, int HPT>
constexpr int smem_of() { return Cfg<D, BF16, NT, HPT>::kSmemFused; }

template <int D, bool BF16, int NT, int HPT>
int ctas_of() {
    const int by_smem = (228 * 1024) / (smem_of<D, BF16, NT, HPT>() + 1024);
    // the launch bounds' register budget
    const int by_regs = decode_min_ctas<D, BF16, NT>();
    const int n = by_smem < by_regs ? by_smem : by_regs;
    return n < 1 ? 1 : n;
}

template <int D, int NT>
int ctas_of(bool bf) { return bf ? ctas_of<D, true, NT, 1>() : ctas_of<D, false, NT, 1>(); }

}  // namespace

int decode_heads_per_unit(int D, int kv_dtype, int G, int Hkv, int B) {
    const int row_bytes = D * (kv_dtype == FP8KV_KV_BF16 ? 2 : 1);
    // few units (B Hkv < 32): halving them doubles the parts each merge combines
    return (G == 2 || G == 4) && Hkv % 2 == 0 && row_bytes <= 128 &&
                   static_cast<long long>(B) * Hkv >= 32 ? 2 : 1;
}

int decode_ctas_per_sm(int D, int kv_dtype, int G, int Hkv, int B) {
    const bool bf = kv_dtype == FP8KV_KV_BF16;
    if (G > 8) {
        switch (D) {
            case 64: return ctas_of<64, 2>(bf);
            case 128: return ctas_of<128, 2>(bf);
            default: return ctas_of<256, 2>(bf);
        }
    }
    if (decode_heads_per_unit(D, kv_dtype, G, Hkv, B) == 2) {   // rows of at most 128 bytes
        if (D == 64) return bf ? ctas_of<64, true, 1, 2>() : ctas_of<64, false, 1, 2>();
        return ctas_of<128, false, 1, 2>();
    }
    switch (D) {
        case 64: return ctas_of<64, 1>(bf);
        case 128: return ctas_of<128, 1>(bf);
        default: return ctas_of<256, 1>(bf);
    }
}

cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int D, int kv_dtype, bool fused,
                                cudaStream_t stream) {
    switch (D) {
        case 64: return dispatch_fused<64>(p, kmap, vmap, kv_dtype, fused, stream);
        case 128: return dispatch_fused<128>(p, kmap, vmap, kv_dtype, fused, stream);
        default: return dispatch_fused<256>(p, kmap, vmap, kv_dtype, fused, stream);
    }
}

}  // namespace fp8kv
