// prefill.cu -- fp8_prefill_attn: chunked causal prefill over the paged e4m3
// cache on the 5th-generation tensor cores (tcgen05, FP8 MMA, TMEM accumulators).
//
// What it computes ("vLLM FP8 KV-Cache 및 Attention 양자화 업데이트": attention in
// FP8 e4m3 over the FP8 cache (opening paragraph), query quantization fused into
// the kernel ("커널 및 퓨전 최적화"), two-level FP32 accumulation for long
// contractions ("정확도를 위한 2단계 누적") that Blackwell does not need ("아키텍처별
// 결과"); "[vLLM] KV Cache Quantization": q_scale / prob_scale of FP8 attention
// ("Q/Prob 스케일과 FP8 Attention")): for query i of sequence b at position
// pos_i = ctx_b - n_b + i and every query head of a KV head,
//     q8 = e4m3(q / q_scale),  s_t = q8 . code_k(t) * q_scale * s_k * softmax_scale,
//     p8_t = e4m3(exp(s_t - m) / prob_scale),  o = sum_t p8_t code_v(t) / sum_t p8_t
// over keys t = 0 .. pos_i (times s_v), fp32 accumulation.
//
// Two operand precisions, chosen per CTA:
//   * single: Q and P are one e4m3 term each, as above (the pages' FP8
//     attention).  Its rounding (3 mantissa bits) averages out over long rows:
//     used where every row of the CTA sees at least kSplitKeys keys.
//   * split: Q and P enter the MMAs as two e4m3 terms each, hi = e4m3(x) and
//     lo = e4m3(x - hi), both accumulated into the same fp32 tensor-memory sum
//     (about 8 significant bits per operand).  Q is first scaled per row by a
//     power of two (max |q| in [128, 256)) and the weights are lifted by 2^8 under
//     a running max that moves every half binade, so that both stay in e4m3's
//     normal range; the logits and the output undo these exact powers of two.
//     Used for rows with fewer keys (or on request), where single terms would
//     miss the accuracy target.
//
// Design (GB300):
//   * one CTA per (tile of 128 / G query tokens x the G query heads of a KV
//     head) = 128 MMA rows; a softmax thread owns one row and one part of every
//     tile's keys and of O's columns (two parts, four with per-token-head
//     scales; the parts' row maxima and sums meet in shared memory), two
//     loader warps issue TMA (K tiles, V tiles), one warp allocates tensor
//     memory and issues the MMAs from one thread.
//   * per KV tile (128 keys single, 64 keys split): S = Q8 K^T (kind::f8f6f4, M
//     128, N = keys, K = D in steps of 32) into TMEM; softmax reads S with
//     tcgen05.ld, writes P8 (e4m3) to shared memory; O += P8 V (M 128, N = D,
//     K = keys) with V read MN-major straight from the cache tile.  Q8, K and
//     P8 are K-major; a P row is always 128 bytes (split: 64 hi then 64 lo
//     weights, which the PV k-steps pair with the same 64 value rows).  All
//     tiles use the 128-byte swizzle that TMA writes.
//   * two-level off: O accumulates in TMEM across tiles; the lazy running max
//     rescales a row of O in TMEM only when the row max moves.  two-level on:
//     every tile's P V lands in a fresh TMEM tile and the softmax threads add it
//     into an fp32 accumulator on the CUDA cores.
//   * per-token-head scales (PT): the K loader also copies each tile's K and V
//     scale rows (64 bytes a page) into a 4-slot ring; the softmax multiplies
//     logit column t by s_k(t) before the row max, and folds s_v(t) into the
//     e4m3 weights relative to a running power-of-two bound E of the V scales
//     seen so far; O is rescaled when E grows, like the lazy row max, and the
//     row sums use the unfolded weights.
//   * every mbarrier wait is bounded and watches a shared abort flag, so a stuck
//     stage ends the kernel with FP8KV_ERR_TIMEOUT instead of hanging.
//   * launch: one CTA per query tile, or (with a workspace, more query tiles than
//     SMs) one persistent CTA per SM on an equal share of all (query tile, key
//     tile) units.  A query tile cut between CTAs is computed in pieces over key
//     ranges; each piece leaves its unnormalised O, running max m and sum l (the
//     state the online softmax carries from tile to tile), and the last CTA of
//     the tile to finish combines them, O = sum_i O_i 2^(m_i - M) / sum_i l_i
//     2^(m_i - M).
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace fp8kv {

namespace {

constexpr int kRows = 128;          // MMA M: query rows of a CTA
constexpr float kMaxInitP = -1.0e30f;
// Rows that see at least this many keys take single e4m3 operands.
constexpr int kSplitKeys = 8192;

// Softmax reference and weight lift.  Weights are p * lift with p = 2^(s - m)
// <= 2^lazy (the running max m moves only when a tile exceeds it by more than
// `lazy` binades); lift * 2^lazy stays below e4m3's largest value 448.
//   single, per-tensor / per-head: lazy 8, lift 1 / prob_scale (the pages' P8)
//   single, per-token-head: lazy 3, lift 2^5 s_v / E (the V scales fold in)
//   split (both): lazy 1/2, lift 2^8 (x s_v / E): small weights stay normal
template <bool SPLIT, bool PT>
struct Soft {
    static constexpr float kLazy = SPLIT ? 0.5f : (PT ? 3.f : 8.f);
    static constexpr float kLift = SPLIT ? 256.f : (PT ? 32.f : 1.f);
};

// WIDE: four softmax parts per row (per-token-head scales, two-level off)
template <int D, bool BF16, bool SPLIT, bool WIDE>
struct PCfg {
    // e4m3 tiles hold 128 keys (8 pages), bf16 and split tiles 64 keys (4 pages):
    // every P row is 128 bytes (bf16: 64 weights; split: 64 hi + 64 lo weights)
    static constexpr int kElem = BF16 ? 2 : 1;
    static constexpr int kKeys = (BF16 || SPLIT) ? 64 : 128;
    static constexpr int kRowB = D * kElem;                 // bytes of a Q / K / V row
    // Q, K and V rows are kept as panels of 128 bytes (128-byte swizzle), or as
    // one 64-byte panel with the 64-byte swizzle (e4m3 at D 64); P rows are 128 bytes
    static constexpr int kPanelB = kRowB < 128 ? kRowB : 128;
    static constexpr int kCPR = kPanelB / 16;               // 16-byte chunks of a panel row
    static constexpr int kKPP = kPanelB / 32;               // 32-byte k-steps of a panel row
    static constexpr uint32_t kLayout = kPanelB == 128 ? kLayoutSw128 : kLayoutSw64;
    // tensor memory: S (or the two-level P V tile) from column 0, O from the
    // kernel's kOCol; D 128 takes 256 columns so two co-resident CTAs never wait
    // on each other
    static constexpr uint32_t kTmemCols = D <= 128 ? 256u : 512u;
    static constexpr int kPanels = kRowB / kPanelB;         // panels of a row
    static constexpr int kQTerms = SPLIT ? 2 : 1;           // Q tiles (hi, lo)
    static constexpr int kQBytes = kRows * kRowB;           // one Q tile
    static constexpr int kKVBytes = kKeys * kRowB;          // one K (or V) tile
    static constexpr int kPBytes = kRows * 128;             // one P tile (128-byte rows)
    static constexpr int kPVSteps = kKeys * kElem / 32;     // PV k-steps of one term
    static constexpr int kOffQ = 0;
    static constexpr int kOffKV = kOffQ + kQTerms * kQBytes;  // [stage][K | V]
    static constexpr int kOffP = kOffKV + 2 * 2 * kKVBytes;   // [2] P tiles
    // e4m3 only: 16 x 128-byte rows of 1.0 (the bf16 D 256 tiles leave no room)
    static constexpr int kOffOnes = kOffP + 2 * kPBytes;
    static constexpr int kOffOnes2 = kOffOnes + (BF16 ? 0 : 16 * 128);
    // softmax warps: kParts per row quarter, each on a contiguous part of a
    // tile's keys and of O's columns (the row maxima and sums meet in shared
    // memory).  Two, except: per-token-head scales, whose column factors make
    // the softmax the longest stage, take four (32 keys of a single tile, 16 of
    // a split one) so that four warps per scheduler hide each other's
    // latencies (not with two-level accumulation, whose extra registers spill
    // at the 96 a thread of 19 warps gets); bf16 at D 256 takes one (its tiles
    // leave no shared memory for the exchange).
    static constexpr int kParts = (BF16 && D == 256) ? 1 : (WIDE ? 4 : 2);
    static constexpr int kSoftWarps = 4 * kParts;
    static constexpr int kThreads = 32 * (kSoftWarps + 3);   // + K loader, MMA, V loader
    static constexpr int kOffPMax = kOffOnes2;               // [2][kParts][128] partial maxima
    // split: per row, 2^-e of the row's Q scaling, then the parts' |q| maxima [kParts][128]
    static constexpr int kOffRow = kOffPMax + (kParts > 1 ? 2 * kParts * kRows * 4 : 0);
    static constexpr int kRowBytes = SPLIT ? (1 + kParts) * kRows * 4 : 0;
    static constexpr int kOffBar = kOffRow + kRowBytes;
    static constexpr int kNumBars = 20;
    // per-token-head scales (e4m3 only): 4 slots of [k scales][v scales] of a
    // tile (128 floats each), then the parts' V-scale maxima [2][kParts]
    static constexpr int kOffScl = kOffBar + kNumBars * 8;
    static constexpr int kSclBytes = BF16 ? 0 : 4 * 1024 + 16 * 4;
    // per-token-head scales: each softmax warp's column factors of the current
    // tile, [64] for the logits (k scale x logit scale), [64] for the weights
    // (v scale / bound)
    static constexpr int kOffPtf = (kOffScl + kSclBytes + 15) / 16 * 16;
    static constexpr int kPtfBytes = BF16 ? 0 : kSoftWarps * 128 * 4;
    static constexpr int kSmem = 1024 + kOffPtf + kPtfBytes;
    static_assert(kKeys / kParts % 16 == 0, "a part is a whole number of 16-key loads");
    static_assert(D / kParts % 16 == 0, "a part of O is a whole number of 16-column loads");
    static_assert(2 * kParts <= 16, "the V-scale maxima fit their slot");
    static_assert(kSmem <= 227 * 1024, "one CTA's shared memory fits an SM");
};

// Dynamic shared memory of the kernel: the larger of its two operand layouts.
template <int D, bool BF16, bool WIDE>
__host__ __device__ constexpr int prefill_smem() {
    using C1 = PCfg<D, BF16, false, WIDE>;
    static_assert(C1::kPanelB == 128 || C1::kPanelB == 64, "panel rows of 64 or 128 bytes");
    if constexpr (BF16) {
        return C1::kSmem;
    } else {
        using C2 = PCfg<D, false, true, WIDE>;
        static_assert(C1::kThreads == C2::kThreads && C1::kTmemCols == C2::kTmemCols,
                      "single and split bodies run in one launch, on one allocation");
        return C1::kSmem > C2::kSmem ? C1::kSmem : C2::kSmem;
    }
}

// barrier indices
// K and V stages fill and free separately: a K slot is free as soon as its QK
// has run, so the next K tile loads while the softmax of the current one runs
enum { kKFull0 = 0, kKFull1, kVFull0, kVFull1, kKEmpty0, kKEmpty1, kVEmpty0, kVEmpty1,
       kSFull, kSEmpty, kPFull0, kPFull1,
       kPvDone0, kPvDone1, kPvtFree, kMmaIdle, kPair0 };   // kPair0 .. kPair0 + 3

__device__ __forceinline__ float ex2p(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait that also gives up as soon as another thread raised `abort`.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              volatile int* abort_flag, int32_t* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_ns() - t0 > kWaitBudgetNs) {
                *abort_flag = 1;
                report(err, FP8KV_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

// Smallest power of two >= x for x > 0 (normal floats), 0 for x <= 0.
__device__ __forceinline__ float pow2_ceil(float x) {
    if (!(x > 0.f)) return 0.f;
    uint32_t u = __float_as_uint(x);
    uint32_t e = u >> 23;
    if (u & 0x7fffffu) ++e;
    return __uint_as_float(e << 23);
}

// 2^e as a float, e in [-126, 127].
__device__ __forceinline__ float exp2i(int e) {
    return __uint_as_float(static_cast<uint32_t>(127 + e) << 23);
}

// Byte offset of 16-byte chunk cc of row r in a panel of `panel_b`-byte rows laid
// out as TMA's 128-byte (8 chunks, XOR row % 8) or 64-byte (4 chunks, XOR
// (row / 2) % 4) swizzle writes it.
template <int PANEL_B>
__device__ __forceinline__ int swz_off(int r, int cc) {
    if constexpr (PANEL_B == 128)
        return r * 128 + ((cc ^ (r & 7)) << 4);
    else
        return r * 64 + ((cc ^ ((r >> 1) & 3)) << 4);
}

// Orders this thread's generic-proxy view of memory (all state spaces) before its
// later async-proxy accesses (bulk copies of data other threads stored).
__device__ __forceinline__ void fence_proxy_async_all() {
    asm volatile("fence.proxy.async;" ::: "memory");
}

// Named barrier of the softmax warps only (the loader and MMA warps run on).
__device__ __forceinline__ void soft_sync(int nthreads) {
    asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// Two fp32 values -> their e4m3 codes (hi) and the codes of what hi misses (lo),
// low value in the low byte; *sum += the four decoded values when asked.
__device__ __forceinline__ void e4m3x2_split(float a, float b, uint32_t& hi, uint32_t& lo,
                                             float* sum) {
    hi = e4m3x2_from_f32(a, b);
    const float2 h = unpack_f16x2(f16x2_from_e4m3x2(hi));   // exact
    lo = e4m3x2_from_f32(a - h.x, b - h.y);                 // exact differences
    if (sum != nullptr) {
        const float2 q = unpack_f16x2(f16x2_from_e4m3x2(lo));
        *sum += (h.x + h.y) + (q.x + q.y);
    }
}

// One piece of work: query tile (sequence b, KV head h, query tokens from tok0)
// against key tiles t0 .. t0 + n_tiles - 1.
struct CtaGeo {
    int b, h;
    int q0, nq;          // the sequence's first q row and chunk length
    int tok0;            // the tile's first query token (in the chunk)
    int ctx, pos_base;   // keys of the sequence; position of the chunk's first query
    int t0, n_tiles;     // the key tiles taken (all of them: t0 = 0, n_tiles = the
                         // tiles the tile's last row reaches)
    float* part;         // null: write the output; else this piece's partial
                         // (O times its output factor [128][D], then m, l [128])
};

// tmem_slot holds the CTA's tensor memory (allocated once by the kernel);
// abort_flag is raised by a wait that gave up.
template <int D, bool TWO_LEVEL, bool BF16, bool PT, bool SPLIT>
__device__ __forceinline__ void prefill_body(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                             const PrefillParams& p, uint8_t* smem,
                                             const CtaGeo& cg, const uint32_t* tmem_slot,
                                             volatile int* abort_flag) {
    using C = PCfg<D, BF16, SPLIT, PT && !TWO_LEVEL>;
    using S = Soft<SPLIT, PT>;
    constexpr int kKeys = C::kKeys;
    constexpr int kParts = C::kParts;
    constexpr int kSoft = 32 * C::kSoftWarps;          // softmax threads
    // K and V tiles come from two loader warps: a single warp issuing every copy
    // of a tile held the pipeline back
    constexpr int kTmaWarp = C::kSoftWarps, kMmaWarp = C::kSoftWarps + 1,
                  kVWarp = C::kSoftWarps + 2;
    // TMEM columns: S [0, kKeys); O from kOCol (two-level on: the P V tile takes
    // [0, D) and O [kOCol, kOCol + D)).  e4m3, D 256, two-level off: the row sums
    // l of the quantized weights come from the tensor core too, as P times a
    // block of ones, into [kLCol, kLCol + 16).
    constexpr uint32_t kOCol = D <= 128 ? 128u : (TWO_LEVEL ? 256u : 128u);
    constexpr bool kLMma = D == 256 && !TWO_LEVEL && !BF16 && !PT;
    constexpr uint32_t kLCol = kOCol + D;
    const uint32_t sbase = smem_addr(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = p.G;
    const int b = cg.b, h = cg.h, q0 = cg.q0, nq = cg.nq, tok0 = cg.tok0;
    const int ctx = cg.ctx, pos_base = cg.pos_base, n_tiles = cg.n_tiles;
    const int ctx_pages = (ctx + kPage - 1) / kPage;
    auto tile_of = [&](int j) { return cg.t0 + j; };   // key tile of the j-th step

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    if (tid == 0) {
        for (int i = kKFull0; i <= kVEmpty1; ++i) mbar_init(bar(i), 1);
        mbar_init(bar(kSFull), 1);
        mbar_init(bar(kSEmpty), kSoft);
        mbar_init(bar(kPFull0), kSoft);
        mbar_init(bar(kPFull1), kSoft);
        mbar_init(bar(kPvDone0), 1);
        mbar_init(bar(kPvDone1), 1);
        mbar_init(bar(kPvtFree), kSoft);
        mbar_init(bar(kMmaIdle), 1);
        for (int i = 0; i < 4; ++i) mbar_init(bar(kPair0 + i), 32 * kParts);   // a quarter's warps
        *abort_flag = 0;
        mbar_init_fence();
    }

    // ---- Q tile(s) (K-major, 128-byte swizzle)
    //   single: e4m3(q / q_scale); bf16: q itself;
    //   split:  hi = e4m3(q 2^e_r), lo = e4m3(q 2^e_r - hi), with 2^e_r putting the
    //           row's max |q| into [128, 256) (exact scaling; 2^-e_r goes to the logits)
    float* rowinfo = reinterpret_cast<float*>(smem + C::kOffRow);   // split: [1 + kParts][128]
    if (warp < C::kSoftWarps) {
        const int r = tid & (kRows - 1);
        const int part = tid / kRows;                   // which chunks of the row
        const int tk = tok0 + r / G, head = r % G;
        uint8_t* qtile = smem + C::kOffQ;
        constexpr int kChunks = C::kRowB / 16 / kParts;
        static_assert(C::kRowB / 16 % kParts == 0, "the Q row's chunks split evenly");
        const __nv_bfloat16* qrow =
            p.q + (static_cast<size_t>(q0 + tk) * p.Hq + h * G + head) * D;
        float qmul = 1.f;                               // split: 2^e_r
        if constexpr (SPLIT) {
            float amax = 0.f;
            if (tk < nq) {
#pragma unroll 4
                for (int c = part * kChunks; c < (part + 1) * kChunks; ++c) {
                    const uint4 a = *reinterpret_cast<const uint4*>(qrow + c * 16);
                    const uint4 bq = *reinterpret_cast<const uint4*>(qrow + c * 16 + 8);
                    const uint32_t in[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        amax = fmaxf(amax, fabsf(bf16_bits_to_float(in[i] & 0xffffu)));
                        amax = fmaxf(amax, fabsf(bf16_bits_to_float(in[i] >> 16)));
                    }
                }
            }
            rowinfo[kRows + part * kRows + r] = amax;
            soft_sync(kSoft);
#pragma unroll
            for (int o = 0; o < kParts; ++o) amax = fmaxf(amax, rowinfo[kRows + o * kRows + r]);
            int e = 0;
            if (amax > 0.f) {
                int ex;
                frexpf(amax, &ex);                      // amax in [2^(ex-1), 2^ex)
                e = 8 - ex;
                e = e > 120 ? 120 : (e < -120 ? -120 : e);
            }
            qmul = exp2i(e);
            if (part == 0) rowinfo[r] = exp2i(-e);
        }
#pragma unroll 4
        for (int c = part * kChunks; c < (part + 1) * kChunks; ++c) {   // 16-byte chunks
            uint32_t w[4] = {0u, 0u, 0u, 0u}, wl[4] = {0u, 0u, 0u, 0u};
            if (tk < nq) {
                const __nv_bfloat16* src = qrow + c * (16 / C::kElem);
                if constexpr (BF16) {
                    const uint4 a = *reinterpret_cast<const uint4*>(src);
                    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
                } else {
                    const uint4 a = *reinterpret_cast<const uint4*>(src);
                    const uint4 bq = *reinterpret_cast<const uint4*>(src + 8);
                    const uint32_t in[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const float x0 = bf16_bits_to_float(in[i] & 0xffffu);
                        const float x1 = bf16_bits_to_float(in[i] >> 16);
                        if constexpr (SPLIT) {
                            uint32_t hi, lo;
                            e4m3x2_split(x0 * qmul, x1 * qmul, hi, lo, nullptr);
                            w[i >> 1] |= hi << (16 * (i & 1));
                            wl[i >> 1] |= lo << (16 * (i & 1));
                        } else {
                            const float lo = __fdiv_rn(x0, p.q_scale);
                            const float hi = __fdiv_rn(x1, p.q_scale);
                            w[i >> 1] |= static_cast<uint32_t>(e4m3x2_from_f32(lo, hi))
                                         << (16 * (i & 1));
                        }
                    }
                }
            }
            const int panel = c / C::kCPR, cc = c % C::kCPR;
            const int off = panel * (kRows * C::kPanelB) + swz_off<C::kPanelB>(r, cc);
            *reinterpret_cast<uint4*>(qtile + off) = make_uint4(w[0], w[1], w[2], w[3]);
            if constexpr (SPLIT)
                *reinterpret_cast<uint4*>(qtile + C::kQBytes + off) =
                    make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
        if constexpr (kLMma) {                          // 16 rows of 128 bytes of 1.0
            const uint32_t one = 0x38383838u;
            for (int i = tid; i < 16 * 128 / 16; i += kSoft)
                *reinterpret_cast<uint4*>(smem + C::kOffOnes + i * 16) =
                    make_uint4(one, one, one, one);
        }
        fence_proxy_async();                            // generic writes -> tensor core reads
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == kTmaWarp || warp == kVWarp) {
        // =============================== TMA producers: K tiles (kTmaWarp), V tiles (kVWarp)
        const bool is_v = warp == kVWarp;
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        const int full0 = is_v ? kVFull0 : kKFull0, empty0 = is_v ? kVEmpty0 : kKEmpty0;
        const int32_t* bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
        int issued = 0;
        // block ids of 32 pages at a time (lane = page), the next 32 loaded while
        // these are used, so that no tile's copies wait for a page-table row
        constexpr int kPPT = kKeys / kPage;            // pages per tile (8 or 4)
        static_assert(32 % kPPT == 0, "a tile's pages lie in one batch of 32");
        auto bt_load = [&](int base) -> int {
            const int pg = base + lane;
            return pg < ctx_pages ? bt_row[pg] : 0;
        };
        int bt_base = -64;                             // no batch loaded yet
        int bt_cur = 0, bt_nxt = 0;
        for (int j = 0; j < n_tiles; ++j) {
            const int st = j & 1;
            const int page0 = tile_of(j) * kPPT;
            int n_pages = ctx_pages - page0;
            n_pages = n_pages > kPPT ? kPPT : n_pages;
            if ((page0 & ~31) != bt_base) {
                const int base = page0 & ~31;
                bt_cur = base == bt_base + 32 ? bt_nxt : bt_load(base);
                bt_base = base;
                bt_nxt = bt_load(base + 32);
            }
            int blk = __shfl_sync(0xffffffffu, bt_cur, (page0 - bt_base + lane) & 31);
            int z = 0;
            if (lane < n_pages) {
                if (blk < 0 || static_cast<int64_t>(blk) >= p.num_blocks) {
                    if (!is_v) report(p.err, FP8KV_ERR_BAD_INDEX);
                    blk = 0;
                }
                z = blk * p.Hkv + h;
            }
            const uint32_t tile_bytes = static_cast<uint32_t>(n_pages) * kPage * C::kRowB;
            const uint32_t dst = sbase + C::kOffKV + st * 2 * C::kKVBytes + (is_v ? C::kKVBytes : 0);
            // the slot held the tile j - 2 until its QK (K) or PV (V) ran
            bool go = true;
            if (j >= 2 && lane == 0)
                go = wait_or_abort(bar(empty0 + st), ((j - 2) >> 1) & 1, abort_flag, p.err);
            if (!__shfl_sync(0xffffffffu, go, 0)) break;
            const uint32_t scl_bytes = PT && !is_v ? static_cast<uint32_t>(n_pages) * 128u : 0u;
            if (lane == 0) mbar_arrive_expect_tx(bar(full0 + st), tile_bytes + scl_bytes);
            __syncwarp();
            if (lane < n_pages) {
#pragma unroll
                for (int pn = 0; pn < C::kPanels; ++pn)
                    tma_load_3d(dst + pn * (kKeys * C::kPanelB) + lane * (kPage * C::kPanelB), map,
                                pn * C::kPanelB, 0, z, bar(full0 + st));
                if constexpr (PT) {
                    // the tile's K and V scale rows, into slot j % 4 (the softmax of
                    // tile j - 4 has finished with it: QK of j - 2 ran after it)
                    if (!is_v) {
                        const uint32_t sd = sbase + C::kOffScl + (j & 3) * 1024 + lane * 64;
                        bulk_load(sd, p.k_scale_cache + static_cast<size_t>(z) * kPage, 64,
                                  bar(full0 + st));
                        bulk_load(sd + 512, p.v_scale_cache + static_cast<size_t>(z) * kPage, 64,
                                  bar(full0 + st));
                    }
                }
            }
            __syncwarp();
            issued = j + 1;
        }
        // copies still in flight land before the CTA can leave (each wait bounded)
        if (lane == 0 && *abort_flag) {
            for (int j = issued - 2 > 0 ? issued - 2 : 0; j < issued; ++j)
                (void)mbar_wait_bounded(bar(full0 + (j & 1)), (j >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // =============================== MMA issuer (one thread)
        if (lane == 0) {
            // e4m3 operands (kind::f8f6f4, format 0) or bf16 (kind::f16, format 1)
            constexpr uint32_t kFmt = BF16 ? 1u : 0u;
            constexpr uint32_t idesc_qk = instr_desc(kFmt, kFmt, 0, 0, kKeys, kRows);
            constexpr uint32_t idesc_pv = instr_desc(kFmt, kFmt, 0, 1, D, kRows);
            constexpr uint32_t idesc_l = instr_desc(kFmt, kFmt, 0, 0, 16, kRows);
            auto mma = [&](uint32_t d, uint64_t a, uint64_t bdsc, uint32_t id, uint32_t acc) {
                if constexpr (BF16)
                    mma_f16kind(d, a, bdsc, id, acc);
                else
                    mma_f8f6f4(d, a, bdsc, id, acc);
            };
            const uint32_t tS = tmem;                           // S: columns [0, kKeys)
            const uint32_t tO = tmem + (TWO_LEVEL ? 0u : kOCol); // PV target
            auto issue_qk = [&](int j) {
                const uint32_t kbase = sbase + C::kOffKV + (j & 1) * 2 * C::kKVBytes;
#pragma unroll
                for (int kk = 0; kk < C::kRowB / 32; ++kk) {    // 32-byte k-steps over D
                    const int pn = kk / C::kKPP, ks = kk % C::kKPP;
                    const uint32_t off = pn * (kRows * C::kPanelB) + ks * 32;
                    const uint64_t bd = smem_desc(kbase + pn * (kKeys * C::kPanelB) + ks * 32, 16,
                                                  8 * C::kPanelB, C::kLayout);
#pragma unroll
                    for (int t = 0; t < C::kQTerms; ++t) {       // split: Q hi, then Q lo
                        const uint64_t ad = smem_desc(sbase + C::kOffQ + t * C::kQBytes + off, 16,
                                                      8 * C::kPanelB, C::kLayout);
                        mma(tS, ad, bd, idesc_qk, (kk > 0 || t > 0) ? 1u : 0u);
                    }
                }
                mma_commit(bar(kSFull));
                mma_commit(bar(kKEmpty0 + (j & 1)));
            };
            auto issue_pv = [&](int j) {
                const uint32_t vbase = sbase + C::kOffKV + (j & 1) * 2 * C::kKVBytes + C::kKVBytes;
                const uint32_t pbase = sbase + C::kOffP + (j & 1) * C::kPBytes;
                // 32-byte k-steps over the 128-byte P rows; split: steps kPVSteps..
                // hold the lo weights of the same keys
#pragma unroll
                for (int kk = 0; kk < 128 / 32; ++kk) {
                    const int vk = kk % C::kPVSteps;
                    const uint64_t ad = smem_desc_sw128(pbase + kk * 32, 16, 1024);
                    // V: MN-major; 8-key groups 8 panel rows apart, D panels
                    // kKeys panel rows apart; one k-step = 32 / elem keys
                    const uint64_t bd =
                        smem_desc(vbase + vk * (32 / C::kElem) * C::kPanelB, kKeys * C::kPanelB,
                                  8 * C::kPanelB, C::kLayout);
                    const uint32_t acc = TWO_LEVEL ? (kk > 0 ? 1u : 0u)
                                                   : ((j > 0 || kk > 0) ? 1u : 0u);
                    mma(tO, ad, bd, idesc_pv, acc);
                    if constexpr (kLMma) {
                        const uint64_t od = smem_desc_sw128(sbase + C::kOffOnes + kk * 32, 16, 1024);
                        mma(tmem + kLCol, ad, od, idesc_l, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                }
                mma_commit(bar(kPvDone0 + (j & 1)));
                mma_commit(bar(kVEmpty0 + (j & 1)));
            };
            if constexpr (!TWO_LEVEL) {
                // S of tile j+1 is computed while the softmax warps work on tile j:
                // the QK of j+1 waits only for S(j) to have been read, not for P(j)
                if (n_tiles > 0 && wait_or_abort(bar(kKFull0), 0, abort_flag, p.err)) {
                    tc_fence_after();
                    issue_qk(0);
                    for (int j = 0; j < n_tiles; ++j) {
                        if (j + 1 < n_tiles) {
                            if (!wait_or_abort(bar(kKFull0 + ((j + 1) & 1)), ((j + 1) >> 1) & 1,
                                               abort_flag, p.err))
                                break;
                            if (!wait_or_abort(bar(kSEmpty), j & 1, abort_flag, p.err)) break;
                            tc_fence_after();
                            issue_qk(j + 1);
                        }
                        if (!wait_or_abort(bar(kPFull0 + (j & 1)), (j >> 1) & 1, abort_flag, p.err))
                            break;
                        if (!wait_or_abort(bar(kVFull0 + (j & 1)), (j >> 1) & 1, abort_flag, p.err))
                            break;
                        tc_fence_after();
                        issue_pv(j);
                    }
                }
            } else {
                for (int j = 0; j < n_tiles; ++j) {
                    const int st = j & 1;
                    if (!wait_or_abort(bar(kKFull0 + st), (j >> 1) & 1, abort_flag, p.err)) break;
                    if (j > 0) {
                        if (!wait_or_abort(bar(kSEmpty), (j - 1) & 1, abort_flag, p.err)) break;
                        if (!wait_or_abort(bar(kPvtFree), (j - 1) & 1, abort_flag, p.err)) break;
                    }
                    tc_fence_after();
                    issue_qk(j);
                    if (!wait_or_abort(bar(kPFull0 + st), (j >> 1) & 1, abort_flag, p.err)) break;
                    if (!wait_or_abort(bar(kVFull0 + st), (j >> 1) & 1, abort_flag, p.err)) break;
                    tc_fence_after();
                    issue_pv(j);
                }
            }
            // every issued MMA finishes before tensor memory is released (bounded
            // wait that does not stop early on an abort)
            mma_commit(bar(kMmaIdle));
            (void)mbar_wait_bounded(bar(kMmaIdle), 0);
        }
        __syncwarp();
    } else {
        // =============================== softmax / correction / epilogue
        // row r of TMEM lane quarter warp % 4; key part kh of every tile (columns
        // [kh * kKH, (kh + 1) * kKH)) and of O's columns
        const int r = 32 * (warp & 3) + lane;
        const int kh = warp / 4;
        constexpr int kKH = kKeys / kParts;             // keys of a tile this thread owns
        constexpr int kDH = D / kParts;                 // O columns this thread owns
        constexpr int kSW = kKH >= 32 ? 32 : kKH;       // columns of one S load
        constexpr int kCW = kDH >= 32 ? 32 : kDH;       // columns of one O load / store
        const int tk = tok0 + r / G;
        const bool row_ok = tk < nq;
        const int pos_r = row_ok ? pos_base + tk : -1;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        float* pmax = reinterpret_cast<float*>(smem + C::kOffPMax);   // [2][kParts][128]
        int pair_phase = 0;
        // the warps of a quarter meet (an mbarrier with a bounded wait, so a
        // stuck partner ends in FP8KV_ERR_TIMEOUT rather than a hang)
        auto pair_sync = [&]() -> bool {
            mbar_arrive(bar(kPair0 + (warp & 3)));
            const bool okp = wait_or_abort(bar(kPair0 + (warp & 3)), pair_phase & 1, abort_flag,
                                           p.err);
            ++pair_phase;
            return __all_sync(0xffffffffu, okp);
        };
        // the bf16 cache has no scales and keeps Q and P in bf16
        float kconst = 1.f, vconst = 1.f, qs = 1.f, ps = 1.f;
        if constexpr (!BF16) {
            if constexpr (!PT) {
                kconst = p.scale_mode == FP8KV_SCALE_PER_HEAD ? p.k_scale[h] : p.k_scale[0];
                vconst = p.scale_mode == FP8KV_SCALE_PER_HEAD ? p.v_scale[h] : p.v_scale[0];
            }
            // split: Q is scaled per row and the weights by 2^8 instead; q_scale
            // and prob_scale would cancel exactly and are not used
            if constexpr (!SPLIT) {
                qs = p.q_scale;
                ps = p.prob_scale;
            }
        }
        // the row's logit factor: raw S times sc is s in base-2 units.  PT: the
        // column factors carry scol, the row factor rowf = 2^-e_r (split) or 1.
        const float rowf = SPLIT ? rowinfo[r] : 1.f;
        const float scol = qs * kconst * p.scale_log2;
        const float sc = scol * rowf;
        const float rf = PT ? rowf : sc;               // raw (PT: column-scaled) S -> s
        // weights p * lift: single non-PT e4m3(p / prob_scale); PT p s_v lift / E
        const float lift = BF16 ? 1.f : S::kLift / ps;
        const float llift = log2f(lift);
        // PT: running power-of-two bound of the V scales folded into the weights
        float e_run = 0.f;
        float* ebuf = reinterpret_cast<float*>(smem + C::kOffScl + 4 * 1024);   // [2][kParts]
        float m = kMaxInitP, l = 0.f;                  // l: this part's keys (summed at the end)
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
            const int st = j & 1;
            if (!__all_sync(0xffffffffu, wait_or_abort(bar(kSFull), j & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sb[kKH];                   // raw S of this row's part: all loads, one wait
#pragma unroll
            for (int cch = 0; cch < kKH / kSW; ++cch) {
                uint32_t* dst = sb + cch * kSW;
                tmem_ld_n<kSW>(tmem + lane_addr + kh * kKH + cch * kSW,
                               *reinterpret_cast<uint32_t(*)[kSW]>(dst));
            }
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(kSEmpty));

            // causal mask on the raw logits (keys past ctx always masked), the row
            // max of raw S, then base-2 logits s * rf - m inside one FFMA below
            const int key0 = tile_of(j) * kKeys + kh * kKH;
            float s[kKH];
            float mxp[8];                       // 8 independent partial maxima
#pragma unroll
            for (int i = 0; i < 8; ++i) mxp[i] = -__int_as_float(0x7f800000);
            const bool full = key0 + kKH - 1 <= pos_r;
            // PT: this tile's scale rows (keys past ctx hold stale values: never read
            // for a logit, excluded from the V-scale bound)
            const float* ksl = reinterpret_cast<const float*>(smem + C::kOffScl + (j & 3) * 1024) +
                               kh * kKH;
            const float* vsl = ksl + 128;
            // PT: this warp's column factors (every lane of the warp works on this part)
            float* ptf = reinterpret_cast<float*>(smem + C::kOffPtf) + warp * 128;
            if constexpr (PT) {
                __syncwarp();                   // the previous tile's factors are read
#pragma unroll
                for (int i = lane; i < kKH; i += 32) ptf[i] = ksl[i] * scol;
                __syncwarp();
                // the factors come as 16-byte broadcast loads (four keys each)
                const float4* ptf4 = reinterpret_cast<const float4*>(ptf);
                if (full) {
#pragma unroll
                    for (int i4 = 0; i4 < kKH / 4; ++i4) {
                        const float4 f4 = ptf4[i4];
                        const float fk[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int i = 4 * i4 + u;
                            s[i] = __uint_as_float(sb[i]) * fk[u];
                            mxp[i & 7] = fmaxf(mxp[i & 7], s[i]);
                        }
                    }
                } else {
#pragma unroll
                    for (int i4 = 0; i4 < kKH / 4; ++i4) {
                        const float4 f4 = ptf4[i4];
                        const float fk[4] = {f4.x, f4.y, f4.z, f4.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const int i = 4 * i4 + u;
                            s[i] = key0 + i <= pos_r ? __uint_as_float(sb[i]) * fk[u]
                                                     : -__int_as_float(0x7f800000);
                            mxp[i & 7] = fmaxf(mxp[i & 7], s[i]);
                        }
                    }
                }
            } else if (full) {
#pragma unroll
                for (int i = 0; i < kKH; ++i) {
                    s[i] = __uint_as_float(sb[i]);
                    mxp[i & 7] = fmaxf(mxp[i & 7], s[i]);
                }
            } else {
#pragma unroll
                for (int i = 0; i < kKH; ++i) {
                    s[i] = key0 + i <= pos_r ? __uint_as_float(sb[i]) : -__int_as_float(0x7f800000);
                    mxp[i & 7] = fmaxf(mxp[i & 7], s[i]);
                }
            }
            float mx_raw = fmaxf(fmaxf(fmaxf(mxp[0], mxp[1]), fmaxf(mxp[2], mxp[3])),
                                 fmaxf(fmaxf(mxp[4], mxp[5]), fmaxf(mxp[6], mxp[7])));
            float vmax = 0.f;                   // PT: this part's largest V scale
            if constexpr (PT) {
                // every lane of the warp works on this part: the lanes share the
                // keys with written scales and meet in a shuffle reduction
                const int nval = min(ctx - key0, kKH);
                for (int i = lane; i < nval; i += 32) vmax = fmaxf(vmax, vsl[i]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1)
                    vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
                ebuf[st * kParts + kh] = vmax;  // every thread of the part: the same value
            }
            if constexpr (kParts > 1) {         // the row's max over every part
                pmax[(st * kParts + kh) * kRows + r] = mx_raw;
                if (!pair_sync()) {
                    ok = false;
                    break;
                }
#pragma unroll
                for (int o = 1; o < kParts; ++o) {
                    const int ko = (kh + o) % kParts;
                    mx_raw = fmaxf(mx_raw, pmax[(st * kParts + ko) * kRows + r]);
                    if constexpr (PT) vmax = fmaxf(vmax, ebuf[st * kParts + ko]);
                }
            }
            const float mx = mx_raw * rf;
            float beta = 1.f;                   // PT: O's factor when the V bound grows
            if constexpr (PT) {
                const float e_t = pow2_ceil(vmax);
                if (e_t > e_run) {
                    beta = e_run > 0.f ? e_run / e_t : 1.f;
                    e_run = e_t;
                }
            }
            float alpha = 1.f;
            if (mx > m + S::kLazy) {            // lazy running max (the same in every part)
                alpha = ex2p(m - mx);
                m = mx;
                l *= alpha;
            }
            // a row whose max moved rescales its O row in TMEM (two-level off); the
            // tcgen05 loads are warp-wide, so the warp does it when any row needs it
            if (!TWO_LEVEL && j > 0 && __any_sync(0xffffffffu, alpha != 1.f || beta != 1.f)) {
                // O (TMEM) must hold PV of tile j-1 before it is rescaled
                if (!__all_sync(0xffffffffu,
                                wait_or_abort(bar(kPvDone0 + ((j - 1) & 1)), ((j - 1) >> 1) & 1,
                                              abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // this part's O columns, and l's columns (tensor-core l) in part 0
                constexpr int kChunks = kDH / kCW;
#pragma unroll 1
                for (int cch = 0; cch < kChunks + ((kLMma) ? 1 : 0); ++cch) {
                    if (cch == kChunks && kh != 0) break;
                    uint32_t rr[kCW];
                    const uint32_t ta = tmem + lane_addr +
                                        (cch < kChunks ? kOCol + kh * kDH + cch * kCW : kLCol);
                    tmem_ld_n<kCW>(ta, rr);
                    tmem_wait_ld();
                    // O takes alpha and beta; the tensor-core l (not PT) only alpha
                    const float fo = cch < kChunks ? alpha * beta : alpha;
#pragma unroll
                    for (int i = 0; i < kCW; ++i)
                        rr[i] = __float_as_uint(__uint_as_float(rr[i]) * fo);
                    tmem_st_n<kCW>(ta, rr);
                }
                tmem_wait_st();
            }
            // P tile j&1 was read by PV of tile j-2
            if (j >= 2 && !__all_sync(0xffffffffu, wait_or_abort(bar(kPvDone0 + st),
                                                                 ((j - 2) >> 1) & 1, abort_flag,
                                                                 p.err))) {
                ok = false;
                break;
            }
            uint8_t* prow = smem + C::kOffP + st * C::kPBytes + r * 128;
            constexpr int kPerChunk = 16 / C::kElem;    // keys per 16-byte chunk
            constexpr int kMyChunks = kKH / kPerChunk;  // this part's chunks of the row
            static_assert(kKH % kPerChunk == 0, "a part is whole 16-byte chunks of P");
            // PT: weight = p * s_v * lift / E, the unfolded p into l
            const float vinv = PT && e_run > 0.f ? lift / e_run : 0.f;
            if constexpr (PT) {
                __syncwarp();                   // the previous tile's factors are read
#pragma unroll
                for (int i = lane; i < kKH; i += 32) ptf[64 + i] = vsl[i] * vinv;
                __syncwarp();
            }
            // not PT: weight = 2^(s rf - m) * lift, one FFMA and an ex2
            const float moff = m - llift;
#pragma unroll
            for (int c8 = 0; c8 < kMyChunks; ++c8) {
                const int cc = kh * kMyChunks + c8;
                uint32_t w[4], wl[4];
#pragma unroll
                for (int i = 0; i < kPerChunk / 2; ++i) {
                    const int ia = c8 * kPerChunk + 2 * i, ib = ia + 1;
                    float wa, wb;
                    if constexpr (PT) {
                        const float pa = ex2p(fmaf(s[ia], rf, -m)), pb = ex2p(fmaf(s[ib], rf, -m));
                        l += pa + pb;
                        // masked keys: p = 0 and a stale scale that must not enter
                        const bool va = full || key0 + ia <= pos_r, vb = full || key0 + ib <= pos_r;
                        const float2 f2 = *reinterpret_cast<const float2*>(ptf + 64 + ia);
                        wa = va ? pa * f2.x : 0.f;
                        wb = vb ? pb * f2.y : 0.f;
                    } else {
                        wa = ex2p(fmaf(s[ia], rf, -moff));
                        wb = ex2p(fmaf(s[ib], rf, -moff));
                    }
                    // the denominator (not PT) sums the same rounded weights the MMA
                    // uses (on the tensor core for D 256, e4m3, two-level off)
                    if constexpr (BF16) {
                        w[i] = pack_bf16x2(wa, wb);
                        if constexpr (!kLMma) {
                            const float2 q2 = unpack_bf16x2(w[i]);
                            l += q2.x + q2.y;
                        }
                    } else if constexpr (SPLIT) {
                        uint32_t hi, lo;
                        e4m3x2_split(wa, wb, hi, lo, (PT || kLMma) ? nullptr : &l);
                        if (i & 1) {
                            w[i >> 1] |= hi << 16;
                            wl[i >> 1] |= lo << 16;
                        } else {
                            w[i >> 1] = hi;
                            wl[i >> 1] = lo;
                        }
                    } else {
                        const uint32_t code = e4m3x2_from_f32(wa, wb);
                        if (i & 1)
                            w[i >> 1] |= code << 16;
                        else
                            w[i >> 1] = code;
                        if constexpr (!kLMma && !PT) {
                            const float2 q2 = unpack_f16x2(f16x2_from_e4m3x2(code));
                            l += q2.x + q2.y;
                        }
                    }
                }
                *reinterpret_cast<uint4*>(prow + ((cc ^ (r & 7)) << 4)) =
                    make_uint4(w[0], w[1], w[2], w[3]);
                if constexpr (SPLIT)            // the lo weights: chunks 4..7 of the row
                    *reinterpret_cast<uint4*>(prow + (((cc + 4) ^ (r & 7)) << 4)) =
                        make_uint4(wl[0], wl[1], wl[2], wl[3]);
            }
            // value rows past ctx in the last tile hold unwritten cache slots (any
            // bytes, NaN codes included): zero them so 0 * v stays 0
            if (tile_of(j) * kKeys + kKeys > ctx) {
                if (!__all_sync(0xffffffffu,
                                wait_or_abort(bar(kVFull0 + st), (j >> 1) & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                uint8_t* vt = smem + C::kOffKV + st * 2 * C::kKVBytes + C::kKVBytes;
                for (int idx = tid; idx < kKeys * C::kPanels * C::kCPR; idx += kSoft) {
                    const int chunk = idx % C::kCPR, row = (idx / C::kCPR) % kKeys,
                              pn = (idx / C::kCPR) / kKeys;
                    if (tile_of(j) * kKeys + row >= ctx)
                        *reinterpret_cast<uint4*>(vt + pn * (kKeys * C::kPanelB) +
                                                  row * C::kPanelB + chunk * 16) =
                            make_uint4(0u, 0u, 0u, 0u);
                }
            }
            fence_proxy_async();
            tc_fence_before();
            mbar_arrive(bar(kPFull0 + st));

            if constexpr (TWO_LEVEL) {
                // O_acc (fp32, TMEM columns [kOCol, kOCol + D)) = alpha * O_acc + P V of
                // this tile; this part's columns
                if (!__all_sync(0xffffffffu,
                                wait_or_abort(bar(kPvDone0 + st), (j >> 1) & 1, abort_flag, p.err))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int cch = 0; cch < kDH / kCW; ++cch) {
                    const int col = kh * kDH + cch * kCW;
                    uint32_t pv[kCW], acc[kCW];
                    tmem_ld_n<kCW>(tmem + lane_addr + col, pv);
                    if (j > 0) tmem_ld_n<kCW>(tmem + lane_addr + kOCol + col, acc);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < kCW; ++i) {
                        const float prev = j > 0 ? __uint_as_float(acc[i]) * (alpha * beta) : 0.f;
                        acc[i] = __float_as_uint(prev + __uint_as_float(pv[i]));
                    }
                    tmem_st_n<kCW>(tmem + lane_addr + kOCol + col, acc);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(kPvtFree));
            }
        }
        // ---- epilogue: out = O * v_scale / l (PT: O * E / (lift l))
        if (ok) {
            const int last = n_tiles - 1;
            if (!TWO_LEVEL &&
                !__all_sync(0xffffffffu, wait_or_abort(bar(kPvDone0 + (last & 1)),
                                                       (last >> 1) & 1, abort_flag, p.err)))
                ok = false;
        }
        if (ok) {
            tc_fence_after();
            if constexpr (kLMma) {
                uint32_t rr[32];
                tmem_ld32(tmem + lane_addr + kLCol, rr);
                tmem_wait_ld();
                l = __uint_as_float(rr[0]);
            } else if constexpr (kParts > 1) {       // the parts' sums
                // through the buffer of tile n-2, which every warp has finished with
                const int lb = ((n_tiles - 1) & 1) ^ 1;
                pmax[(lb * kParts + kh) * kRows + r] = l;
                if (pair_sync()) {
#pragma unroll
                    for (int o = 1; o < kParts; ++o)
                        l += pmax[(lb * kParts + (kh + o) % kParts) * kRows + r];
                } else {
                    ok = false;
                }
            }
        }
        if (ok && cg.part != nullptr) {
            // a piece of a split tile: O times its output factor, then m and l
            // (the row's logits are base-2 numbers relative to m)
            const float g = PT ? e_run / lift : vconst;
            float* prow = cg.part + static_cast<size_t>(r) * D;
            for (int cch = 0; cch < kDH / kCW; ++cch) {
                const int col = kh * kDH + cch * kCW;
                uint32_t rr[kCW];
                tmem_ld_n<kCW>(tmem + lane_addr + kOCol + col, rr);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < kCW; i += 4)
                    *reinterpret_cast<float4*>(prow + col + i) = make_float4(
                        __uint_as_float(rr[i]) * g, __uint_as_float(rr[i + 1]) * g,
                        __uint_as_float(rr[i + 2]) * g, __uint_as_float(rr[i + 3]) * g);
            }
            if (kh == 0) {
                cg.part[kRows * D + r] = m;
                cg.part[kRows * D + kRows + r] = l;
            }
        } else if (ok) {
            // not PT: l sums the weights the MMA used, so O / l is the weighted mean
            // of the value codes; PT: l sums p itself and O carries lift / E
            const float f = l > 0.f ? (PT ? e_run / lift : vconst) / l : 0.f;
            const int head = r % G;
            for (int cch = 0; cch < kDH / kCW; ++cch) {
                const int col = kh * kDH + cch * kCW;
                uint32_t rr[kCW];
                tmem_ld_n<kCW>(tmem + lane_addr + kOCol + col, rr);
                tmem_wait_ld();
                if (row_ok) {
                    const size_t o = (static_cast<size_t>(q0 + tk) * p.Hq + h * G + head) * D + col;
                    if (p.out_bf16) {
                        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
#pragma unroll
                        for (int i = 0; i < kCW; i += 2)
                            *reinterpret_cast<__nv_bfloat162*>(dst + i) = __floats2bfloat162_rn(
                                __uint_as_float(rr[i]) * f, __uint_as_float(rr[i + 1]) * f);
                    } else {
                        float* dst = reinterpret_cast<float*>(p.out) + o;
#pragma unroll
                        for (int i = 0; i < kCW; i += 4)
                            *reinterpret_cast<float4*>(dst + i) = make_float4(
                                __uint_as_float(rr[i]) * f, __uint_as_float(rr[i + 1]) * f,
                                __uint_as_float(rr[i + 2]) * f, __uint_as_float(rr[i + 3]) * f);
                    }
                }
            }
        }
        tc_fence_before();
    }

    __syncthreads();
    // every copy and MMA has completed: the barriers' memory may take other
    // data in the next piece (whose layout may differ)
    if (tid == 0)
        for (int i = 0; i < C::kNumBars; ++i) mbar_inval(bar(i));
}

// Geometry of query tile x of a sequence with chunk length nq and context
// ctx_raw (its query rows from q0), KV head h, with all of its key tiles; false
// when the tile holds no query (or its chunk is longer than the context,
// reported when `report_errors`).  split: the tile takes split e4m3 operands
// (some row sees fewer than kSplitKeys keys, or forced).
template <int D, bool BF16, bool PT>
__device__ __forceinline__ bool geo_of(const PrefillParams& p, int q0, int nq, int ctx_raw, int x,
                                       bool report_errors, CtaGeo& cg, bool& split) {
    cg.q0 = q0;
    cg.nq = nq;
    const int TPT = kRows / p.G;                        // query tokens per tile
    cg.tok0 = x * TPT;
    cg.t0 = 0;
    cg.n_tiles = 0;
    cg.part = nullptr;
    split = false;
    if (cg.tok0 >= nq) return false;
    int ctx = ctx_raw;
    if (ctx > p.max_blocks_per_seq * kPage) {
        if (report_errors) report(p.err, FP8KV_ERR_BAD_INDEX);
        ctx = p.max_blocks_per_seq * kPage;
    }
    cg.ctx = ctx;
    cg.pos_base = ctx - nq;                             // position of the chunk's first query
    const int n_tok = min(TPT, nq - cg.tok0);
    const int pos_max = cg.pos_base + cg.tok0 + n_tok - 1;
    const int pos_min = cg.pos_base + cg.tok0;
    if (pos_min < 0) {                                  // chunk longer than the context
        if (report_errors) report(p.err, FP8KV_ERR_BAD_INDEX);
        return false;
    }
    int keys;
    if constexpr (BF16) {
        keys = PCfg<D, true, false, false>::kKeys;      // bf16: no PT
    } else {
        split = p.split == FP8KV_PREFILL_SPLIT_ALWAYS ||
                (p.split == 0 && pos_min + 1 < kSplitKeys);
        keys = split ? PCfg<D, false, true, false>::kKeys : PCfg<D, false, false, false>::kKeys;
    }
    cg.n_tiles = pos_max / keys + 1;
    return true;
}

// geo_of for query tile x of sequence b, KV head h.
template <int D, bool BF16, bool PT>
__device__ bool tile_geo(const PrefillParams& p, int b, int h, int x, bool report_errors,
                         CtaGeo& cg, bool& split) {
    cg.b = b;
    cg.h = h;
    const int q0 = p.cu_seqlens_q[b];
    return geo_of<D, BF16, PT>(p, q0, p.cu_seqlens_q[b + 1] - q0, p.context_lens[b], x,
                               report_errors, cg, split);
}

// Key tiles of query tile x (TPT tokens) of a sequence whose chunk of nq queries
// ends its context of ctx keys (already clamped to the page table): the unit of
// the balanced split, 0 for an empty tile.  The same count as geo_of's, in
// shifts (a tile is 128 keys, 64 for bf16 and split operands).
template <bool BF16>
__device__ __forceinline__ int tile_units(int nq, int ctx, int x, int TPT, int split_mode) {
    const int tok0 = x * TPT;
    if (tok0 >= nq) return 0;
    const int pos_min = ctx - nq + tok0;
    if (pos_min < 0) return 0;
    const int pos_max = ctx - nq + min(tok0 + TPT, nq) - 1;
    const bool split = !BF16 && (split_mode == FP8KV_PREFILL_SPLIT_ALWAYS ||
                                 (split_mode == 0 && pos_min + 1 < kSplitKeys));
    return (pos_max >> ((BF16 || split) ? 6 : 7)) + 1;
}

// Balanced split (persistent launch): the key tiles of every query tile, in the
// order (sequence, KV head, query tile), form one list of W units; CTA c of n
// takes units [c W / n, (c + 1) W / n).  A query tile cut between CTAs leaves a
// partial per piece; the last of its CTAs to finish merges them.
struct Piece {
    int b, h, x;        // the query tile
    int t0, n;          // its key tiles taken
    int cf, cl;         // first and last CTA holding a piece of the tile
};
constexpr int kMaxPieces = 16;     // pieces planned at a time
struct Plan {
    long long W, w0, w1;           // all units; this CTA's range
    long long S;                   // first unit of the next query tile to look at
    int b, h, x;                   // that query tile
    int n_pieces;
    int last;                      // the merge of the current piece falls to this CTA
    Piece pieces[kMaxPieces];
};

// CTA owning unit u under the split of W units over n CTAs.
__device__ __forceinline__ int cta_of(long long u, long long W, int n) {
    return static_cast<int>(((u + 1) * n + W - 1) / W) - 1;
}

// Warp 0 of the CTA: the next pieces of this CTA's range into pl (n_pieces 0
// when the range is done).  First call (pl.S < 0): W, the range and its first
// query tile.
template <int D, bool BF16, bool PT>
__device__ __noinline__ void plan_pieces(const PrefillParams& p, Plan& pl, int lane) {
    static_assert(PCfg<D, false, false, false>::kKeys == 128 &&
                      PCfg<D, false, true, false>::kKeys == 64 &&
                      PCfg<D, true, false, false>::kKeys == 64, "tile_units' shifts");
    const int TPT = kRows / p.G;
    const int n = gridDim.x, c = blockIdx.x;
    const int max_ctx = p.max_blocks_per_seq * kPage;
    if (pl.S < 0) {
        long long W = 0;                               // every sequence's units
        for (int b = 0; b < p.B; ++b) {
            const int nq = p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b];
            const int ctx = min(p.context_lens[b], max_ctx);
            if (c == 0 && lane == 0 && nq > 0 &&       // CTA 0 reports bad geometry
                (p.context_lens[b] > max_ctx || ctx < nq))
                report(p.err, FP8KV_ERR_BAD_INDEX);
            const int nqt = (nq + TPT - 1) / TPT;
            int cost = 0;
            for (int x0 = 0; x0 < nqt; x0 += 32)
                cost += x0 + lane < nqt ? tile_units<BF16>(nq, ctx, x0 + lane, TPT, p.split) : 0;
            for (int o = 16; o > 0; o >>= 1) cost += __shfl_xor_sync(0xffffffffu, cost, o);
            W += static_cast<long long>(cost) * p.Hkv;
        }
        const long long w0 = W * c / n, w1 = W * (c + 1) / n;
        // the query tile holding unit w0
        long long S = 0;
        int b = 0, h = 0, x = 0;
        bool found = w0 >= w1;
        for (; b < p.B && !found; ++b) {
            const int nq = p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b];
            const int ctx = min(p.context_lens[b], max_ctx);
            const int nqt = (nq + TPT - 1) / TPT;
            int cost = 0;
            for (int x0 = 0; x0 < nqt; x0 += 32)
                cost += x0 + lane < nqt ? tile_units<BF16>(nq, ctx, x0 + lane, TPT, p.split) : 0;
            for (int o = 16; o > 0; o >>= 1) cost += __shfl_xor_sync(0xffffffffu, cost, o);
            if (S + static_cast<long long>(cost) * p.Hkv <= w0) {
                S += static_cast<long long>(cost) * p.Hkv;
                continue;
            }
            h = static_cast<int>((w0 - S) / cost);
            S += static_cast<long long>(h) * cost;
            // query tiles of (b, h) 32 at a time: the first whose units pass w0
            for (int x0 = 0; x0 < nqt; x0 += 32) {
                const int ci = x0 + lane < nqt ? tile_units<BF16>(nq, ctx, x0 + lane, TPT, p.split) : 0;
                int inc = ci;                          // inclusive prefix over the lanes
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, inc, o);
                    if (lane >= o) inc += v;
                }
                const unsigned hit = __ballot_sync(0xffffffffu, S + inc > w0);
                if (hit) {
                    const int l0 = __ffs(hit) - 1;
                    x = x0 + l0;
                    S += __shfl_sync(0xffffffffu, inc - ci, l0);
                    break;
                }
                S += __shfl_sync(0xffffffffu, inc, 31);
            }
            found = true;
            break;
        }
        if (lane == 0) {
            pl.W = W;
            pl.w0 = w0;
            pl.w1 = w1;
            pl.S = found && w0 < w1 ? S : w1;          // nothing to do: S = w1
            pl.b = b;
            pl.h = h;
            pl.x = x;
        }
        __syncwarp();
    }
    if (lane == 0) {
        int np = 0;
        long long S = pl.S;
        int b = pl.b, h = pl.h, x = pl.x;
        int nq = 0, ctx = 0, seq = -1;                 // the sequence b's chunk and context
        while (np < kMaxPieces && S < pl.w1 && b < p.B) {
            if (seq != b) {
                nq = p.cu_seqlens_q[b + 1] - p.cu_seqlens_q[b];
                ctx = min(p.context_lens[b], max_ctx);
                seq = b;
            }
            if (x >= (nq + TPT - 1) / TPT) {           // next KV head, next sequence
                x = 0;
                if (++h >= p.Hkv) {
                    h = 0;
                    ++b;
                }
                continue;
            }
            const int cost = tile_units<BF16>(nq, ctx, x, TPT, p.split);
            if (cost > 0) {
                const long long a = S > pl.w0 ? S : pl.w0;
                const long long e = S + cost < pl.w1 ? S + cost : pl.w1;
                Piece& pc = pl.pieces[np++];
                pc.b = b;
                pc.h = h;
                pc.x = x;
                pc.t0 = static_cast<int>(a - S);
                pc.n = static_cast<int>(e - a);
                pc.cf = cta_of(S, pl.W, gridDim.x);
                pc.cl = cta_of(S + cost - 1, pl.W, gridDim.x);
            }
            S += cost;
            ++x;
        }
        // the range's last piece, when cut, goes first: its partner pieces were
        // taken early by the next CTA, so the merge happens early too instead of
        // at the end of the launch
        if (S >= pl.w1 && np > 1 && pl.pieces[np - 1].cf != pl.pieces[np - 1].cl) {
            const Piece last = pl.pieces[np - 1];
            for (int i = np - 1; i > 0; --i) pl.pieces[i] = pl.pieces[i - 1];
            pl.pieces[0] = last;
        }
        pl.S = S;
        pl.b = b;
        pl.h = h;
        pl.x = x;
        pl.n_pieces = np;
    }
    __syncwarp();
}

// Partial slot of CTA c's piece of a query tile whose pieces run from CTA cf:
// the tile is the last piece of cf (slot 2 cf + 1) and the first of the others.
__device__ __forceinline__ float* part_slot(const PrefillParams& p, int c, int cf, int D) {
    const int slot = c == cf ? 2 * c + 1 : 2 * c;
    return p.ws_part + static_cast<size_t>(slot) * kRows * (D + 2);
}

// The output rows of a cut query tile from its pieces' partials (CTAs cf..cl):
// out = sum_i O_i 2^(m_i - M) / sum_i l_i 2^(m_i - M), M the largest m_i.  Every
// thread of the CTA takes part (the body has finished, so its shared memory
// holds the pieces' weights [cl - cf + 1][128]); each thread keeps 8 float4 loads
// per piece in flight, as the partials come from L2.
template <int D>
__device__ __noinline__ void merge_pieces(const PrefillParams& p, const CtaGeo& cg, int cf,
                                          int cl, float* wts, uint32_t bar, int& bar_phase) {
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int G = p.G;
    if (tid < kRows) {
        const int r = tid;
        float M = kMaxInitP, L = 0.f;
        for (int c = cf; c <= cl; ++c)
            M = fmaxf(M, __ldcg(part_slot(p, c, cf, D) + kRows * D + r));
        for (int c = cf; c <= cl; ++c) {
            const float* ps = part_slot(p, c, cf, D);
            const float e = ex2p(__ldcg(ps + kRows * D + r) - M);
            wts[(c - cf) * kRows + r] = e;
            L += __ldcg(ps + kRows * D + kRows + r) * e;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int c = cf; c <= cl; ++c) wts[(c - cf) * kRows + r] *= inv;
    }
    __syncthreads();
    constexpr int kRow4 = D / 4;                        // float4 of a row
    if (cl == cf + 1) {
        // two pieces (the usual cut): half a tile's rows of both partials at a time
        // come into shared memory by bulk copies, which keep far more bytes in
        // flight than loads; out = w0 * O0 + w1 * O1 from there
        constexpr int kHalfRows = kRows / 2;
        constexpr uint32_t kBytes = kHalfRows * D * 4;
        const float4* st0 = reinterpret_cast<const float4*>(wts + 2 * kRows);
        const float4* st1 = st0 + kHalfRows * kRow4;
        const uint32_t dst0 = smem_addr(wts + 2 * kRows);
        for (int hh = 0; hh < 2; ++hh) {
            if (tid == 0) {
                fence_proxy_async_all();                // the partials: other CTAs' stores
                mbar_arrive_expect_tx(bar, 2 * kBytes);
                bulk_load(dst0, part_slot(p, cf, cf, D) + hh * kHalfRows * D, kBytes, bar);
                bulk_load(dst0 + kBytes, part_slot(p, cl, cf, D) + hh * kHalfRows * D, kBytes,
                          bar);
            }
            // (the same answer in every thread: a bounded wait that ran out in one
            // thread ends the merge in all of them)
            const bool landed = __syncthreads_and(mbar_wait_bounded(bar, bar_phase & 1));
            ++bar_phase;
            if (!landed) {
                if (tid == 0) report(p.err, FP8KV_ERR_TIMEOUT);
                return;
            }
            for (int i = tid; i < kHalfRows * kRow4; i += nthreads) {
                const int r = hh * kHalfRows + i / kRow4, col = (i % kRow4) * 4;
                const int tk = cg.tok0 + r / G;
                if (tk >= cg.nq) continue;
                const float w0 = wts[r], w1 = wts[kRows + r];
                const float4 a = st0[i], b = st1[i];
                const float4 acc = make_float4(a.x * w0 + b.x * w1, a.y * w0 + b.y * w1,
                                               a.z * w0 + b.z * w1, a.w * w0 + b.w * w1);
                const size_t o =
                    (static_cast<size_t>(cg.q0 + tk) * p.Hq + cg.h * G + r % G) * D + col;
                if (p.out_bf16) {
                    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
                    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc.x, acc.y);
                    *reinterpret_cast<__nv_bfloat162*>(dst + 2) =
                        __floats2bfloat162_rn(acc.z, acc.w);
                } else {
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) = acc;
                }
            }
            __syncthreads();                            // the staging is read
        }
        return;
    }
    constexpr int kN = kRows * kRow4;
    constexpr int kU = 8;
    for (int base = tid; base < kN; base += kU * nthreads) {
        float4 acc[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = cf; c <= cl; ++c) {
            const float4* ps = reinterpret_cast<const float4*>(part_slot(p, c, cf, D));
            float4 v[kU];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = base + u * nthreads;
                v[u] = i < kN ? __ldcg(ps + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int i = base + u * nthreads;
                const float wgt = i < kN ? wts[(c - cf) * kRows + i / kRow4] : 0.f;
                acc[u].x += v[u].x * wgt;
                acc[u].y += v[u].y * wgt;
                acc[u].z += v[u].z * wgt;
                acc[u].w += v[u].w * wgt;
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int i = base + u * nthreads;
            if (i >= kN) continue;
            const int r = i / kRow4, col = (i % kRow4) * 4;
            const int tk = cg.tok0 + r / G;
            if (tk >= cg.nq) continue;
            const size_t o = (static_cast<size_t>(cg.q0 + tk) * p.Hq + cg.h * G + r % G) * D + col;
            if (p.out_bf16) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(p.out) + o;
                *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[u].x, acc[u].y);
                *reinterpret_cast<__nv_bfloat162*>(dst + 2) =
                    __floats2bfloat162_rn(acc[u].z, acc[u].w);
            } else {
                *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + o) = acc[u];
            }
        }
    }
}

template <int D, bool TWO_LEVEL, bool BF16, bool PT>
__global__ void __launch_bounds__(PCfg<D, BF16, false, PT && !TWO_LEVEL>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using C1 = PCfg<D, BF16, false, PT && !TWO_LEVEL>;   // thread roles of both bodies
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ Plan s_plan;
    __shared__ uint64_t s_merge_bar;                    // the merge's bulk copies
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int kMmaWarp = C1::kSoftWarps + 1;
    if (warp == kMmaWarp) tmem_alloc(smem_addr(&s_tmem), C1::kTmemCols);
    const bool persistent = p.ws_part != nullptr;
    if (tid == 0) {
        s_plan.S = -1;
        s_plan.n_pieces = 0;
        if (persistent) {
            mbar_init(smem_addr(&s_merge_bar), 1);
            mbar_init_fence();
        }
    }
    int merge_phase = 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    int next = 0;                                       // next planned piece
    bool grid_done = false;
    for (;;) {
        CtaGeo cg;
        bool split = false, valid = false;
        if (!persistent) {
            if (grid_done) break;
            grid_done = true;
            // tiles go out last-first: later query tiles see more keys (causal), so
            // the heaviest CTAs take the first wave and the lightest the last one
            valid = tile_geo<D, BF16, PT>(p, blockIdx.z, blockIdx.y,
                                          gridDim.x - 1 - blockIdx.x, tid == 0, cg, split);
            if (!valid) break;
        } else {
            if (next == s_plan.n_pieces) {
                __syncthreads();                        // every thread has read the pieces
                if (warp == 0) plan_pieces<D, BF16, PT>(p, s_plan, lane);
                __syncthreads();
                next = 0;
                if (s_plan.n_pieces == 0) break;
            }
            const Piece pc = s_plan.pieces[next++];
            valid = tile_geo<D, BF16, PT>(p, pc.b, pc.h, pc.x, tid == 0 && pc.cf == blockIdx.x,
                                          cg, split);
            if (!valid) continue;                       // (planned tiles always hold queries)
            cg.t0 = pc.t0;
            cg.n_tiles = pc.n;
            if (pc.cf != pc.cl) cg.part = part_slot(p, blockIdx.x, pc.cf, D);
        }
        if constexpr (BF16) {
            prefill_body<D, TWO_LEVEL, true, PT, false>(kmap, vmap, p, smem, cg, &s_tmem, &s_abort);
        } else if (split) {
            prefill_body<D, TWO_LEVEL, false, PT, true>(kmap, vmap, p, smem, cg, &s_tmem, &s_abort);
        } else {
            prefill_body<D, TWO_LEVEL, false, PT, false>(kmap, vmap, p, smem, cg, &s_tmem,
                                                         &s_abort);
        }
        if (!persistent) continue;
        // ---- a piece of a cut query tile: the last CTA of its pieces to get here
        // merges their partials into the output (the piece and its geometry are
        // read again rather than kept in registers across the body)
        const Piece pc = s_plan.pieces[next - 1];
        const int cf = pc.cf, cl = pc.cl;
        if (cf == cl) continue;
        tile_geo<D, BF16, PT>(p, pc.b, pc.h, pc.x, false, cg, split);
        __threadfence();                                // this CTA's partial, device-wide
        __syncthreads();
        if (tid == 0) {
            const int old = atomicAdd(p.ws_count + cf, 1);
            s_plan.last = old == cl - cf;
            if (s_plan.last) atomicExch(p.ws_count + cf, 0);   // ready for the next call
        }
        __syncthreads();
        if (s_plan.last) {                              // (uniform over the CTA)
            // the pieces' weights fit the shared memory for any GPU of up to
            // (dynamic shared memory) / 512 SMs
            constexpr int kSmemBytes = prefill_smem<D, BF16, PT && !TWO_LEVEL>();
            static_assert(2 * kRows * 4 + kRows * D * 4 <= kSmemBytes - 1024,
                          "two pieces' weights and half rows fit the shared memory");
            if ((cl - cf + 1) * kRows * 4 > kSmemBytes - 1024) {
                if (tid == 0) report(p.err, FP8KV_ERR_UNSUPPORTED);
                continue;
            }
            __threadfence();
            merge_pieces<D>(p, cg, cf, cl, reinterpret_cast<float*>(smem),
                            smem_addr(&s_merge_bar), merge_phase);
            __syncthreads();                            // the weights are read
        }
    }
    tc_fence_before();
    __syncthreads();
    if (persistent && tid == 0) mbar_inval(smem_addr(&s_merge_bar));
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(s_tmem, C1::kTmemCols);
    }
}

template <int D, bool TWO, bool BF16, bool PT>
cudaError_t launch_prefill_t(const PrefillParams& p, const CUtensorMap& kmap,
                             const CUtensorMap& vmap, int grid_x, cudaStream_t stream) {
    auto kern = prefill_kernel<D, TWO, BF16, PT>;
    constexpr int kSmem = prefill_smem<D, BF16, PT && !TWO>();
    static unsigned long long attr_done[64] = {};
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), kSmem, attr_done);
    if (e != cudaSuccess) return e;
    // persistent (balanced split): grid_x CTAs, one per SM
    const dim3 grid = p.ws_part != nullptr ? dim3(grid_x, 1, 1) : dim3(grid_x, p.Hkv, p.B);
    kern<<<grid, PCfg<D, BF16, false, PT && !TWO>::kThreads, kSmem, stream>>>(kmap, vmap, p);
    return cudaGetLastError();
}

template <int D, bool BF16, bool PT>
cudaError_t launch_two(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       int two_level, int grid_x, cudaStream_t stream) {
    return two_level ? launch_prefill_t<D, true, BF16, PT>(p, kmap, vmap, grid_x, stream)
                     : launch_prefill_t<D, false, BF16, PT>(p, kmap, vmap, grid_x, stream);
}

template <int D>
cudaError_t launch_d(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                     bool bf, int two_level, int grid_x, cudaStream_t stream) {
    if (bf) return launch_two<D, true, false>(p, kmap, vmap, two_level, grid_x, stream);
    if (p.scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD)
        return launch_two<D, false, true>(p, kmap, vmap, two_level, grid_x, stream);
    return launch_two<D, false, false>(p, kmap, vmap, two_level, grid_x, stream);
}

}  // namespace

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int D, int kv_dtype, int two_level,
                           int grid_x, cudaStream_t stream) {
    const bool bf = kv_dtype == FP8KV_KV_BF16;
    if (D == 64) return launch_d<64>(p, kmap, vmap, bf, two_level, grid_x, stream);
    if (D == 128) return launch_d<128>(p, kmap, vmap, bf, two_level, grid_x, stream);
    return launch_d<256>(p, kmap, vmap, bf, two_level, grid_x, stream);
}

}  // namespace fp8kv
