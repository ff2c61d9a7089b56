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
//   * grid (split, kv head, seq); 4 warps per CTA share one split's pages
//     round-robin; each warp runs its own TMA ring: lane 0 issues 3-D tiled
//     tensor copies (128-byte swizzle) of the K and V page tiles -- plus the
//     64-byte per-token scale rows -- onto an mbarrier, S stages ahead.
//   * math on the legacy tensor pipe (mma.sync m16n8k16, fp32 accumulate):
//     S^T = K_page . Q^T with M = 16 page tokens, N = 8 query heads of the GQA
//     group, K = D; then O^T += V_page^T . P^T with M = D, N = heads, K = the 16
//     tokens.  e4m3 codes convert exactly to f16 (one cvt per pair), Q is
//     scaled by a per-head power of two into f16's top binade (exact), and P is
//     split into hi + lo halves so the PV product keeps ~22 bits.
//   * per-token-head scales fold out of the dot products: one multiply per
//     logit (k) and per weight (v).  Per-tensor / per-head scales multiply the
//     logit scale and the final output.
//   * online softmax in base 2 with a lazy max (the running max moves only when
//     a page exceeds it by 2^8), fp32 everywhere.
//   * the fragment row/column orders are permuted (token pi(g), d-chunk pi(g))
//     so that every 16-byte shared-memory read of the swizzled tiles is free of
//     bank conflicts for D = 128 e4m3; the permutation is undone when writing.
//   * each split writes (m, l, unnormalised O) to the workspace; split_merge
//     combines the valid splits of a (seq, head).  One split writes `out`
//     directly.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fp8kv {

namespace {

constexpr int kWarps = kDecodeWarps;
__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }
constexpr float kMaxInit = -1.0e30f;   // running-max start: finite, below any real logit

template <int D, bool BF16>
struct Cfg {
    static constexpr int kElem = BF16 ? 2 : 1;
    static constexpr int kRowB = D * kElem;           // bytes of one token row
    static constexpr int kTileB = kPage * kRowB;      // bytes of one (page, head) tile
    // pages per iteration: two when a page tile is small, so each warp works on
    // two independent pages between waits
    static constexpr int kPPI = kRowB <= 128 ? 2 : 1;
    static constexpr int kStageB = 2 * kPPI * kTileB; // K tiles, then V tiles
    static constexpr int kStagesRaw = 16384 / kStageB;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kSegs = kRowB / 64;          // 64-byte segments of a row
    static constexpr int kKPerSeg = 4 / kElem;        // QK k-steps per segment
    static constexpr int kKSteps = D / 16;
    static constexpr int kMTiles = D / 16;            // PV m-tiles (rows of O^T)
    static constexpr int kVBytes = (D / 8) * kElem;   // V bytes a lane reads per token
    static constexpr int kVWords = kVBytes / 4;
    static constexpr int kBoxes = kRowB >= 128 ? kRowB / 128 : 1;
    static constexpr int kWarpSmem = kStages * kStageB;
    static constexpr int kScaleB = 128;               // k scales + v scales of one page
    static constexpr int kSmem = 1024 + kWarps * kWarpSmem + kWarps * kStages * kPPI * kScaleB +
                                 kWarps * kStages * 8 + 16;
    static_assert(kSegs * kKPerSeg == kKSteps, "k-step split");
    static_assert(kWarps * 8 * (D + 2) * 4 <= kWarps * kWarpSmem, "merge area fits the rings");
};

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

// Visible page range of sequence b: positions [lo, ctx) live in pages
// [p_lo, p_hi).  Clamps a context longer than the page table (and reports it).
__device__ __forceinline__ void visible(const DecodeParams& p, int b, int& lo, int& ctx, int& p_lo,
                                        int& p_hi, bool report_errors) {
    ctx = p.context_lens[b];
    if (ctx < 0) ctx = 0;
    if (ctx > p.max_blocks_per_seq * kPage) {
        if (report_errors) report(p.err, FP8KV_ERR_BAD_INDEX);
        ctx = p.max_blocks_per_seq * kPage;
    }
    lo = (p.window > 0 && ctx > p.window) ? ctx - p.window : 0;
    p_lo = lo / kPage;
    p_hi = (ctx + kPage - 1) / kPage;
}

template <bool BF16>
__device__ __forceinline__ void store_out(void* out, int out_bf16, size_t idx, float v) {
    if (out_bf16)
        reinterpret_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else
        reinterpret_cast<float*>(out)[idx] = v;
}

template <int D, bool BF16, bool PER_TOKEN>
__global__ void __launch_bounds__(kWarps * 32)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using C = Cfg<D, BF16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, c = lane & 3;
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int G = p.G;

    int lo, ctx, p_lo, p_hi;
    visible(p, b, lo, ctx, p_lo, p_hi, split == 0 && h == 0 && threadIdx.x == 0);
    const int pb = p_lo + split * p.pages_per_split;
    const int pe = min(pb + p.pages_per_split, p_hi);
    if (pb >= pe) {
        if (p.num_splits == 1 && split == 0) {   // empty context: zero rows
            for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
                const int hq = h * G + i / D;
                store_out<BF16>(p.out, p.out_bf16, (static_cast<size_t>(b) * p.Hq + hq) * D + i % D,
                                0.f);
            }
        }
        return;
    }

    constexpr int PPI = C::kPPI;
    uint8_t* ring = smem + warp * C::kWarpSmem;
    uint8_t* scl = smem + kWarps * C::kWarpSmem + warp * C::kStages * PPI * C::kScaleB;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * C::kWarpSmem +
                                                 kWarps * C::kStages * PPI * C::kScaleB) +
                     warp * C::kStages;
    int* abort_flag = reinterpret_cast<int*>(smem + kWarps * C::kWarpSmem +
                                             kWarps * C::kStages * PPI * C::kScaleB +
                                             kWarps * C::kStages * 8);
    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        mbar_init_fence();
        prefetch_tmap(&kmap);
        prefetch_tmap(&vmap);
    }
    __syncthreads();

    // ---- query fragments (B operand of S^T = K Q^T): head g, elements d0..d0+3
    const int hq_g = h * G + g;
    uint32_t qb[C::kKSteps][2];
    float qscale;                           // log2-domain logit multiplier of head g
    {
        const __nv_bfloat16* qrow = p.q + (static_cast<size_t>(b) * p.Hq + hq_g) * D;
        uint2 raw[C::kKSteps];
#pragma unroll
        for (int ks = 0; ks < C::kKSteps; ++ks) {
            const int s = ks / C::kKPerSeg, jj = ks % C::kKPerSeg;
            const int d0 = s * (64 / C::kElem) + c * (16 / C::kElem) + 4 * jj;
            raw[ks] = g < G ? *reinterpret_cast<const uint2*>(qrow + d0) : make_uint2(0u, 0u);
        }
        float kconst = 1.f;
        if constexpr (!BF16 && !PER_TOKEN)
            kconst = p.scale_mode == FP8KV_SCALE_PER_HEAD ? p.k_scale[h] : p.k_scale[0];
        if constexpr (BF16) {
#pragma unroll
            for (int ks = 0; ks < C::kKSteps; ++ks) {
                qb[ks][0] = raw[ks].x;
                qb[ks][1] = raw[ks].y;
            }
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
                qb[ks][0] = pack_f16x2(bf16_bits_to_float(raw[ks].x & 0xffffu) * f,
                                       bf16_bits_to_float(raw[ks].x >> 16) * f);
                qb[ks][1] = pack_f16x2(bf16_bits_to_float(raw[ks].y & 0xffffu) * f,
                                       bf16_bits_to_float(raw[ks].y >> 16) * f);
            }
            qscale = p.scale_log2 * kconst / f;
        }
    }
    // this lane's S^T / O^T columns are heads 2c and 2c+1
    const float hs0 = __shfl_sync(0xffffffffu, qscale, (2 * c) * 4);
    const float hs1 = __shfl_sync(0xffffffffu, qscale, (2 * c + 1) * 4);

    // ---- work: groups of PPI consecutive pages; this warp takes groups
    //      warp, warp + 4, ...; its j-th group starts at page pb + PPI*(warp + 4j)
    const int n_groups = (pe - pb + PPI - 1) / PPI;
    const int n_my = n_groups > warp ? (n_groups - warp + kWarps - 1) / kWarps : 0;
    const int32_t* bt_row = p.block_table + static_cast<size_t>(b) * p.max_blocks_per_seq;
    constexpr int kGroupsPerBatch = 32 / PPI;
    auto bt_load = [&](int batch) -> int {   // lane L: page L%PPI of group batch*GPB + L/PPI
        const int grp = warp + (batch * kGroupsPerBatch + lane / PPI) * kWarps;
        const int pg = pb + PPI * grp + lane % PPI;
        return pg < pe ? bt_row[pg] : -1;
    };
    int bt_cur = 0, bt_next = 0;
    uint32_t bad_mask = 0u;                 // bit st*PPI+k: page k of stage st is absent/invalid

    auto issue = [&](int j) {               // called by all lanes of the warp
        if ((j % kGroupsPerBatch) == 0) {
            bt_cur = (j == 0) ? bt_load(0) : bt_next;
            bt_next = bt_load(j / kGroupsPerBatch + 1);
        }
        const int st = j % C::kStages;
        const int pg0 = pb + PPI * (warp + j * kWarps);
        int blk[PPI];
        bool here[PPI];
        uint32_t tx = 0;
#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            blk[k] = __shfl_sync(0xffffffffu, bt_cur, (j % kGroupsPerBatch) * PPI + k);
            here[k] = pg0 + k < pe;
            const bool ok = here[k] && blk[k] >= 0 && static_cast<int64_t>(blk[k]) < p.num_blocks;
            const uint32_t bit = 1u << (st * PPI + k);
            bad_mask = ok ? (bad_mask & ~bit) : (bad_mask | bit);
            if (here[k] && !ok) {
                if (lane == 0) report(p.err, FP8KV_ERR_BAD_INDEX);
                blk[k] = 0;                  // load an in-range page, masked later
            }
            if (here[k]) tx += 2 * C::kTileB + (PER_TOKEN ? C::kScaleB : 0);
        }
        if (lane == 0) {
            const uint32_t bar = smem_addr(&bars[st]);
            const uint32_t base = smem_addr(ring + st * C::kStageB);
            fence_proxy_async();
            mbar_arrive_expect_tx(bar, tx);
#pragma unroll
            for (int k = 0; k < PPI; ++k) {
                if (!here[k]) continue;
                const int z = blk[k] * p.Hkv + h;
#pragma unroll
                for (int box = 0; box < C::kBoxes; ++box) {
                    tma_load_3d(base + k * C::kTileB + box * 2048, &kmap, box * 128, 0, z, bar);
                    tma_load_3d(base + (PPI + k) * C::kTileB + box * 2048, &vmap, box * 128, 0, z,
                                bar);
                }
                if constexpr (PER_TOKEN) {
                    const uint32_t sdst = smem_addr(scl + (st * PPI + k) * C::kScaleB);
                    bulk_load(sdst, p.k_scale_cache + static_cast<size_t>(z) * kPage, 64, bar);
                    bulk_load(sdst + 64, p.v_scale_cache + static_cast<size_t>(z) * kPage, 64,
                              bar);
                }
            }
        }
    };

    // fp8 path: P = hi + lo with lo scaled by 2^11 into f16's normal range and
    // accumulated separately (O = o + 2^-11 olo); bf16 P has no subnormal issue
    constexpr int kLoTiles = BF16 ? 1 : C::kMTiles;
    constexpr float kLoScale = 2048.f;
    float o[C::kMTiles][4];
    float olo[kLoTiles][4];
#pragma unroll
    for (int i = 0; i < C::kMTiles; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < kLoTiles; ++i) olo[i][0] = olo[i][1] = olo[i][2] = olo[i][3] = 0.f;
    // running max starts finite so that a fully masked group gives ex2(-inf) = 0
    float m0 = kMaxInit, m1 = kMaxInit, l0 = 0.f, l1 = 0.f;
    bool timed_out = false;
    int drain_from = 0;

    const int pre = n_my < C::kStages ? n_my : C::kStages;
    for (int j = 0; j < pre; ++j) issue(j);

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

    for (int j = 0; j < n_my; ++j) {
        const int st = j % C::kStages;
        const bool arrived =
            mbar_wait_bounded(smem_addr(&bars[st]), static_cast<uint32_t>((j / C::kStages) & 1));
        if (!__all_sync(0xffffffffu, arrived)) {   // leave together
            timed_out = true;
            drain_from = j;
            break;
        }
        const uint8_t* stage = ring + st * C::kStageB;
        const int pos0 = (pb + PPI * (warp + j * kWarps)) * kPage;

        bool bad[PPI], interior[PPI];
#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            bad[k] = (bad_mask >> (st * PPI + k)) & 1u;
            interior[k] = !bad[k] && pos0 + k * kPage >= lo && pos0 + (k + 1) * kPage <= ctx;
        }

        // ---- S^T = K_page Q^T for each page (rows: tokens tA, tB; cols: heads 2c, 2c+1)
        float acc[PPI][4];
#pragma unroll
        for (int k = 0; k < PPI; ++k) acc[k][0] = acc[k][1] = acc[k][2] = acc[k][3] = 0.f;
#pragma unroll
        for (int s = 0; s < C::kSegs; ++s) {
            uint4 kx[PPI], ky[PPI];
#pragma unroll
            for (int k = 0; k < PPI; ++k) {
                kx[k] = *reinterpret_cast<const uint4*>(stage + k * C::kTileB + koffA[s]);
                ky[k] = *reinterpret_cast<const uint4*>(stage + k * C::kTileB + koffB[s]);
            }
#pragma unroll
            for (int jj = 0; jj < C::kKPerSeg; ++jj) {
                const int ks = s * C::kKPerSeg + jj;
#pragma unroll
                for (int k = 0; k < PPI; ++k) {
                    const uint32_t wx[4] = {kx[k].x, kx[k].y, kx[k].z, kx[k].w};
                    const uint32_t wy[4] = {ky[k].x, ky[k].y, ky[k].z, ky[k].w};
                    if constexpr (BF16) {
                        mma_bf16(acc[k], wx[2 * jj], wy[2 * jj], wx[2 * jj + 1], wy[2 * jj + 1],
                                 qb[ks][0], qb[ks][1]);
                    } else {
                        uint32_t xl, xh, yl, yh;
                        f16x2x2_from_e4m3x4(wx[jj], xl, xh);
                        f16x2x2_from_e4m3x4(wy[jj], yl, yh);
                        mma_f16(acc[k], xl, yl, xh, yh, qb[ks][0], qb[ks][1]);
                    }
                }
            }
        }

        // ---- logits (base 2), masked outside [lo, ctx) on boundary pages
        float z[PPI][4], vs[PPI][2];
        float mx0 = neg_inf(), mx1 = neg_inf();
#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            const int posA = pos0 + k * kPage + tA, posB = pos0 + k * kPage + tB;
            const bool vA = interior[k] || (!bad[k] && posA >= lo && posA < ctx);
            const bool vB = interior[k] || (!bad[k] && posB >= lo && posB < ctx);
            float ksA = 1.f, ksB = 1.f;
            vs[k][0] = vs[k][1] = 1.f;
            if constexpr (PER_TOKEN) {
                const float* sk = reinterpret_cast<const float*>(scl + (st * PPI + k) * C::kScaleB);
                ksA = sk[tA];
                ksB = sk[tB];
                // scales of masked tokens may be any bits (slots never written,
                // pages not fetched): zero them so that 0 * scale stays 0
                vs[k][0] = vA ? sk[16 + tA] : 0.f;
                vs[k][1] = vB ? sk[16 + tB] : 0.f;
            }
            z[k][0] = vA ? acc[k][0] * hs0 * ksA : neg_inf();
            z[k][1] = vA ? acc[k][1] * hs1 * ksA : neg_inf();
            z[k][2] = vB ? acc[k][2] * hs0 * ksB : neg_inf();
            z[k][3] = vB ? acc[k][3] * hs1 * ksB : neg_inf();
            mx0 = fmaxf(mx0, fmaxf(z[k][0], z[k][2]));
            mx1 = fmaxf(mx1, fmaxf(z[k][1], z[k][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        // lazy running max: move it only when the group exceeds it by 2^8
        if (mx0 > m0 + 8.f) {
            const float a = ex2(m0 - mx0);
            l0 *= a;
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i) {
                o[i][0] *= a;
                o[i][2] *= a;
            }
            if constexpr (!BF16) {
#pragma unroll
                for (int i = 0; i < kLoTiles; ++i) {
                    olo[i][0] *= a;
                    olo[i][2] *= a;
                }
            }
            m0 = mx0;
        }
        if (mx1 > m1 + 8.f) {
            const float a = ex2(m1 - mx1);
            l1 *= a;
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i) {
                o[i][1] *= a;
                o[i][3] *= a;
            }
            if constexpr (!BF16) {
#pragma unroll
                for (int i = 0; i < kLoTiles; ++i) {
                    olo[i][1] *= a;
                    olo[i][3] *= a;
                }
            }
            m1 = mx1;
        }

#pragma unroll
        for (int k = 0; k < PPI; ++k) {
            // masked logits are -inf and give weight 0 (the running max is finite)
            const float p0 = ex2(z[k][0] - m0), p1 = ex2(z[k][1] - m1);
            const float p2 = ex2(z[k][2] - m0), p3 = ex2(z[k][3] - m1);
            l0 += p0 + p2;
            l1 += p1 + p3;
            const float w0 = p0 * vs[k][0], w1 = p1 * vs[k][0];
            const float w2 = p2 * vs[k][1], w3 = p3 * vs[k][1];

            // ---- P^T as the B operand: hi + lo halves, transposed by movmatrix
            uint32_t bh0, bh1, bl0, bl1;
            if constexpr (BF16) {
                const uint32_t hA = pack_bf16x2(w0, w1), hB = pack_bf16x2(w2, w3);
                const float2 fA = unpack_bf16x2(hA), fB = unpack_bf16x2(hB);
                bh0 = movmatrix_trans(hA);
                bh1 = movmatrix_trans(hB);
                bl0 = movmatrix_trans(pack_bf16x2(w0 - fA.x, w1 - fA.y));
                bl1 = movmatrix_trans(pack_bf16x2(w2 - fB.x, w3 - fB.y));
            } else {
                const uint32_t hA = pack_f16x2(w0, w1), hB = pack_f16x2(w2, w3);
                const float2 fA = unpack_f16x2(hA), fB = unpack_f16x2(hB);
                bh0 = movmatrix_trans(hA);
                bh1 = movmatrix_trans(hB);
                bl0 = movmatrix_trans(pack_f16x2((w0 - fA.x) * kLoScale, (w1 - fA.y) * kLoScale));
                bl1 = movmatrix_trans(pack_f16x2((w2 - fB.x) * kLoScale, (w3 - fB.y) * kLoScale));
            }

            // ---- V rows of tokens c, c+4, c+8, c+12 (k-slots 2c, 2c+1, 2c+8, 2c+9)
            const uint8_t* vt = stage + (PPI + k) * C::kTileB;
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
                    mma_bf16(o[i], a0, a1, a2, a3, bh0, bh1);
                    mma_bf16(o[i], a0, a1, a2, a3, bl0, bl1);
                } else {
                    const int w = i >> 1;
                    const uint32_t sel = (i & 1) ? 0x7362u : 0x5140u;
                    const uint32_t x01 = __byte_perm(vr[0][w], vr[1][w], sel);
                    const uint32_t x23 = __byte_perm(vr[2][w], vr[3][w], sel);
                    f16x2x2_from_e4m3x4(x01, a0, a1);
                    f16x2x2_from_e4m3x4(x23, a2, a3);
                    mma_f16(o[i], a0, a1, a2, a3, bh0, bh1);
                    mma_f16(olo[i < kLoTiles ? i : 0], a0, a1, a2, a3, bl0, bl1);
                }
            }
        }

        __syncwarp();
        if (j + C::kStages < n_my) issue(j + C::kStages);
    }

    if (timed_out) {
        if (lane == 0) report(p.err, FP8KV_ERR_TIMEOUT);
        // let this warp's copies still in flight land (each wait bounded) before
        // the CTA leaves; the output of this split is not written
        const int last = min(drain_from + C::kStages, n_my);
        for (int j = drain_from; j < last; ++j)
            (void)mbar_wait_bounded(smem_addr(&bars[j % C::kStages]),
                                    static_cast<uint32_t>((j / C::kStages) & 1));
        if (lane == 0) *abort_flag = 1;
    }

    // ---- per-warp softmax denominators: sum the 8 lane groups
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, off);
        l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }

    // ---- combine the 4 warps in shared memory (the rings are free now)
    __syncthreads();
    if (*abort_flag) return;
    float* mw = reinterpret_cast<float*>(smem);              // [warp][8]
    float* lw = mw + kWarps * 8;                            // [warp][8]
    float* ow = lw + kWarps * 8;                            // [warp][8][D]
    if (g == 0) {
        mw[warp * 8 + 2 * c] = m0;
        mw[warp * 8 + 2 * c + 1] = m1;
        lw[warp * 8 + 2 * c] = l0;
        lw[warp * 8 + 2 * c + 1] = l1;
    }
    {
        const int dbase = perm8(g) * (D / 8);
        float* o0 = ow + (warp * 8 + 2 * c) * D;
        float* o1 = ow + (warp * 8 + 2 * c + 1) * D;
        if constexpr (!BF16) {
#pragma unroll
            for (int i = 0; i < C::kMTiles; ++i)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[i][r] += olo[i < kLoTiles ? i : 0][r] * (1.f / kLoScale);
        }
#pragma unroll
        for (int i = 0; i < C::kMTiles; ++i) {
            const int d = dbase + 2 * i;
            o0[d] = o[i][0];
            o1[d] = o[i][1];
            o0[d + 1] = o[i][2];
            o1[d + 1] = o[i][3];
        }
    }
    __syncthreads();

    float vconst = 1.f;
    if constexpr (!BF16 && !PER_TOKEN)
        vconst = p.scale_mode == FP8KV_SCALE_PER_HEAD ? p.v_scale[h] : p.v_scale[0];
    for (int i = threadIdx.x; i < G * D; i += blockDim.x) {
        const int head = i / D, d = i % D;
        float M = neg_inf();
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, mw[w * 8 + head]);
        float L = 0.f, O = 0.f;
        if (M != neg_inf()) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float a = ex2(mw[w * 8 + head] - M);
                L += a * lw[w * 8 + head];
                O += a * ow[(w * 8 + head) * D + d];
            }
        }
        O *= vconst;
        const int hq = h * G + head;
        const size_t row = static_cast<size_t>(b) * p.Hq + hq;
        if (p.num_splits == 1) {
            store_out<BF16>(p.out, p.out_bf16, row * D + d, L > 0.f ? O / L : 0.f);
        } else {
            const size_t ws = row * p.num_splits + split;
            p.ws_o[ws * D + d] = O;
            if (d == 0) {
                p.ws_m[ws] = M;
                p.ws_l[ws] = L;
            }
        }
    }
}

// split_merge: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s over the splits
// that hold visible pages of the sequence.
template <int D>
__global__ void __launch_bounds__(128) split_merge_kernel(const DecodeParams p) {
    __shared__ float wgt[1024];
    __shared__ float inv_l;
    const int row = blockIdx.x;                 // b * Hq + hq
    const int b = row / p.Hq;
    int lo, ctx, p_lo, p_hi;
    visible(p, b, lo, ctx, p_lo, p_hi, false);
    const int n_vis = p_hi > p_lo ? p_hi - p_lo : 0;
    int n_valid = (n_vis + p.pages_per_split - 1) / p.pages_per_split;
    if (n_valid > p.num_splits) n_valid = p.num_splits;
    if (n_valid > 1024) n_valid = 1024;
    const float* m = p.ws_m + static_cast<size_t>(row) * p.num_splits;
    const float* l = p.ws_l + static_cast<size_t>(row) * p.num_splits;
    if (threadIdx.x < 32) {
        float M = neg_inf();
        for (int s = threadIdx.x; s < n_valid; s += 32) M = fmaxf(M, m[s]);
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float L = 0.f;
        for (int s = threadIdx.x; s < n_valid; s += 32) {
            const float a = (M == neg_inf()) ? 0.f : ex2(m[s] - M);
            wgt[s] = a;
            L += a * l[s];
        }
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(0xffffffffu, L, off);
        if (threadIdx.x == 0) inv_l = L > 0.f ? 1.f / L : 0.f;
    }
    __syncthreads();
    const float* o = p.ws_o + static_cast<size_t>(row) * p.num_splits * D;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float acc = 0.f;
        for (int s = 0; s < n_valid; ++s) acc += wgt[s] * o[static_cast<size_t>(s) * D + d];
        store_out<false>(p.out, p.out_bf16, static_cast<size_t>(row) * D + d, acc * inv_l);
    }
}

template <int D, bool BF16, bool PER_TOKEN>
cudaError_t launch_split(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         cudaStream_t stream) {
    using C = Cfg<D, BF16>;
    auto kern = paged_decode_kernel<D, BF16, PER_TOKEN>;
    // opt in to the large dynamic shared-memory size once per device
    static bool attr_done[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    dim3 grid(p.num_splits, p.Hkv, p.B);
    kern<<<grid, kWarps * 32, C::kSmem, stream>>>(kmap, vmap, p);
    e = cudaGetLastError();
    if (e != cudaSuccess || p.num_splits == 1) return e;
    split_merge_kernel<D><<<p.B * p.Hq, 128, 0, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch_dtype(const DecodeParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int kv_dtype, cudaStream_t s) {
    if (kv_dtype == FP8KV_KV_BF16) return launch_split<D, true, false>(p, kmap, vmap, s);
    if (p.scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD)
        return launch_split<D, false, true>(p, kmap, vmap, s);
    return launch_split<D, false, false>(p, kmap, vmap, s);
}

template <int D, bool BF16>
constexpr int smem_of() { return Cfg<D, BF16>::kSmem; }

}  // namespace

int decode_ctas_per_sm(int D, int kv_dtype) {
    int bytes;
    const bool bf = kv_dtype == FP8KV_KV_BF16;
    switch (D) {
        case 64: bytes = bf ? smem_of<64, true>() : smem_of<64, false>(); break;
        case 128: bytes = bf ? smem_of<128, true>() : smem_of<128, false>(); break;
        default: bytes = bf ? smem_of<256, true>() : smem_of<256, false>(); break;
    }
    int n = (228 * 1024) / (bytes + 1024);
    return n < 1 ? 1 : (n > 4 ? 4 : n);
}

cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int D, int kv_dtype,
                                cudaStream_t stream) {
    switch (D) {
        case 64: return dispatch_dtype<64>(p, kmap, vmap, kv_dtype, stream);
        case 128: return dispatch_dtype<128>(p, kmap, vmap, kv_dtype, stream);
        default: return dispatch_dtype<256>(p, kmap, vmap, kv_dtype, stream);
    }
}

}  // namespace fp8kv
