// common.cuh -- device helpers shared by the libfp8kv kernels (sm_103a):
// error reporting, bounded mbarrier waits, TMA bulk copies, e4m3 conversions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/fp8kv.h"

namespace fp8kv {

constexpr int kPage = FP8KV_PAGE_SIZE;

// A bounded wait gives up after this many nanoseconds of %globaltimer, reports
// FP8KV_ERR_TIMEOUT and lets the kernel leave instead of hanging the GPU.
constexpr unsigned long long kWaitBudgetNs = 2000000000ull;

__device__ __forceinline__ void report(int32_t* err, int code) {
    if (err != nullptr) atomicCAS(err, 0, code);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Invalidate a barrier whose phases have all completed, so it can be re-initialised.
__device__ __forceinline__ void mbar_inval(uint32_t bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of the barrier; false if the budget ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0u && global_ns() - t0 > kWaitBudgetNs) return false;
    }
}

// Orders this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy (TMA) writes to the same buffer.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- programmatic launch
// A kernel launched with programmatic stream serialization may start before the
// previous kernel in the stream has finished; it must wait here before reading
// anything that kernel (or an earlier one) writes.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel in the stream (if launched programmatically) start early.
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- TMA
// 3-D tiled tensor copy global -> shared, completing on an mbarrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z,
                                            uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// Plain (untiled) bulk copy; both addresses 16-byte aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
        : "memory");
}

// L2 policy for data read once (streamed cache pages): evicted first, so that
// small tables, queries and partial results stay resident in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// tma_load_3d / bulk_load with an L2 cache policy.
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y,
                                                 int z, uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void bulk_load_hint(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(pol)
        : "memory");
}

// One lane's 16-byte asynchronous copy global -> shared (both 16-byte aligned),
// with an L2 cache policy.  Completion is tracked per thread (cp_async_mbar_arrive).
__device__ __forceinline__ void cp_async16_hint(uint32_t dst, const void* src, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "l"(pol)
                 : "memory");
}

// The barrier receives this thread's arrival once all of its earlier cp.async
// copies have landed (the arrival is one of the barrier's expected count).
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Fetch the 128-byte line holding `p` into L2.
__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(p)) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// ---------------------------------------------------------------- conversions
// Two fp32 values -> two e4m3fn bytes (lo in the low byte), round to nearest
// even, saturating to +-448 (NaN stays NaN).
__device__ __forceinline__ uint16_t e4m3x2_from_f32(float lo, float hi) {
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Packed fp32 pairs (sm_100+ f32x2 arithmetic): value a in the low word.
__device__ __forceinline__ uint64_t pack_f32x2(float a, float b) {
    uint64_t d;
    asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
    return d;
}

// Both products rounded to nearest even (IEEE fp32 multiplies, subnormals kept).
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// e4m3_rn_satfinite of both values of a pair (low value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2_from_f32x2(uint64_t v) {
    uint16_t d;
    asm("{\n\t.reg .f32 lo, hi;\n\t"
        "mov.b64 {lo, hi}, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 %0, hi, lo;\n\t}"
        : "=h"(d)
        : "l"(v));
    return d;
}

// e4m3 codes of IEEE fp32 quotients fp32(x / s) in two phases: multiplies by
// two reciprocals for every value (no branches), then the IEEE divide for the
// few pairs whose codes the multiplies cannot certify.
//
// Why the multiplies are exact where they are used: r = __fdividef(1, s) is
// within 2 ulps of 1 / s for |s| in [2^-126, 2^126), so x * r is within 2^-21
// (relative) of x / s.  With r_lo = fp32(r * (1 - 2^-19)) and
// r_hi = fp32(r * (1 + 2^-19)), the products y_lo = fp32(x * r_lo) and
// y_hi = fp32(x * r_hi) therefore lie on either side of Q = fp32(x / s): the
// 2^-19 margins exceed that error plus the roundings.  Rounding to e4m3
// (satfinite) is monotone in the value, so if y_lo and y_hi encode to the same
// code, Q, which lies between them, encodes to it too.  This holds for zeros,
// infinities, fp32 subnormals and overflowing products alike (they encode like
// Q does); NaN inputs give NaN codes on both paths.  The codes differ when a
// rounding midpoint of e4m3 lies between the two products (about 1 % of pairs
// on bf16 data, whose ratios often land on one exactly); those pairs take the
// divide.  Scales outside [2^-126, 2^126) send every pair to the divide.
//
// Phase 1 for N values: codes into w (4 per word, value 0 in the low byte);
// returns the mask of pairs (bit i = values 2i, 2i+1) that need phase 2.
template <int N>
__device__ __forceinline__ uint32_t e4m3_codes_by_multiply(const float (&f)[N], float s,
                                                           uint32_t (&w)[N / 4]) {
    const uint32_t e = (__float_as_uint(s) >> 23) & 0xffu;
    const bool fast = e >= 1u && e <= 252u;              // |s| in [2^-126, 2^126)
    const float r = __fdividef(1.0f, s);
    const float r_lo = __fmul_rn(r, 1.0f - 0x1p-19f);
    const float r_hi = __fmul_rn(r, 1.0f + 0x1p-19f);
    const uint64_t rl = pack_f32x2(r_lo, r_lo), rh = pack_f32x2(r_hi, r_hi);
    // the two bracketing products' codes differ somewhere iff diff != 0 (one
    // three-input logic op per pair); which pairs, only in that rare case
    uint32_t diff = 0u;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const uint64_t x2 = pack_f32x2(f[2 * i], f[2 * i + 1]);
        const uint32_t lo = e4m3x2_from_f32x2(mul_f32x2(x2, rl));
        const uint32_t hi = e4m3x2_from_f32x2(mul_f32x2(x2, rh));
        if (i & 1)
            w[i >> 1] |= lo << 16;
        else
            w[i >> 1] = lo;
        diff |= lo ^ hi;
    }
    if (!fast) return N >= 64 ? ~0u : (1u << (N / 2)) - 1u;
    if (diff == 0u) return 0u;
    uint32_t redo = 0u;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const uint32_t lo = (w[i >> 1] >> (16 * (i & 1))) & 0xffffu;
        const uint32_t hi = e4m3x2_from_f32x2(mul_f32x2(pack_f32x2(f[2 * i], f[2 * i + 1]), rh));
        redo |= static_cast<uint32_t>(lo != hi) << i;
    }
    return redo;
}

// fp32(a / 448) -- the per-token-head scale of a row whose max |x| is a -- for
// a = 0, +inf or any finite non-negative bf16 value (a row maximum of bf16
// inputs always is one).  Division by a constant through its correctly rounded
// reciprocal y and one remainder correction (Markstein's method: q0 = a y,
// r = a - 448 q0 exactly by a fused multiply-add, q = q0 + r y), which rounds
// exactly like the IEEE quotient for every such a (checked exhaustively over
// all finite bf16 values; the writer's tests compare the scales bit for bit).
__device__ __forceinline__ float amax_over_448(float a) {
    constexpr float y = 0x1.24924ap-9f;             // fp32(1 / 448)
    const float q0 = __fmul_rn(a, y);
    const float r = __fmaf_rn(-q0, 448.0f, a);
    const float q = __fmaf_rn(r, y, q0);
    return a == __int_as_float(0x7f800000) ? a : q;
}

// Phase 2 for one pair: codes of fp32(x0 / s), fp32(x1 / s) by IEEE divides.
// Callers store it over the pair's two bytes after storing phase 1's codes (no
// register array is indexed by the pair number, which would move it to local
// memory).
__device__ __forceinline__ uint16_t e4m3x2_by_divide(float x0, float x1, float s) {
    return e4m3x2_from_f32(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
}

// Two e4m3fn bytes (low byte first) -> f16x2, exact.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t two_bytes) {
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two_bytes),
                                               __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Four e4m3fn bytes -> two f16x2 words (bytes 0,1 -> lo; bytes 2,3 -> hi), exact.
// The halves are taken as 16-bit register views so no extraction is needed.
__device__ __forceinline__ void f16x2x2_from_e4m3x4(uint32_t four_bytes, uint32_t& lo,
                                                    uint32_t& hi) {
    asm("{\n\t.reg .b16 l, h;\n\t"
        "mov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_bytes));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_f16x2(uint32_t v) {
    return __half22float2(*reinterpret_cast<__half2*>(&v));
}

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
    return __bfloat1622float2(*reinterpret_cast<__nv_bfloat162*>(&v));
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b16) {
    return __uint_as_float(b16 << 16);
}

}  // namespace fp8kv
