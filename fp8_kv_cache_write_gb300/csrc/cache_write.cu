// cache_write.cu -- kv_cache_write: quantize bf16 K/V rows into the paged e4m3
// cache (or copy them into the bf16 cache).
//
// What it computes ("[vLLM] KV Cache Quantization: KV 캐시 FP8/INT8 양자화",
// section "Per-Token-Head vs Per-Tensor 양자화"; "vLLM FP8 KV-Cache 및 Attention
// 양자화 업데이트", opening paragraph and "커널 및 퓨전 최적화"): every (token, KV
// head) row of D values is stored at slot = block * 16 + offset as e4m3 codes
// e4m3_rn_satfinite(fp32(x / s)).  s is the per-tensor scale, the head's scale,
// or -- per-token-head -- fp32(max|x| / 448), which the kernel computes while
// storing and writes beside the page.
//
// Two kernels, both HBM-streaming (read 4*Hkv*D, write 2*Hkv*D (+8*Hkv scale)
// bytes per token):
//   * staged (bulk writes from device memory): K and V are contiguous
//     [T*Hkv][D] arrays, so one producer lane bulk-copies 12 KiB chunks of each
//     (cp.async.bulk, L2 evict-first) into a 3-stage shared-memory ring, and 8
//     consumer warps quantize rows out of shared memory.  The bytes in flight
//     (3 CTAs x 2 of their 3 stages of 24 KiB per SM) no longer depend on registers.
//   * direct (small writes, e.g. one decode step, or inputs in pinned host
//     memory): D/8 lanes own one row and keep the loads of 4 rows in flight.
// Each lane quantizes in two phases: a branch-free multiply by fp32(1/s) whose
// codes are certified equal to those of the IEEE quotient, then the IEEE divide
// for the few pairs the certificate rejects (e4m3_codes_by_multiply).
// Both launch with programmatic stream serialization and wait in-kernel for
// their predecessor.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fp8kv {

// ---------------------------------------------------------------- one row
// Scale of a row held by a group of lanes (each lane holds N values): the
// mode's constant, or fp32(max|x| / 448) reduced over the group.
template <int MODE, int kLanes, int N>
__device__ __forceinline__ float row_scale(const float (&f)[N], const WriteParams& p, int which,
                                           int h, unsigned group_mask) {
    if constexpr (MODE == FP8KV_SCALE_PER_TOKEN_HEAD) {
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < N; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
        for (int o = kLanes / 2; o > 0; o >>= 1)
            amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, o));
        return amax_over_448(amax);
    } else if constexpr (MODE == FP8KV_SCALE_PER_HEAD) {
        return (which ? p.v_scale : p.k_scale)[h];
    } else {
        return (which ? p.v_scale : p.k_scale)[0];
    }
}

__device__ __forceinline__ void unpack8(uint4 x, float* f) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
        f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
    }
}

// ---------------------------------------------------------------- staged kernel
namespace staged {
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;   // + one producer warp
constexpr int kStages = 4;
constexpr int kTileBytes = 8192;                      // per tensor (K or V) per stage
constexpr int kSmemBytes = kStages * 2 * kTileBytes + 2 * kStages * 8;
constexpr int kCtasPerSm = 3;
// bulk writes only: below this many (token, head) rows the direct kernel runs
constexpr int64_t kMinRows = 8192;
}  // namespace staged

// CTA c takes chunks c, c + gridDim.x, ...; chunk i holds rows
// [i * rows_per_chunk, min(rows, (i + 1) * rows_per_chunk)) of K and of V
// (rows_per_chunk <= 8 KiB / (2 D)).  hkv_shift = log2(Hkv) when Hkv is a power
// of two, else -1.
template <int D, int MODE, bool BF16>
__global__ void __launch_bounds__(staged::kThreads, staged::kCtasPerSm)
    kv_cache_write_staged_kernel(WriteParams p, int rows_per_chunk, int64_t nchunks,
                                 int hkv_shift) {
    using namespace staged;
    constexpr int kMaxRows = kTileBytes / (D * 2);
    constexpr int kLanes = D / 32;                    // lanes per row, 32 values each
    constexpr int kRowsPerPass = 32 / kLanes;
    constexpr int kPasses = 2 * kMaxRows / (kRowsPerPass * kConsumerWarps);
    static_assert(kPasses * kRowsPerPass * kConsumerWarps == 2 * kMaxRows, "row split");

    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * 2 * kTileBytes);
    uint64_t* empty = full + kStages;
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_addr(&full[s]), 1);
            mbar_init(smem_addr(&empty[s]), kConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    pdl_wait();                              // inputs of earlier kernels are visible
    pdl_trigger();
    const int64_t rows = p.T * p.Hkv;

    if (warp == kConsumerWarps) {            // producer: one lane issues every copy
        if (lane != 0) return;
        const uint64_t pol = l2_evict_first();   // inputs are read once
        int j = 0;
        for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++j) {
            const int st = j % kStages;
            if (j >= kStages &&
                !mbar_wait_bounded(smem_addr(&empty[st]), ((j / kStages) - 1) & 1)) {
                report(p.err, FP8KV_ERR_TIMEOUT);
                return;
            }
            const int64_t r0 = c * rows_per_chunk;
            const int64_t n = rows - r0 < rows_per_chunk ? rows - r0 : rows_per_chunk;
            const uint32_t bytes = static_cast<uint32_t>(n) * (D * 2);
            const uint32_t bar = smem_addr(&full[st]);
            uint8_t* tile = smem + st * 2 * kTileBytes;
            mbar_arrive_expect_tx(bar, 2 * bytes);
            bulk_load_hint(smem_addr(tile), p.k + r0 * D, bytes, bar, pol);
            bulk_load_hint(smem_addr(tile + kTileBytes), p.v + r0 * D, bytes, bar, pol);
        }
        return;
    }

    const int sub = lane / kLanes;           // row within the pass
    const int l = lane % kLanes;             // lane within the row
    const unsigned group_mask =
        kLanes == 32 ? 0xffffffffu : (((1u << kLanes) - 1u) << (sub * kLanes));
    int j = 0;
    for (int64_t c = blockIdx.x; c < nchunks; c += gridDim.x, ++j) {
        const int st = j % kStages;
        const int64_t r0 = c * rows_per_chunk;
        const int n = static_cast<int>(rows - r0 < rows_per_chunk ? rows - r0 : rows_per_chunk);
        const int64_t t0 = hkv_shift >= 0 ? (r0 >> hkv_shift) : r0 / p.Hkv;
        const int h0 = static_cast<int>(r0 - t0 * p.Hkv);
        // slots of this lane's rows, fetched while the chunk is still in flight
        int64_t slot[kPasses];
        int hh[kPasses];
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
            const int jb = (it * kConsumerWarps + warp) * kRowsPerPass + sub;
            const int rr = jb % kMaxRows;
            slot[it] = -1;
            hh[it] = 0;
            if (rr < n) {
                const int u = h0 + rr;
                const int dt = hkv_shift >= 0 ? (u >> hkv_shift) : u / p.Hkv;
                hh[it] = u - dt * p.Hkv;
                slot[it] = p.slot_mapping[t0 + dt];
            }
        }
        if (!mbar_wait_bounded(smem_addr(&full[st]), (j / kStages) & 1)) {
            if (lane == 0) report(p.err, FP8KV_ERR_TIMEOUT);
            return;
        }
        const uint8_t* tile = smem + st * 2 * kTileBytes;
#pragma unroll
        for (int it = 0; it < kPasses; ++it) {
            const int jb = (it * kConsumerWarps + warp) * kRowsPerPass + sub;
            const int which = jb / kMaxRows;             // 0 = K, 1 = V
            const int rr = jb % kMaxRows;
            if (slot[it] < 0) continue;                  // the row's lanes leave together
            const int64_t blk = slot[it] >> 4;
            const int off = static_cast<int>(slot[it] & 15);
            if (blk >= p.num_blocks) {
                if (l == 0) report(p.err, FP8KV_ERR_BAD_INDEX);
                continue;
            }
            const int h = hh[it];
            const int64_t row = (blk * p.Hkv + h) * kPage + off;
            // the lane's values: [16l, 16l + 16) and [D/2 + 16l, D/2 + 16l + 16) (four
            // 16-byte shared-memory reads); its codes are two 16-byte stores
            const uint8_t* src = tile + which * kTileBytes + rr * (D * 2);
            const uint4 a0 = *reinterpret_cast<const uint4*>(src + l * 32);
            const uint4 a1 = *reinterpret_cast<const uint4*>(src + l * 32 + 16);
            const uint4 b0 = *reinterpret_cast<const uint4*>(src + D + l * 32);
            const uint4 b1 = *reinterpret_cast<const uint4*>(src + D + l * 32 + 16);
            if constexpr (BF16) {
                uint8_t* dst = reinterpret_cast<uint8_t*>(which ? p.v_cache : p.k_cache) +
                               row * (D * 2);
                *reinterpret_cast<uint4*>(dst + l * 32) = a0;
                *reinterpret_cast<uint4*>(dst + l * 32 + 16) = a1;
                *reinterpret_cast<uint4*>(dst + D + l * 32) = b0;
                *reinterpret_cast<uint4*>(dst + D + l * 32 + 16) = b1;
            } else {
                float f[32];
                unpack8(a0, f);
                unpack8(a1, f + 8);
                unpack8(b0, f + 16);
                unpack8(b1, f + 24);
                const float s = row_scale<MODE, kLanes>(f, p, which, h, group_mask);
                if constexpr (MODE == FP8KV_SCALE_PER_TOKEN_HEAD) {
                    if (l == 0) (which ? p.v_scale_cache : p.k_scale_cache)[row] = s;
                }
                uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};   // a zero scale writes code 0
                uint32_t redo = 0u;
                if (s != 0.0f) redo = e4m3_codes_by_multiply(f, s, w);
                uint8_t* dst = reinterpret_cast<uint8_t*>(which ? p.v_cache : p.k_cache) + row * D;
                *reinterpret_cast<uint4*>(dst + l * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                *reinterpret_cast<uint4*>(dst + D / 2 + l * 16) = make_uint4(w[4], w[5], w[6], w[7]);
                while (redo) {                       // rare: reread the pair, divide, restore
                    const int i = __ffs(redo) - 1;
                    redo &= redo - 1u;
                    // the pair's two codes, from dst + 16 l, and its two bf16 values
                    const int e = i < 8 ? 2 * i : D / 2 + 2 * (i - 8);
                    const uint32_t pr = *reinterpret_cast<const uint32_t*>(
                        src + (i < 8 ? l * 32 + 4 * i : D + l * 32 + 4 * (i - 8)));
                    *reinterpret_cast<uint16_t*>(dst + l * 16 + e) = e4m3x2_by_divide(
                        bf16_bits_to_float(pr & 0xffffu), bf16_bits_to_float(pr >> 16), s);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
    }
}

// ---------------------------------------------------------------- direct kernel
template <int D, int MODE, bool BF16>
__global__ void __launch_bounds__(256) kv_cache_write_kernel(WriteParams p) {
    constexpr int kLanes = D / 8;            // lanes per row (8 bf16 each)
    constexpr int kRowsPerWarp = 32 / kLanes;
    const int lane = threadIdx.x & 31;
    const int sub = lane / kLanes;           // row within the warp
    const int l = lane % kLanes;             // lane within the row
    const unsigned group_mask =
        kLanes == 32 ? 0xffffffffu : (((1u << kLanes) - 1u) << (sub * kLanes));

    // wait first: a dependent decode may start its set-up (which reads tables that
    // kernels before this one may have written) as soon as this kernel triggers
    pdl_wait();                              // inputs of earlier kernels are visible
    pdl_trigger();                           // the decode step may start setting up
    const int64_t rows = p.T * p.Hkv * 2;    // (token, head, K|V)
    const int64_t warp_global = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) / 32;
    const int64_t warp_stride = static_cast<int64_t>(gridDim.x) * blockDim.x / 32;
    const int64_t step = warp_stride * kRowsPerWarp;   // rows between a lane's unrolled rows
    constexpr int kUnroll = 4;               // row groups whose loads are in flight together

    for (int64_t base = warp_global * kRowsPerWarp + sub; base < rows; base += kUnroll * step) {
        // all loads of the kUnroll rows first (the data load does not wait for the slot)
        uint4 x[kUnroll];
        int64_t slot[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * step;
            slot[u] = -1;
            x[u] = make_uint4(0u, 0u, 0u, 0u);
            if (r < rows) {
                const int64_t th = r >> 1;
                const int64_t t = th / p.Hkv;
                const int h = static_cast<int>(th - t * p.Hkv);
                slot[u] = p.slot_mapping[t];
                const __nv_bfloat16* src = ((r & 1) ? p.v : p.k) + (t * p.Hkv + h) * D;
                x[u] = *reinterpret_cast<const uint4*>(src + l * 8);
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t r = base + u * step;
            if (r >= rows || slot[u] < 0) continue;   // whole row group leaves together
            const int which = static_cast<int>(r & 1);          // 0 = K, 1 = V
            const int64_t th = r >> 1;
            const int h = static_cast<int>(th - (th / p.Hkv) * p.Hkv);
            const int64_t blk = slot[u] / kPage;
            const int off = static_cast<int>(slot[u] - blk * kPage);
            if (blk >= p.num_blocks) {
                if (l == 0) report(p.err, FP8KV_ERR_BAD_INDEX);
                continue;
            }
            const int64_t row = (blk * p.Hkv + h) * kPage + off;
            if constexpr (BF16) {
                __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(which ? p.v_cache : p.k_cache);
                *reinterpret_cast<uint4*>(dst + row * D + l * 8) = x[u];
                continue;
            } else {
                float f[8];
                unpack8(x[u], f);
                const float s = row_scale<MODE, kLanes>(f, p, which, h, group_mask);
                if constexpr (MODE == FP8KV_SCALE_PER_TOKEN_HEAD) {
                    if (l == 0) (which ? p.v_scale_cache : p.k_scale_cache)[row] = s;
                }
                uint32_t w[2] = {0u, 0u};            // a zero scale writes code 0
                uint32_t redo = 0u;
                if (s != 0.0f) redo = e4m3_codes_by_multiply(f, s, w);
                uint8_t* dst = reinterpret_cast<uint8_t*>(which ? p.v_cache : p.k_cache) +
                               row * D + l * 8;
                *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
                while (redo) {                       // rare: divide the pair, restore its codes
                    const int i = __ffs(redo) - 1;
                    redo &= redo - 1u;
                    const uint32_t pr = i == 0 ? x[u].x : i == 1 ? x[u].y : i == 2 ? x[u].z : x[u].w;
                    *reinterpret_cast<uint16_t*>(dst + 2 * i) = e4m3x2_by_divide(
                        bf16_bits_to_float(pr & 0xffffu), bf16_bits_to_float(pr >> 16), s);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- launchers
// Host queries made while the calling thread may be capturing a CUDA graph in
// global mode (which refuses calls it deems unsafe) switch this thread to
// relaxed capture mode for their duration.
struct RelaxedCapture {
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    RelaxedCapture() { cudaThreadExchangeStreamCaptureMode(&mode); }
    ~RelaxedCapture() { cudaThreadExchangeStreamCaptureMode(&mode); }
};

static cudaLaunchConfig_t pdl_config(cudaLaunchAttribute* attr, int64_t blocks, int threads,
                                     size_t smem, cudaStream_t stream) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int D, int MODE, bool BF16>
static cudaError_t launch_write(const WriteParams& p, cudaStream_t stream, int num_sms) {
    constexpr int kRowsPerBlock = 256 / (D / 8);
    const int64_t rows = p.T * p.Hkv * 2;
    int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
    const int64_t cap = static_cast<int64_t>(num_sms) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(attr, blocks, 256, 0, stream);
    return cudaLaunchKernelEx(&cfg, kv_cache_write_kernel<D, MODE, BF16>, p);
}

template <int D, int MODE, bool BF16>
static cudaError_t launch_write_staged(const WriteParams& p, cudaStream_t stream, int num_sms) {
    using namespace staged;
    constexpr int64_t kMaxRows = kTileBytes / (D * 2);
    auto kern = kv_cache_write_staged_kernel<D, MODE, BF16>;
    static unsigned long long attr_done[64] = {};   // large dynamic shared memory, once per context
    cudaError_t e = opt_in_smem(reinterpret_cast<const void*>(kern), kSmemBytes, attr_done);
    if (e != cudaSuccess) return e;
    // equal chunk counts per CTA: as many chunk rounds as full-size chunks need,
    // then the chunk size that spreads the rows evenly over them
    const int64_t rows = p.T * p.Hkv;
    const int64_t ctas = static_cast<int64_t>(num_sms) * kCtasPerSm;
    const int64_t rounds = (rows + ctas * kMaxRows - 1) / (ctas * kMaxRows);
    const int64_t rows_per_chunk = (rows + ctas * rounds - 1) / (ctas * rounds);
    const int64_t nchunks = (rows + rows_per_chunk - 1) / rows_per_chunk;
    const int64_t grid = nchunks < ctas ? nchunks : ctas;
    int hkv_shift = -1;
    for (int s = 0; s < 31; ++s)
        if ((1 << s) == p.Hkv) hkv_shift = s;
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pdl_config(attr, grid, kThreads, kSmemBytes, stream);
    return cudaLaunchKernelEx(&cfg, kern, p, static_cast<int>(rows_per_chunk), nchunks, hkv_shift);
}

// The staged kernel reads K and V with bulk copies; it runs for bulk writes
// whose inputs are device memory of the current GPU (pinned host inputs take the
// direct kernel, whose plain loads read them over the host link).
static bool use_staged(const WriteParams& p) {
    if (p.T * p.Hkv < staged::kMinRows) return false;
    RelaxedCapture relaxed;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    for (const void* ptr : {static_cast<const void*>(p.k), static_cast<const void*>(p.v)}) {
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        // device memory of this GPU only (peer or managed memory takes the plain loads)
        if (a.type != cudaMemoryTypeDevice || a.device != dev) return false;
    }
    return true;
}

template <int D, int MODE, bool BF16>
static cudaError_t launch_any(const WriteParams& p, cudaStream_t s, int sms) {
    return use_staged(p) ? launch_write_staged<D, MODE, BF16>(p, s, sms)
                         : launch_write<D, MODE, BF16>(p, s, sms);
}

template <int D>
static cudaError_t dispatch_mode(const WriteParams& p, int kv_dtype, int mode, cudaStream_t s,
                                 int sms) {
    if (kv_dtype == FP8KV_KV_BF16) return launch_any<D, 0, true>(p, s, sms);
    switch (mode) {
        case FP8KV_SCALE_PER_TENSOR: return launch_any<D, FP8KV_SCALE_PER_TENSOR, false>(p, s, sms);
        case FP8KV_SCALE_PER_HEAD: return launch_any<D, FP8KV_SCALE_PER_HEAD, false>(p, s, sms);
        default: return launch_any<D, FP8KV_SCALE_PER_TOKEN_HEAD, false>(p, s, sms);
    }
}

cudaError_t launch_kv_cache_write(const WriteParams& p, int D, int kv_dtype, int mode,
                                  cudaStream_t stream, int num_sms) {
    switch (D) {
        case 64: return dispatch_mode<64>(p, kv_dtype, mode, stream, num_sms);
        case 128: return dispatch_mode<128>(p, kv_dtype, mode, stream, num_sms);
        default: return dispatch_mode<256>(p, kv_dtype, mode, stream, num_sms);
    }
}

// ---------------------------------------------------------------- quantize
// The writer's encoder on its own, elementwise: out[i] = e4m3(fp32(x[i] / scale)),
// through the same two phases as the cache writer.
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const float* __restrict__ x,
                                                            float scale,
                                                            uint8_t* __restrict__ out,
                                                            int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < n;
         i += stride) {
        float f[4] = {0.f, 0.f, 0.f, 0.f};
        if (i + 4 <= n && (reinterpret_cast<uintptr_t>(x + i) & 15u) == 0u) {
            const float4 v = *reinterpret_cast<const float4*>(x + i);
            f[0] = v.x;
            f[1] = v.y;
            f[2] = v.z;
            f[3] = v.w;
        } else {
            for (int j = 0; j < 4 && i + j < n; ++j) f[j] = x[i + j];
        }
        uint32_t w[1] = {0u};                // a zero scale writes code 0
        if (scale != 0.0f) {
            const uint32_t redo = e4m3_codes_by_multiply(f, scale, w);
            if (redo & 1u) w[0] = (w[0] & 0xffff0000u) | e4m3x2_by_divide(f[0], f[1], scale);
            if (redo & 2u)
                w[0] = (w[0] & 0x0000ffffu) |
                       (static_cast<uint32_t>(e4m3x2_by_divide(f[2], f[3], scale)) << 16);
        }
        if (i + 4 <= n && (reinterpret_cast<uintptr_t>(out + i) & 3u) == 0u) {
            *reinterpret_cast<uint32_t*>(out + i) = w[0];
        } else {
            for (int j = 0; j < 4 && i + j < n; ++j) out[i + j] = static_cast<uint8_t>(w[0] >> (8 * j));
        }
    }
}

cudaError_t launch_quantize_e4m3(const float* x, float scale, uint8_t* out, int64_t n,
                                 cudaStream_t stream, int num_sms) {
    int64_t blocks = (n + 1023) / 1024;
    const int64_t cap = static_cast<int64_t>(num_sms) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    quantize_e4m3_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(x, scale, out, n);
    return cudaGetLastError();
}

}  // namespace fp8kv
