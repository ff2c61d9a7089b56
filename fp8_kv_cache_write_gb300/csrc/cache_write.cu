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
// Design: HBM-streaming.  A group of D/8 lanes owns one row: each lane loads 16
// bytes (8 bf16), the group reduces max|x| with shuffles, each lane divides its
// 8 values by s (IEEE fp32 divide), converts pairs with the satfinite e4m3 cvt
// and stores 8 bytes.  Rows are K and V of every (token, head); the grid strides
// over them, and each lane has the loads of 4 rows in flight before it converts
// any (the data load does not wait for the slot lookup).  Launched with
// programmatic stream serialization: it waits in-kernel for its predecessor.  Reads 4*Hkv*D and writes 2*Hkv*D (+8*Hkv scale) bytes per token.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace fp8kv {

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
                const uint32_t w[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
                float f[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    f[2 * i] = bf16_bits_to_float(w[i] & 0xffffu);
                    f[2 * i + 1] = bf16_bits_to_float(w[i] >> 16);
                }
                float s;
                if constexpr (MODE == FP8KV_SCALE_PER_TOKEN_HEAD) {
                    float amax = 0.f;
#pragma unroll
                    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
#pragma unroll
                    for (int o = kLanes / 2; o > 0; o >>= 1)
                        amax = fmaxf(amax, __shfl_xor_sync(group_mask, amax, o));
                    s = __fdiv_rn(amax, 448.0f);
                    if (l == 0) (which ? p.v_scale_cache : p.k_scale_cache)[row] = s;
                } else if constexpr (MODE == FP8KV_SCALE_PER_HEAD) {
                    s = (which ? p.v_scale : p.k_scale)[h];
                } else {
                    s = (which ? p.v_scale : p.k_scale)[0];
                }
                uint32_t packed[2] = {0u, 0u};
                if (s != 0.0f) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t c = e4m3x2_from_f32(__fdiv_rn(f[2 * i], s),
                                                           __fdiv_rn(f[2 * i + 1], s));
                        packed[i >> 1] |= c << (16 * (i & 1));
                    }
                }
                uint8_t* dst = reinterpret_cast<uint8_t*>(which ? p.v_cache : p.k_cache);
                *reinterpret_cast<uint2*>(dst + row * D + l * 8) = make_uint2(packed[0], packed[1]);
            }
        }
    }
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
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv_cache_write_kernel<D, MODE, BF16>, p);
}

template <int D>
static cudaError_t dispatch_mode(const WriteParams& p, int kv_dtype, int mode, cudaStream_t s,
                                 int sms) {
    if (kv_dtype == FP8KV_KV_BF16) return launch_write<D, 0, true>(p, s, sms);
    switch (mode) {
        case FP8KV_SCALE_PER_TENSOR: return launch_write<D, FP8KV_SCALE_PER_TENSOR, false>(p, s, sms);
        case FP8KV_SCALE_PER_HEAD: return launch_write<D, FP8KV_SCALE_PER_HEAD, false>(p, s, sms);
        default: return launch_write<D, FP8KV_SCALE_PER_TOKEN_HEAD, false>(p, s, sms);
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
// The writer's encoder on its own, elementwise: out[i] = e4m3(x[i] / scale).
__global__ void __launch_bounds__(256) quantize_e4m3_kernel(const float* __restrict__ x,
                                                            float scale,
                                                            uint8_t* __restrict__ out,
                                                            int64_t n) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 4;
    for (int64_t i = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 4; i < n;
         i += stride) {
        uint32_t packed = 0u;
        if (i + 4 <= n && (reinterpret_cast<uintptr_t>(x + i) & 15u) == 0u) {
            const float4 v = *reinterpret_cast<const float4*>(x + i);
            if (scale != 0.0f) {
                packed = e4m3x2_from_f32(__fdiv_rn(v.x, scale), __fdiv_rn(v.y, scale)) |
                         (static_cast<uint32_t>(e4m3x2_from_f32(__fdiv_rn(v.z, scale),
                                                                __fdiv_rn(v.w, scale)))
                          << 16);
            }
            if ((reinterpret_cast<uintptr_t>(out + i) & 3u) == 0u) {
                *reinterpret_cast<uint32_t*>(out + i) = packed;
                continue;
            }
            for (int j = 0; j < 4; ++j) out[i + j] = static_cast<uint8_t>(packed >> (8 * j));
        } else {
            for (int64_t j = i; j < n && j < i + 4; ++j) {
                const float q = scale != 0.0f ? __fdiv_rn(x[j], scale) : 0.0f;
                out[j] = scale != 0.0f ? static_cast<uint8_t>(e4m3x2_from_f32(q, 0.0f) & 0xffu)
                                       : static_cast<uint8_t>(0);
            }
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
