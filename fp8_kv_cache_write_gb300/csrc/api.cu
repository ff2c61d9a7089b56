// api.cu -- the extern "C" boundary of libfp8kv: host-side validation, the
// decode split planner, TMA tensor-map encoding and kernel launches.  Every
// check runs before the first launch, so an invalid call launches nothing.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/fp8kv.h"
#include "internal.h"

namespace fp8kv {

unsigned long long current_context_id() {
    using GetCurrent = CUresult (*)(CUcontext*);
    using GetId = CUresult (*)(CUcontext, unsigned long long*);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* a = nullptr;
        void* b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                             &qa) == cudaSuccess &&
            qa == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
                cudaSuccess &&
            qb == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrent>(a);
            get_id = reinterpret_cast<GetId>(b);
        } else {
            cudaGetLastError();
        }
    });
    if (get_current == nullptr || get_id == nullptr) return 0;
    CUcontext c = nullptr;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || c == nullptr || get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id + 1;
}

cudaError_t opt_in_smem(const void* func, int bytes, unsigned long long (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long id = current_context_id();
    if (dev >= 0 && dev < 64 && id != 0 && done[dev] == id) return cudaSuccess;
    // a setting, not a stream operation: allowed while another thread captures
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    cudaThreadExchangeStreamCaptureMode(&mode);
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    cudaThreadExchangeStreamCaptureMode(&mode);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) done[dev] = current_context_id();
    return cudaSuccess;
}

}  // namespace fp8kv

namespace {

using namespace fp8kv;

thread_local std::string g_warning;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// SM count of the current device (cached per device; 152 if none is visible).
int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 152;
    }
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            n <= 0) {
            cudaGetLastError();
            n = 152;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        else
            cudaGetLastError();
    });
    return fn;
}

// Tensor map over a paged cache [num_blocks * Hkv][16][row_bytes] (bytes):
// boxes of 16 rows x 128 bytes with 128-byte swizzle.  64-byte rows are viewed
// as 8 rows of 128 bytes, two tokens each (decode), or copied as 16 rows of 64
// bytes with the 64-byte swizzle (prefill's MMA operands, sw64).  Encodings are
// cached per thread.
struct MapKey {
    const void* base;
    int row_bytes;
    int64_t nbh;
    bool sw64;
    int depth;
};

// depth: (block, head) tiles per box, adjacent heads of one block (decode units
// of packed heads take 2)
bool make_kv_map(const void* base, int row_bytes, int64_t nbh, CUtensorMap* out,
                 bool sw64 = false, int depth = 1) {
    sw64 = sw64 && row_bytes == 64;
    struct Entry {
        MapKey key;
        CUtensorMap map;
        bool used;
    };
    thread_local Entry cache[8] = {};
    thread_local int next = 0;
    for (auto& e : cache)
        if (e.used && e.key.base == base && e.key.row_bytes == row_bytes && e.key.nbh == nbh &&
            e.key.sw64 == sw64 && e.key.depth == depth) {
            *out = e.map;
            return true;
        }
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3];
    cuuint64_t strides[2];
    cuuint32_t box[3];
    const cuuint32_t estr[3] = {1, 1, 1};
    if (sw64) {
        dims[0] = 64; dims[1] = 16; dims[2] = static_cast<cuuint64_t>(nbh);
        strides[0] = 64; strides[1] = 1024;
        box[0] = 64; box[1] = 16; box[2] = 1;
    } else if (row_bytes == 64) {
        dims[0] = 128; dims[1] = 8; dims[2] = static_cast<cuuint64_t>(nbh);
        strides[0] = 128; strides[1] = 1024;
        box[0] = 128; box[1] = 8; box[2] = static_cast<cuuint32_t>(depth);
    } else {
        dims[0] = static_cast<cuuint64_t>(row_bytes); dims[1] = 16;
        dims[2] = static_cast<cuuint64_t>(nbh);
        strides[0] = static_cast<cuuint64_t>(row_bytes);
        strides[1] = static_cast<cuuint64_t>(row_bytes) * 16;
        box[0] = 128; box[1] = 16; box[2] = static_cast<cuuint32_t>(depth);
    }
    CUtensorMap m;
    CUresult r = fn(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    sw64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return false;
    cache[next] = Entry{MapKey{base, row_bytes, nbh, sw64, depth}, m, true};
    next = (next + 1) % 8;
    *out = m;
    return true;
}

struct Plan {
    int num_splits;          // CTAs of the decode grid (work partitions)
    size_t workspace_bytes;
    bool cta_units;          // one CTA per unit, combining in shared memory
};

// Decode planner.  The launch's (seq, KV head, page) tiles are split evenly over
// the 4 warps of `num_splits` CTAs.  Automatic: one wave of resident CTAs, but no fewer than
// 16 tiles per CTA for the upper bound of the work (B * Hkv * visible pages);
// an explicit count n asks for about n partitions per (seq, KV head) unit;
// max_ctas > 0 caps the CTA count.  Sliding windows of at most 16 visible pages
// under the automatic plan take one CTA per unit instead (no workspace).
// Workspace: one (m, l, O) slot per (warp, unit) pair a warp can touch, i.e.
// 4 * num_splits + B * Hkv / hpt slots of G * hpt query heads, for the heads per
// unit hpt of the e4m3 cache (at least the bf16 cache's, so the size covers both).
int plan(int B, int Hq, int Hkv, int D, int max_blocks, int window, int req, Plan* out,
         int64_t max_ctas = 0) {
    int maxvis = max_blocks;
    if (window > 0) {
        const int wp = (window + FP8KV_PAGE_SIZE - 1) / FP8KV_PAGE_SIZE + 1;
        if (wp < maxvis) maxvis = wp;
    }
    if (maxvis < 1) maxvis = 1;
    const int64_t units = static_cast<int64_t>(B) * Hkv;
    const int64_t work = units * maxvis;
    const int G1 = Hkv > 0 ? Hq / Hkv : 1;
    const int hpt = decode_heads_per_unit(D, FP8KV_KV_E4M3, G1, Hkv, B);
    int64_t n;
    if (req > 0) {
        n = static_cast<int64_t>(req) * units;
    } else {
        n = static_cast<int64_t>(sm_count()) * decode_ctas_per_sm(D, 0, G1, Hkv, B);
        const int64_t by_work = (work + 15) / 16;
        if (by_work < n) n = by_work;
        // units of at most 16 visible pages (a sliding window): one worker warp
        // per unit, so that every unit ends in its own warp (no partials to merge)
        if (maxvis <= 16) n = (units / hpt + kDecodeWarps - 1) / kDecodeWarps;
    }
    // sliding windows (few pages per unit), automatic plan, one 8-column group:
    // one CTA per unit, whose 4 warps split the unit's pages and combine their
    // partials in shared memory -- no workspace, no split_merge launch
    const int64_t cta_units = units / hpt;
    if (req == 0 && window > 0 && maxvis <= 16 && G1 * hpt <= 8 && cta_units >= 1 &&
        cta_units <= 65535) {
        out->num_splits = static_cast<int>(cta_units);
        out->workspace_bytes = 16;
        out->cta_units = true;
        return FP8KV_OK;
    }
    out->cta_units = false;
    if (n > work) n = work;
    if (n > 1024) n = 1024;
    if (max_ctas > 0 && n > max_ctas) n = max_ctas;
    if (n < 1) n = 1;
    out->num_splits = static_cast<int>(n);
    const int64_t workers = n * kDecodeWarps;      // every warp is a worker
    out->workspace_bytes = static_cast<size_t>(workers + units / hpt) * G1 * hpt *
                           (static_cast<size_t>(D) + 2) * sizeof(float);
    return FP8KV_OK;
}

bool valid_d(int D) { return D == 64 || D == 128 || D == 256; }

}  // namespace

extern "C" {

const char* fp8kv_status_string(int status) {
    switch (status) {
        case FP8KV_OK: return "ok";
        case FP8KV_ERR_INVALID: return "invalid argument";
        case FP8KV_ERR_UNSUPPORTED: return "unsupported shape or mode";
        case FP8KV_ERR_WORKSPACE: return "workspace too small";
        case FP8KV_ERR_CUDA: return "CUDA error";
        case FP8KV_ERR_TIMEOUT: return "device wait timed out";
        case FP8KV_ERR_BAD_INDEX: return "block id or slot outside the cache";
        default: return "unknown status";
    }
}

const char* fp8kv_last_warning(void) { return g_warning.c_str(); }

int fp8kv_resolve_scales(int kv_dtype, int scale_mode, int n, const float* k_loaded,
                         const float* v_loaded, float q_loaded, float prob_loaded,
                         float* k_out, float* v_out, float* q_out, float* prob_out) {
    g_warning.clear();
    if (kv_dtype != FP8KV_KV_E4M3 && kv_dtype != FP8KV_KV_BF16) return FP8KV_ERR_INVALID;
    if (scale_mode < FP8KV_SCALE_PER_TENSOR || scale_mode > FP8KV_SCALE_PER_TOKEN_HEAD)
        return FP8KV_ERR_INVALID;
    if (!q_out || !prob_out || q_loaded != q_loaded || prob_loaded != prob_loaded)
        return FP8KV_ERR_INVALID;
    const bool quantized = kv_dtype == FP8KV_KV_E4M3;
    if (!quantized || scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD) {
        // nothing per-tensor to resolve; q / prob are dropped for these caches
        *q_out = 1.0f;
        *prob_out = 1.0f;
        return FP8KV_OK;
    }
    if (n < 1 || (scale_mode == FP8KV_SCALE_PER_TENSOR && n != 1)) return FP8KV_ERR_INVALID;
    if (!k_loaded || !v_loaded || !k_out || !v_out) return FP8KV_ERR_INVALID;
    for (int i = 0; i < n; ++i) {
        const float k = k_loaded[i], v = v_loaded[i];
        if (k != k || v != v) return FP8KV_ERR_INVALID;
        const bool both_loaded = k > 0.0f && v > 0.0f, none_loaded = k < 0.0f && v < 0.0f;
        if (!both_loaded && !none_loaded && !(k > 0.0f)) return FP8KV_ERR_INVALID;
    }
    for (int i = 0; i < n; ++i) {
        const float k = k_loaded[i], v = v_loaded[i];
        if (k > 0.0f && v > 0.0f) {
            k_out[i] = k;
            v_out[i] = v;
        } else if (k < 0.0f && v < 0.0f) {
            k_out[i] = 1.0f;
            v_out[i] = 1.0f;
        } else {
            k_out[i] = v_out[i] = k > v ? k : v;
        }
    }
    *q_out = q_loaded > 0.0f ? q_loaded : 1.0f;
    *prob_out = prob_loaded > 0.0f ? prob_loaded : 1.0f;
    if (*q_out == 1.0f || *prob_out == 1.0f)
        g_warning = "fp8 attention with uncalibrated q_scale and/or prob_scale of 1.0";
    return FP8KV_OK;
}

int fp8kv_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t T,
                         int Hkv, int D, void* k_cache, void* v_cache, int64_t num_blocks,
                         int kv_dtype, int scale_mode, const float* k_scale, const float* v_scale,
                         float* k_scale_cache, float* v_scale_cache, int32_t* err_flag,
                         void* cuda_stream) {
    g_warning.clear();
    if (T < 0 || Hkv <= 0 || num_blocks < 0) return FP8KV_ERR_INVALID;
    if (!valid_d(D)) return FP8KV_ERR_UNSUPPORTED;
    if (kv_dtype != FP8KV_KV_E4M3 && kv_dtype != FP8KV_KV_BF16) return FP8KV_ERR_INVALID;
    if (kv_dtype == FP8KV_KV_E4M3 && (scale_mode < FP8KV_SCALE_PER_TENSOR ||
                                      scale_mode > FP8KV_SCALE_PER_TOKEN_HEAD))
        return FP8KV_ERR_INVALID;
    if (T == 0) return FP8KV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return FP8KV_ERR_INVALID;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8) ||
        !aligned(k_cache, 16) || !aligned(v_cache, 16))
        return FP8KV_ERR_INVALID;
    if (kv_dtype == FP8KV_KV_E4M3) {
        if (scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD) {
            if (!k_scale_cache || !v_scale_cache || !aligned(k_scale_cache, 4) ||
                !aligned(v_scale_cache, 4))
                return FP8KV_ERR_INVALID;
        } else if (!k_scale || !v_scale) {
            return FP8KV_ERR_INVALID;
        }
    }
    WriteParams p{};
    p.k = static_cast<const __nv_bfloat16*>(k);
    p.v = static_cast<const __nv_bfloat16*>(v);
    p.slot_mapping = slot_mapping;
    p.T = T;
    p.Hkv = Hkv;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.num_blocks = num_blocks;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_scale_cache = k_scale_cache;
    p.v_scale_cache = v_scale_cache;
    p.err = err_flag;
    cudaError_t e = launch_kv_cache_write(p, D, kv_dtype, scale_mode,
                                          static_cast<cudaStream_t>(cuda_stream), sm_count());
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

int fp8kv_decode_plan(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int window,
                      int num_splits, int* num_splits_out, size_t* workspace_bytes_out) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_blocks_per_seq < 0 || window < 0 ||
        num_splits < 0)
        return FP8KV_ERR_INVALID;
    if (!valid_d(D)) return FP8KV_ERR_UNSUPPORTED;
    Plan pl;
    plan(B, Hq, Hkv, D, max_blocks_per_seq, window, num_splits, &pl);
    if (num_splits_out) *num_splits_out = pl.num_splits;
    if (workspace_bytes_out) *workspace_bytes_out = pl.workspace_bytes;
    return FP8KV_OK;
}

}  // extern "C"

namespace {

// Shared body of fp8kv_paged_decode_attn and fp8kv_decode_step (k_new / v_new
// non-null: the split kernel stores the new tokens itself).
int paged_decode(const void* q, const void* k_new, const void* v_new, const void* k_cache,
                 const void* v_cache, int kv_dtype, int scale_mode, const float* k_scale,
                 const float* v_scale, const float* k_scale_cache, const float* v_scale_cache,
                 const int32_t* block_table, int max_blocks_per_seq, const int32_t* context_lens,
                 int B, int Hq, int Hkv, int D, int64_t num_blocks, float softmax_scale,
                 int window, int num_splits, void* workspace, size_t workspace_bytes, void* out,
                 int out_dtype, unsigned flags, int32_t* err_flag, void* cuda_stream,
                 int64_t max_ctas = 0) {
    const bool fused = k_new != nullptr || v_new != nullptr;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || window < 0 || num_splits < 0 ||
        max_blocks_per_seq < 0 || num_blocks < 0 ||
        (flags & ~(FP8KV_DECODE_EARLY_SETUP | FP8KV_DECODE_EARLY_PAGES)) != 0)
        return FP8KV_ERR_INVALID;
    if (!valid_d(D)) return FP8KV_ERR_UNSUPPORTED;
    if (Hq / Hkv > 16) return FP8KV_ERR_UNSUPPORTED;
    if (kv_dtype != FP8KV_KV_E4M3 && kv_dtype != FP8KV_KV_BF16) return FP8KV_ERR_INVALID;
    if (kv_dtype == FP8KV_KV_E4M3 && (scale_mode < FP8KV_SCALE_PER_TENSOR ||
                                      scale_mode > FP8KV_SCALE_PER_TOKEN_HEAD))
        return FP8KV_ERR_INVALID;
    if (out_dtype != FP8KV_OUT_F32 && out_dtype != FP8KV_OUT_BF16) return FP8KV_ERR_INVALID;
    if (!(softmax_scale == softmax_scale)) return FP8KV_ERR_INVALID;   // NaN
    if (B == 0) return FP8KV_OK;
    if (B > 65535 || Hkv > 65535 || max_blocks_per_seq < 1 || num_blocks < 1)
        return FP8KV_ERR_INVALID;
    if (num_blocks * static_cast<int64_t>(Hkv) >= (int64_t{1} << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks_per_seq) * FP8KV_PAGE_SIZE >= (int64_t{1} << 31))
        return FP8KV_ERR_UNSUPPORTED;
    // the partition arithmetic multiplies tile counts (<= B * Hkv * pages) by
    // worker counts (<= 4096) in 64 bits
    if (static_cast<int64_t>(B) * Hkv * max_blocks_per_seq >= (int64_t{1} << 50))
        return FP8KV_ERR_UNSUPPORTED;
    // one sequence's (KV head, page) tiles are indexed in 32 bits
    if (static_cast<int64_t>(max_blocks_per_seq) * Hkv >= (int64_t{1} << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out)
        return FP8KV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_table, 4) || !aligned(context_lens, 4) || !aligned(out, 4))
        return FP8KV_ERR_INVALID;
    if (fused && (!k_new || !v_new || !aligned(k_new, 16) || !aligned(v_new, 16)))
        return FP8KV_ERR_INVALID;
    if (kv_dtype == FP8KV_KV_E4M3) {
        if (scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD) {
            if (!k_scale_cache || !v_scale_cache || !aligned(k_scale_cache, 16) ||
                !aligned(v_scale_cache, 16))
                return FP8KV_ERR_INVALID;
        } else if (!k_scale || !v_scale) {
            return FP8KV_ERR_INVALID;
        }
    }
    Plan pl;
    plan(B, Hq, Hkv, D, max_blocks_per_seq, window, num_splits, &pl, max_ctas);
    if (!workspace || workspace_bytes < pl.workspace_bytes) return FP8KV_ERR_WORKSPACE;
    if (!aligned(workspace, 16)) return FP8KV_ERR_INVALID;
    const int row_bytes = D * (kv_dtype == FP8KV_KV_BF16 ? 2 : 1);
    const int64_t nbh = num_blocks * Hkv;
    const int hpt = decode_heads_per_unit(D, kv_dtype, Hq / Hkv, Hkv, B);
    CUtensorMap kmap, vmap;
    if (!make_kv_map(k_cache, row_bytes, nbh, &kmap, false, hpt) ||
        !make_kv_map(v_cache, row_bytes, nbh, &vmap, false, hpt))
        return FP8KV_ERR_CUDA;

    DecodeParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_scale_cache = k_scale_cache;
    p.v_scale_cache = v_scale_cache;
    p.block_table = block_table;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = Hq / Hkv;
    p.hpt = hpt;
    p.Hu = Hkv / hpt;
    p.Gu = p.G * hpt;
    p.num_blocks = num_blocks;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.window = window;
    p.num_splits = pl.num_splits;
    p.cta_units = pl.cta_units ? 1 : 0;
    if (p.cta_units) p.num_splits = B * p.Hu;   // one CTA per unit of this cache's kind
    {
        float* ws = static_cast<float*>(workspace);
        const size_t rows = (static_cast<size_t>(pl.num_splits) * kDecodeWarps +
                             static_cast<size_t>(B) * p.Hu) * p.Gu;
        p.ws_o = ws;
        p.ws_m = ws + rows * D;
        p.ws_l = p.ws_m + rows;
    }
    p.out = out;
    p.out_bf16 = out_dtype == FP8KV_OUT_BF16;
    p.scale_mode = kv_dtype == FP8KV_KV_E4M3 ? scale_mode : FP8KV_SCALE_PER_TENSOR;
    p.flags = flags;
    p.err = err_flag;
    // the kernels stream pages from these (and the fused step also stores into them)
    p.k_cache = static_cast<uint8_t*>(const_cast<void*>(k_cache));
    p.v_cache = static_cast<uint8_t*>(const_cast<void*>(v_cache));
    if (fused) {
        p.k_new = static_cast<const __nv_bfloat16*>(k_new);
        p.v_new = static_cast<const __nv_bfloat16*>(v_new);
    }
    cudaError_t e = launch_paged_decode(p, kmap, vmap, D, kv_dtype, fused,
                                        static_cast<cudaStream_t>(cuda_stream));
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

}  // namespace

namespace fp8kv {

int paged_decode_attn_fitting(const void* q, const void* k_cache, const void* v_cache,
                              int kv_dtype, int scale_mode, const float* k_scale,
                              const float* v_scale, const float* k_scale_cache,
                              const float* v_scale_cache, const int32_t* block_table,
                              int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                              int Hkv, int D, int64_t num_blocks, float softmax_scale, int window,
                              int num_splits, void* scratch, size_t scratch_bytes, void* out,
                              int out_dtype, int32_t* err_flag, void* cuda_stream) {
    g_warning.clear();
    int64_t max_ctas = 0;
    Plan cta;                                    // a short sliding window needs no scratch
    const bool cta_units = Hkv > 0 && Hq > 0 && Hq % Hkv == 0 && B > 0 && valid_d(D) &&
                           plan(B, Hq, Hkv, D, max_blocks_per_seq, window, num_splits, &cta) ==
                               FP8KV_OK &&
                           cta.cta_units;
    if (num_splits == 0 && !cta_units && Hkv > 0 && Hq > 0 && Hq % Hkv == 0 && B > 0 &&
        valid_d(D)) {
        // slots that fit, less the one per unit, over the 4 worker warps of a CTA
        // (a worker's slot holds hpt KV heads' query heads, as the planner sizes it)
        const int hpt = decode_heads_per_unit(D, FP8KV_KV_E4M3, Hq / Hkv, Hkv, B);
        const int64_t slot_bytes = static_cast<int64_t>(Hq / Hkv) * (D + 2) * sizeof(float);
        const int64_t spare = static_cast<int64_t>(scratch_bytes) / slot_bytes -
                              static_cast<int64_t>(B) * Hkv;
        max_ctas = spare / (static_cast<int64_t>(kDecodeWarps) * hpt);
        if (max_ctas < 1) return FP8KV_ERR_WORKSPACE;
    }
    return paged_decode(q, nullptr, nullptr, k_cache, v_cache, kv_dtype, scale_mode, k_scale,
                        v_scale, k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
                        context_lens, B, Hq, Hkv, D, num_blocks, softmax_scale, window,
                        num_splits, scratch, scratch_bytes, out, out_dtype, 0u, err_flag,
                        cuda_stream, max_ctas);
}

}  // namespace fp8kv

namespace {

// Persistent prefill workspace: a counter per CTA (padded to 256 bytes), then
// two partial slots per CTA of [128][D + 2] floats.
size_t prefill_ws_count_bytes(int n_ctas) {
    return (static_cast<size_t>(n_ctas) * 4 + 255) / 256 * 256;
}

size_t prefill_ws_bytes(int D, int n_ctas) {
    return prefill_ws_count_bytes(n_ctas) +
           static_cast<size_t>(2) * n_ctas * 128 * (static_cast<size_t>(D) + 2) * 4;
}

}  // namespace

extern "C" {

int fp8kv_paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                            int kv_dtype, int scale_mode, const float* k_scale,
                            const float* v_scale, const float* k_scale_cache,
                            const float* v_scale_cache, const int32_t* block_table,
                            int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                            int Hkv, int D, int64_t num_blocks, float softmax_scale, int window,
                            int num_splits, void* workspace, size_t workspace_bytes, void* out,
                            int out_dtype, unsigned flags, int32_t* err_flag, void* cuda_stream) {
    g_warning.clear();
    return paged_decode(q, nullptr, nullptr, k_cache, v_cache, kv_dtype, scale_mode, k_scale,
                        v_scale, k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
                        context_lens, B, Hq, Hkv, D, num_blocks, softmax_scale, window,
                        num_splits, workspace, workspace_bytes, out, out_dtype, flags, err_flag,
                        cuda_stream);
}

int fp8kv_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, int kv_dtype, int scale_mode, const float* k_scale,
                      const float* v_scale, float* k_scale_cache, float* v_scale_cache,
                      const int32_t* block_table, int max_blocks_per_seq,
                      const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                      int64_t num_blocks, float softmax_scale, int window, int num_splits,
                      void* workspace, size_t workspace_bytes, void* out, int out_dtype,
                      unsigned flags, int32_t* err_flag, void* cuda_stream) {
    g_warning.clear();
    if (!k_new || !v_new) return FP8KV_ERR_INVALID;
    return paged_decode(q, k_new, v_new, k_cache, v_cache, kv_dtype, scale_mode, k_scale,
                        v_scale, k_scale_cache, v_scale_cache, block_table, max_blocks_per_seq,
                        context_lens, B, Hq, Hkv, D, num_blocks, softmax_scale, window,
                        num_splits, workspace, workspace_bytes, out, out_dtype, flags, err_flag,
                        cuda_stream);
}

int fp8kv_prefill_workspace_bytes(int D, size_t* bytes) {
    if (!bytes) return FP8KV_ERR_INVALID;
    if (!valid_d(D)) return FP8KV_ERR_UNSUPPORTED;
    const int n = sm_count();
    if (n <= 0) return FP8KV_ERR_CUDA;
    *bytes = prefill_ws_bytes(D, n);
    return FP8KV_OK;
}

int fp8kv_prefill_attn(const void* q, const int32_t* cu_seqlens_q, int max_seqlen_q,
                       const void* k_cache, const void* v_cache, int kv_dtype, int scale_mode,
                       const float* k_scale, const float* v_scale, const float* k_scale_cache,
                       const float* v_scale_cache, float q_scale,
                       float prob_scale, const int32_t* block_table, int max_blocks_per_seq,
                       const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                       int64_t num_blocks, float softmax_scale, int flags, void* out,
                       int out_dtype, int32_t* err_flag, void* cuda_stream) {
    return fp8kv_prefill_attn_ws(q, cu_seqlens_q, max_seqlen_q, k_cache, v_cache, kv_dtype,
                                 scale_mode, k_scale, v_scale, k_scale_cache, v_scale_cache,
                                 q_scale, prob_scale, block_table, max_blocks_per_seq,
                                 context_lens, B, Hq, Hkv, D, num_blocks, softmax_scale, flags,
                                 nullptr, 0, out, out_dtype, err_flag, cuda_stream);
}

int fp8kv_prefill_attn_ws(const void* q, const int32_t* cu_seqlens_q, int max_seqlen_q,
                          const void* k_cache, const void* v_cache, int kv_dtype, int scale_mode,
                          const float* k_scale, const float* v_scale,
                          const float* k_scale_cache, const float* v_scale_cache, float q_scale,
                          float prob_scale, const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                          int64_t num_blocks, float softmax_scale, int flags, void* workspace,
                          size_t workspace_bytes, void* out, int out_dtype, int32_t* err_flag,
                          void* cuda_stream) {
    g_warning.clear();
    constexpr int kKnown =
        FP8KV_PREFILL_TWO_LEVEL | FP8KV_PREFILL_SPLIT_ALWAYS | FP8KV_PREFILL_SPLIT_NEVER;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || max_seqlen_q < 0 ||
        max_blocks_per_seq < 0 || num_blocks < 0 || (flags & ~kKnown) != 0 ||
        ((flags & FP8KV_PREFILL_SPLIT_ALWAYS) && (flags & FP8KV_PREFILL_SPLIT_NEVER)))
        return FP8KV_ERR_INVALID;
    const int two_level = flags & FP8KV_PREFILL_TWO_LEVEL;
    if (kv_dtype != FP8KV_KV_E4M3 && kv_dtype != FP8KV_KV_BF16) return FP8KV_ERR_INVALID;
    if (scale_mode < FP8KV_SCALE_PER_TENSOR || scale_mode > FP8KV_SCALE_PER_TOKEN_HEAD)
        return FP8KV_ERR_INVALID;
    if (out_dtype != FP8KV_OUT_F32 && out_dtype != FP8KV_OUT_BF16) return FP8KV_ERR_INVALID;
    if (!(q_scale > 0.f) || !(prob_scale > 0.f) || !(q_scale < 3.0e38f) ||
        !(prob_scale < 3.0e38f) || !(softmax_scale == softmax_scale))
        return FP8KV_ERR_INVALID;
    const int G = Hq / Hkv;
    if (!valid_d(D) || G > 128 || (128 % G) != 0) return FP8KV_ERR_UNSUPPORTED;
    if (B == 0 || max_seqlen_q == 0) return FP8KV_OK;
    if (B > 65535 || Hkv > 65535 || max_blocks_per_seq < 1 || num_blocks < 1)
        return FP8KV_ERR_INVALID;
    if (num_blocks * static_cast<int64_t>(Hkv) >= (int64_t{1} << 31) ||
        static_cast<int64_t>(max_blocks_per_seq) * FP8KV_PAGE_SIZE >= (int64_t{1} << 31))
        return FP8KV_ERR_UNSUPPORTED;
    if (!q || !cu_seqlens_q || !k_cache || !v_cache || !block_table || !context_lens || !out)
        return FP8KV_ERR_INVALID;
    const bool per_token = kv_dtype == FP8KV_KV_E4M3 && scale_mode == FP8KV_SCALE_PER_TOKEN_HEAD;
    if (kv_dtype == FP8KV_KV_E4M3 && !per_token && (!k_scale || !v_scale)) return FP8KV_ERR_INVALID;
    if (per_token && (!k_scale_cache || !v_scale_cache || !aligned(k_scale_cache, 16) ||
                      !aligned(v_scale_cache, 16)))
        return FP8KV_ERR_INVALID;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16))
        return FP8KV_ERR_INVALID;
    CUtensorMap kmap, vmap;
    const int64_t nbh = num_blocks * Hkv;
    const int row_bytes = D * (kv_dtype == FP8KV_KV_BF16 ? 2 : 1);
    if (!make_kv_map(k_cache, row_bytes, nbh, &kmap, true) ||
        !make_kv_map(v_cache, row_bytes, nbh, &vmap, true))
        return FP8KV_ERR_CUDA;
    PrefillParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.cu_seqlens_q = cu_seqlens_q;
    p.block_table = block_table;
    p.max_blocks_per_seq = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.B = B;
    p.Hq = Hq;
    p.Hkv = Hkv;
    p.G = G;
    p.num_blocks = num_blocks;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.q_scale = q_scale;
    p.prob_scale = prob_scale;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.k_scale_cache = k_scale_cache;
    p.v_scale_cache = v_scale_cache;
    p.scale_mode = kv_dtype == FP8KV_KV_E4M3 ? scale_mode : FP8KV_SCALE_PER_TENSOR;
    p.split = flags & (FP8KV_PREFILL_SPLIT_ALWAYS | FP8KV_PREFILL_SPLIT_NEVER);
    p.out = out;
    p.out_bf16 = out_dtype == FP8KV_OUT_BF16;
    p.err = err_flag;
    const int tpt = 128 / G;
    int grid_x = (max_seqlen_q + tpt - 1) / tpt;
    // more query tiles than SMs and a workspace: a persistent CTA per SM with
    // the key tiles split evenly (no partly filled last wave).  Each CTA plans
    // its share by walking the sequences one after another (~1 us each), so
    // batches of more than kBalancedMaxSeqs sequences keep one CTA per tile.
    constexpr int kBalancedMaxSeqs = 8;
    const int n_sm = sm_count();
    if (workspace != nullptr && n_sm > 0 && B <= kBalancedMaxSeqs &&
        static_cast<int64_t>(grid_x) * Hkv * B > n_sm) {
        if (workspace_bytes < prefill_ws_bytes(D, n_sm)) return FP8KV_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return FP8KV_ERR_INVALID;
        p.ws_count = static_cast<int32_t*>(workspace);
        p.ws_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                             prefill_ws_count_bytes(n_sm));
        grid_x = n_sm;
    }
    cudaError_t e = launch_prefill(p, kmap, vmap, D, kv_dtype, two_level, grid_x,
                                   static_cast<cudaStream_t>(cuda_stream));
    if (e != cudaSuccess) return FP8KV_ERR_CUDA;
    if (kv_dtype == FP8KV_KV_E4M3 && (q_scale == 1.0f || prob_scale == 1.0f))
        g_warning = "fp8 attention with uncalibrated q_scale and/or prob_scale of 1.0";
    return FP8KV_OK;
}

int fp8kv_quantize_e4m3(const float* x, float scale, uint8_t* out, int64_t n,
                        void* cuda_stream) {
    g_warning.clear();
    if (n < 0) return FP8KV_ERR_INVALID;
    if (n == 0) return FP8KV_OK;
    if (!x || !out) return FP8KV_ERR_INVALID;
    cudaError_t e =
        launch_quantize_e4m3(x, scale, out, n, static_cast<cudaStream_t>(cuda_stream), sm_count());
    return e == cudaSuccess ? FP8KV_OK : FP8KV_ERR_CUDA;
}

}  // extern "C"
