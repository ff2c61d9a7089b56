// decode_noalloc.cu -- paged decode attention for callers that cannot allocate
// device memory.
//
// fp8kv_paged_decode_attn needs a caller-provided workspace for its split
// partials.  Some callers cannot provide one: a C host program or plugin that
// receives only the tensors it reads and writes from the framework that owns
// the GPU's memory pool has no allocator handle, and a serving loop cannot
// afford cudaMalloc / cudaFree there because they synchronize the device and
// stall every other stream.  This entry point keeps the split partials in a
// fixed-size array compiled into the library instead, so it allocates nothing.
//
// Costs and rules of that choice:
//   * every GPU that loads this library holds the array
//     (FP8KV_NOALLOC_DECODE_SCRATCH_BYTES) until the process exits;
//   * the array is shared by every call on a device, so calls whose kernels
//     overlap on the GPU (different streams, or different host threads) race;
//     serialize them, e.g. on one stream;
//   * the first call on each device looks up the array's device address (with
//     that device current), and so does the first call after the device's
//     context was recreated (cudaDeviceReset); make those calls outside stream
//     capture;
//   * with num_splits 0 the automatic plan is lowered to the largest CTA count
//     whose partials fit the array; a call that cannot fit even one CTA (the
//     B * Hq * (D + 2) * 4 bytes of one slot per unit alone exceed the array),
//     or whose explicit num_splits plan does not fit, is rejected with
//     FP8KV_ERR_WORKSPACE and launches nothing: the allocating entry point is
//     the remedy.
// The partials need no initial value: every split the merge reads is written by
// the same call first, so nothing is cleared between calls.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/fp8kv.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = FP8KV_NOALLOC_DECODE_SCRATCH_BYTES;

// The split partials' home on every device (fp32, 256-byte aligned).
static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

// Device address of g_decode_scratch in the current context, looked up once per
// device and again whenever that device's context is a new one (after
// cudaDeviceReset the old address is gone).  In host code the symbol is only a
// host-side stand-in, never a device address, so kernels always receive the
// looked-up pointer.
int scratch_on_current_device(void** out) {
    struct Entry {
        unsigned long long ctx;
        void* addr;
    };
    static std::mutex mu;
    static Entry cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return FP8KV_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long ctx = fp8kv::current_context_id();
    if (cache[dev].addr == nullptr || ctx == 0 || cache[dev].ctx != ctx) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return FP8KV_ERR_CUDA;
        }
        // the lookup makes the context current if it was not yet
        cache[dev] = Entry{fp8kv::current_context_id(), p};
    }
    *out = cache[dev].addr;
    return FP8KV_OK;
}

}  // namespace

extern "C" {

int fp8kv_paged_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    int kv_dtype, int scale_mode, const float* k_scale,
                                    const float* v_scale, const float* k_scale_cache,
                                    const float* v_scale_cache, const int32_t* block_table,
                                    int max_blocks_per_seq, const int32_t* context_lens, int B,
                                    int Hq, int Hkv, int D, int64_t num_blocks,
                                    float softmax_scale, int window, int num_splits, void* out,
                                    int out_dtype, int32_t* err_flag, void* cuda_stream) {
    int splits = 0;
    size_t need = 0;
    int st = fp8kv_decode_plan(B, Hq, Hkv, D, max_blocks_per_seq, window, num_splits, &splits,
                               &need);
    if (st != FP8KV_OK) return st;
    if (num_splits > 0 && need > kScratchBytes) return FP8KV_ERR_WORKSPACE;
    void* scratch = nullptr;
    if (B > 0) {
        st = scratch_on_current_device(&scratch);
        if (st != FP8KV_OK) return st;
    }
    return fp8kv::paged_decode_attn_fitting(
        q, k_cache, v_cache, kv_dtype, scale_mode, k_scale, v_scale, k_scale_cache,
        v_scale_cache, block_table, max_blocks_per_seq, context_lens, B, Hq, Hkv, D, num_blocks,
        softmax_scale, window, num_splits, scratch, kScratchBytes, out, out_dtype, err_flag,
        cuda_stream);
}

}  // extern "C"
