// internal.h -- kernel parameter blocks and launchers shared between the
// kernels' translation units and the C-ABI layer (api.cu).  Not installed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8kv.h"

namespace fp8kv {

struct WriteParams {
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const int64_t* slot_mapping;
    int64_t T;
    int Hkv;
    void* k_cache;
    void* v_cache;
    int64_t num_blocks;
    const float* k_scale;
    const float* v_scale;
    float* k_scale_cache;
    float* v_scale_cache;
    int32_t* err;
};

cudaError_t launch_kv_cache_write(const WriteParams& p, int D, int kv_dtype, int mode,
                                  cudaStream_t stream, int num_sms);
cudaError_t launch_quantize_e4m3(const float* x, float scale, uint8_t* out, int64_t n,
                                 cudaStream_t stream, int num_sms);

// Split-K decode over a balanced partition: the (seq, KV head, page) tiles of
// the launch (pages [p_lo, p_hi) hold positions [lo, ctx)) are split evenly over
// num_splits CTAs; a CTA's share may span several (seq, KV head) units.
struct DecodeParams {
    const __nv_bfloat16* q;
    const float* k_scale;        // per tensor / per head (fp8 only)
    const float* v_scale;
    const float* k_scale_cache;  // per token-head (fp8 only)
    const float* v_scale_cache;
    const int32_t* block_table;
    int max_blocks_per_seq;
    const int32_t* context_lens;
    int B, Hq, Hkv, G;
    int64_t num_blocks;
    float scale_log2;            // softmax_scale * log2(e)
    int window;
    int num_splits;              // CTAs of the decode grid
    float* ws_m;                 // [4*num_splits + B*Hkv][G] running max (log2 units)
    float* ws_l;                 // [4*num_splits + B*Hkv][G] softmax denominator
    float* ws_o;                 // [4*num_splits + B*Hkv][G][D] unnormalised output
    void* out;                   // [B][Hq][D]
    int out_bf16;
    int scale_mode;
    int32_t* err;
    // fused decode step only (null otherwise): the new token of every sequence,
    // [B][Hkv][D] bf16, stored at position ctx - 1 by the kernel itself
    const __nv_bfloat16* k_new;
    const __nv_bfloat16* v_new;
    uint8_t* k_cache;
    uint8_t* v_cache;
};

// Launches the split kernel and the merge kernel (fused: the split kernel also
// stores k_new / v_new).
cudaError_t launch_paged_decode(const DecodeParams& p, const CUtensorMap& kmap,
                                const CUtensorMap& vmap, int D, int kv_dtype, bool fused,
                                cudaStream_t stream);

// Chunked causal prefill on the tcgen05 FP8 tensor cores.  CTA (x, h, b) takes
// query tokens [x*128/G, (x+1)*128/G) of sequence b with the G query heads of
// KV head h (128 MMA rows).
struct PrefillParams {
    const __nv_bfloat16* q;        // [Tq][Hq][D]
    const int32_t* cu_seqlens_q;   // [B+1]
    const int32_t* block_table;
    int max_blocks_per_seq;
    const int32_t* context_lens;   // keys of each sequence, the chunk included
    int B, Hq, Hkv, G;
    int64_t num_blocks;
    float scale_log2;              // softmax_scale * log2(e)
    float q_scale, prob_scale;
    const float* k_scale;          // [1] or [Hkv]
    const float* v_scale;
    const float* k_scale_cache;    // per token-head: [num_blocks][Hkv][16]
    const float* v_scale_cache;
    int scale_mode;
    void* out;                     // [Tq][Hq][D]
    int out_bf16;
    int32_t* err;
};

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int D, int kv_dtype, int two_level,
                           int grid_x, cudaStream_t stream);

// Decode kernel geometry used by the planner and the tensor maps.
constexpr int kDecodeWarps = 4;
int decode_ctas_per_sm(int D, int kv_dtype);

}  // namespace fp8kv
