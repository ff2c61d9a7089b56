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
    int cta_units;               // 1: CTA u takes unit u whole (B * Hu CTAs), no split_merge
    int hpt;                     // KV heads per unit (decode_heads_per_unit)
    int Hu;                      // units per sequence, Hkv / hpt
    int Gu;                      // query heads per unit, G * hpt
    float* ws_m;                 // [4*num_splits + B*Hu][Gu] running max (log2 units)
    float* ws_l;                 // [4*num_splits + B*Hu][Gu] softmax denominator
    float* ws_o;                 // [4*num_splits + B*Hu][Gu][D] unnormalised output
    void* out;                   // [B][Hq][D]
    int out_bf16;
    int scale_mode;
    unsigned flags;              // FP8KV_DECODE_EARLY_* (what may run before the wait)
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
    int split;                     // 0 automatic, else FP8KV_PREFILL_SPLIT_ALWAYS / _NEVER
    void* out;                     // [Tq][Hq][D]
    int out_bf16;
    int32_t* err;
    // balanced split over a persistent grid (null: one CTA per query tile): the
    // partial of each cut piece, [2 * CTAs][128][D + 2] floats, and a counter
    // per CTA (zero between calls)
    float* ws_part;
    int32_t* ws_count;
};

cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& kmap,
                           const CUtensorMap& vmap, int D, int kv_dtype, int two_level,
                           int grid_x, cudaStream_t stream);

// Identifier of the calling thread's current CUDA context, unique over the
// process's lifetime (a context recreated after cudaDeviceReset gets a new one);
// 0 when there is no current context or the driver cannot say.
unsigned long long current_context_id();

// cudaFuncSetAttribute(MaxDynamicSharedMemorySize) for `func` when the current
// context has not had it yet: done[dev] keeps the id of the context it was set in.
cudaError_t opt_in_smem(const void* func, int bytes, unsigned long long (&done)[64]);

// fp8kv_paged_decode_attn with the split partials in `scratch` (scratch_bytes
// long).  num_splits 0: the automatic plan, with the CTA count lowered until
// its partials fit (FP8KV_ERR_WORKSPACE if not even one CTA fits, i.e. the
// B * Hq * (D + 2) * 4 bytes of one slot per unit alone exceed it); num_splits
// > 0: that plan, FP8KV_ERR_WORKSPACE if it does not fit.
int paged_decode_attn_fitting(const void* q, const void* k_cache, const void* v_cache,
                              int kv_dtype, int scale_mode, const float* k_scale,
                              const float* v_scale, const float* k_scale_cache,
                              const float* v_scale_cache, const int32_t* block_table,
                              int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                              int Hkv, int D, int64_t num_blocks, float softmax_scale, int window,
                              int num_splits, void* scratch, size_t scratch_bytes, void* out,
                              int out_dtype, int32_t* err_flag, void* cuda_stream);

// Decode kernel geometry used by the planner and the tensor maps.
constexpr int kDecodeWarps = 4;
// KV heads per decode unit: 2 packs adjacent KV heads h, h + 1 (G = 2 or 4
// query heads each, an even Hkv, tiles of at most 2 KiB, at least 32 (sequence,
// KV head) pairs in the batch) into one unit whose tiles are copied together
// and share the 8 MMA columns; else 1.
int decode_heads_per_unit(int D, int kv_dtype, int G, int Hkv, int B);
// CTAs of the decode kernel resident per SM (shared memory and the register
// budget of its launch bounds) for head dim D, G query heads per KV head, Hkv
// KV heads and B sequences.
int decode_ctas_per_sm(int D, int kv_dtype, int G, int Hkv, int B);

}  // namespace fp8kv
