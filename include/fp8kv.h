/*
 * fp8kv.h -- C ABI of libfp8kv: an FP8 (e4m3) paged KV cache and attention
 * directly over it, hand-written for GB300 (sm_103a).
 *
 * What the library computes follows these pages (cited by title and section):
 *   [KO]  "vLLM FP8 KV-Cache 및 Attention 양자화 업데이트" (agentlenshq.com):
 *         storing K/V as FP8 e4m3 halves the KV cache and attention then runs
 *         over FP8 data (opening paragraph); per-KV-head scale arrays
 *         ("커널 및 퓨전 최적화"); uncalibrated scale 1.0 ("정확도 및 검증");
 *         sliding-window layers kept in BF16 ("하이브리드 Attention 및 레이어
 *         스킵"); two-level FP32 accumulation for long contractions
 *         ("정확도를 위한 2단계 누적"), not needed on Blackwell ("아키텍처별 결과").
 *   [KVQ] "[vLLM] KV Cache Quantization: KV 캐시 FP8/INT8 양자화"
 *         (blog.secrett2633.cloud): per-tensor K/V scale from a checkpoint or
 *         1.0, or per-token-head scales that the kernel computes when it stores
 *         the cache ("Per-Token-Head vs Per-Tensor 양자화"); q and prob scales
 *         for FP8 attention and the uncalibrated-scale warning ("Q/Prob 스케일과
 *         FP8 Attention").
 *   [PR]  "vLLM Qwen3.8-Flash-Next: QSA Indexer 캐시를 위한 FP8 지원" (same blog):
 *         torch.float8_e4m3fn storage and paged caches with a shuffled page
 *         table ("코드 분석").
 *
 * Conventions for every entry point
 *   - Ownership: the caller owns every buffer.  Array arguments are DEVICE
 *     pointers on the current CUDA device (from cudaMalloc or a framework's
 *     allocator); the library allocates nothing and keeps no pointer after the
 *     call returns.  Scalars are host values.
 *   - Streams: work is enqueued on `cuda_stream` (a cudaStream_t; NULL is the
 *     legacy default stream) and nothing synchronizes.
 *   - Errors: a negative fp8kv_status is returned, never an exception.  Host
 *     checks run before any launch, so an invalid call launches nothing.  Errors
 *     found by a kernel (a block id or slot outside the cache, a timed-out wait)
 *     are written to `*err_flag` (device int32, first error wins; NULL = do not
 *     report) and the offending page/row is skipped; read it after a sync.
 *   - Cache layout (page size 16): k_cache / v_cache are
 *     [num_blocks][Hkv][16][D] of e4m3 bytes (kv_dtype E4M3) or bf16
 *     (kv_dtype BF16); one (block, head) tile is 16*D contiguous elements.
 *     Per-token-head scales live beside the pages in fp32
 *     k_scale_cache / v_scale_cache [num_blocks][Hkv][16], indexed by the same
 *     block id and in-page offset.
 *   - Supported shapes: D in {64, 128, 256}; Hq % Hkv == 0; decode attention
 *     takes Hq / Hkv <= 16, prefill Hq / Hkv dividing 128; base addresses
 *     16-byte aligned.
 */
#ifndef FP8KV_H
#define FP8KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8KV_PAGE_SIZE 16

typedef enum {
    FP8KV_OK = 0,
    FP8KV_ERR_INVALID = -1,     /* a pointer, size or enum value is invalid */
    FP8KV_ERR_UNSUPPORTED = -2, /* valid but not implemented (shape, mode) */
    FP8KV_ERR_WORKSPACE = -3,   /* workspace too small */
    FP8KV_ERR_CUDA = -4,        /* a CUDA runtime call or launch failed */
    FP8KV_ERR_TIMEOUT = -5,     /* device: a bounded wait expired (err_flag) */
    FP8KV_ERR_BAD_INDEX = -6    /* device: block id / slot outside the cache (err_flag) */
} fp8kv_status;

typedef enum { FP8KV_KV_E4M3 = 0, FP8KV_KV_BF16 = 1 } fp8kv_kv_dtype;

typedef enum {
    FP8KV_SCALE_PER_TENSOR = 0,     /* k_scale[0], v_scale[0] ([KVQ] per-tensor; 1.0 uncalibrated) */
    FP8KV_SCALE_PER_HEAD = 1,       /* k_scale[h], v_scale[h] ([KO] per-KV-head scale arrays) */
    FP8KV_SCALE_PER_TOKEN_HEAD = 2  /* computed at write time ([KVQ] per-token-head) */
} fp8kv_scale_mode;

typedef enum { FP8KV_OUT_F32 = 0, FP8KV_OUT_BF16 = 1 } fp8kv_out_dtype;

/*
 * fp8kv_kv_cache_write -- store T new tokens of K and V into the paged cache.
 * [KO] opening paragraph (e4m3 storage), [KVQ] "Per-Token-Head vs Per-Tensor
 * 양자화" (scale modes).
 *
 *   k, v          bf16 [T][Hkv][D], row-major.  k, v and slot_mapping may be
 *                 device memory or pinned host memory (read by the kernel over
 *                 the host link; one pass, so no staging copy is needed).
 *   slot_mapping  int64 [T]: slot = block * 16 + offset; a negative slot skips
 *                 the token (padding).  A slot at or past num_blocks * 16 sets
 *                 FP8KV_ERR_BAD_INDEX in err_flag and is skipped.
 *   kv_dtype      E4M3: codes e4m3_rn_satfinite(fp32(x / scale)); BF16: a copy.
 *   scale_mode    (E4M3 only) PER_TENSOR: scale = k_scale[0] / v_scale[0];
 *                 PER_HEAD: k_scale[h] / v_scale[h]; PER_TOKEN_HEAD: scale =
 *                 fp32(max_d |x_d| / 448) per (token, head), written to
 *                 k_scale_cache / v_scale_cache.  A zero scale writes code 0.
 *   k_scale, v_scale  fp32 device arrays of 1 or Hkv entries (ignored for
 *                 PER_TOKEN_HEAD and BF16).
 * Codes are those of the IEEE fp32 quotient (a multiply by fp32(1/scale) is used
 * only where it provably gives the same codes) rounded to nearest even, so codes
 * and scales are bit-identical to a plain CPU restatement.  Bulk writes
 * (T * Hkv >= 8192 rows, k and v in device memory) stream K and V through
 * shared memory with bulk copies; other writes use plain loads.
 */
int fp8kv_kv_cache_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t T,
                         int Hkv, int D, void* k_cache, void* v_cache, int64_t num_blocks,
                         int kv_dtype, int scale_mode, const float* k_scale, const float* v_scale,
                         float* k_scale_cache, float* v_scale_cache, int32_t* err_flag,
                         void* cuda_stream);

/*
 * fp8kv_decode_plan -- how fp8kv_paged_decode_attn splits the context and the
 * workspace it needs (pure host function, no CUDA call besides reading the
 * current device's SM count).
 *
 *   max_blocks_per_seq  columns of block_table (upper bound on pages per sequence)
 *   window              0 = full attention, else the last `window` keys
 *   num_splits          0 = choose automatically, else the requested split count
 *   *num_splits_out     the split count the kernel will use (CTAs of its grid)
 *   *workspace_bytes_out  bytes of workspace needed (split partials)
 * Automatic plans: one wave of CTAs over all (sequence, KV head, page) tiles,
 * with partials merged by a second kernel; a sliding window of at most 16
 * visible pages per sequence instead takes one CTA per (sequence, KV head)
 * unit that combines its warps' partials itself (workspace_bytes_out 16).  With
 * 2 or 4 query heads per KV head, an even Hkv, rows of at most 128 bytes and
 * B * Hkv >= 32, a unit is two adjacent KV heads; the workspace is sized for
 * that (an upper bound for the bf16 cache too).
 */
int fp8kv_decode_plan(int B, int Hq, int Hkv, int D, int max_blocks_per_seq, int window,
                      int num_splits, int* num_splits_out, size_t* workspace_bytes_out);

/*
 * fp8kv_paged_decode_attn -- one query token per sequence attends to its paged
 * FP8 (or bf16) cache: split-K flash decoding plus a split-merge kernel.
 * [KO] opening paragraph (attention over the FP8 cache), "커널 및 퓨전 최적화"
 * (per-KV-head scales), "하이브리드 Attention 및 레이어 스킵" (window on a bf16
 * cache); [KVQ] "Per-Token-Head vs Per-Tensor 양자화" (per-token-head scales).
 *
 *   q              bf16 [B][Hq][D]; query head hq reads KV head hq / (Hq / Hkv).
 *                  q, context_lens and out may be device memory or pinned host
 *                  memory (read / written by the kernels over the host link);
 *                  every other pointer is device memory.
 *   k_cache, v_cache, kv_dtype, scale_mode  as written by fp8kv_kv_cache_write;
 *                  the bf16 cache ignores scales.
 *   k_scale, v_scale              fp32 [1] or [Hkv] (PER_TENSOR / PER_HEAD).
 *   k_scale_cache, v_scale_cache  fp32 [num_blocks][Hkv][16] (PER_TOKEN_HEAD).
 *   block_table    int32 [B][max_blocks_per_seq]: page p of sequence b is block
 *                  block_table[b][p]; entries past the sequence are not read.
 *   context_lens   int32 [B]: keys of sequence b are positions 0 .. ctx-1
 *                  (the new token already written); ctx 0 gives a zero row.
 *   softmax_scale  logits are softmax_scale * q . k (usually 1/sqrt(D)).
 *   window         0 = all keys; w > 0 = keys at positions >= ctx - w.
 *   num_splits     0 = automatic (see fp8kv_decode_plan).
 *   workspace      scratch of at least the planned bytes, 16-byte aligned; its
 *                  contents need no initialisation.  Calls that share one
 *                  workspace must not overlap on the GPU.
 *   out            [B][Hq][D] fp32 or bf16 (out_dtype).
 *   flags          0 or FP8KV_DECODE_EARLY_SETUP / FP8KV_DECODE_EARLY_PAGES
 *                  (below); any other bit is FP8KV_ERR_INVALID.
 * Ordering: the kernels launch with programmatic stream serialization, so they
 * may be resident while the preceding kernel of the stream finishes.  With
 * flags 0 they read nothing before that kernel has completed: any kernel may
 * produce any input.  The flags let the start overlap that kernel's tail when
 * the caller knows which inputs it does not write.
 * Output: softmax(z) V over the visible keys, accumulated in fp32.
 */
/* context_lens, block_table and k_scale / v_scale are complete before the
 * preceding kernel of the stream starts (written by a copy or an earlier
 * kernel): the work partition and the page-table reads start before it ends. */
#define FP8KV_DECODE_EARLY_SETUP 1u
/* EARLY_SETUP, and the cache pages the call reads (every slot but those
 * fp8kv_decode_step itself writes) are complete before the preceding kernel
 * starts too: the first pages stream before it ends.  True in a decode loop
 * whose older pages were written by earlier steps. */
#define FP8KV_DECODE_EARLY_PAGES 2u
int fp8kv_paged_decode_attn(const void* q, const void* k_cache, const void* v_cache,
                            int kv_dtype, int scale_mode, const float* k_scale,
                            const float* v_scale, const float* k_scale_cache,
                            const float* v_scale_cache, const int32_t* block_table,
                            int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                            int Hkv, int D, int64_t num_blocks, float softmax_scale, int window,
                            int num_splits, void* workspace, size_t workspace_bytes, void* out,
                            int out_dtype, unsigned flags, int32_t* err_flag, void* cuda_stream);

/*
 * fp8kv_decode_step -- a whole decode step of one attention layer in one
 * call: fp8kv_kv_cache_write of every sequence's new token followed by
 * fp8kv_paged_decode_attn, with the store done inside the attention kernel.
 * [KVQ] "Per-Token-Head vs Per-Tensor 양자화" (the kernel computes the
 * per-token-head scales when it stores the cache); [KO] opening paragraph.
 *
 *   k_new, v_new   bf16 [B][Hkv][D] (device or pinned host memory): the new
 *                  token of sequence b, stored at position ctx - 1
 *                  (ctx = context_lens[b]), i.e. in block
 *                  block_table[b][(ctx-1) / 16] at offset (ctx-1) % 16, with
 *                  exactly the codes and scales fp8kv_kv_cache_write would
 *                  store there (bf16 cache: the values as they are).  A
 *                  sequence with ctx 0 stores nothing and gets a zero row.
 *   k_cache, v_cache, k_scale_cache, v_scale_cache  written at those slots.
 *   Everything else as in fp8kv_paged_decode_attn; the attention sees the new
 *   token.  A block id outside the cache skips the store and sets
 *   FP8KV_ERR_BAD_INDEX in err_flag.
 * Ordering: as fp8kv_paged_decode_attn, flags included.  q, k_new and v_new
 * are read, and anything is written, only after the preceding kernel has
 * completed, whatever the flags.  In a decode loop whose tables were copied in
 * before the step and whose older pages were written by earlier steps,
 * FP8KV_DECODE_EARLY_PAGES holds.
 */
int fp8kv_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                      void* v_cache, int kv_dtype, int scale_mode, const float* k_scale,
                      const float* v_scale, float* k_scale_cache, float* v_scale_cache,
                      const int32_t* block_table, int max_blocks_per_seq,
                      const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                      int64_t num_blocks, float softmax_scale, int window, int num_splits,
                      void* workspace, size_t workspace_bytes, void* out, int out_dtype,
                      unsigned flags, int32_t* err_flag, void* cuda_stream);

/*
 * fp8kv_prefill_attn -- chunked causal prefill in FP8 on the tcgen05 tensor
 * cores.  [KO] opening paragraph (FP8 e4m3 attention compute), "커널 및 퓨전
 * 최적화" (query quantization fused into the kernel), "정확도를 위한 2단계 누적"
 * and "아키텍처별 결과" (two-level FP32 accumulation and its switch); [KVQ] "Q/Prob
 * 스케일과 FP8 Attention" (q_scale, prob_scale and the uncalibrated warning).
 *
 *   q              bf16 [Tq][Hq][D]: the new queries of every sequence back to back.
 *   cu_seqlens_q   int32 [B+1] (device): sequence b owns q rows cu[b] .. cu[b+1]-1.
 *   max_seqlen_q   host upper bound of cu[b+1] - cu[b] (sizes the grid).
 *   k_cache, v_cache  e4m3 [num_blocks][Hkv][16][D] holding every key of the
 *                  sequence, the chunk's own keys included (written before).
 *   scale_mode     PER_TENSOR (k_scale[0], v_scale[0]), PER_HEAD (k_scale[h]) or
 *                  PER_TOKEN_HEAD (k_scale_cache / v_scale_cache [num_blocks][Hkv][16],
 *                  16-byte aligned, as fp8kv_kv_cache_write stored them; the V
 *                  scales are folded into the e4m3 weights relative to a running
 *                  power-of-two bound of the scales seen, see prefill.cu).
 *   q_scale, prob_scale  host floats > 0: Q and the softmax weights are stored
 *                  as e4m3(q / q_scale) and e4m3(p / prob_scale) for the MMAs
 *                  (single operands; see flags).
 *   context_lens   int32 [B]: keys of sequence b, the chunk included; query i of
 *                  the chunk sits at position ctx - n_b + i and sees keys 0..that.
 *   flags          FP8KV_PREFILL_TWO_LEVEL: each KV tile's P V is added into a
 *                  separate fp32 accumulator on the CUDA cores (else the tensor
 *                  core accumulates across tiles, enough on Blackwell).
 *                  Operand precision of the e4m3 cache: by default a block of
 *                  query rows whose rows all see at least 8192 keys takes single
 *                  e4m3 Q and P (the rounding averages out over long rows); other
 *                  blocks take split operands, Q and P each as two e4m3 terms
 *                  (hi and the e4m3 of what hi misses, ~8 significant bits, after
 *                  exact power-of-two scaling that replaces q_scale and
 *                  prob_scale), which meets max-abs 1e-2 on N(0,1) data at any
 *                  length.  FP8KV_PREFILL_SPLIT_ALWAYS / _NEVER force one of
 *                  them; setting both is FP8KV_ERR_INVALID, as is any other bit.
 *                  The 8192-key threshold holds for N(0,1)-like data; with
 *                  per-token-head scales on data with x20 outlier channels
 *                  single operands lost up to ~0.3 of a channel's value rms on
 *                  9000-key rows (many small weights underflow e4m3 once the V
 *                  scales are folded in), split operands ~1.5e-2: force
 *                  SPLIT_ALWAYS for such data.
 *   out            [Tq][Hq][D] fp32 or bf16.
 * Supported: e4m3 cache (every scale mode) and its bf16 twin (bf16 Q, P and
 * cache, kind::f16; scales ignored), D in {64, 128, 256}, Hq / Hkv dividing 128.
 * Other shapes return FP8KV_ERR_UNSUPPORTED.  With q_scale or prob_scale equal
 * to 1.0 an e4m3 call succeeds and sets fp8kv_last_warning().
 */
#define FP8KV_PREFILL_TWO_LEVEL 1
#define FP8KV_PREFILL_SPLIT_ALWAYS 2
#define FP8KV_PREFILL_SPLIT_NEVER 4
int fp8kv_prefill_attn(const void* q, const int32_t* cu_seqlens_q, int max_seqlen_q,
                       const void* k_cache, const void* v_cache, int kv_dtype, int scale_mode,
                       const float* k_scale, const float* v_scale, const float* k_scale_cache,
                       const float* v_scale_cache, float q_scale,
                       float prob_scale, const int32_t* block_table, int max_blocks_per_seq,
                       const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                       int64_t num_blocks, float softmax_scale, int flags, void* out,
                       int out_dtype, int32_t* err_flag, void* cuda_stream);

/*
 * fp8kv_prefill_attn_ws -- fp8kv_prefill_attn with a device workspace, which
 * lets a launch of at most 8 sequences with more query tiles than the GPU has
 * SMs (B * Hkv * ceil(max_seqlen_q * G / 128) > SMs) run as one persistent CTA
 * per SM that takes an equal share of all (query tile, key tile) work instead
 * of one CTA per query tile (whose last wave leaves SMs idle).  A query tile
 * cut between CTAs leaves an fp32 partial per piece (O, its running max and
 * sum, as in the split decode's merge); the last CTA of the tile to finish
 * merges them.  Each piece rounds its e4m3 weights against its own running
 * maximum, so results differ from one CTA per tile within the rounding of FP8
 * attention.  Other launches (no more query tiles than SMs, or more than 8
 * sequences: every CTA plans its share by walking the sequences one after
 * another) ignore the workspace.
 *
 *   workspace        device memory, 16-byte aligned, workspace_bytes >=
 *                    fp8kv_prefill_workspace_bytes(D) (else FP8KV_ERR_WORKSPACE):
 *                    a counter per CTA, then the partials.  It must be zero
 *                    before its first use; every call that ends without error
 *                    leaves its counters zero again.  Calls that may run at the
 *                    same time (other streams) need separate workspaces.  NULL:
 *                    exactly fp8kv_prefill_attn.
 * Other arguments, supported shapes and errors: fp8kv_prefill_attn.
 */
int fp8kv_prefill_attn_ws(const void* q, const int32_t* cu_seqlens_q, int max_seqlen_q,
                          const void* k_cache, const void* v_cache, int kv_dtype, int scale_mode,
                          const float* k_scale, const float* v_scale,
                          const float* k_scale_cache, const float* v_scale_cache, float q_scale,
                          float prob_scale, const int32_t* block_table, int max_blocks_per_seq,
                          const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                          int64_t num_blocks, float softmax_scale, int flags, void* workspace,
                          size_t workspace_bytes, void* out, int out_dtype, int32_t* err_flag,
                          void* cuda_stream);

/*
 * fp8kv_prefill_workspace_bytes -- *bytes = the workspace fp8kv_prefill_attn_ws
 * needs at head_dim D on the current device (2 x SMs x 128 x (D + 2) floats of
 * partials plus the counters: 40 MB at D 256 on 152 SMs).  D outside {64, 128,
 * 256}: FP8KV_ERR_UNSUPPORTED.
 */
int fp8kv_prefill_workspace_bytes(int D, size_t* bytes);

/*
 * fp8kv_quantize_e4m3 -- the cache writer's encoder on its own: out[i] =
 * e4m3_rn_satfinite(fp32(x[i] / scale)) for n fp32 values (device arrays).
 * [PR] "코드 분석" (torch.float8_e4m3fn storage).  A zero scale writes code 0.
 */
int fp8kv_quantize_e4m3(const float* x, float scale, uint8_t* out, int64_t n,
                        void* cuda_stream);

/*
 * fp8kv_paged_decode_attn_noalloc -- fp8kv_paged_decode_attn for callers that
 * cannot allocate device memory.  The pages have no counterpart of it: it is a
 * deployment variant of the same computation, not part of the method.
 *
 * Who needs it: a C host program or plugin that only receives the tensors it
 * reads and writes from the framework owning the GPU's memory pool (it has no
 * allocator to get a workspace from), and serving loops that cannot call
 * cudaMalloc / cudaFree because those synchronize the device.
 *
 * Arguments are those of fp8kv_paged_decode_attn without workspace and flags
 * (it always waits for the preceding kernel first, as flags 0 does): the split
 * partials live in a static device array of FP8KV_NOALLOC_DECODE_SCRATCH_BYTES
 * inside the library, which every GPU that loads the library holds until the
 * process exits.  The caller still passes q, the caches, the tables and `out`.
 *   - num_splits 0: the automatic plan, lowered to the largest CTA count whose
 *     partials fit the array (a short sliding window needs none of it: its
 *     plan combines inside each CTA).  If not even one CTA fits (one slot per
 *     (sequence, KV head) unit alone, B * Hq * (D + 2) * 4 bytes, exceeds the
 *     array), or an explicit num_splits plan (fp8kv_decode_plan) needs more
 *     than the array holds, the call returns FP8KV_ERR_WORKSPACE and launches
 *     nothing; use fp8kv_paged_decode_attn with a workspace then.
 *   - All calls on a device share the array: calls whose kernels overlap on the
 *     GPU (other streams, other host threads) race.  Serialize them.
 *   - The first call on each device looks the array's address up with that
 *     device current, and so does the first call after that device's context
 *     was recreated (cudaDeviceReset); make those calls outside stream capture.
 *   - The array needs no initialisation and keeps the last call's partials.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine.
 */
#define FP8KV_NOALLOC_DECODE_SCRATCH_BYTES (8u << 20)
int fp8kv_paged_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    int kv_dtype, int scale_mode, const float* k_scale,
                                    const float* v_scale, const float* k_scale_cache,
                                    const float* v_scale_cache, const int32_t* block_table,
                                    int max_blocks_per_seq, const int32_t* context_lens, int B,
                                    int Hq, int Hkv, int D, int64_t num_blocks,
                                    float softmax_scale, int window, int num_splits, void* out,
                                    int out_dtype, int32_t* err_flag, void* cuda_stream);

/*
 * fp8kv_resolve_scales -- turn the scales a checkpoint loader found (or did
 * not find) into the scales the cache writer and the attention calls take.
 * Host-only: every array here is HOST memory, no GPU is touched.  [KVQ]
 * "BaseKVCacheMethod" (every scale starts at the sentinel -1.0, "not loaded"),
 * "Per-Token-Head vs Per-Tensor 양자화" (which scales each mode uses),
 * "Q/Prob 스케일과 FP8 Attention" (q_scale fallback and the uncalibrated
 * warning) and "스케일 통합 로직" (a lone kv_scale serves both K and V).
 *
 *   kv_dtype, scale_mode  the cache the scales are for.
 *   k_loaded, v_loaded    host float [n]: the loaded values, -1.0 (or any
 *                  negative value) where nothing was loaded.  n = 1 for
 *                  PER_TENSOR, Hkv for PER_HEAD; ignored (may be NULL) for
 *                  PER_TOKEN_HEAD and for a bf16 cache.
 *   q_loaded, prob_loaded  loaded q / prob scales, negative = not loaded.
 *   k_out, v_out   host float [n]: resolved K/V scales (written for
 *                  PER_TENSOR and PER_HEAD only).
 *   q_out, prob_out  host float: resolved q / prob scales.
 * Rules, per element i (PER_TENSOR and PER_HEAD on an e4m3 cache):
 *   both k and v > 0  -> used as loaded;
 *   both < 0          -> 1.0 each (the uncalibrated default);
 *   otherwise         -> one scale was loaded for both: k must be > 0
 *                        (else FP8KV_ERR_INVALID) and k_out = v_out = max(k, v).
 * PER_TOKEN_HEAD and bf16 caches: the writer computes (or needs) no per-tensor
 * scale; q_out = prob_out = 1.0.  Otherwise q_out = q_loaded if > 0 else 1.0,
 * and the same for prob.  An e4m3 cache whose resolved q or prob scale is 1.0
 * sets fp8kv_last_warning().  NaN anywhere returns FP8KV_ERR_INVALID; nothing
 * is written on error.  The FNUZ (x2) adjustment of [KVQ] is for AMD GPUs and
 * is not applied.
 */
int fp8kv_resolve_scales(int kv_dtype, int scale_mode, int n, const float* k_loaded,
                         const float* v_loaded, float q_loaded, float prob_loaded,
                         float* k_out, float* v_out, float* q_out, float* prob_out);

/* Human-readable name of a status code (static string). */
const char* fp8kv_status_string(int status);

/*
 * Last warning raised by a call on this thread, or "" if none: FP8 attention
 * with uncalibrated q/prob scales of 1.0 warns as [KVQ] "Q/Prob 스케일과 FP8
 * Attention" describes.  The string stays valid until the next call.
 */
const char* fp8kv_last_warning(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8KV_H */
