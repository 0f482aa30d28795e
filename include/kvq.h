/*
 * kvq.h -- C ABI of libkvq: tokenwise symmetric INT8 paged KV cache for LLM
 * decode on GB300 (sm_103a).
 *
 * The library has two hot operations and a 16-bit twin of the second:
 *
 *   kvq_quantize_append    quantize-on-write of new K/V rows into a paged
 *                          INT8 cache with one FP16 scale per (page, KV head,
 *                          token).
 *   kvq_paged_decode       fused paged decode attention over the INT8 cache:
 *                          page walk through a block table, dequantization in
 *                          registers, FP32 accumulation, online softmax, and
 *                          a split-K (flash-decoding) variant with a combine
 *                          kernel for long contexts and small batches.
 *   kvq_paged_decode_kv16  the same decode over a native 16-bit cache (A/B).
 *
 * Where the operations are defined (page title, then section):
 *   [MI] "feat: opt-in INT8 KV-cache quantization" (MoE-Infinity PR #183),
 *        "What landed" -- tokenwise symmetric INT8 with upward-rounded FP16
 *        scales, no -128, exact zero, element error <= stored_scale/2 + 1e-6;
 *        paged INT8 decode with FP16 scales and FP32 accumulation, MHA/GQA;
 *        "Precision & memory" -- one FP16 scale per (layer, page, KV head,
 *        token); 33,280 bytes per 16-token, 8-head, d=128 page.
 *   [ML] "fix(cuda/kv): correct Int8 KV per-token scale ..." (mlxcel PR
 *        #717), "The Int8 bug and fix" -- scale = absmax/127, 1.0 only for
 *        an all-zero token; the largest coordinate maps to +-127.
 *
 * ---------------------------------------------------------------------------
 * Conventions common to every call
 * ---------------------------------------------------------------------------
 *  - Pointers: every tensor pointer is a DEVICE pointer owned by the caller.
 *    The library never frees or retains them.  Calls are asynchronous on
 *    `stream` (a cudaStream_t; NULL = legacy default stream) and never
 *    synchronize, except kvq_get_error.
 *  - Allocation: no call allocates device memory.  Split-K scratch is the
 *    caller's `workspace` (size from kvq_decode_workspace_bytes).
 *  - One layer per call: per-layer caches are separate base pointers.
 *  - Cache layout (one layer), block_size bs = 16, D = head_dim:
 *        payload     int8   [num_blocks][num_kv_heads][bs][D]     (K and V)
 *        scale plane uint16 [num_blocks][num_kv_heads][bs]        (FP16 bits)
 *    A token with slot s lives in block s / bs at offset s % bs.  Each
 *    (block, KV head) tile of the payload is bs*D contiguous bytes.
 *    Page bytes (K+V, all heads) = bs*Hkv*(2*D + 4): 33,280 at (16, 8, 128).
 *    16-bit twin cache: dtype [num_blocks][num_kv_heads][bs][D].
 *  - Block table: int32 [num_seqs][max_blocks_per_seq], row-major; entry i of
 *    row b is the physical block of logical page i of sequence b.
 *  - GQA: query head h reads KV head h / (num_q_heads / num_kv_heads).
 *  - Errors: host-detectable problems (NULL pointers, bad sizes, misaligned
 *    pointers, unsupported shapes, small workspace) return a status and launch
 *    nothing.  Device-detectable problems (slot, block id or context length
 *    out of range) skip the offending item, never fault, and set a bit in a
 *    per-device error word that kvq_get_error reads and clears.  There is no
 *    fallback path: an unsupported input is an error.
 *  - Supported: head_dim 64 or 128; block_size 16; Hq/Hkv in 1..8;
 *    num_seqs <= 4096; FP16 or BF16 activations.
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARGUMENT = 1,   /* NULL pointer, negative size, misaligned  */
  KVQ_ERR_UNSUPPORTED = 2,        /* shape outside the supported set          */
  KVQ_ERR_CUDA = 3,               /* a CUDA runtime call failed               */
  KVQ_ERR_WORKSPACE_TOO_SMALL = 4,
  KVQ_ERR_DEVICE_INDEX = 5,       /* kvq_get_error: an index was out of range */
  KVQ_ERR_DEVICE_TIMEOUT = 6      /* kvq_get_error: a bounded wait gave up    */
} kvq_status;

typedef enum { KVQ_FP16 = 0, KVQ_BF16 = 1 } kvq_dtype;

/* Bits of the device error word (kvq_get_error). */
#define KVQ_DEVERR_SLOT 0x1u        /* slot >= num_blocks * block_size          */
#define KVQ_DEVERR_BLOCK 0x2u       /* block id < 0 or >= num_blocks            */
#define KVQ_DEVERR_CONTEXT 0x4u     /* context_len < 0 or > max_blocks * bs     */
#define KVQ_DEVERR_TIMEOUT 0x8u     /* an mbarrier wait hit its limit           */

/*
 * kvq_quantize_append -- tokenwise symmetric INT8 quantize-on-write.
 * Defined by [MI] "What landed" and [ML] "The Int8 bug and fix".
 *
 * For each new token t < num_tokens and KV head j, separately for K and V,
 * with row x = k[t][j][0..D) (resp. v):
 *     a = max_d |x_d|
 *     s = 1.0                                  if a == 0
 *         smallest FP16 value >= a / 127       otherwise (upward rounding;
 *                                              saturates at 65504)
 *     code_d = clamp(round_half_even(x_d / s), -127, 127)
 * then stores the D codes and the FP16 bits of s at slot slot_mapping[t].
 * Codes and scales are bit-identical to an exact-arithmetic evaluation.
 *
 *   k, v            [num_tokens][num_kv_heads][head_dim] of `dtype`; heads
 *                   are contiguous (stride head_dim); consecutive tokens are
 *                   k_token_stride / v_token_stride ELEMENTS apart
 *                   (>= num_kv_heads*head_dim, multiple of 4); 8-byte aligned.
 *   slot_mapping    int64 [num_tokens]; negative = skip the token;
 *                   >= num_blocks*block_size sets KVQ_DEVERR_SLOT (skipped).
 *   k_cache,v_cache int8 payload (layout above), 16-byte aligned.
 *   k_scale,v_scale uint16 scale planes (layout above), 16-byte aligned.
 * num_tokens == 0 is a no-op.  Tokens mapped to the same slot race.
 */
kvq_status kvq_quantize_append(const void* k, const void* v, int64_t k_token_stride,
                               int64_t v_token_stride, int32_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, kvq_dtype dtype,
                               const int64_t* slot_mapping, int8_t* k_cache, int8_t* v_cache,
                               uint16_t* k_scale, uint16_t* v_scale, int32_t num_blocks,
                               int32_t block_size, kvq_stream_t stream);

/*
 * kvq_paged_decode -- fused paged decode attention over the INT8 cache.
 * Defined by [MI] "What landed" (INT8 + FP16-scale paged decode, FP32
 * accumulation, MHA/GQA, checked against dequantized softmax attention).
 *
 * For each sequence b with L = context_lens[b] and query head h (KV head j):
 *     k_hat_t = s_k[t] * code_k[t],  v_hat_t = s_v[t] * code_v[t]
 *     z_t     = sm_scale * <q[b][h], k_hat_t>,   t < L
 *     out[b][h] = sum_t softmax(z)_t * v_hat_t        (0 when L == 0)
 * Token t of sequence b is read from block block_tables[b][t / 16], offset
 * t % 16.  Arithmetic: codes and q in FP16 on the tensor cores, FP32
 * accumulation and softmax, output rounded to `dtype`.
 *
 *   q, out          [num_seqs][num_q_heads][head_dim] of `dtype`, contiguous,
 *                   16-byte aligned.
 *   block_tables    int32 [num_seqs][max_blocks_per_seq].
 *   context_lens    int32 [num_seqs] (device); max_context_len is a host-side
 *                   upper bound on every entry (used by the launcher; an entry
 *                   above max_blocks_per_seq*16 sets KVQ_DEVERR_CONTEXT and
 *                   that sequence's output is left unspecified).
 *   workspace       device scratch of kvq_decode_workspace_bytes(...) bytes,
 *                   256-byte aligned, not shared by calls that overlap on the
 *                   GPU.  NULL (or 0 bytes): no split-K -- one warp per
 *                   (sequence, KV head), correct but unbalanced.  A smaller
 *                   non-zero size is accepted down to four work ranges and
 *                   only lowers the number of warps used.  Calls whose
 *                   sequences all fit in four pages (max_context_len <= 64)
 *                   never split and do not touch it.
 * Work distribution: the (sequence, KV head, page) tiles form one stream,
 * cut into ranges of R = max(4, ceil(tiles / warps)) pages from the exact
 * context lengths, one range per resident warp, so every warp reads the same
 * number of pages.  A sequence whose tiles span two or more ranges goes
 * through split-K partials and a combine kernel (flash-decoding).
 */
kvq_status kvq_paged_decode(const void* q, kvq_dtype dtype, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            const int8_t* k_cache, const int8_t* v_cache,
                            const uint16_t* k_scale, const uint16_t* v_scale,
                            int32_t num_blocks, int32_t block_size,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t max_context_len,
                            float sm_scale, void* out, void* workspace,
                            size_t workspace_bytes, kvq_stream_t stream);

/* Scratch bytes for kvq_paged_decode (and kvq_paged_decode_kv16) with these
 * sizes on the current device: two partial slots of G rows per work range,
 * one range per resident warp.  0 when no sequence can hold more than four
 * pages (max_context_len <= 64: the call then never splits) or on invalid
 * sizes. */
size_t kvq_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len);

/* The work-range length (pages) kvq_paged_decode uses on the current device
 * when every sequence holds max_context_len tokens: max(4, ceil(tiles /
 * resident warps)); with shorter contexts the kernel uses the value for the
 * actual total.  0 on invalid input. */
int32_t kvq_decode_partition_pages(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_context_len);

/* kvq_paged_decode with the work-range length forced (partition_pages >= 1
 * pages per range; ranges are dealt to the warps round-robin), for tests and
 * tuning.  Workspace from kvq_decode_workspace_bytes_split with the same
 * length (required, also when nothing ends up split). */
kvq_status kvq_paged_decode_split(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  const int8_t* k_cache, const int8_t* v_cache,
                                  const uint16_t* k_scale, const uint16_t* v_scale,
                                  int32_t num_blocks, int32_t block_size,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t max_context_len,
                                  float sm_scale, void* out, void* workspace,
                                  size_t workspace_bytes, int32_t partition_pages,
                                  kvq_stream_t stream);

size_t kvq_decode_workspace_bytes_split(int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_context_len, int32_t partition_pages);

/*
 * kvq_paged_prefill -- chunked-prefill attention over the INT8 cache: the
 * queries of a chunk of new tokens per sequence, written into the cache
 * before the call (kvq_quantize_append), attend causally to the sequence's
 * cached tokens.  Defined by [ML] "Server integration" (Int8 chunked prefill
 * + decode over the same cache) with [MI]'s dequantized attention:
 *     n_b = query_start[b+1] - query_start[b] queries, the last n_b of the
 *     sequence's L_b = context_lens[b] tokens; query i sits at position
 *     p = L_b - n_b + i and attends to tokens 0..p:
 *     out[query_start[b] + i][h] = softmax_{t<=p}(sm_scale q . k_hat_t) . v_hat
 * Arithmetic: q and codes in FP16 on the 5th-generation tensor cores
 * (tcgen05, FP32 accumulators in tensor memory), K scales on the FP32
 * scores, softmax in FP32, V scales folded into the FP16 probabilities
 * (P s_v), output rounded to `dtype`.  Each CTA covers 256 (query, head)
 * rows of one KV head, so the grid is ceil(max_query_len / (256 / G)) x
 * num_kv_heads x num_seqs.
 *
 *   q, out          [total_q][num_q_heads][head_dim] of `dtype`, 16-byte aligned
 *                   (may be null when total_q == 0: nothing is launched).
 *   query_start     device int32 [num_seqs + 1], non-decreasing, from 0.
 *   total_q         rows of q and out; a sequence whose queries fall outside
 *                   them is flagged (KVQ_DEVERR_CONTEXT) and skipped.
 *   max_query_len   host upper bound on every n_b (sizes the grid; a larger
 *                   n_b is flagged and skipped).
 *   other arguments as kvq_paged_decode (no workspace).
 * Device errors: n_b > L_b or L_b above the table / max_context_len
 * (KVQ_DEVERR_CONTEXT, that sequence's output unspecified), block id out of
 * range (KVQ_DEVERR_BLOCK).
 */
kvq_status kvq_paged_prefill(const void* q, kvq_dtype dtype, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             const int8_t* k_cache, const int8_t* v_cache,
                             const uint16_t* k_scale, const uint16_t* v_scale,
                             int32_t num_blocks, int32_t block_size,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len,
                             const int32_t* query_start, int32_t total_q, int32_t max_query_len,
                             float sm_scale, void* out, kvq_stream_t stream);

/*
 * kvq_paged_decode_kv16 -- the same decode over a native 16-bit cache (K and
 * V in `dtype`, no scales); the A/B twin of kvq_paged_decode.  Arguments as
 * kvq_paged_decode; k_cache/v_cache are [num_blocks][num_kv_heads][16][D] of
 * `dtype`.  Workspace from kvq_decode_workspace_bytes (same sizes).
 * Arithmetic: q, K, V, P in `dtype` on the tensor cores, FP32 accumulation.
 */
kvq_status kvq_paged_decode_kv16(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 const void* k_cache, const void* v_cache, int32_t num_blocks,
                                 int32_t block_size, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 int32_t max_context_len, float sm_scale, void* out,
                                 void* workspace, size_t workspace_bytes, kvq_stream_t stream);

kvq_status kvq_paged_decode_kv16_split(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, const void* k_cache,
                                       const void* v_cache, int32_t num_blocks,
                                       int32_t block_size, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float sm_scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t partition_pages, kvq_stream_t stream);

/*
 * Static-scale variant (one binary32 scale per tensor, no scale planes):
 * "fix: #552 int8 kv cache quantization cannot be enabled" (InfiniLM PR #553)
 * -- a static per-tensor scale (default 1.0, or calibrated from max|K|/127);
 * "Add calibrated INT8 KV cache to PyTorch backend" (TensorRT-LLM PR #18953)
 * -- a calibrated scalar applied through its reciprocal (K and V may share
 * it: pass the same value twice).
 *
 * kvq_quantize_append_static: as kvq_quantize_append, with
 *     inv = fl32(1 / scale),  code = clamp(rne(fl32(x * inv)), -127, 127)
 * (binary32 reciprocal and product, round half to even); no scale planes.
 * k_scale, v_scale must be finite and > 0 (KVQ_ERR_INVALID_ARGUMENT).
 *
 * kvq_paged_decode_static: as kvq_paged_decode over such a cache:
 *     k_hat = k_scale * code_k,  v_hat = v_scale * code_v
 * (the K scale is folded into the score scale, the V scale applied to the
 * output).  Same workspace (kvq_decode_workspace_bytes) and errors.
 */
kvq_status kvq_quantize_append_static(const void* k, const void* v, int64_t k_token_stride,
                                      int64_t v_token_stride, int32_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim, kvq_dtype dtype,
                                      const int64_t* slot_mapping, int8_t* k_cache,
                                      int8_t* v_cache, float k_scale, float v_scale,
                                      int32_t num_blocks, int32_t block_size,
                                      kvq_stream_t stream);

kvq_status kvq_paged_decode_static(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   const int8_t* k_cache, const int8_t* v_cache, float k_scale,
                                   float v_scale, int32_t num_blocks, int32_t block_size,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   float sm_scale, void* out, void* workspace,
                                   size_t workspace_bytes, kvq_stream_t stream);

/* Scatter copy of new 16-bit K/V rows into the twin's cache (no
 * quantization): the write half of the 16-bit A/B path.  Arguments as
 * kvq_quantize_append; caches are [num_blocks][num_kv_heads][16][D] of dtype. */
kvq_status kvq_cache_append_kv16(const void* k, const void* v, int64_t k_token_stride,
                                 int64_t v_token_stride, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, kvq_dtype dtype,
                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                 int32_t num_blocks, int32_t block_size, kvq_stream_t stream);

/*
 * kvq_dequantize_window -- the dequantize-window baseline: for every page of
 * every sequence (pages 0 .. ceil(context_lens[b]/16)-1 through the block
 * table), write s[t] * code[t][d] rounded (nearest even) to `dtype` into a
 * 16-bit cache of the same [num_blocks][num_kv_heads][16][D] layout, K and V.
 * Defined by [ML] "The Int8 bug and fix" (its CUDA path dequantizes the
 * whole window, then runs attention over FP16); followed by
 * kvq_paged_decode_kv16 on k_out/v_out it is that path, the comparison the
 * fused kvq_paged_decode is measured against.
 *
 *   k_cache, v_cache, k_scale, v_scale   the INT8 cache (as kvq_paged_decode).
 *   k_out, v_out     device, 16-byte aligned, [num_blocks][num_kv_heads][16][D]
 *                    of `dtype`; only the pages the sequences reach are
 *                    written (all 16 rows of each).
 *   block_tables, context_lens, max_context_len   as kvq_paged_decode.
 * Device errors: block id out of range (page skipped, KVQ_DEVERR_BLOCK),
 * context above max_context_len (clamped, KVQ_DEVERR_CONTEXT).
 */
kvq_status kvq_dequantize_window(const int8_t* k_cache, const int8_t* v_cache,
                                 const uint16_t* k_scale, const uint16_t* v_scale,
                                 int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, const int32_t* block_tables,
                                 int32_t num_seqs, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t max_context_len,
                                 kvq_dtype dtype, void* k_out, void* v_out,
                                 kvq_stream_t stream);

/*
 * kvq_trim_front_keep_sink -- front trim of each sequence that keeps the
 * attention sink.  Defined by "fix(cuda/kv): correct Int8 KV per-token scale
 * ..." (mlxcel PR #717), follow-up commit, "The fix": a sequence of L tokens
 * becomes [its first keep tokens] ++ [the tokens after the next n], exactly n
 * removed, the INT8 payload and its scale rows moved in lockstep; keep = 0 is
 * the plain front trim (drop the n oldest).  Per sequence b:
 *     keep_b = min(keep, L),  n = clamp(trim[b], 0, L - keep_b)
 *     token keep_b + n + i moves to keep_b + i,  context_lens[b] = L - n.
 *
 *   k_cache, v_cache   INT8 payload [num_blocks][num_kv_heads][16][D], moved
 *                      in place through the block table.
 *   k_scale, v_scale   FP16 scale planes, moved with the payload; both NULL
 *                      for a static-scale cache (codes only).
 *   context_lens       device int32 [B], read, then updated in place.
 *   trim               device int32 [B], tokens to drop after the sink.
 *   keep               sink tokens kept at the front (>= 0; 4 in the page's
 *                      scheduler).
 * The pages of a trimmed sequence must not be shared with another sequence.
 * Rows past the new length are left as they were.  Device errors: block id
 * out of range (that token skipped, KVQ_DEVERR_BLOCK).
 */
kvq_status kvq_trim_front_keep_sink(int8_t* k_cache, int8_t* v_cache, uint16_t* k_scale,
                                    uint16_t* v_scale, int32_t num_blocks, int32_t block_size,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    const int32_t* block_tables, int32_t num_seqs,
                                    int32_t max_blocks_per_seq, int32_t* context_lens,
                                    const int32_t* trim, int32_t keep, kvq_stream_t stream);

/*
 * kvq_paged_decode_cuda_cores -- kvq_paged_decode with the page math on the
 * CUDA cores: FP32 FFMA dot products over the exactly converted codes and
 * warp-shuffle reductions, in place of the tensor-core MMAs (same pages, same
 * work split, same arithmetic up to rounding order, same arguments, results
 * and error behaviour).  The A/B counterpart that measures what the tensor
 * cores gain for each query-group size; kvq_paged_decode takes the faster
 * engine.  The computation is that of "feat: opt-in INT8 KV-cache
 * quantization" (MoE-Infinity PR #183), "What landed".
 */
kvq_status kvq_paged_decode_cuda_cores(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, const int8_t* k_cache,
                                       const int8_t* v_cache, const uint16_t* k_scale,
                                       const uint16_t* v_scale, int32_t num_blocks,
                                       int32_t block_size, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float sm_scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       kvq_stream_t stream);

/*
 * kvq_paged_decode_noalloc -- kvq_paged_decode for callers that cannot
 * allocate device memory.  The pages have no counterpart of this call; it
 * exists for hosts that own all device memory through their own pool
 * (inference servers, framework plugins) or run on a fixed memory budget, and
 * for latency-critical loops that must not risk the device synchronization
 * cudaMalloc/cudaFree can cause.
 *
 * Same arguments and result as kvq_paged_decode, minus the workspace: the
 * split-K scratch is a static device array of KVQ_NOALLOC_SCRATCH_BYTES built
 * into the library (held on every GPU that loads it, until exit), passed to
 * kvq_paged_decode as its workspace.  Where kvq_decode_workspace_bytes(...)
 * recommends more, the launcher uses fewer, longer work ranges (or one range
 * per sequence), with the same results; KVQ_ERR_WORKSPACE_TOO_SMALL is
 * returned only when not even one range per KV head fits (about
 * 16 MiB / (8 G (D + 1)) KV heads).  Allocates nothing.  The first call on a
 * device looks up the array's device address (make that first call before
 * any stream capture); the address is not valid across cudaDeviceReset, after
 * which this call must not be used in the process.  All calls on a device
 * share the array: calls that overlap on the GPU race.  Nothing in it needs
 * clearing between calls.
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)

kvq_status kvq_paged_decode_noalloc(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    const int8_t* k_cache, const int8_t* v_cache,
                                    const uint16_t* k_scale, const uint16_t* v_scale,
                                    int32_t num_blocks, int32_t block_size,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t max_context_len,
                                    float sm_scale, void* out, kvq_stream_t stream);

/* Synchronizes `stream`, then reads and clears the current device's error
 * word.  *flags (may be NULL) receives the KVQ_DEVERR_* bits.  Returns
 * KVQ_OK when no bit was set, KVQ_ERR_DEVICE_TIMEOUT if the timeout bit was
 * set, else KVQ_ERR_DEVICE_INDEX. */
kvq_status kvq_get_error(kvq_stream_t stream, uint32_t* flags);

/* Self-test of the device-side failure path (no page defines it): one warp
 * waits on an mbarrier that nothing completes, gives up after limit_us
 * microseconds (1 .. 1,000,000) and sets KVQ_DEVERR_TIMEOUT, exactly as a
 * kernel whose copies never landed would; the context stays usable.  Follow
 * with kvq_get_error, which then returns KVQ_ERR_DEVICE_TIMEOUT. */
kvq_status kvq_selftest_wait_timeout(uint32_t limit_us, kvq_stream_t stream);

/* Static, NUL-terminated description of a status code. */
const char* kvq_status_string(kvq_status status);

/* Library version, major*10000 + minor*100 + patch. */
int32_t kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
