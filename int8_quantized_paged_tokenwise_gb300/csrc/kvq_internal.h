// Internal interface between the C-ABI layer (kvq_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kvq {

constexpr int kBlockSize = 16;   // tokens per page
constexpr int kWarps = 4;        // consumer warps per decode CTA
constexpr int kThreads = kWarps * 32;
constexpr int kMaxGroup = 8;     // query heads per KV head handled by one MMA n-tile
constexpr int kMaxSeqs = 4096;   // sequences per decode call (prefix table in smem)

struct QuantParams {
  const void* k;
  const void* v;
  int64_t k_stride;   // elements between tokens
  int64_t v_stride;
  const int64_t* slots;
  void* k_cache;      // int8 (quantize) or 16-bit (twin append)
  void* v_cache;
  uint16_t* k_scale;  // unused by the twin append
  uint16_t* v_scale;
  int64_t num_rows;   // tokens * kv heads
  int32_t num_kv_heads;
  int64_t num_slots;  // num_blocks * block_size
  unsigned int* err;
};

// Work distribution of the decode: the pages of all sequences form one
// column stream (sequence-major), cut into ranges of R columns; work unit
// u = (range u / Hkv, KV head u % Hkv) goes to warp u mod (warps in the
// grid).  The part of a range inside one sequence is a "piece": a piece
// covering the whole sequence writes the output directly; otherwise it writes
// a normalized partial and its log2-sum-exp into one of the unit's two
// partial slots (slot 0: the piece continues a sequence begun in an earlier
// range; slot 1: the piece begins a sequence that continues in a later
// range), which the combine kernel merges.
constexpr int kMinRangePages = 4;   // shortest range of the balanced split

struct DecodeParams {
  const void* q;
  void* out;
  const void* k_cache;      // payload base pointers
  const void* v_cache;
  const uint16_t* k_scale;  // INT8 path only
  const uint16_t* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;            // [2 * range_cap][G][D]   (unit u, slot k -> rows (2u + k) * G)
  float* part_lse;          // [2 * range_cap][G]      (log2 domain)
  unsigned int* err;
  int32_t B, Hq, Hkv, G;     // Hkv, G: head groups and query heads per group
  int32_t Gr;               // query heads per KV head (G / KV heads per group)
  int32_t max_blocks;       // block-table row length
  int32_t max_ctx;          // host upper bound on context_lens
  int32_t num_blocks;
  int32_t R;                // > 0: pages per range; 0: balanced (ceil(columns / groups), at
                            // least kMinRangePages); < 0: one unit per (sequence, KV head)
  int64_t groups;           // R == 0: ranges of the balanced split (>= 1)
  int64_t range_cap;        // work units the partial slots hold (0 when R < 0)
  float scale_log2;         // sm_scale * log2(e) (static scales: times the K scale)
  float v_static;           // static scales: the V scale (applied to the output)
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  const int32_t* context_lens;
  void* out;
  int32_t B, Hq, Hkv, G;
  int32_t max_tok;          // the decode kernel's clamp of context_lens
  int32_t R;                // as DecodeParams::R (>= 0)
  int64_t groups;           // as DecodeParams::groups
  int32_t per_cta;          // 1: one CTA per (sequence, query head), else one warp
};

struct DequantParams {
  const int8_t* k_cache;
  const int8_t* v_cache;
  const uint16_t* k_scale;
  const uint16_t* v_scale;
  void* k_out;              // 16-bit cache, same [NB][Hkv][16][D] layout
  void* v_out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  unsigned int* err;
  int32_t B, Hkv, max_blocks, max_tok, num_blocks;
};

struct TrimParams {
  int8_t* k_cache;
  int8_t* v_cache;
  uint16_t* k_scale;        // nullptr: a cache without scale planes (static scales)
  uint16_t* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* trim;      // [B] tokens to drop after the sink
  unsigned int* err;
  int32_t B, Hkv, max_blocks, max_tok, num_blocks, keep;
};

struct PrefillParams {
  const void* q;            // [total_q][Hq][D]
  void* out;                // [total_q][Hq][D]
  const uint16_t* k_scale;
  const uint16_t* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;   // [B + 1]
  unsigned int* err;
  int32_t B, Hq, Hkv, G, max_blocks, max_ctx, num_blocks;
  int32_t total_q, max_q;   // rows of q/out; host bound on a sequence's queries
  float scale_log2;         // sm_scale * log2(e)
};

// chunked prefill (kvq_prefill.cu); grid = (tiles, Hkv, B)
size_t prefill_smem_bytes(int D);
int prefill_rows_per_cta();   // (query, head) rows of one CTA tile
cudaError_t prefill_configure(int D, bool bf16);
cudaError_t prefill_launch(int D, bool bf16, const CUtensorMap* maps, const PrefillParams& p,
                           int tiles, cudaStream_t s);

// Head groups: KV heads one decode warp processes together (each page step
// covers their adjacent tiles).  The launcher uses up to kMaxHeadGroup.
#ifndef KVQ_MAX_HEAD_GROUP
#define KVQ_MAX_HEAD_GROUP 2
#endif
constexpr int kMaxHeadGroup = KVQ_MAX_HEAD_GROUP;
// Pages one warp step covers when the head group is one KV head.
#ifndef KVQ_MAX_PAGE_STEP
#define KVQ_MAX_PAGE_STEP 2
#endif
constexpr int kMaxPageStep = KVQ_MAX_PAGE_STEP;

// One decode kernel variant (cache kind x head group), for head_dim 64/128
// and FP16/BF16 activations.  D = head_dim, GH = query heads per head group,
// smem in bytes, maps = {K tiles, V tiles}.
struct DecodeOps {
  size_t (*smem)(int D, int B, int GH);
  cudaError_t (*configure)(int D, bool bf16, size_t smem);
  cudaError_t (*occupancy)(int D, bool bf16, size_t smem, int* n);
  cudaError_t (*launch)(int D, bool bf16, const CUtensorMap* maps, const DecodeParams& p,
                        int grid, size_t smem, cudaStream_t s);
};
extern const DecodeOps kDecodeInt8H1;    // kvq_decode_int8.cu
extern const DecodeOps kDecodeInt8H2;    // kvq_decode_int8_h2.cu
extern const DecodeOps kDecodeStaticH1;  // kvq_decode_static.cu
extern const DecodeOps kDecodeStaticH2;  // kvq_decode_static_h2.cu
extern const DecodeOps kDecodeKv16;      // kvq_decode_kv16.cu
extern const DecodeOps kDecodeInt8Cc;    // kvq_decode_int8_cc.cu (CUDA cores, A/B)
extern const DecodeOps kDecodeInt8T2;    // kvq_decode_int8_t2.cu (two pages per step)

// combine (kvq_combine.cu)
cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, int sms, cudaStream_t s);

// dequantize-window baseline (kvq_dequant.cu)
cudaError_t dequant_window_launch(int D, bool bf16, const DequantParams& p, int max_pages,
                                  cudaStream_t s);

// front trim keeping the sink (kvq_trim.cu): moves the rows, then updates
// context_lens (the same array as p.context_lens)
cudaError_t trim_launch(int D, const TrimParams& p, int32_t* context_lens, cudaStream_t s);

// quantize-append and twin append (kvq_quant.cu)
cudaError_t quantize_append_launch(int D, bool bf16, const QuantParams& p, cudaStream_t s);
// static scales: p.k_scale/v_scale unused, inv_k/inv_v = fl32(1 / scale)
cudaError_t quantize_static_launch(int D, bool bf16, const QuantParams& p, float inv_k,
                                   float inv_v, cudaStream_t s);
cudaError_t append_kv16_launch(int D, const QuantParams& p, cudaStream_t s);

}  // namespace kvq
