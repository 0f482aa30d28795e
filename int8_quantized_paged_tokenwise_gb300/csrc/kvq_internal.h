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

struct DecodeParams {
  const void* q;
  void* out;
  const void* k_cache;      // payload base pointers (L2 prefetch addresses)
  const void* v_cache;
  const uint16_t* k_scale;  // INT8 path only
  const uint16_t* v_scale;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* part_o;            // [sp][Hkv][G][D]
  float* part_lse;          // [sp][Hkv][G]   (log2 domain)
  int32_t* prefix_out;      // [B] inclusive partition prefix, written by CTA 0
  unsigned int* err;
  int32_t B, Hq, Hkv, G;
  int32_t max_blocks;       // block-table row length
  int32_t max_ctx;          // host upper bound on context_lens
  int32_t num_blocks;
  int32_t P;                // pages per partition (one warp's work item); 0 = kernel picks
  int32_t sp_cap;           // sequence-partitions the workspace holds (>= B)
  float scale_log2;         // sm_scale * log2(e)
};

struct CombineParams {
  const float* part_o;
  const float* part_lse;
  const int32_t* prefix;
  void* out;
  int32_t B, Hq, Hkv, G;
};

// decode (kvq_decode_int8.cu / kvq_decode_kv16.cu); D = head_dim, smem in bytes; maps =
// {K tiles, V tiles}.
size_t decode_smem_bytes_int8(int D, int B, int G);
cudaError_t decode_configure_int8(int D, bool bf16, size_t smem);
cudaError_t decode_occupancy_int8(int D, bool bf16, size_t smem, int* n);
cudaError_t decode_launch_int8(int D, bool bf16, const CUtensorMap* maps,
                               const DecodeParams& p, int grid, size_t smem, cudaStream_t s);
size_t decode_smem_bytes_kv16(int D, int B, int G);
cudaError_t decode_configure_kv16(int D, bool bf16, size_t smem);
cudaError_t decode_occupancy_kv16(int D, bool bf16, size_t smem, int* n);
cudaError_t decode_launch_kv16(int D, bool bf16, const CUtensorMap* maps,
                               const DecodeParams& p, int grid, size_t smem, cudaStream_t s);

// combine (kvq_combine.cu)
cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, cudaStream_t s);

// quantize-append and twin append (kvq_quant.cu)
cudaError_t quantize_append_launch(int D, bool bf16, const QuantParams& p, cudaStream_t s);
cudaError_t append_kv16_launch(int D, const QuantParams& p, cudaStream_t s);

}  // namespace kvq
