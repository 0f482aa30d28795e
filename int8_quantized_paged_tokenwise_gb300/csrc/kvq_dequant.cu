// Dequantize-window baseline: the pages of a batch's sequences, INT8 codes
// times their token's FP16 scale, written as a 16-bit paged cache with the
// same block layout, for the 16-bit decode to read afterwards.
//
// This is the comparison path of "fix(cuda/kv): correct Int8 KV per-token
// scale ..." (mlxcel PR #717), "The Int8 bug and fix": its CUDA route
// dequantizes the whole cached window and then runs attention over FP16,
// which moves the INT8 bytes once and 16-bit bytes twice.  The fused decode
// (kvq_paged_decode) is the alternative it is measured against.
//
// Exactness: |code| <= 127 (7 bits) times an FP16 scale (11 significant bits)
// is exact in FP32; one round-to-nearest-even to the 16-bit dtype follows,
// the single rounding the definition has.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kDqThreads = 256;
constexpr int kDqPages = 4;   // pages of one sequence per CTA

template <bool BF16>
__device__ __forceinline__ uint32_t pack16(float a, float b) {
  if constexpr (BF16) return bf2_as_u32(__floats2bfloat162_rn(a, b));
  else return h2_as_u32(__floats2half2_rn(a, b));
}

// grid (ceil(max pages / kDqPages), B); each thread converts chunks of 8
// codes (one 8-byte load, one 16-byte store) of the CTA's pages, all KV
// heads, K then V.
template <int D, bool BF16>
__global__ void __launch_bounds__(kDqThreads) dequant_window_kernel(const DequantParams p) {
  constexpr int kRowChunks = D / 8;                 // chunks per token row
  constexpr int kTileChunks = kBlockSize * kRowChunks;
  const int b = blockIdx.y;
  int L = __ldg(&p.context_lens[b]);
  if (L < 0 || L > p.max_tok) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, 0x4u);
    L = L < 0 ? 0 : p.max_tok;
  }
  const int pages = (L + kBlockSize - 1) / kBlockSize;
  const int pg0 = blockIdx.x * kDqPages;
  if (pg0 >= pages) return;
  const int npg = min(pages - pg0, kDqPages);
  const int per_page = p.Hkv * kTileChunks;
  const int per_kv = npg * per_page;
  for (int i = threadIdx.x; i < 2 * per_kv; i += kDqThreads) {
    const bool is_v = i >= per_kv;
    const int r = is_v ? i - per_kv : i;
    const int pg = r / per_page;
    const int r2 = r - pg * per_page;
    const int j = r2 / kTileChunks;
    const int ch = r2 - j * kTileChunks;
    const int tok = ch / kRowChunks, dc = ch - tok * kRowChunks;
    const int blk = __ldg(&p.block_tables[(int64_t)b * p.max_blocks + pg0 + pg]);
    if (blk < 0 || blk >= p.num_blocks) {
      if (j == 0 && ch == 0 && !is_v) atomicOr(p.err, 0x2u);
      continue;
    }
    const int64_t row = ((int64_t)blk * p.Hkv + j) * kBlockSize + tok;
    const int8_t* src = (is_v ? p.v_cache : p.k_cache) + row * D + dc * 8;
    const uint16_t sbits = __ldg((is_v ? p.v_scale : p.k_scale) + row);
    const float s = __half2float(__ushort_as_half(sbits));
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
    float x[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[e] = (float)(int8_t)((w.x >> (8 * e)) & 0xFFu) * s;
      x[4 + e] = (float)(int8_t)((w.y >> (8 * e)) & 0xFFu) * s;
    }
    uint4 o;
    o.x = pack16<BF16>(x[0], x[1]);
    o.y = pack16<BF16>(x[2], x[3]);
    o.z = pack16<BF16>(x[4], x[5]);
    o.w = pack16<BF16>(x[6], x[7]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(is_v ? p.v_out : p.k_out) + row * D + dc * 8) = o;
  }
}

}  // namespace

cudaError_t dequant_window_launch(int D, bool bf16, const DequantParams& p, int max_pages,
                                  cudaStream_t s) {
  if (p.B == 0 || max_pages == 0) return cudaSuccess;
  const dim3 grid((unsigned)((max_pages + kDqPages - 1) / kDqPages), (unsigned)p.B);
  if (D == 128) {
    if (bf16) dequant_window_kernel<128, true><<<grid, kDqThreads, 0, s>>>(p);
    else dequant_window_kernel<128, false><<<grid, kDqThreads, 0, s>>>(p);
  } else {
    if (bf16) dequant_window_kernel<64, true><<<grid, kDqThreads, 0, s>>>(p);
    else dequant_window_kernel<64, false><<<grid, kDqThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvq
