// Split-K combine: merges the normalized partial outputs of a sequence's
// partitions with their log2-sum-exp weights,
//   M = max_i lse_i,  w_i = 2^(lse_i - M) / sum_k 2^(lse_k - M),
//   out = sum_i w_i * O_i,
// the flash-decoding form of one softmax over all of the sequence's tokens.
// Sequences with a single partition were written by the decode kernel.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

// One warp per (query head, sequence); each lane owns D/32 consecutive dims.
template <int D, bool BF16>
__global__ void __launch_bounds__(32) combine_kernel(const CombineParams p) {
  constexpr int PER = D / 32;
  const int h = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  const int sp0 = b > 0 ? p.prefix[b - 1] : 0;
  const int n = p.prefix[b] - sp0;
  if (n <= 1) return;
  const int j = h / p.G, g = h - j * p.G;
  const int64_t row0 = ((int64_t)sp0 * p.Hkv + j) * p.G + g;   // partition i: + i*Hkv*G
  const int64_t rstride = (int64_t)p.Hkv * p.G;

  float M = -INFINITY;
  for (int i = lane; i < n; i += 32) M = fmaxf(M, p.part_lse[row0 + i * rstride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (int i = 0; i < n; ++i) {
      const int64_t r = row0 + i * rstride;
      const float w = fast_exp2(p.part_lse[r] - M);
      wsum += w;
      const float* src = p.part_o + r * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x; acc[1] += w * v.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + ((int64_t)b * p.Hq + h) * D + lane * PER;
#pragma unroll
  for (int e = 0; e < PER; e += 2) {
    uint32_t v;
    if constexpr (BF16) v = bf2_as_u32(__floats2bfloat162_rn(acc[e] * inv, acc[e + 1] * inv));
    else v = h2_as_u32(__floats2half2_rn(acc[e] * inv, acc[e + 1] * inv));
    *reinterpret_cast<uint32_t*>(dst + e) = v;
  }
}

}  // namespace

cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, cudaStream_t s) {
  if (p.B == 0 || p.Hq == 0) return cudaSuccess;
  const dim3 grid(p.Hq, p.B);
  if (D == 128) {
    if (bf16) combine_kernel<128, true><<<grid, 32, 0, s>>>(p);
    else combine_kernel<128, false><<<grid, 32, 0, s>>>(p);
  } else {
    if (bf16) combine_kernel<64, true><<<grid, 32, 0, s>>>(p);
    else combine_kernel<64, false><<<grid, 32, 0, s>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace kvq
