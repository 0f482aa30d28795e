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

constexpr int kCombineWarps = 8;

// One CTA per (query head, sequence).  The partitions are dealt round-robin
// to the 8 warps; each lane owns D/32 consecutive head dims; the warps'
// partial sums meet in shared memory.
template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  constexpr int PER = D / 32;
  __shared__ float red[kCombineWarps];
  __shared__ float part[kCombineWarps][D];
  __shared__ float wpart[kCombineWarps];
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  griddep_wait();               // the decode grid's partials are complete and visible
  const int sp0 = b > 0 ? p.prefix[b - 1] : 0;
  const int n = p.prefix[b] - sp0;
  if (n <= 1) return;
  const int j = h / p.G, g = h - j * p.G;
  const int64_t row0 = ((int64_t)sp0 * p.Hkv + j) * p.G + g;   // partition i: + i*Hkv*G
  const int64_t rstride = (int64_t)p.Hkv * p.G;

  float M = -INFINITY;
  for (int i = tid; i < n; i += kCombineWarps * 32) M = fmaxf(M, p.part_lse[row0 + i * rstride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  if (lane == 0) red[warp] = M;
  __syncthreads();
  M = red[0];
#pragma unroll
  for (int w = 1; w < kCombineWarps; ++w) M = fmaxf(M, red[w]);

  float acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
#pragma unroll 4
    for (int i = warp; i < n; i += kCombineWarps) {
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
#pragma unroll
  for (int e = 0; e < PER; ++e) part[warp][lane * PER + e] = acc[e];
  if (lane == 0) wpart[warp] = wsum;
  __syncthreads();
  if (tid < D / 2) {
    const int d = 2 * tid;
    float s0 = 0.f, s1 = 0.f, ws = 0.f;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) {
      s0 += part[w][d];
      s1 += part[w][d + 1];
      ws += wpart[w];
    }
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.out) + ((int64_t)b * p.Hq + h) * D + d;
    uint32_t v;
    if constexpr (BF16) v = bf2_as_u32(__floats2bfloat162_rn(s0 * inv, s1 * inv));
    else v = h2_as_u32(__floats2half2_rn(s0 * inv, s1 * inv));
    *reinterpret_cast<uint32_t*>(dst) = v;
  }
}

}  // namespace

cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, cudaStream_t s) {
  if (p.B == 0 || p.Hq == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, p.B);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) {
    return bf16 ? cudaLaunchKernelEx(&cfg, combine_kernel<128, true>, p)
                : cudaLaunchKernelEx(&cfg, combine_kernel<128, false>, p);
  }
  return bf16 ? cudaLaunchKernelEx(&cfg, combine_kernel<64, true>, p)
              : cudaLaunchKernelEx(&cfg, combine_kernel<64, false>, p);
}

}  // namespace kvq
