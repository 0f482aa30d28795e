// Split-K combine: merges the normalized partial outputs of a sequence's
// pieces with their log2-sum-exp weights,
//   M = max_i lse_i,  w_i = 2^(lse_i - M) / sum_k 2^(lse_k - M),
//   out = sum_i w_i * O_i,
// the flash-decoding form of one softmax over all of the sequence's tokens.
// The pieces of (sequence b, KV head j) are the parts of b's pages in the
// consecutive column ranges c0..c1 that cover them: unit (c0, j) holds the
// first piece in its slot 1, units (c0+1..c1, j) the others in slot 0.
// Sequences inside one range were written by the decode kernel.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kCombineWarps = 8;
constexpr int kCombineThreads = kCombineWarps * 32;
constexpr int kCombineBatch = 8;   // pieces a lane loads before using any
// CTAs resident per SM the register budget is set for (64 registers): the
// merge is a chain of dependent L2 loads per pair, so the number of warps in
// flight sets its speed (measured on GB300: 8 pieces per batch and 4 CTAs per
// SM took the serving mix's merge from ~11 to ~7 us after the decode)
constexpr int kCombineMinCtas = 4;

// Every CTA first rebuilds, from context_lens, the page prefix and range
// length the decode kernel used (this overlaps the decode's tail: the launch
// is programmatic); then (sequence, query head) pairs are merged, lanes
// owning D/32 consecutive head dims: one warp per pair, or, when there are
// few pairs (long contexts, many pieces each), one CTA per pair with the
// warps splitting the pieces and meeting in shared memory.

// Online merge of pieces i = first, first + step, ... < n of one pair into
// (m, wsum, acc), loading kCombineBatch pieces before using any.
template <int D>
__device__ __forceinline__ void merge_pieces(const CombineParams& p, int64_t row0, int64_t rstride,
                                             int n, int first, int step, int lane, float& m,
                                             float& wsum, float (&acc)[D / 32]) {
  constexpr int E = D / 32;
  for (int i0 = first; i0 < n; i0 += kCombineBatch * step) {
    float lse[kCombineBatch];
    float v[kCombineBatch][E];
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const int i = i0 + k * step;
      if (i < n) {
        const int64_t r = i == 0 ? row0 : row0 - p.G + i * rstride;
        lse[k] = p.part_lse[r];
        const float* src = p.part_o + r * D + lane * E;
        if constexpr (E == 4) {
          const float4 x = *reinterpret_cast<const float4*>(src);
          v[k][0] = x.x; v[k][1] = x.y; v[k][2] = x.z; v[k][3] = x.w;
        } else {
          const float2 x = *reinterpret_cast<const float2*>(src);
          v[k][0] = x.x; v[k][1] = x.y;
        }
      } else {
        lse[k] = -INFINITY;
#pragma unroll
        for (int e = 0; e < E; ++e) v[k][e] = 0.f;
      }
    }
    float bm = m;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) bm = fmaxf(bm, lse[k]);
    if (bm == -INFINITY) continue;
    const float a = fast_exp2(m - bm);
    wsum *= a;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] *= a;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const float w = fast_exp2(lse[k] - bm);
      wsum += w;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] += w * v[k][e];
    }
    m = bm;
  }
}

template <int D, bool BF16>
__device__ __forceinline__ void store_out(const CombineParams& p, int b, int h, int lane,
                                          const float (&acc)[D / 32], float wsum) {
  constexpr int E = D / 32;
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint16_t* dst = static_cast<uint16_t*>(p.out) + ((int64_t)b * p.Hq + h) * D + lane * E;
  uint32_t pk[E / 2];
#pragma unroll
  for (int e = 0; e < E / 2; ++e) {
    if constexpr (BF16)
      pk[e] = bf2_as_u32(__floats2bfloat162_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv));
    else
      pk[e] = h2_as_u32(__floats2half2_rn(acc[2 * e] * inv, acc[2 * e + 1] * inv));
  }
  if constexpr (E == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
  else *reinterpret_cast<uint32_t*>(dst) = pk[0];
}
template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineThreads, kCombineMinCtas)
    combine_kernel(const CombineParams p) {
  constexpr int E = D / 32;                      // dims per lane
  __shared__ int s_prefix[kMaxSeqs];
  __shared__ int s_warp[kCombineWarps];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = p.B;

  // ---- page prefix over sequences (clamped as by the decode kernel) ----
  const int per = (B + kCombineThreads - 1) / kCombineThreads;
  const int b0 = tid * per, b1 = min(B, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) {
    int L = __ldg(&p.context_lens[b]);
    L = L < 0 ? 0 : (L > p.max_tok ? p.max_tok : L);
    sum += (L + kBlockSize - 1) / kBlockSize;
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int run = incl - sum, T = 0;
  for (int w = 0; w < kCombineWarps; ++w) {
    if (w < warp) run += s_warp[w];
    T += s_warp[w];
  }
  for (int b = b0; b < b1; ++b) {
    int L = __ldg(&p.context_lens[b]);
    L = L < 0 ? 0 : (L > p.max_tok ? p.max_tok : L);
    run += (L + kBlockSize - 1) / kBlockSize;
    s_prefix[b] = run;
  }
  int R = p.R;
  if (R == 0) {
    const int64_t even = ((int64_t)T + p.groups - 1) / p.groups;
    R = (int)(even > kMinRangePages ? even : kMinRangePages);
  }
  __syncthreads();
  griddep_wait();               // the decode grid's partials are complete and visible

  const int pairs = B * p.Hq;
  if (!p.per_cta) {
    for (int pair = blockIdx.x * kCombineWarps + warp; pair < pairs;
         pair += gridDim.x * kCombineWarps) {
      const int b = pair / p.Hq, h = pair - b * p.Hq;
      const int first = b > 0 ? s_prefix[b - 1] : 0;
      const int pages = s_prefix[b] - first;
      if (pages == 0) continue;
      const int c0 = first / R, c1 = (first + pages - 1) / R;
      const int n = c1 - c0 + 1;
      if (n <= 1) continue;
      const int j = h / p.G, g = h - j * p.G;
      // piece i -> partial row (2 ((c0 + i) Hkv + j) + slot) G + g, slot 1 for i == 0
      const int64_t row0 = (2 * ((int64_t)c0 * p.Hkv + j) + 1) * p.G + g;
      float m = -INFINITY, wsum = 0.f, acc[E];
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = 0.f;
      merge_pieces<D>(p, row0, 2 * (int64_t)p.Hkv * p.G, n, 0, 1, lane, m, wsum, acc);
      store_out<D, BF16>(p, b, h, lane, acc, wsum);
    }
    return;
  }
  __shared__ float s_m[kCombineWarps], s_w[kCombineWarps];
  __shared__ float s_acc[kCombineWarps][D];
  for (int pair = blockIdx.x; pair < pairs; pair += gridDim.x) {
    const int b = pair / p.Hq, h = pair - b * p.Hq;
    const int first = b > 0 ? s_prefix[b - 1] : 0;
    const int pages = s_prefix[b] - first;
    if (pages == 0) continue;                          // uniform over the CTA
    const int c0 = first / R, c1 = (first + pages - 1) / R;
    const int n = c1 - c0 + 1;
    if (n <= 1) continue;
    const int j = h / p.G, g = h - j * p.G;
    const int64_t row0 = (2 * ((int64_t)c0 * p.Hkv + j) + 1) * p.G + g;
    float m = -INFINITY, wsum = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    merge_pieces<D>(p, row0, 2 * (int64_t)p.Hkv * p.G, n, warp, kCombineWarps, lane, m, wsum,
                    acc);
#pragma unroll
    for (int e = 0; e < E; ++e) s_acc[warp][lane * E + e] = acc[e];
    if (lane == 0) {
      s_m[warp] = m;
      s_w[warp] = wsum;
    }
    __syncthreads();
    if (warp == 0) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, s_m[w]);
      float o[E], ws = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) o[e] = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kCombineWarps; ++w) {
          const float a = s_m[w] == -INFINITY ? 0.f : fast_exp2(s_m[w] - M);
          ws += a * s_w[w];
#pragma unroll
          for (int e = 0; e < E; ++e) o[e] += a * s_acc[w][lane * E + e];
        }
      }
      store_out<D, BF16>(p, b, h, lane, o, ws);
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, int sms, cudaStream_t s) {
  if (p.B == 0 || p.Hq == 0) return cudaSuccess;
  const int64_t pairs = (int64_t)p.B * p.Hq;
  const int64_t want = p.per_cta ? pairs : (pairs + kCombineWarps - 1) / kCombineWarps;
  const int64_t cap = 2 * kCombineMinCtas * (int64_t)sms;   // two waves at most
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(want < cap ? want : cap));
  cfg.blockDim = dim3(kCombineThreads);
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
