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

constexpr int kCombineThreads = 256;
constexpr int kCombineBatch = 8;   // pieces a thread loads before using any

// One CTA per (query head, sequence).  Thread t owns 4 consecutive head dims
// (column group t % (D/4)) of every ROWS-th piece, ROWS = 256 / (D/4); it
// loads a batch of pieces at once, keeps its own running (max, sum, acc), and
// the row groups meet in shared memory with the usual rescaling.
template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  constexpr int COLS = D / 4;                      // float4 columns per row
  constexpr int ROWS = kCombineThreads / COLS;     // pieces in flight per pass
  __shared__ float s_m[ROWS], s_w[ROWS];
  __shared__ float4 s_acc[ROWS][COLS];
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int col = tid % COLS, row = tid / COLS;
  griddep_wait();               // the decode grid's partials are complete and visible
  const int pg0 = b > 0 ? p.prefix[b - 1] : 0;
  const int pages = p.prefix[b] - pg0;
  const int64_t R = *p.range;
  if (pages == 0 || R <= 0) return;
  const int j = h / p.G, g = h - j * p.G;
  const int64_t c0 = pg0 / R, c1 = (pg0 + pages - 1) / R;   // columns [pg0, pg0 + pages)
  const int n = (int)(c1 - c0 + 1);
  if (n <= 1) return;
  // piece i -> partial row (2 ((c0 + i) Hkv + j) + slot) G + g, slot 1 for i == 0
  const int64_t row0 = (2 * (c0 * p.Hkv + j) + 1) * p.G + g;
  const int64_t rstride = 2 * (int64_t)p.Hkv * p.G;

  float m = -INFINITY, wsum = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int i0 = row; i0 < n; i0 += ROWS * kCombineBatch) {
    float lse[kCombineBatch];
    float4 v[kCombineBatch];
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const int i = i0 + k * ROWS;
      if (i < n) {
        const int64_t r = i == 0 ? row0 : row0 - p.G + i * rstride;
        lse[k] = p.part_lse[r];
        v[k] = reinterpret_cast<const float4*>(p.part_o + r * D)[col];
      } else {
        lse[k] = -INFINITY;
        v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float bm = m;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) bm = fmaxf(bm, lse[k]);
    if (bm == -INFINITY) continue;
    const float a = fast_exp2(m - bm);
    wsum *= a;
    acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
#pragma unroll
    for (int k = 0; k < kCombineBatch; ++k) {
      const float w = fast_exp2(lse[k] - bm);
      wsum += w;
      acc.x += w * v[k].x; acc.y += w * v[k].y; acc.z += w * v[k].z; acc.w += w * v[k].w;
    }
    m = bm;
  }
  s_acc[row][col] = acc;
  if (col == 0) {
    s_m[row] = m;
    s_w[row] = wsum;
  }
  __syncthreads();
  if (row == 0) {
    float M = -INFINITY;
#pragma unroll
    for (int r = 0; r < ROWS; ++r) M = fmaxf(M, s_m[r]);
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    float ws = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int r = 0; r < ROWS; ++r) {
        const float a = s_m[r] == -INFINITY ? 0.f : fast_exp2(s_m[r] - M);
        const float4 x = s_acc[r][col];
        ws += a * s_w[r];
        o.x += a * x.x; o.y += a * x.y; o.z += a * x.z; o.w += a * x.w;
      }
    }
    const float inv = ws > 0.f ? 1.f / ws : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.out) + ((int64_t)b * p.Hq + h) * D + 4 * col;
    uint2 out;
    if constexpr (BF16) {
      out.x = bf2_as_u32(__floats2bfloat162_rn(o.x * inv, o.y * inv));
      out.y = bf2_as_u32(__floats2bfloat162_rn(o.z * inv, o.w * inv));
    } else {
      out.x = h2_as_u32(__floats2half2_rn(o.x * inv, o.y * inv));
      out.y = h2_as_u32(__floats2half2_rn(o.z * inv, o.w * inv));
    }
    *reinterpret_cast<uint2*>(dst) = out;
  }
}

}  // namespace

cudaError_t combine_launch(int D, bool bf16, const CombineParams& p, cudaStream_t s) {
  if (p.B == 0 || p.Hq == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.Hq, p.B);
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
