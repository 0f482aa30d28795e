// Front trim that keeps the attention sink, on the paged INT8 cache.
//
// "fix(cuda/kv): correct Int8 KV per-token scale ..." (mlxcel PR #717),
// follow-up commit, "The fix": a sequence of L tokens becomes [its first keep
// tokens] ++ [the tokens after the next n], exactly n removed, the INT8
// payload and its scale rows moved in lockstep; keep = 0 is the plain front
// trim.  keep and n are clamped to the sequence (keep <= L, n <= L - keep).
//
// In place: token keep + n + i moves to keep + i (i < L - keep - n), read and
// written through the block table.  One CTA per (KV head, sequence) moves
// its tiles' rows in chunks, each chunk fully staged in shared memory before
// it is written; the writes of a chunk land below the sources of every later
// chunk, so chunks in order never read overwritten data.  A second kernel
// then sets context_lens[b] = L - n.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kTrimThreads = 256;
constexpr int kTrimChunk = 128;   // tokens staged per step

__device__ __forceinline__ void trim_clamp(const TrimParams& p, int b, int& L, int& keep,
                                           int& n) {
  L = __ldg(&p.context_lens[b]);
  L = L < 0 ? 0 : (L > p.max_tok ? p.max_tok : L);
  keep = p.keep < L ? p.keep : L;
  n = __ldg(&p.trim[b]);
  n = n < 0 ? 0 : (n > L - keep ? L - keep : n);
}

template <int D>
__global__ void __launch_bounds__(kTrimThreads) trim_kernel(const TrimParams p) {
  constexpr int kRowVec = D / 16;                      // 16-byte vectors per token row
  __shared__ uint4 s_k[kTrimChunk * kRowVec], s_v[kTrimChunk * kRowVec];
  __shared__ uint16_t s_ks[kTrimChunk], s_vs[kTrimChunk];
  __shared__ int s_ok[kTrimChunk];
  const int j = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  int L, keep, n;
  trim_clamp(p, b, L, keep, n);
  const int moved = L - keep - n;
  if (n == 0 || moved <= 0) return;
  const bool scales = p.k_scale != nullptr;
  const int32_t* bt = p.block_tables + (int64_t)b * p.max_blocks;
  // row of token t of this (sequence, KV head), or -1 (block id flagged)
  auto row_of = [&](int t) -> int64_t {
    const int blk = __ldg(&bt[t / kBlockSize]);
    if (blk < 0 || blk >= p.num_blocks) {
      atomicOr(p.err, 0x2u);
      return -1;
    }
    return ((int64_t)blk * p.Hkv + j) * kBlockSize + t % kBlockSize;
  };
  for (int s0 = 0; s0 < moved; s0 += kTrimChunk) {
    const int cnt = min(kTrimChunk, moved - s0);
    for (int i = tid; i < cnt; i += kTrimThreads) {
      const int64_t r = row_of(keep + n + s0 + i);
      s_ok[i] = r >= 0;
      if (r >= 0 && scales) {
        s_ks[i] = p.k_scale[r];
        s_vs[i] = p.v_scale[r];
      }
    }
    __syncthreads();
    for (int e = tid; e < cnt * kRowVec; e += kTrimThreads) {
      const int i = e / kRowVec, c = e - i * kRowVec;
      if (!s_ok[i]) continue;
      const int t = keep + n + s0 + i;
      const int64_t r = ((int64_t)__ldg(&bt[t / kBlockSize]) * p.Hkv + j) * kBlockSize +
                        t % kBlockSize;
      s_k[e] = reinterpret_cast<const uint4*>(p.k_cache + r * D)[c];
      s_v[e] = reinterpret_cast<const uint4*>(p.v_cache + r * D)[c];
    }
    __syncthreads();
    for (int e = tid; e < cnt * kRowVec; e += kTrimThreads) {
      const int i = e / kRowVec, c = e - i * kRowVec;
      if (!s_ok[i]) continue;
      const int64_t r = row_of(keep + s0 + i);
      if (r < 0) continue;
      reinterpret_cast<uint4*>(p.k_cache + r * D)[c] = s_k[e];
      reinterpret_cast<uint4*>(p.v_cache + r * D)[c] = s_v[e];
      if (c == 0 && scales) {
        p.k_scale[r] = s_ks[i];
        p.v_scale[r] = s_vs[i];
      }
    }
    __syncthreads();
  }
}

__global__ void trim_lens_kernel(const TrimParams p, int32_t* context_lens) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= p.B) return;
  int L, keep, n;
  trim_clamp(p, b, L, keep, n);
  if (n > 0) context_lens[b] = L - n;
}

}  // namespace

cudaError_t trim_launch(int D, const TrimParams& p, int32_t* context_lens, cudaStream_t s) {
  if (p.B == 0) return cudaSuccess;
  const dim3 grid((unsigned)p.Hkv, (unsigned)p.B);
  if (D == 128) trim_kernel<128><<<grid, kTrimThreads, 0, s>>>(p);
  else trim_kernel<64><<<grid, kTrimThreads, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  trim_lens_kernel<<<(p.B + 255) / 256, 256, 0, s>>>(p, context_lens);
  return cudaGetLastError();
}

}  // namespace kvq
