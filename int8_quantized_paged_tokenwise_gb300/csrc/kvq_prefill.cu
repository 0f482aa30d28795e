// Chunked-prefill attention over the tokenwise INT8 paged cache.
//
// What it computes ("fix(cuda/kv): correct Int8 KV per-token scale ..."
// (mlxcel PR #717), "Server integration": Int8 chunked prefill + decode over
// the same cache): sequence b holds L tokens, the last n of them being this
// chunk's queries (already quantized into the cache); query i at position
// p = L - n + i attends causally to tokens 0..p:
//   out[i][h] = softmax_{t<=p}(sm_scale * q[i][h] . s_k[t] code_k[t]) . (s_v code_v)
//
// A real dense contraction, so the whole tile works on the tensor cores:
//  * CTA = (query tile, KV head, sequence); its 64 rows are (query, head of
//    the GQA group) pairs, 16 per warp, so each K/V page is read once for all
//    of them.  The Q tile is converted to FP16 once and its MMA A fragments
//    stay in registers.
//  * pages stream through an S-stage ring shared by the CTA's 4 warps: warp 0
//    issues the TMA copies (K and V tiles, 128/64-byte swizzle) and the two
//    32-byte scale rows, all completing on the stage's mbarrier; a block
//    barrier per page frees the stage.
//  * S = Q K^T with K as the B operand: codes become exact FP16 integers in
//    registers (byte permute under exponent 0x64, minus 1152); the head dims
//    are taken in the order {4c, 4c+1, 4c+2, 4c+3} <-> MMA k {2c, 2c+1, 2c+8,
//    2c+9} on both operands, so each ldmatrix word is one B fragment pair.
//  * K scales and sm_scale*log2(e) scale the FP32 scores; causal mask; online
//    softmax per row (quad shuffles); P stays in registers as the A operand of
//    P V; V pairs of consecutive tokens come from ldmatrix.trans, multiplied by
//    their V scales; O accumulates in FP32.
#include "kvq_decode.cuh"

namespace kvq {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfThreads = kPfWarps * 32;
constexpr int kPfRows = 16 * kPfWarps;   // (query, head) rows per CTA
constexpr int kPfStages = 4;

template <int D>
struct PfLayout {
  using C = TileCfg<D, true>;
  static constexpr int kQStride = D * 2 + 32;               // bytes per Q row (padded)
  static constexpr int kStage = 2 * C::kTile;               // K tile, V tile
  static constexpr size_t kTiles = 0;
  static constexpr size_t kScales = kTiles + (size_t)kPfStages * kStage;
  static constexpr size_t kQ = kScales + (size_t)kPfStages * 64;
  static constexpr size_t kBars = kQ + (size_t)kPfRows * kQStride;
  static constexpr size_t kTotal = kBars + kPfStages * 8 + 1024;   // + base alignment slack
};

template <int D, bool BF16>
__global__ void __launch_bounds__(kPfThreads, 2)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = TileCfg<D, true>;
  using Ly = PfLayout<D>;
  constexpr int KSTEPS = D / 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBars);
  __shared__ int s_blk[kPfStages];               // block id of the page in each stage (-1: none)
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int b = blockIdx.z, j = blockIdx.y, G = p.G;
  const int TQ = kPfRows / G;                     // queries per tile
  const int qt = blockIdx.x;

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (tid < kPfStages) mbar_init(smem_u32(&bars[tid]), 1);
  griddep_wait();
  fence_mbar_init();

  const int q0 = __ldg(&p.query_start[b]);
  const int n = __ldg(&p.query_start[b + 1]) - q0;
  int L = __ldg(&p.context_lens[b]);
  const int max_tok = min(p.max_blocks * kBlockSize, p.max_ctx);
  if (L < 0 || L > max_tok || n < 0 || n > L || n > p.max_q || q0 < 0 || q0 + n > p.total_q) {
    if (tid == 0 && qt == 0 && j == 0) atomicOr(p.err, 0x4u);
    return;                                      // no copies issued yet
  }
  const int i_begin = qt * TQ;
  if (i_begin >= n) return;
  const int i_end = min(n, i_begin + TQ);
  const int p_last = L - n + i_end - 1;          // last query position of the tile
  const int npages = p_last / kBlockSize + 1;

  // ---- Q tile: rows r = (query i_begin + r / G, head j*G + r % G), as FP16 ----
  uint8_t* qs = smem + Ly::kQ;
  for (int e = tid; e < kPfRows * (D / 4); e += kPfThreads) {
    const int r = e / (D / 4), d4 = e - r * (D / 4);
    const int i = i_begin + r / G;
    uint2 v = make_uint2(0, 0);
    if (r < TQ * G && i < i_end) {
      const uint16_t* src = static_cast<const uint16_t*>(p.q) +
                            ((int64_t)(q0 + i) * p.Hq + (int64_t)j * G + r % G) * D + 4 * d4;
      v = __ldg(reinterpret_cast<const uint2*>(src));
      if constexpr (BF16) {
        v.x = h2_as_u32(__floats2half2_rn(__uint_as_float(v.x << 16),
                                          __uint_as_float(v.x & 0xFFFF0000u)));
        v.y = h2_as_u32(__floats2half2_rn(__uint_as_float(v.y << 16),
                                          __uint_as_float(v.y & 0xFFFF0000u)));
      }
    }
    *reinterpret_cast<uint2*>(qs + r * Ly::kQStride + 8 * d4) = v;
  }
  __syncthreads();
  // A fragments of this warp's 16 rows: per k-step, rows g / g+8, 8 bytes at d = 16ks + 4c
  uint32_t qa[KSTEPS][4];
  {
    const uint8_t* r0 = qs + (16 * warp + g) * Ly::kQStride;
    const uint8_t* r8 = r0 + 8 * Ly::kQStride;
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks) {
      const uint2 lo = *reinterpret_cast<const uint2*>(r0 + 32 * ks + 8 * c);
      const uint2 hi = *reinterpret_cast<const uint2*>(r8 + 32 * ks + 8 * c);
      qa[ks][0] = lo.x;   // row g,   k {2c, 2c+1}
      qa[ks][1] = hi.x;   // row g+8
      qa[ks][2] = lo.y;   // row g,   k {2c+8, 2c+9}
      qa[ks][3] = hi.y;   // row g+8
    }
  }
  // positions of the thread's two rows (-1: padding row, attends nothing)
  int pos[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int r = 16 * warp + g + 8 * h;
    const int i = i_begin + r / G;
    pos[h] = (r < TQ * G && i < i_end) ? L - n + i : -1;
  }

  // ---- producer (warp 0): block ids 32 pages at a time, copies by lanes 0..3 ----
  const uint32_t tiles_u32 = smem_u32(smem + Ly::kTiles);
  const uint32_t scales_u32 = smem_u32(smem + Ly::kScales);
  const int32_t* bt = p.block_tables + (int64_t)b * p.max_blocks;
  int blk_chunk = -1, chunk_base = -32;
  auto issue = [&](int k) {                      // warp 0 only; page k into stage k % S
    // (s_blk is written before the arrive, which releases it to the waiting warps)
    if (k >= chunk_base + 32) {
      chunk_base = k - k % 32;
      const int pg = chunk_base + lane;
      blk_chunk = -1;
      if (pg < npages) {
        blk_chunk = __ldg(&bt[pg]);
        if (blk_chunk < 0 || blk_chunk >= p.num_blocks) {
          atomicOr(p.err, 0x2u);
          blk_chunk = -1;
        }
      }
    }
    const int blk = __shfl_sync(0xFFFFFFFFu, blk_chunk, k - chunk_base);
    const int s = k % kPfStages;
    const uint32_t bar = smem_u32(&bars[s]);
    if (lane == 0) {
      s_blk[s] = blk;
      if (blk >= 0) mbar_arrive_expect_tx(bar, 2 * C::kTile + 64);
      else mbar_arrive(bar);
    }
    if (blk >= 0) {
      const int row = (blk * p.Hkv + j) * kBlockSize;
      const int64_t srow = (int64_t)(blk * p.Hkv + j) * kBlockSize;
      if (lane == 0) tma_load_2d(tiles_u32 + s * Ly::kStage, &tmK, 0, row, bar);
      else if (lane == 1) tma_load_2d(tiles_u32 + s * Ly::kStage + C::kTile, &tmV, 0, row, bar);
      else if (lane == 2) bulk_load(scales_u32 + s * 64, p.k_scale + srow, 32, bar);
      else if (lane == 3) bulk_load(scales_u32 + s * 64 + 32, p.v_scale + srow, 32, bar);
    }
  };
  int k_next = 0;                                // next page to issue (warp 0)
  if (warp == 0)
    for (; k_next < kPfStages && k_next < npages; ++k_next) issue(k_next);

  // ---- consumer: all warps ----
  float o[D / 16][2][4];                          // [16-dim block][even/odd dims][quad]
#pragma unroll
  for (int cb = 0; cb < D / 16; ++cb)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int x = 0; x < 4; ++x) o[cb][e][x] = 0.f;
  float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
  const int lt = (lane & 7) + ((lane >> 3) & 1) * 8;
  bool aborted = false;
  int k = 0;
  for (; k < npages; ++k) {
    const int s = k % kPfStages;
    if (!mbar_wait_bounded(smem_u32(&bars[s]), (k / kPfStages) & 1)) aborted = true;
    if (!aborted && s_blk[s] >= 0) {
      const uint32_t kt = tiles_u32 + s * Ly::kStage, vt = kt + C::kTile;
      const uint16_t* sc = reinterpret_cast<const uint16_t*>(smem + Ly::kScales + s * 64);
      // ---------- S = Q K^T: n-tile 0 = tokens 0-7, n-tile 1 = tokens 8-15 ----------
      float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < KSTEPS / 2; ++kk) {
        uint32_t r0, r1, r2, r3;   // (tok 0-7, k-step 2kk), (8-15, 2kk), (0-7, 2kk+1), (8-15, 2kk+1)
        ldsm_x4(kt + tile_off<C>(lt, 2 * kk + (lane >> 4)), r0, r1, r2, r3);
        uint32_t b0, b1;
        i8x4_to_h2x2<0x4140u, 0x4342u>(r0, b0, b1);
        mma_16816_acc<false>(s0, qa[2 * kk][0], qa[2 * kk][1], qa[2 * kk][2], qa[2 * kk][3], b0, b1);
        i8x4_to_h2x2<0x4140u, 0x4342u>(r1, b0, b1);
        mma_16816_acc<false>(s1, qa[2 * kk][0], qa[2 * kk][1], qa[2 * kk][2], qa[2 * kk][3], b0, b1);
        i8x4_to_h2x2<0x4140u, 0x4342u>(r2, b0, b1);
        mma_16816_acc<false>(s0, qa[2 * kk + 1][0], qa[2 * kk + 1][1], qa[2 * kk + 1][2],
                             qa[2 * kk + 1][3], b0, b1);
        i8x4_to_h2x2<0x4140u, 0x4342u>(r3, b0, b1);
        mma_16816_acc<false>(s1, qa[2 * kk + 1][0], qa[2 * kk + 1][1], qa[2 * kk + 1][2],
                             qa[2 * kk + 1][3], b0, b1);
      }
      // scores in log2 units; the thread's tokens: 2c, 2c+1 (s0) and 8+2c, 9+2c (s1)
      const int t0 = k * kBlockSize;
      float z[2][4];                              // [row g / g+8][tok 2c, 2c+1, 8+2c, 9+2c]
#pragma unroll
      for (int x = 0; x < 4; ++x) {
        const int tok = (x < 2 ? 2 * c + x : 8 + 2 * c + (x - 2));
        const float ks = p.scale_log2 * __half2float(__ushort_as_half(sc[tok]));
        const float v0 = x < 2 ? s0[x] : s1[x - 2];
        const float v8 = x < 2 ? s0[2 + x] : s1[x];
        z[0][x] = t0 + tok <= pos[0] ? v0 * ks : -INFINITY;
        z[1][x] = t0 + tok <= pos[1] ? v8 * ks : -INFINITY;
      }
      // ---------- online softmax per row (reduce over the quad) ----------
      uint32_t pa[4];                             // A fragments of P (16 rows x 16 tokens)
      float alpha[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = fmaxf(fmaxf(z[h][0], z[h][1]), fmaxf(z[h][2], z[h][3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float mn = fmaxf(m[h], mx);
        const float ref = mn == -INFINITY ? 0.f : mn;
        alpha[h] = fast_exp2(m[h] - ref);
        float pr[4];
#pragma unroll
        for (int x = 0; x < 4; ++x) pr[x] = fast_exp2(z[h][x] - ref);
        l[h] = l[h] * alpha[h] + (pr[0] + pr[1] + pr[2] + pr[3]);
        m[h] = mn;
        // a0 / a1: rows g / g+8, tokens 2c, 2c+1; a2 / a3: tokens 8+2c, 9+2c
        pa[h] = h2_as_u32(__floats2half2_rn(pr[0], pr[1]));
        pa[2 + h] = h2_as_u32(__floats2half2_rn(pr[2], pr[3]));
      }
      if (__any_sync(0xFFFFFFFFu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            o[cb][e][0] *= alpha[0];
            o[cb][e][1] *= alpha[0];
            o[cb][e][2] *= alpha[1];
            o[cb][e][3] *= alpha[1];
          }
      }
      // ---------- O += P V: V pairs of tokens per head dim, times V scales ----------
      const uint32_t* vsc = reinterpret_cast<const uint32_t*>(sc + kBlockSize);
      const __half2 vs01 = u32_as_h2(vsc[c]), vs89 = u32_as_h2(vsc[4 + c]);
#pragma unroll
      for (int kk = 0; kk < KSTEPS / 2; ++kk) {
        uint32_t r[4];
        ldsm_x4_trans(vt + tile_off<C>(lt, 2 * kk + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // r[2hh]: tokens 2c, 2c+1; r[2hh+1]: tokens 8+2c, 9+2c; at dims
          // d0 = 16cb + 2g (even n-tile) and d0 + 1 (odd n-tile)
          uint32_t ev0, od0, ev1, od1;
          i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * hh], ev0, od0);
          i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * hh + 1], ev1, od1);
          ev0 = h2_as_u32(__hmul2(u32_as_h2(ev0), vs01));
          od0 = h2_as_u32(__hmul2(u32_as_h2(od0), vs01));
          ev1 = h2_as_u32(__hmul2(u32_as_h2(ev1), vs89));
          od1 = h2_as_u32(__hmul2(u32_as_h2(od1), vs89));
          const int cb = 2 * kk + hh;
          mma_16816_acc<false>(o[cb][0], pa[0], pa[1], pa[2], pa[3], ev0, ev1);
          mma_16816_acc<false>(o[cb][1], pa[0], pa[1], pa[2], pa[3], od0, od1);
        }
      }
    }
    // stage s consumed by every warp (and a timed-out wait anywhere stops all)
    if (__syncthreads_or(aborted)) {
      aborted = true;
      break;
    }
    if (warp == 0 && k_next < npages) issue(k_next++);
  }

  if (aborted) {
    // a wait gave up: record it, then wait (bounded) for the copies still in
    // flight (pages k .. k_next-1, known to warp 0) so none lands after exit
    if (warp == 0) {
      if (lane == 0) atomicOr(p.err, 0x8u);
      for (int kp = k; kp < k_next; ++kp)
        mbar_wait_bounded(smem_u32(&bars[kp % kPfStages]), (kp / kPfStages) & 1);
    }
    return;
  }
  // ---------- finalize: rows g and g+8; dims 16cb + 4c + {0, 1, 2, 3} ----------
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    l[h] += __shfl_xor_sync(0xFFFFFFFFu, l[h], 1);
    l[h] += __shfl_xor_sync(0xFFFFFFFFu, l[h], 2);
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (pos[h] < 0) continue;
    const int r = 16 * warp + g + 8 * h;
    const int i = i_begin + r / G;
    const float inv = l[h] > 0.f ? 1.f / l[h] : 0.f;
    uint16_t* dst = static_cast<uint16_t*>(p.out) +
                    ((int64_t)(q0 + i) * p.Hq + (int64_t)j * G + r % G) * D + 4 * c;
#pragma unroll
    for (int cb = 0; cb < D / 16; ++cb) {
      const float a = o[cb][0][2 * h] * inv, bq = o[cb][1][2 * h] * inv;
      const float c2 = o[cb][0][2 * h + 1] * inv, d2 = o[cb][1][2 * h + 1] * inv;
      uint2 w;
      if constexpr (BF16) {
        w.x = bf2_as_u32(__floats2bfloat162_rn(a, bq));
        w.y = bf2_as_u32(__floats2bfloat162_rn(c2, d2));
      } else {
        w.x = h2_as_u32(__floats2half2_rn(a, bq));
        w.y = h2_as_u32(__floats2half2_rn(c2, d2));
      }
      *reinterpret_cast<uint2*>(dst + 16 * cb) = w;
    }
  }
}

template <int D, bool BF16>
const void* pf_ptr() {
  return reinterpret_cast<const void*>(&paged_prefill_kernel<D, BF16>);
}
const void* pf_pick(int D, bool bf16) {
  if (D == 128) return bf16 ? pf_ptr<128, true>() : pf_ptr<128, false>();
  return bf16 ? pf_ptr<64, true>() : pf_ptr<64, false>();
}

}  // namespace

size_t prefill_smem_bytes(int D) {
  return D == 128 ? PfLayout<128>::kTotal : PfLayout<64>::kTotal;
}

cudaError_t prefill_configure(int D, bool bf16) {
  return cudaFuncSetAttribute(pf_pick(D, bf16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)prefill_smem_bytes(D));
}

cudaError_t prefill_launch(int D, bool bf16, const CUtensorMap* maps, const PrefillParams& p,
                           int tiles, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)p.Hkv, (unsigned)p.B);
  cfg.blockDim = dim3(kPfThreads);
  cfg.dynamicSmemBytes = prefill_smem_bytes(D);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) {
    return bf16 ? cudaLaunchKernelEx(&cfg, paged_prefill_kernel<128, true>, maps[0], maps[1], p)
                : cudaLaunchKernelEx(&cfg, paged_prefill_kernel<128, false>, maps[0], maps[1], p);
  }
  return bf16 ? cudaLaunchKernelEx(&cfg, paged_prefill_kernel<64, true>, maps[0], maps[1], p)
              : cudaLaunchKernelEx(&cfg, paged_prefill_kernel<64, false>, maps[0], maps[1], p);
}

}  // namespace kvq
