// Fused paged decode attention for sm_103a, over the tokenwise INT8 cache
// (codes + FP16 scale planes) or over a native 16-bit cache (the A/B twin).
//
// What it computes ("feat: opt-in INT8 KV-cache quantization", MoE-Infinity
// PR #183, "What landed"): for sequence b, query head h (KV head j = h / G),
//   z_t = sm_scale * <q, s_k[t] * code_k[t]>,  out = softmax(z) . (s_v * code_v)
// over the b's L tokens, read page by page through the block table, with the
// codes dequantized in registers and FP32 accumulation.  The online softmax
// and the split into partitions with a log-sum-exp combine are the
// flash-decoding formulation of the same sum.
//
// Structure (one CTA = 4 warps, persistent over a flat list of work items):
//  * work item = (sequence-partition, KV head); a sequence of L tokens has
//    max(1, ceil(ceil(L/16) / P)) partitions of P pages.  Every CTA rebuilds
//    the partition prefix from context_lens in shared memory and strides over
//    the items, so skewed context lengths need no host-side planning.
//  * each warp owns every 4th page of the item and a private ring of S
//    stages; lane 0 streams its pages with TMA: the K and V tiles of the
//    (page, KV head) as 2-D tensor copies with the 128-/64-byte swizzle (so
//    that the ldmatrix reads below are bank-conflict free) and, for INT8, the
//    two 32-byte scale rows as 1-D bulk copies, all completing on one
//    mbarrier.  Waits are bounded (error bit + clean exit on timeout).
//  * QK^T and PV run on the tensor cores (mma.sync m16n8k16, FP32 accumulate)
//    with the GQA group as the M dimension (padded to 16) so each page is
//    read once for all query heads of its KV head.  INT8 codes become exact
//    FP16 integers with two byte permutes and one subtraction; K scales
//    multiply the FP32 scores, V scales multiply the converted V pairs.
//  * at the end of an item the warps merge (m, l, O) through shared memory
//    and write either the final output or a normalized partial + log2-sum-exp
//    for the combine kernel.
#pragma once

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {

template <int D, bool INT8>
struct TileCfg {
  static constexpr int kElem = INT8 ? 1 : 2;                 // bytes per cache element
  static constexpr int kRowBytes = D * kElem;                // bytes per token row
  static constexpr int kSubRow = kRowBytes < 128 ? kRowBytes : 128;   // TMA box row bytes
  static constexpr int kSubTiles = kRowBytes / kSubRow;       // TMA copies per tile
  static constexpr int kSubBytes = kBlockSize * kSubRow;
  static constexpr int kTile = kBlockSize * kRowBytes;        // bytes of one K (or V) tile
  static constexpr int kStages = INT8 ? 3 : 2;
  static constexpr int kStageBytes = 2 * kTile;               // K tile then V tile
  static constexpr int kScaleBytes = INT8 ? 2 * kBlockSize * 2 : 0;  // K then V scale rows
  static constexpr uint32_t kTxBytes = 2 * kTile + kScaleBytes;
  static constexpr int kChunks = kRowBytes / 16;              // 16-byte chunks per row
  static constexpr uint32_t kSwzMask = kSubRow == 128 ? 0x70u : 0x30u;
  static constexpr int kMinCtas = (INT8 && D == 64) ? 4 : 3;   // 170-register cap otherwise
};

// Byte offset inside a (K or V) tile of 16-byte chunk `c` of token row `t`,
// with the TMA swizzle applied (16-byte chunk index XOR row bits).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
  constexpr int cps = C::kSubRow / 16;  // chunks per sub-tile row
  const uint32_t off = (uint32_t)((c / cps) * C::kSubBytes + t * C::kSubRow + (c % cps) * 16);
  return off ^ ((off >> 3) & C::kSwzMask);
}

template <int D, bool INT8>
__host__ __device__ constexpr size_t decode_smem_layout_tiles() {
  return (size_t)kWarps * TileCfg<D, INT8>::kStages * TileCfg<D, INT8>::kStageBytes;
}

// Shared-memory carve-up (offsets from a 1024-aligned base).
template <int D, bool INT8>
struct SmemLayout {
  using C = TileCfg<D, INT8>;
  static constexpr size_t kTiles = 0;
  static constexpr size_t kTilesBytes = decode_smem_layout_tiles<D, INT8>();
  static constexpr size_t kScales = kTiles + kTilesBytes;
  static constexpr size_t kScalesBytes = (size_t)kWarps * C::kStages * C::kScaleBytes;
  static constexpr size_t kBars = (kScales + kScalesBytes + 15) & ~(size_t)15;
  static constexpr size_t kBarsBytes = (size_t)kWarps * C::kStages * 8;
  static constexpr size_t kStats = kBars + kBarsBytes;           // m, l per warp and head
  static constexpr size_t kStatsBytes = (size_t)2 * kWarps * kMaxGroup * 4;
  static constexpr size_t kMisc = kStats + kStatsBytes;          // abort flag + pad
  static constexpr size_t kBlk = kMisc + 16;                     // int32 [P]
  // the merge buffer [W][G][D] float reuses the tile region
  static_assert((size_t)kWarps * kMaxGroup * D * 4 <= kTilesBytes, "merge must fit");
  __host__ __device__ static size_t prefix_off(int P) { return kBlk + (size_t)P * 4; }
  __host__ __device__ static size_t total(int B, int P) { return prefix_off(P) + (size_t)B * 4 + 1024; }
};

template <bool BF16>
__device__ __forceinline__ void store_out4(void* out, int64_t idx, float a, float b, float c,
                                           float d) {
  uint2 v;
  if constexpr (BF16) {
    v.x = bf2_as_u32(__floats2bfloat162_rn(a, b));
    v.y = bf2_as_u32(__floats2bfloat162_rn(c, d));
  } else {
    v.x = h2_as_u32(__floats2half2_rn(a, b));
    v.y = h2_as_u32(__floats2half2_rn(c, d));
  }
  *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + idx) = v;
}

// INT8: QBF16 = activations are bf16 (converted to FP16 for the tensor cores);
// twin: QBF16 selects the bf16 MMA, otherwise FP16.
template <int D, bool INT8, bool QBF16>
__global__ void __launch_bounds__(kThreads, TileCfg<D, INT8>::kMinCtas)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = TileCfg<D, INT8>;
  using Lay = SmemLayout<D, INT8>;
  constexpr bool MMA_BF16 = (!INT8) && QBF16;
  constexpr int S = C::kStages;
  constexpr int KSTEPS = D / 16;       // MMA k-steps over the head dim
  constexpr int NOUT = D / 4;          // output floats per thread (one head)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint8_t* tiles = smem + Lay::kTiles;
  uint16_t* scales = reinterpret_cast<uint16_t*>(smem + Lay::kScales);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBars);
  float* st_m = reinterpret_cast<float*>(smem + Lay::kStats);
  float* st_l = st_m + kWarps * kMaxGroup;
  int* abort_flag = reinterpret_cast<int*>(smem + Lay::kMisc);
  int* blk_s = reinterpret_cast<int*>(smem + Lay::kBlk);
  int* prefix = reinterpret_cast<int*>(smem + Lay::prefix_off(p.P));
  float* merge = reinterpret_cast<float*>(tiles);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;   // MMA fragment coordinates
  const int B = p.B, Hkv = p.Hkv, G = p.G, P = p.P;
  // tokens any sequence may have: the table row and the host's bound (which
  // sized the workspace); a larger context_lens entry is flagged and clamped
  const int max_tok = min(p.max_blocks * kBlockSize, p.max_ctx);

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    *abort_flag = 0;
  }
  if (tid < kWarps * S) mbar_init(smem_u32(&bars[tid]), 1);

  // ---- partition prefix over sequences (inclusive), built by every CTA ----
  {
    auto parts_of = [&](int b, bool flag) {
      int L = __ldg(&p.context_lens[b]);
      if (L < 0 || L > max_tok) {
        if (flag) atomicOr(p.err, 0x4u);
        L = L < 0 ? 0 : max_tok;
      }
      const int pages = (L + kBlockSize - 1) / kBlockSize;
      return max(1, (pages + P - 1) / P);
    };
    const int per = (B + kThreads - 1) / kThreads;   // consecutive sequences per thread
    const int b0 = tid * per, b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) sum += parts_of(b, true);
    int incl = sum;                                  // block-wide scan of per-thread sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    int* wsum = reinterpret_cast<int*>(st_m);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int b = b0; b < b1; ++b) {
      run += parts_of(b, false);
      prefix[b] = run;
    }
  }
  fence_mbar_init();
  fence_proxy_async_smem();
  __syncthreads();
  if (blockIdx.x == 0 && p.prefix_out != nullptr)
    for (int b = tid; b < B; b += kThreads) p.prefix_out[b] = prefix[b];

  const int total_sp = B > 0 ? prefix[B - 1] : 0;
  const int64_t n_items = (int64_t)total_sp * Hkv;
  uint32_t phase = 0;  // bit s = parity of the next wait on stage s of this warp

  const uint32_t tiles_u32 = smem_u32(tiles);
  const uint32_t scales_u32 = smem_u32(scales);

  for (int64_t item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int sp = (int)(item / Hkv);
    const int j = (int)(item - (int64_t)sp * Hkv);
    // sequence = first b with prefix[b] > sp
    int lo = 0, hi = B - 1;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (prefix[mid] > sp) hi = mid; else lo = mid + 1;
    }
    const int b = lo;
    const int sp0 = b > 0 ? prefix[b - 1] : 0;
    const int part = sp - sp0;
    const int nparts = prefix[b] - sp0;
    int L = __ldg(&p.context_lens[b]);
    L = L < 0 ? 0 : (L > max_tok ? max_tok : L);
    const int pages_b = (L + kBlockSize - 1) / kBlockSize;
    const int pg0 = part * P;
    const int npg = max(0, min(P, pages_b - pg0));

    __syncthreads();                        // merge buffer of the previous item consumed
    if (*abort_flag) break;
    for (int t = tid; t < npg; t += kThreads) {
      int blk = __ldg(&p.block_tables[(int64_t)b * p.max_blocks + pg0 + t]);
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.err, 0x2u);
        blk = -1;
      }
      blk_s[t] = blk;
    }
    fence_proxy_async_smem();
    __syncthreads();

    // ---- per-warp page stream ----
    const int nk = npg > warp ? (npg - warp + kWarps - 1) / kWarps : 0;
    const int row_base = j * kBlockSize;   // + blk * Hkv * 16
    auto issue = [&](int k) {              // lane 0 only
      const int s = k % S;
      const int lp = warp + k * kWarps;
      const int blk = blk_s[lp];
      const uint32_t bar = smem_u32(&bars[warp * S + s]);
      if (blk < 0) {
        mbar_arrive(bar);
        return;
      }
      mbar_arrive_expect_tx(bar, C::kTxBytes);
      const uint32_t kdst = tiles_u32 + (uint32_t)((warp * S + s) * C::kStageBytes);
      const uint32_t vdst = kdst + C::kTile;
      const int y = blk * Hkv * kBlockSize + row_base;
#pragma unroll
      for (int st = 0; st < C::kSubTiles; ++st) {
        tma_load_2d(kdst + st * C::kSubBytes, &tmK, st * (C::kSubRow / C::kElem), y, bar);
        tma_load_2d(vdst + st * C::kSubBytes, &tmV, st * (C::kSubRow / C::kElem), y, bar);
      }
      if constexpr (INT8) {
        const int64_t srow = ((int64_t)blk * Hkv + j) * kBlockSize;
        const uint32_t sdst = scales_u32 + (uint32_t)((warp * S + s) * C::kScaleBytes);
        bulk_load(sdst, p.k_scale + srow, kBlockSize * 2, bar);
        bulk_load(sdst + kBlockSize * 2, p.v_scale + srow, kBlockSize * 2, bar);
      }
    };
    if (lane == 0)
      for (int k = 0; k < min(S, nk); ++k) issue(k);

    // ---- query fragments (rows g < G of the padded 16-row A operand) ----
    uint32_t qa0[KSTEPS], qa2[KSTEPS];
    {
      const bool has = g < G && nk > 0;
      const uint16_t* qrow =
          static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + (int64_t)j * G + g) * D;
#pragma unroll
      for (int ks = 0; ks < KSTEPS; ++ks) {
        if constexpr (INT8) {
          // logical k {2c,2c+1,2c+8,2c+9} of step ks <-> head-dim 16ks+4c+{0..3}
          uint2 v = has ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * ks + 4 * c))
                        : make_uint2(0, 0);
          if constexpr (QBF16) {
            qa0[ks] = h2_as_u32(__floats2half2_rn(__uint_as_float(v.x << 16),
                                                  __uint_as_float(v.x & 0xFFFF0000u)));
            qa2[ks] = h2_as_u32(__floats2half2_rn(__uint_as_float(v.y << 16),
                                                  __uint_as_float(v.y & 0xFFFF0000u)));
          } else {
            qa0[ks] = v.x;
            qa2[ks] = v.y;
          }
        } else {
          // natural order: k {2c,2c+1} <-> 16ks+2c, k {2c+8,2c+9} <-> 16ks+8+2c
          qa0[ks] = has ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * c)) : 0u;
          qa2[ks] = has ? __ldg(reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * c))
                        : 0u;
        }
      }
    }

    float m_run = -INFINITY, l_run = 0.f;
    float o[NOUT];
#pragma unroll
    for (int i = 0; i < NOUT; ++i) o[i] = 0.f;

    bool timed_out = false;
    int k = 0;
    for (; k < nk; ++k) {
      const int s = k % S;
      const uint32_t bar = smem_u32(&bars[warp * S + s]);
      const uint32_t par = (phase >> s) & 1u;
      if (!mbar_wait_bounded(bar, par)) {
        timed_out = true;
        break;
      }
      phase ^= 1u << s;
      const int lp = warp + k * kWarps;
      const int blk = blk_s[lp];
      if (blk >= 0) {
        const uint32_t kt = tiles_u32 + (uint32_t)((warp * S + s) * C::kStageBytes);
        const uint32_t vt = kt + C::kTile;
        const int tok0 = (pg0 + lp) * kBlockSize;
        const int nvalid = min(kBlockSize, L - tok0);

        // ---------------- S = Q K^T (16 padded heads x 16 tokens) ----------------
        float sc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        if constexpr (INT8) {
#pragma unroll
          for (int kk = 0; kk < KSTEPS / 2; ++kk) {
            // matrices: tokens 0-7 / 8-15 of chunk 2kk, then of chunk 2kk+1
            const int t = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = 2 * kk + (lane >> 4);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<C>(t, ch), r0, r1, r2, r3);
            uint32_t b0, b1;
            i8x4_to_h2x2<0x4140u, 0x4342u>(r0, b0, b1);
            mma_16816<false>(sc[0][0], sc[0][1], qa0[2 * kk], qa2[2 * kk], b0, b1);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r1, b0, b1);
            mma_16816<false>(sc[1][0], sc[1][1], qa0[2 * kk], qa2[2 * kk], b0, b1);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r2, b0, b1);
            mma_16816<false>(sc[0][0], sc[0][1], qa0[2 * kk + 1], qa2[2 * kk + 1], b0, b1);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r3, b0, b1);
            mma_16816<false>(sc[1][0], sc[1][1], qa0[2 * kk + 1], qa2[2 * kk + 1], b0, b1);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            // matrices: tokens 0-7 chunk 2ks, 0-7 chunk 2ks+1, 8-15 chunk 2ks, 8-15 chunk 2ks+1
            const int t = (lane & 7) + (lane >> 4) * 8;
            const int ch = 2 * ks + ((lane >> 3) & 1);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<C>(t, ch), r0, r1, r2, r3);
            mma_16816<MMA_BF16>(sc[0][0], sc[0][1], qa0[ks], qa2[ks], r0, r1);
            mma_16816<MMA_BF16>(sc[1][0], sc[1][1], qa0[ks], qa2[ks], r2, r3);
          }
        }

        // scores in log2 units; thread holds head g, tokens 8nb + 2c + e
        float z[2][2];
        if constexpr (INT8) {
          const uint16_t* ksc = scales + (warp * S + s) * (C::kScaleBytes / 2);
          const float2 k01 = __half22float2(
              u32_as_h2(reinterpret_cast<const uint32_t*>(ksc)[c]));
          const float2 k89 = __half22float2(
              u32_as_h2(reinterpret_cast<const uint32_t*>(ksc)[4 + c]));
          z[0][0] = sc[0][0] * (k01.x * p.scale_log2);
          z[0][1] = sc[0][1] * (k01.y * p.scale_log2);
          z[1][0] = sc[1][0] * (k89.x * p.scale_log2);
          z[1][1] = sc[1][1] * (k89.y * p.scale_log2);
        } else {
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e) z[nb][e] = sc[nb][e] * p.scale_log2;
        }
        if (nvalid < kBlockSize) {
#pragma unroll
          for (int nb = 0; nb < 2; ++nb)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              if (8 * nb + 2 * c + e >= nvalid) z[nb][e] = -INFINITY;
        }

        // ---------------- online softmax (per head g, over the 4 c-lanes) --------
        float mx = fmaxf(fmaxf(z[0][0], z[0][1]), fmaxf(z[1][0], z[1][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        const float alpha = fast_exp2(m_run - m_new);
        float pr[2][2];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) pr[nb][e] = fast_exp2(z[nb][e] - m_new);
        l_run = l_run * alpha + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
        m_run = m_new;
        if (__any_sync(0xFFFFFFFFu, alpha != 1.f)) {
#pragma unroll
          for (int i = 0; i < NOUT; ++i) o[i] *= alpha;
        }

        // ---------------- O += P V ----------------
        if constexpr (INT8) {
          const uint32_t pa0 = h2_as_u32(__floats2half2_rn(pr[0][0], pr[0][1]));
          const uint32_t pa2 = h2_as_u32(__floats2half2_rn(pr[1][0], pr[1][1]));
          const uint16_t* vsc = scales + (warp * S + s) * (C::kScaleBytes / 2) + kBlockSize;
          const __half2 vs01 = u32_as_h2(reinterpret_cast<const uint32_t*>(vsc)[c]);
          const __half2 vs89 = u32_as_h2(reinterpret_cast<const uint32_t*>(vsc)[4 + c]);
#pragma unroll
          for (int kk = 0; kk < KSTEPS / 2; ++kk) {
            const int t = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = 2 * kk + (lane >> 4);
            uint32_t r[4];
            ldsm_x4_trans(vt + tile_off<C>(t, ch), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // r[2h]: tokens 2c,2c+1 (b0);  r[2h+1]: tokens 2c+8,2c+9 (b1);
              // bytes {t0 d0, t0 d1, t1 d0, t1 d1} with d0 = 16ch + 2g (even).
              uint32_t e0, od0, e1, od1;
              i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * h], e0, od0);
              i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * h + 1], e1, od1);
              e0 = h2_as_u32(__hmul2(u32_as_h2(e0), vs01));
              od0 = h2_as_u32(__hmul2(u32_as_h2(od0), vs01));
              e1 = h2_as_u32(__hmul2(u32_as_h2(e1), vs89));
              od1 = h2_as_u32(__hmul2(u32_as_h2(od1), vs89));
              const int cb = 2 * kk + h;
              // even-d tile: d = 16cb + 4c + {0, 2};  odd-d tile: d = 16cb + 4c + {1, 3}
              mma_16816<false>(o[4 * cb + 0], o[4 * cb + 2], pa0, pa2, e0, e1);
              mma_16816<false>(o[4 * cb + 1], o[4 * cb + 3], pa0, pa2, od0, od1);
            }
          }
        } else {
          uint32_t pa0, pa2;
          if constexpr (MMA_BF16) {
            pa0 = bf2_as_u32(__floats2bfloat162_rn(pr[0][0], pr[0][1]));
            pa2 = bf2_as_u32(__floats2bfloat162_rn(pr[1][0], pr[1][1]));
          } else {
            pa0 = h2_as_u32(__floats2half2_rn(pr[0][0], pr[0][1]));
            pa2 = h2_as_u32(__floats2half2_rn(pr[1][0], pr[1][1]));
          }
#pragma unroll
          for (int pp = 0; pp < D / 16; ++pp) {
            // matrices: tokens 0-7 / 8-15 of chunk 2pp, then of chunk 2pp+1
            const int t = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int ch = 2 * pp + (lane >> 4);
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vt + tile_off<C>(t, ch), r0, r1, r2, r3);
            // n-tile 2pp: d = 16pp + 2c + {0,1};  n-tile 2pp+1: d = 16pp + 8 + 2c + {0,1}
            mma_16816<MMA_BF16>(o[4 * pp + 0], o[4 * pp + 1], pa0, pa2, r0, r1);
            mma_16816<MMA_BF16>(o[4 * pp + 2], o[4 * pp + 3], pa0, pa2, r2, r3);
          }
        }
      }
      __syncwarp();
      if (lane == 0 && k + S < nk) issue(k + S);
    }
    if (timed_out) {
      // give up on this item: record, drain this warp's copies still in flight
      if (lane == 0) {
        atomicOr(p.err, 0x8u);
        atomicExch(abort_flag, 1);
      }
      for (int k2 = k; k2 < min(nk, k + S); ++k2) {
        const int s2 = k2 % S;
        mbar_wait_bounded(smem_u32(&bars[warp * S + s2]), (phase >> s2) & 1u);
        phase ^= 1u << s2;
      }
    }

    // ---- merge the warps' (m, l, O) and write ----
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 1);
    l_run += __shfl_xor_sync(0xFFFFFFFFu, l_run, 2);
    __syncthreads();                         // every warp is done with its stages
    if (c == 0 && g < kMaxGroup) {
      st_m[warp * kMaxGroup + g] = m_run;
      st_l[warp * kMaxGroup + g] = l_run;
    }
    if (g < G) {
      float* mrow = merge + ((size_t)warp * kMaxGroup + g) * D;
      if constexpr (INT8) {
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb)
          *reinterpret_cast<float4*>(mrow + 16 * cb + 4 * c) =
              make_float4(o[4 * cb], o[4 * cb + 1], o[4 * cb + 2], o[4 * cb + 3]);
      } else {
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt)
          *reinterpret_cast<float2*>(mrow + 8 * nt + 2 * c) = make_float2(o[2 * nt], o[2 * nt + 1]);
      }
    }
    __syncthreads();
    const int64_t hbase = (int64_t)b * p.Hq + (int64_t)j * G;
    for (int idx = tid; idx < G * (D / 4); idx += kThreads) {
      const int gg = idx / (D / 4);
      const int d = (idx - gg * (D / 4)) * 4;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) M = fmaxf(M, st_m[w * kMaxGroup + gg]);
      float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f, lsum = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float f = fast_exp2(st_m[w * kMaxGroup + gg] - M);
          lsum += f * st_l[w * kMaxGroup + gg];
          const float4 v =
              *reinterpret_cast<const float4*>(merge + ((size_t)w * kMaxGroup + gg) * D + d);
          acc0 += f * v.x; acc1 += f * v.y; acc2 += f * v.z; acc3 += f * v.w;
        }
      }
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      if (nparts == 1) {
        store_out4<QBF16>(p.out, (hbase + gg) * D + d, acc0 * inv, acc1 * inv, acc2 * inv,
                          acc3 * inv);
      } else {
        const int64_t prow = ((int64_t)sp * Hkv + j) * G + gg;
        *reinterpret_cast<float4*>(p.part_o + prow * D + d) =
            make_float4(acc0 * inv, acc1 * inv, acc2 * inv, acc3 * inv);
        if (d == 0) p.part_lse[prow] = lsum > 0.f ? M + __log2f(lsum) : -INFINITY;
      }
    }
    fence_proxy_async_smem();                // merge writes precede the next TMA fills
  }
}

}  // namespace kvq
