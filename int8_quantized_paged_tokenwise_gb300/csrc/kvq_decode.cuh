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
// Structure:
//  * work item = (sequence, KV head, partition of P pages), processed by ONE
//    warp; a sequence of L tokens has max(1, ceil(ceil(L/16) / P)) partitions.
//    Every CTA rebuilds the partition prefix from context_lens in shared
//    memory; warps then stride over the flat item list independently (no
//    CTA-wide synchronization after start-up), so skewed context lengths need
//    no host-side planning.
//  * each warp keeps one continuous stream of page loads across its items:
//    lane 0 issues, S pages ahead of the consumer, TMA copies of the
//    (page, KV head) K and V tiles (2-D tensor copies with the 128-/64-byte
//    swizzle so that the ldmatrix reads are bank-conflict free) and, for INT8,
//    the two 32-byte scale rows (1-D bulk copies), all completing on the
//    stage's mbarrier; an item's first page also brings the item's query rows.
//    Block ids come from the block table 32 pages at a time, the next item's
//    first chunk prefetched.  Waits are bounded (error bit + exit on timeout).
//  * QK^T and PV run on the tensor cores (mma.sync m16n8k16, FP32 accumulate)
//    with the GQA group as the M dimension (padded to 16), so each page is
//    read once for all query heads of its KV head.  INT8 codes become exact
//    FP16 integers with a byte permute and a subtraction; K scales multiply
//    the FP32 scores, V scales multiply the converted V pairs.
//  * at the end of an item the warp writes the final output (one partition)
//    or a normalized partial + log2-sum-exp for the combine kernel.
#pragma once

#include "kvq_internal.h"
#include "kvq_ptx.cuh"

// Pages in flight per warp and the CTAs per SM the register budget targets
// (INT8 cache; the 16-bit twin uses 2 stages and 3 CTAs).
#ifndef KVQ_INT8_STAGES
#define KVQ_INT8_STAGES 2
#endif
#ifndef KVQ_INT8_MIN_CTAS
#define KVQ_INT8_MIN_CTAS 4
#endif

namespace kvq {

template <int D, bool INT8>
struct TileCfg {
  static constexpr int kElem = INT8 ? 1 : 2;                 // bytes per cache element
  static constexpr int kRowBytes = D * kElem;                // bytes per token row
  static constexpr int kSubRow = kRowBytes < 128 ? kRowBytes : 128;   // TMA box row bytes
  static constexpr int kSubTiles = kRowBytes / kSubRow;       // TMA copies per tile
  static constexpr int kSubBytes = kBlockSize * kSubRow;
  static constexpr int kTile = kBlockSize * kRowBytes;        // bytes of one K (or V) tile
  static constexpr int kStages = INT8 ? KVQ_INT8_STAGES : 2;  // pages in flight per warp
  static constexpr int kStageBytes = 2 * kTile;               // K tile then V tile
  static constexpr int kScaleBytes = INT8 ? 2 * kBlockSize * 2 : 0;  // K then V scale rows
  static constexpr uint32_t kTxBytes = 2 * kTile + kScaleBytes;
  static constexpr uint32_t kSwzMask = kSubRow == 128 ? 0x70u : 0x30u;
  static constexpr int kMinCtas = INT8 ? KVQ_INT8_MIN_CTAS : 3;
};

// Partition sizes (pages per work item) the kernel chooses among when the
// caller leaves the choice to it.
constexpr int kNumCand = 20;
__host__ __device__ constexpr int cand_pages(int k) {
  return k == 0 ? 4 : k == 1 ? 5 : k == 2 ? 6 : k == 3 ? 7 : k == 4 ? 8 : k == 5 ? 10
       : k == 6 ? 12 : k == 7 ? 14 : k == 8 ? 16 : k == 9 ? 20 : k == 10 ? 24 : k == 11 ? 28
       : k == 12 ? 32 : k == 13 ? 40 : k == 14 ? 48 : k == 15 ? 56 : k == 16 ? 64
       : k == 17 ? 80 : k == 18 ? 96 : 128;
}

// Byte offset inside a (K or V) tile of 16-byte chunk `c` of token row `t`,
// with the TMA swizzle applied (16-byte chunk index XOR row bits).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
  constexpr int cps = C::kSubRow / 16;  // chunks per sub-tile row
  const uint32_t off = (uint32_t)((c / cps) * C::kSubBytes + t * C::kSubRow + (c % cps) * 16);
  return off ^ ((off >> 3) & C::kSwzMask);
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base).  Per warp:
// S page stages, one raw query slot (the TMA target, G*D*2 bytes) and a query
// fragment buffer ([k-step][lane] pairs of the MMA B operand for the lanes
// 0..4G-1 of real heads, also G*D*2 bytes; the padded heads read as zeros).
template <int D, bool INT8>
struct SmemLayout {
  using C = TileCfg<D, INT8>;
  size_t tiles, q, qfrag, scales, bars, stage_blk, misc, seq, total_bytes;
  uint32_t q_bytes;  // one item's query rows: G * D * 2
  __host__ __device__ SmemLayout(int B, int G) {
    q_bytes = (uint32_t)(G * D * 2);
    tiles = 0;
    q = tiles + (size_t)kWarps * C::kStages * C::kStageBytes;
    qfrag = q + (size_t)kWarps * q_bytes;
    scales = qfrag + (size_t)kWarps * q_bytes;
    bars = (scales + (size_t)kWarps * C::kStages * C::kScaleBytes + 15) & ~(size_t)15;
    stage_blk = bars + (size_t)kWarps * C::kStages * 8;
    misc = stage_blk + (size_t)kWarps * C::kStages * 4;   // 4 ints + reduction buffer
    seq = (misc + 16 + (size_t)kWarps * (kNumCand + 1) * 4 + 15) & ~(size_t)15;  // prefix, lens
    total_bytes = seq + (size_t)B * 8 + 1024;        // + alignment slack of the base
  }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) return bf2_as_u32(__floats2bfloat162_rn(a, b));
  else return h2_as_u32(__floats2half2_rn(a, b));
}

// One work item's coordinates.
struct ItemInfo {
  int b, j, sp, pg0, npg, nparts, L;
};

__device__ __forceinline__ ItemInfo item_info(int64_t item, const int* prefix, const int* lens,
                                              int B, int Hkv, int P) {
  ItemInfo it;
  // item counts stay below 2^31 (checked on the host): 32-bit division
  const uint32_t u = (uint32_t)item;
  it.sp = (int)(u / (uint32_t)Hkv);
  it.j = (int)(u - (uint32_t)it.sp * (uint32_t)Hkv);
  int lo = 0, hi = B - 1;                       // first b with prefix[b] > sp
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] > it.sp) hi = mid; else lo = mid + 1;
  }
  it.b = lo;
  const int sp0 = lo > 0 ? prefix[lo - 1] : 0;
  it.nparts = prefix[lo] - sp0;
  it.L = lens[lo];
  it.pg0 = (it.sp - sp0) * P;
  const int pages = (it.L + kBlockSize - 1) / kBlockSize;
  it.npg = max(0, min(P, pages - it.pg0));
  return it;
}

// INT8: QBF16 = activations are bf16 (converted to FP16 for the tensor cores);
// twin: QBF16 selects the bf16 MMA, otherwise FP16.
template <int D, bool INT8, bool QBF16>
__global__ void __launch_bounds__(kThreads, TileCfg<D, INT8>::kMinCtas)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = TileCfg<D, INT8>;
  const SmemLayout<D, INT8> lay(p.B, p.G);
  constexpr bool MMA_BF16 = (!INT8) && QBF16;
  constexpr int S = C::kStages;
  constexpr int KSTEPS = D / 16;       // MMA k-steps over the head dim
  constexpr int NOUT = D / 4;          // output floats per thread (one head)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + lay.bars);
  int* stage_blk = reinterpret_cast<int*>(smem + lay.stage_blk);
  int* misc = reinterpret_cast<int*>(smem + lay.misc);
  int* prefix = reinterpret_cast<int*>(smem + lay.seq);
  int* lens = prefix + p.B;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;   // MMA fragment coordinates
  const int B = p.B, Hkv = p.Hkv, G = p.G;
  // tokens any sequence may have: the table row and the host's bound (which
  // sized the workspace); a larger context_lens entry is flagged and clamped
  const int max_tok = min(p.max_blocks * kBlockSize, p.max_ctx);

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  if (tid < kWarps * S) mbar_init(smem_u32(&bars[tid]), 1);
  // Programmatic dependent launch: let the combine kernel be scheduled as this
  // grid drains, and wait here until the previous kernel in the stream (e.g.
  // the quantize-append that wrote the newest tokens) has completed and its
  // writes are visible, before reading any input.
  griddep_launch_dependents();
  griddep_wait();
  // Warm L2 with the small inputs every warp reads first (block tables and
  // query rows): CTA i prefetches the i-th 4 KB slice of each.
  if (tid == 0) {
    const int64_t bt_bytes = (int64_t)p.B * p.max_blocks * 4;
    const int64_t q_bytes = (int64_t)p.B * p.Hq * D * 2;
    const int64_t off = (int64_t)blockIdx.x * 4096;
    if (off < bt_bytes && (bt_bytes & 15) == 0 &&
        (reinterpret_cast<uintptr_t>(p.block_tables) & 15) == 0) {
      const int64_t n = bt_bytes - off;
      prefetch_l2(reinterpret_cast<const uint8_t*>(p.block_tables) + off,
                  (uint32_t)(n < 4096 ? n : 4096));
    }
    if (off < q_bytes) {
      const int64_t n = q_bytes - off;
      prefetch_l2(static_cast<const uint8_t*>(p.q) + off, (uint32_t)(n < 4096 ? n : 4096));
    }
  }

  // ---- clamped lengths, partition size, partition prefix over sequences ----
  // P > 0: fixed by the caller.  P == 0: chosen here from the exact lengths,
  // identically in every CTA: among candidate sizes whose partition count fits
  // the workspace (p.sp_cap), the one with the lowest modelled time under the
  // static round-robin assignment of items to warps,
  //   cost(P) = ceil(items / warps) * (min(P, longest) + 2)   [pages],
  // the +2 standing for the per-item overhead (query load, partial write).
  int P = p.P;
  {
    const int per = (B + kThreads - 1) / kThreads;   // consecutive sequences per thread
    const int b0 = tid * per, b1 = min(B, b0 + per);
    int cnt[kNumCand];
#pragma unroll
    for (int k = 0; k < kNumCand; ++k) cnt[k] = 0;
    int pmax = 0;
    for (int b = b0; b < b1; ++b) {
      int L = __ldg(&p.context_lens[b]);
      if (L < 0 || L > max_tok) {
        atomicOr(p.err, 0x4u);
        L = L < 0 ? 0 : max_tok;
      }
      lens[b] = L;
      const int pages = (L + kBlockSize - 1) / kBlockSize;
      pmax = max(pmax, pages);
      if (P == 0) {
#pragma unroll
        for (int k = 0; k < kNumCand; ++k) cnt[k] += max(1, (pages + cand_pages(k) - 1) / cand_pages(k));
      }
    }
    if (P == 0) {
      int* red = misc + 4;                           // [kWarps][kNumCand + 1]
#pragma unroll
      for (int k = 0; k < kNumCand; ++k) {
        int v = cnt[k];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
        if (lane == 0) red[warp * (kNumCand + 1) + k] = v;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) pmax = max(pmax, __shfl_xor_sync(0xFFFFFFFFu, pmax, o));
      if (lane == 0) red[warp * (kNumCand + 1) + kNumCand] = pmax;
      __syncthreads();
      if (warp == 0) {
        // lane k scores candidate k (lane kNumCand: no split); warp arg-min,
        // ties to the larger size
        int longest = 0;
        for (int w = 0; w < kWarps; ++w) longest = max(longest, red[w * (kNumCand + 1) + kNumCand]);
        const uint32_t warps = (uint32_t)gridDim.x * kWarps;
        uint32_t cost = 0xFFFFFFFFu;
        int cand = 0;
        if (lane < kNumCand) {
          // branch-free pick of this lane's size (an indexed lookup of the
          // table would become a divergent jump or a memory access)
#pragma unroll
          for (int k = 0; k < kNumCand; ++k) cand = lane == k ? cand_pages(k) : cand;
          int sp = 0;
          for (int w = 0; w < kWarps; ++w) sp += red[w * (kNumCand + 1) + lane];
          if (sp <= p.sp_cap && cand < longest) {
            const uint32_t items = (uint32_t)sp * (uint32_t)Hkv;
            cost = (items + warps - 1) / warps * (uint32_t)(cand + 2);
          }
        } else if (lane == kNumCand) {
          cand = max(longest, 1);
          cost = ((uint32_t)B * (uint32_t)Hkv + warps - 1) / warps * (uint32_t)(cand + 2);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const uint32_t oc = __shfl_xor_sync(0xFFFFFFFFu, cost, o);
          const int op = __shfl_xor_sync(0xFFFFFFFFu, cand, o);
          if (oc < cost || (oc == cost && op > cand)) {
            cost = oc;
            cand = op;
          }
        }
        if (lane == 0) misc[3] = cand;
      }
      __syncthreads();
      P = misc[3];
    }
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      const int pages = (lens[b] + kBlockSize - 1) / kBlockSize;
      sum += max(1, (pages + P - 1) / P);
    }
    int incl = sum;                                  // block-wide scan of per-thread sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    __syncthreads();                                 // misc[] free again
    if (lane == 31) misc[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += misc[w];
    for (int b = b0; b < b1; ++b) {
      const int pages = (lens[b] + kBlockSize - 1) / kBlockSize;
      run += max(1, (pages + P - 1) / P);
      prefix[b] = run;
    }
  }
  fence_mbar_init();
  __syncthreads();
  if (blockIdx.x == 0 && p.prefix_out != nullptr)
    for (int b = tid; b < B; b += kThreads) p.prefix_out[b] = prefix[b];

  const int64_t n_items = B > 0 ? (int64_t)prefix[B - 1] * Hkv : 0;
  const int64_t wg = (int64_t)blockIdx.x * kWarps + warp;     // this warp's first item
  const int64_t nw = (int64_t)gridDim.x * kWarps;             // item stride

  const uint32_t tiles_u32 = smem_u32(smem + lay.tiles) + warp * S * C::kStageBytes;
  const uint32_t q_u32 = smem_u32(smem + lay.q) + warp * lay.q_bytes;
  uint2* qfrag = reinterpret_cast<uint2*>(smem + lay.qfrag + (size_t)warp * lay.q_bytes);
  const uint32_t qfrag_lane_u32 = smem_u32(qfrag) + 8 * lane;   // + 32 * G * ks
  const uint32_t qks = 32u * (uint32_t)G;                        // bytes per k-step
  const uint32_t scales_u32 = smem_u32(smem + lay.scales) + warp * S * C::kScaleBytes;
  const uint16_t* scales_w =
      reinterpret_cast<const uint16_t*>(smem + lay.scales) + warp * S * (C::kScaleBytes / 2);
  const uint32_t bars_u32 = smem_u32(&bars[warp * S]);
  int* blk_w = stage_blk + warp * S;

  // Each page arrives as copies issued together by lanes 0..3: 2-D tensor TMA
  // of the K and V tiles (16-bit tiles in 128-byte-wide sub-tiles; a tiled
  // TMA needs a 128-byte aligned shared destination, which the tiles have)
  // and, for INT8, 1-D bulk copies of the K and V scale rows (16-byte aligned
  // destinations).  Per lane: tensor map, x coordinate and destination (+ the
  // per-stage stride), or the scale plane and destination.
  constexpr int kTensorCopies = 2 * C::kSubTiles;
  const CUtensorMap* cp_map = lane < C::kSubTiles ? &tmK : &tmV;
  const int cp_sub = lane % C::kSubTiles;               // 128-byte column block
  const int cp_x = cp_sub * (C::kSubRow / C::kElem);
  const uint32_t cp_dst = tiles_u32 + (lane < C::kSubTiles ? 0 : C::kTile) + cp_sub * C::kSubBytes;
  const uint16_t* sc_src = lane == kTensorCopies ? p.k_scale : p.v_scale;
  const uint32_t sc_dst = scales_u32 + (lane == kTensorCopies ? 0 : kBlockSize * 2);

  // ---------------------------------------------------------------- issuer
  // Warp-uniform state; lane 0 performs the copies.  The block ids of the
  // current 32-page chunk live one per lane (blk_cur); the first chunk of the
  // following item is prefetched into blk_nxt.
  int64_t is_item = wg;
  int is_ord = 0, is_pg = 0, is_chunk = 0;
  ItemInfo nx_it{};                      // the item after the issuer's (first chunk in blk_nxt)
  int q_issued = -1, q_consumed = -1;   // ordinals: last item whose query was copied / read
  ItemInfo is_it{};
  int blk_cur = -1, blk_nxt = -1;
  uint32_t n_issued = 0, n_done = 0;
  int is_slot = 0;                       // stage the next issued page goes to
  int cs_slot = 0;                       // stage the consumer reads next
  uint32_t cs_phase = 0;                 // parity of that wait (flips each pass over the ring)

  auto load_chunk = [&](const ItemInfo& it, int base) -> int {
    const int pg = base + lane;
    int blk = -1;
    if (pg < it.npg) {
      blk = __ldg(&p.block_tables[(int64_t)it.b * p.max_blocks + it.pg0 + pg]);
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.err, 0x2u);
        blk = -1;
      }
    }
    return blk;
  };
  auto next_item_chunk = [&](int64_t item) -> int {
    if (item >= n_items) {
      nx_it.npg = 0;
      return -1;
    }
    nx_it = item_info(item, prefix, lens, B, Hkv, P);
    return load_chunk(nx_it, 0);
  };
  if (is_item < n_items) {
    is_it = item_info(is_item, prefix, lens, B, Hkv, P);
    blk_cur = load_chunk(is_it, 0);
    blk_nxt = next_item_chunk(is_item + nw);
  }

  // Issue pages while fewer than S are in flight; an item's first page (which
  // also copies the item's query rows into the single raw query slot) waits
  // until the previously copied query rows have been read by the consumer.
  auto refill = [&]() {
    while (n_issued - n_done < (uint32_t)S) {
      while (is_item < n_items && is_pg >= is_it.npg) {   // next item with pages
        is_item += nw;
        ++is_ord;
        is_pg = 0;
        is_chunk = 0;
        if (is_item < n_items) {
          is_it = item_info(is_item, prefix, lens, B, Hkv, P);
          blk_cur = blk_nxt;
          blk_nxt = next_item_chunk(is_item + nw);
        }
      }
      if (is_item >= n_items || (is_pg == 0 && q_issued > q_consumed)) return;
      if (is_pg >= is_chunk + 32) {
        is_chunk += 32;
        blk_cur = load_chunk(is_it, is_chunk);
      }
      const int blk = __shfl_sync(0xFFFFFFFFu, blk_cur, is_pg - is_chunk);
      const int s = is_slot;
      is_slot = is_slot + 1 == S ? 0 : is_slot + 1;
      const uint32_t bar = bars_u32 + 8 * s;
      const uint32_t qbytes = is_pg == 0 ? lay.q_bytes : 0u;
      if (lane == 0) {
        blk_w[s] = blk;
        if (blk >= 0) mbar_arrive_expect_tx(bar, C::kTxBytes + qbytes);
        else if (qbytes) mbar_arrive_expect_tx(bar, qbytes);
        else mbar_arrive(bar);
      }
      if (blk >= 0) {
        const int row = blk * Hkv + is_it.j;          // (block, KV head) tile index
        if (lane < kTensorCopies) {
          tma_load_2d(cp_dst + s * C::kStageBytes, cp_map, cp_x, row * kBlockSize, bar);
        } else if (INT8 && lane < kTensorCopies + 2) {
          bulk_load(sc_dst + s * C::kScaleBytes, sc_src + (int64_t)row * kBlockSize,
                    kBlockSize * 2, bar);
        }
      }
      if (qbytes && lane == 4) {
        const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) +
                               ((int64_t)is_it.b * p.Hq + (int64_t)is_it.j * G) * D;
        bulk_load(q_u32, qsrc, qbytes, bar);
      }
      if (is_pg == 0) q_issued = is_ord;
      ++n_issued;
      ++is_pg;
    }
  };
  refill();

  // -------------------------------------------------------------- consumer
  int ord = 0;
  bool aborted = false;
  for (int64_t item = wg; item < n_items && !aborted; item += nw, ++ord) {
    const ItemInfo it = item_info(item, prefix, lens, B, Hkv, P);
    // Running softmax state of the two query heads this thread's columns hold
    // (heads 2c and 2c+1 of the KV head's group), and the output accumulator
    // O^T[d][head]: o[4cb + e] for 16-wide head-dim block cb, e = (row, col)
    // of the MMA quad: e0 (row g, col 2c), e1 (g, 2c+1), e2 (g+8, 2c),
    // e3 (g+8, 2c+1).
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    float o[NOUT];
#pragma unroll
    for (int i = 0; i < NOUT; ++i) o[i] = 0.f;
    const bool has_head = g < G;   // this lane provides a real query column

    for (int pg = 0; pg < it.npg; ++pg) {
      const int s = cs_slot;
      const uint32_t par = cs_phase;
      if (++cs_slot == S) {
        cs_slot = 0;
        cs_phase ^= 1u;
      }
      if (!mbar_wait_bounded(bars_u32 + 8 * s, par)) {
        aborted = true;
        break;
      }
      if (pg == 0) {
        // query fragments (the MMA B operand, column g = head g < G), from the
        // raw rows to this lane's slots of the fragment buffer
        if (has_head) {
          const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + lay.q) +
                               (size_t)warp * (lay.q_bytes / 2) + g * D;
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint2 f;
            if constexpr (INT8) {
              // logical k {2c,2c+1,2c+8,2c+9} of step ks <-> head-dim 16ks+4c+{0..3}
              const uint2 v = *reinterpret_cast<const uint2*>(qs + 16 * ks + 4 * c);
              if constexpr (QBF16) {
                f.x = h2_as_u32(__floats2half2_rn(__uint_as_float(v.x << 16),
                                                  __uint_as_float(v.x & 0xFFFF0000u)));
                f.y = h2_as_u32(__floats2half2_rn(__uint_as_float(v.y << 16),
                                                  __uint_as_float(v.y & 0xFFFF0000u)));
              } else {
                f = v;
              }
            } else {
              // natural order: k {2c,2c+1} <-> 16ks+2c, k {2c+8,2c+9} <-> 16ks+8+2c
              f.x = *reinterpret_cast<const uint32_t*>(qs + 16 * ks + 2 * c);
              f.y = *reinterpret_cast<const uint32_t*>(qs + 16 * ks + 8 + 2 * c);
            }
            qfrag[ks * 4 * G + lane] = f;
          }
        }
        q_consumed = ord;
      }
      const int blk = blk_w[s];
      if (blk >= 0) {
        const uint32_t kt = tiles_u32 + s * C::kStageBytes;
        const uint32_t vt = kt + C::kTile;
        const int nvalid = min(kBlockSize, it.L - (it.pg0 + pg) * kBlockSize);
        // ldmatrix row address: matrices (tokens 0-7, chunk 2i), (8-15, 2i),
        // (0-7, 2i+1), (8-15, 2i+1) for lanes 0-7, 8-15, 16-23, 24-31
        const int lt = (lane & 7) + ((lane >> 3) & 1) * 8;

        // ---------- S[token][head] = K Q^T: M = 16 tokens, N = 8 heads ----------
        // two accumulators (even/odd k-steps) halve the dependent MMA chain
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < (INT8 ? KSTEPS / 2 : 0); ++kk) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kt + tile_off<C>(lt, 2 * kk + (lane >> 4)), r0, r1, r2, r3);
          const uint2 qa = lds_u2_if(has_head, qfrag_lane_u32 + qks * (2 * kk));
          const uint2 qb = lds_u2_if(has_head, qfrag_lane_u32 + qks * (2 * kk + 1));
          if constexpr (INT8) {
            // r0/r1: tokens g / g+8, head-dim 16(2kk)+4c+{0..3}; r2/r3: next chunk
            uint32_t a0, a2, a1, a3;
            i8x4_to_h2x2<0x4140u, 0x4342u>(r0, a0, a2);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r1, a1, a3);
            mma_16816_acc<false>(sa, a0, a1, a2, a3, qa.x, qa.y);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r2, a0, a2);
            i8x4_to_h2x2<0x4140u, 0x4342u>(r3, a1, a3);
            mma_16816_acc<false>(sb, a0, a1, a2, a3, qb.x, qb.y);
          }
        }
        if constexpr (!INT8) {
          // 16-bit tiles: one 16-byte chunk holds 8 elements, so k-step ks spans
          // chunks 2ks and 2ks+1 and (r0, r1, r2, r3) is directly its A operand
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<C>(lt, 2 * ks + (lane >> 4)), r0, r1, r2, r3);
            const uint2 qa = lds_u2_if(has_head, qfrag_lane_u32 + qks * ks);
            // a0: token g, d 16ks+2c..; a1: token g+8; a2: token g, d 16ks+8+2c..; a3: g+8
            if (ks & 1) mma_16816_acc<MMA_BF16>(sb, r0, r1, r2, r3, qa.x, qa.y);
            else mma_16816_acc<MMA_BF16>(sa, r0, r1, r2, r3, qa.x, qa.y);
          }
        }

        // scores in log2 units: z0 (token g, head 2c), z1 (g, 2c+1), z2 (g+8, 2c), z3
        float ksg = p.scale_log2, ksg8 = p.scale_log2;
        if constexpr (INT8) {
          const uint16_t* ksc = scales_w + s * (C::kScaleBytes / 2);
          ksg *= __half2float(__ushort_as_half(ksc[g]));
          ksg8 *= __half2float(__ushort_as_half(ksc[g + 8]));
        }
        float z0 = (sa[0] + sb[0]) * ksg, z1 = (sa[1] + sb[1]) * ksg;
        float z2 = (sa[2] + sb[2]) * ksg8, z3 = (sa[3] + sb[3]) * ksg8;
        if (nvalid < kBlockSize) {
          if (g >= nvalid) z0 = z1 = -INFINITY;
          if (g + 8 >= nvalid) z2 = z3 = -INFINITY;
        }

        // ---------- online softmax per head column (reduce over the 8 g-lanes) ----------
        float mx0 = fmaxf(z0, z2), mx1 = fmaxf(z1, z3);
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
        const float p0 = fast_exp2(z0 - mn0), p1 = fast_exp2(z1 - mn1);
        const float p2 = fast_exp2(z2 - mn0), p3 = fast_exp2(z3 - mn1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
        if (__any_sync(0xFFFFFFFFu, (al0 != 1.f) || (al1 != 1.f))) {
#pragma unroll
          for (int cb = 0; cb < D / 16; ++cb) {
            o[4 * cb + 0] *= al0;
            o[4 * cb + 1] *= al1;
            o[4 * cb + 2] *= al0;
            o[4 * cb + 3] *= al1;
          }
        }

        // P^T as the B operand: b0 = P[tokens 2c, 2c+1][head g], b1 = tokens 2c+8, 2c+9
        const uint32_t pb0 = movmatrix_trans(pack2<MMA_BF16>(p0, p1));
        const uint32_t pb1 = movmatrix_trans(pack2<MMA_BF16>(p2, p3));

        // ---------- O^T[d][head] += V^T P^T: M = 16 head-dims, N = 8 heads ----------
        if constexpr (INT8) {
          const uint16_t* vsc = scales_w + s * (C::kScaleBytes / 2) + kBlockSize;
          const __half2 vs01 = u32_as_h2(reinterpret_cast<const uint32_t*>(vsc)[c]);
          const __half2 vs89 = u32_as_h2(reinterpret_cast<const uint32_t*>(vsc)[4 + c]);
#pragma unroll
          for (int kk = 0; kk < KSTEPS / 2; ++kk) {
            uint32_t r[4];
            ldsm_x4_trans(vt + tile_off<C>(lt, 2 * kk + (lane >> 4)), r[0], r[1], r[2], r[3]);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              // r[2h]: tokens 2c, 2c+1; r[2h+1]: tokens 2c+8, 2c+9; bytes
              // {t0 d0, t0 d1, t1 d0, t1 d1} with d0 = 16cb + 2g (row g), d1 = d0 + 1 (row g+8)
              uint32_t ev0, od0, ev1, od1;
              i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * h], ev0, od0);
              i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * h + 1], ev1, od1);
              ev0 = h2_as_u32(__hmul2(u32_as_h2(ev0), vs01));
              od0 = h2_as_u32(__hmul2(u32_as_h2(od0), vs01));
              ev1 = h2_as_u32(__hmul2(u32_as_h2(ev1), vs89));
              od1 = h2_as_u32(__hmul2(u32_as_h2(od1), vs89));
              const int cb = 2 * kk + h;
              float* oq = o + 4 * cb;
              mma_16816_acc<false>(*reinterpret_cast<float(*)[4]>(oq), ev0, od0, ev1, od1, pb0, pb1);
            }
          }
        } else {
          // matrices: (tokens 0-7, chunk 2pp), (0-7, 2pp+1), (8-15, 2pp), (8-15, 2pp+1)
          const int vtk = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
          for (int pp = 0; pp < D / 16; ++pp) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vt + tile_off<C>(vtk, 2 * pp + ((lane >> 3) & 1)), r0, r1, r2, r3);
            // rows g: d = 16pp + g; rows g+8: d = 16pp + 8 + g
            float* oq = o + 4 * pp;
            mma_16816_acc<MMA_BF16>(*reinterpret_cast<float(*)[4]>(oq), r0, r1, r2, r3, pb0, pb1);
          }
        }
      }
      ++n_done;
      __syncwarp();
      refill();
    }
    if (aborted) break;

    // ---- finalize the item: this warp holds the whole partition ----
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xFFFFFFFFu, l0, off);
      l1 += __shfl_xor_sync(0xFFFFFFFFu, l1, off);
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int head = 2 * c + hh;              // this thread's column
      if (head >= G) continue;
      const float l = hh ? l1 : l0;
      const float m = hh ? m1 : m0;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int64_t hrow = (int64_t)it.b * p.Hq + (int64_t)it.j * G + head;
      if (it.nparts == 1) {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + hrow * D;
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb) {
          const float v0 = o[4 * cb + hh] * inv, v1 = o[4 * cb + 2 + hh] * inv;
          if constexpr (INT8) {  // rows g, g+8 <-> d = 16cb + 2g, 16cb + 2g + 1
            *reinterpret_cast<uint32_t*>(dst + 16 * cb + 2 * g) = pack2<QBF16>(v0, v1);
          } else {               // rows g, g+8 <-> d = 16cb + g, 16cb + 8 + g
            const uint32_t pk = pack2<QBF16>(v0, v1);
            dst[16 * cb + g] = (uint16_t)(pk & 0xFFFFu);
            dst[16 * cb + 8 + g] = (uint16_t)(pk >> 16);
          }
        }
      } else {
        const int64_t prow = ((int64_t)it.sp * Hkv + it.j) * G + head;
        float* dst = p.part_o + prow * D;
#pragma unroll
        for (int cb = 0; cb < D / 16; ++cb) {
          const float v0 = o[4 * cb + hh] * inv, v1 = o[4 * cb + 2 + hh] * inv;
          if constexpr (INT8) {
            *reinterpret_cast<float2*>(dst + 16 * cb + 2 * g) = make_float2(v0, v1);
          } else {
            dst[16 * cb + g] = v0;
            dst[16 * cb + 8 + g] = v1;
          }
        }
        if (g == 0) p.part_lse[prow] = l > 0.f ? m + __log2f(l) : -INFINITY;
      }
    }
  }

  if (aborted) {
    // A wait gave up: record it, then wait (bounded) for this warp's copies
    // still in flight so that none lands after the CTA has exited.
    if (lane == 0) atomicOr(p.err, 0x8u);
    // the failed wait's stage is the one before cs_slot (cs_slot/cs_phase advanced)
    int s = cs_slot == 0 ? S - 1 : cs_slot - 1;
    uint32_t ph = cs_slot == 0 ? (cs_phase ^ 1u) : cs_phase;
    for (; n_done < n_issued; ++n_done) {
      mbar_wait_bounded(bars_u32 + 8 * s, ph);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
}

}  // namespace kvq
