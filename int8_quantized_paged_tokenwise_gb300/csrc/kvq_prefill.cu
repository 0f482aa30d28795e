// Chunked-prefill attention over the tokenwise INT8 paged cache, on the
// 5th-generation tensor cores (tcgen05 MMAs with TMEM accumulators).
//
// What it computes ("fix(cuda/kv): correct Int8 KV per-token scale ..."
// (mlxcel PR #717), "Server integration": Int8 chunked prefill + decode over
// the same cache): sequence b holds L tokens, the last n of them being this
// chunk's queries (already quantized into the cache); query i at position
// p = L - n + i attends causally to tokens 0..p:
//   out[i][h] = softmax_{t<=p}(sm_scale * q[i][h] . s_k[t] code_k[t]) . (s_v code_v)
//
// One CTA = two consecutive tiles ("halves" A and B) of 128 (query,
// head-of-the-GQA-group) rows of one KV head of one sequence; each half is
// the M = 128 of its own MMAs, and both share every converted K/V tile.  The
// sequence's tokens stream in tiles of 64 (4 pages).  Warp roles:
//  * warp 8, producer: block ids 32 pages at a time, TMA copies of each
//    page's INT8 K and V tiles (2-D tensor copies, 128-/64-byte swizzle) and
//    bulk copies of its two 32-byte scale rows into a 3-stage ring;
//  * warps 10-13, converters: INT8 codes to exact FP16 integers (byte
//    permute under exponent 0x64, minus 1152), K and V both as [64 tokens][D]
//    tiles, 128-byte swizzled, in 4 buffers: K is the K-major B operand of
//    Q K^T, V the MN-major B operand of P V; the tile's K scales (times
//    sm_scale log2 e) and V scales as FP32 columns;
//  * warp 9, MMA issuer (one thread): per KV tile and half, P V of the
//    previous tile (A = P read from TMEM, into the half's 128 x D FP32
//    accumulator) and then S = Q K^T (D/16 MMAs of K = 16) into the half's
//    128 x 64 FP32 S buffer; a commit after S therefore also covers the P V
//    before it, so the softmax may rescale O and overwrite P as soon as S
//    has landed;
//  * warps 0-3 (half A) and 4-7 (half B), softmax (one thread per row =
//    TMEM lane): the row of S times the K-scale column, causal mask, running
//    maximum, P = 2^(z - m); the row sum takes P, and P' = P s_v (FP16) is
//    stored into the half's TMEM P buffer as the A operand of the next P V.
//    O is rescaled in TMEM only when a row maximum grows by more than 2^8
//    over the one in use (the shift cancels in O / l, and P' stays below
//    2^8 s_v); the epilogue normalizes O and stores it.
// All waits are bounded: a timeout sets an error bit, the roles leave their
// loops, the copies and MMAs in flight are waited for, and TMEM is freed.
#include "kvq_decode.cuh"
#include "kvq_tc.cuh"

namespace kvq {
namespace {

constexpr int kTcRows = 128;                    // M: (query, head) rows per half
constexpr int kTcHalves = 2;                    // row tiles per CTA
constexpr int kTcKv = 64;                       // tokens per KV tile
constexpr int kTcPages = kTcKv / kBlockSize;     // pages per KV tile
#ifndef KVQ_PF_RAW
#define KVQ_PF_RAW 3
#endif
#ifndef KVQ_PF_CONV
#define KVQ_PF_CONV 4
#endif
constexpr int kTcRaw = KVQ_PF_RAW;              // INT8 staging ring depth
constexpr int kTcConv = KVQ_PF_CONV;            // converted (FP16) operand buffers
constexpr int kTcWarps = 14;
constexpr int kTcThreads = kTcWarps * 32;
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpCvt = 10;
constexpr uint32_t kTcCols = 512;

// TMEM columns of half h: O at h D, S at 2 D + 64 h, whose first 32 columns
// also hold P' (64 FP16) once the softmax has read S, and the half's Q tile
// (the A operand of S = Q K^T, D FP16 = D / 2 columns) at 2 D + 128 + D h / 2;
// 3 D + 128 <= 512.

// barrier indices
constexpr int kBarRawFull = 0, kBarRawEmpty = kTcRaw, kBarCvtFull = 2 * kTcRaw,
              kBarCvtEmpty = 2 * kTcRaw + kTcConv, kBarSFull = 2 * kTcRaw + 2 * kTcConv,
              kBarPFull = kBarSFull + 2, kBarODone = kBarPFull + 2, kBarFin = kBarODone + 2,
              kNumBars = kBarFin + 1;

// Shared memory (offsets from a 1024-aligned base; every operand tile starts
// on a 1024-byte boundary).
template <int D>
struct TcLayout {
  static constexpr int kConvBytes = kTcKv * D * 2;        // [64][D] FP16, D/64 tiles of 8 KB
  static constexpr int kKc = 0;                          // kTcConv K buffers
  static constexpr int kVc = kKc + kTcConv * kConvBytes; // kTcConv V buffers
  static constexpr int kTile = kBlockSize * D;           // one page's INT8 K (or V) tile
  static constexpr int kRawBytes = 2 * kTcPages * kTile; // K tiles of 4 pages, then V tiles
  static constexpr int kRaw = kVc + kTcConv * kConvBytes;          // kTcRaw stages
  static constexpr int kRawSc = kRaw + kTcRaw * kRawBytes;         // per page: K 32 B, V 32 B
  static constexpr int kColSc = kRawSc + kTcRaw * kTcPages * 64;   // per buffer: K 64, V 64 floats
  static constexpr int kVmax = kColSc + kTcConv * 2 * kTcKv * 4;  // per buffer: 2 floats
  static constexpr int kBars = kVmax + kTcConv * 2 * 4;
  static constexpr int kMisc = kBars + kNumBars * 8;     // TMEM base, abort flag
  static constexpr size_t kTotal = (size_t)kMisc + 16 + 1024;      // + base alignment slack
};

// Two BF16 values times a power of two `f`, as an FP16 pair.
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t v, float f) {
  return h2_as_u32(
      __floats2half2_rn(__uint_as_float(v << 16) * f, __uint_as_float(v & 0xFFFF0000u) * f));
}

// 16 INT8 codes (chunk c of token row t of a page tile) -> FP16 chunks 2c,
// 2c+1 of row t of a [64][D] 128-byte-swizzled operand tile.
template <int D>
__device__ __forceinline__ void convert_chunk(const uint8_t* src, uint8_t* dst, int t, int c) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  uint4 lo, hi;
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.x, lo.x, lo.y);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.y, lo.z, lo.w);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.z, hi.x, hi.y);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.w, hi.z, hi.w);
  uint8_t* row = dst + (c >> 2) * (kTcKv * 128) + t * 128;
  const int c0 = (2 * c) & 7;
  *reinterpret_cast<uint4*>(row + ((c0 ^ (t & 7)) << 4)) = lo;
  *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (t & 7)) << 4)) = hi;
}

// The same for V, each exact code pair then multiplied by the token's scale
// factor `f` (an FP16 pair): V' = code * s_v * 2^(127 - F) <= 254.
template <int D>
__device__ __forceinline__ void convert_chunk_scaled(const uint8_t* src, uint8_t* dst, int t, int c,
                                                     __half2 f) {
  const uint4 w = *reinterpret_cast<const uint4*>(src);
  uint4 lo, hi;
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.x, lo.x, lo.y);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.y, lo.z, lo.w);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.z, hi.x, hi.y);
  i8x4_to_h2x2<0x4140u, 0x4342u>(w.w, hi.z, hi.w);
  uint32_t* l4 = reinterpret_cast<uint32_t*>(&lo);
  uint32_t* h4 = reinterpret_cast<uint32_t*>(&hi);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    l4[i] = h2_as_u32(__hmul2(u32_as_h2(l4[i]), f));
    h4[i] = h2_as_u32(__hmul2(u32_as_h2(h4[i]), f));
  }
  uint8_t* row = dst + (c >> 2) * (kTcKv * 128) + t * 128;
  const int c0 = (2 * c) & 7;
  *reinterpret_cast<uint4*>(row + ((c0 ^ (t & 7)) << 4)) = lo;
  *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (t & 7)) << 4)) = hi;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_prefill_kernel(const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = TileCfg<D, true>;
  using Ly = TcLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Ly::kBars);
  uint32_t* misc = reinterpret_cast<uint32_t*>(smem + Ly::kMisc);
  volatile uint32_t* abort_flag = misc + 1;
  auto bar = [&](int i) { return smem_u32(&bars[i]); };
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, j = blockIdx.y, G = p.G;
  const int TH = kTcRows / G;                     // queries per half
  const int ct_idx = (int)gridDim.x - 1 - (int)blockIdx.x;   // latest (longest) tiles first

  if (tid == 0) {
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    misc[1] = 0;
  }
  if (tid < kNumBars) {
    uint32_t count = 1;                           // TMA transactions, commits
    if (tid >= kBarRawEmpty && tid < kBarRawEmpty + kTcRaw) count = 4;     // converter warps
    if (tid >= kBarCvtFull && tid < kBarCvtFull + kTcConv) count = 4;      // converter warps
    if (tid >= kBarPFull && tid < kBarPFull + kTcHalves) count = 4;        // a half's softmax warps
    mbar_init(bar(tid), count);
  }
  griddep_wait();

  const int q0 = __ldg(&p.query_start[b]);
  const int n = __ldg(&p.query_start[b + 1]) - q0;
  const int L = __ldg(&p.context_lens[b]);
  const int max_tok = min(p.max_blocks * kBlockSize, p.max_ctx);
  if (L < 0 || L > max_tok || n < 0 || n > L || n > p.max_q || q0 < 0 || q0 + n > p.total_q) {
    if (tid == 0 && ct_idx == 0 && j == 0) atomicOr(p.err, 0x4u);
    return;                                      // nothing issued or allocated yet
  }
  const int i_begin = ct_idx * kTcHalves * TH;   // first query of half A
  if (i_begin >= n) return;
  // KV tiles of each half (0: no queries); half B has at least as many
  int n_half[kTcHalves];
#pragma unroll
  for (int h = 0; h < kTcHalves; ++h) {
    const int hb = i_begin + h * TH, he = min(n, hb + TH);
    n_half[h] = hb < n ? (L - n + he - 1) / kTcKv + 1 : 0;
  }
  const int n_it = max(n_half[0], n_half[1]);    // KV tiles of the CTA
  const int npages = min((L - n + min(n, i_begin + kTcHalves * TH) - 1) / kBlockSize + 1,
                         n_it * kTcPages);

  if (warp == kWarpMma) tc_alloc(smem_u32(&misc[0]), kTcCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  auto tO = [&](int h) { return tmem + (uint32_t)(h * D); };
  auto tS = [&](int h) { return tmem + (uint32_t)(2 * D + kTcKv * h); };
  auto tP = [&](int h) { return tS(h); };
  auto tQ = [&](int h) { return tmem + (uint32_t)(2 * D + 2 * kTcKv + (D / 2) * h); };

  // ---- Q tiles into TMEM: row r of half h = TMEM lane r = (query i_begin +
  // h TH + r / G, head j G + r % G), FP16, written by that row's softmax
  // thread.  BF16 rows enter as q * 2^-sh (exact: the row's largest |q| lands
  // in [2^14, 2^15)); the softmax multiplies the row's scores by qf = 2^sh.
  float qf = 1.f;
  if (warp < 2 * 4) {
    const int h = warp >> 2, r = 32 * (warp & 3) + lane;
    const int i = i_begin + h * TH + r / G;
    uint4 v[D / 8];
    const bool row = r < TH * G && i < n;
    const uint4* src = reinterpret_cast<const uint4*>(
        static_cast<const uint16_t*>(p.q) +
        ((int64_t)(q0 + (row ? i : 0)) * p.Hq + (int64_t)j * G + r % G) * D);
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) v[c8] = row ? __ldg(src + c8) : make_uint4(0, 0, 0, 0);
    if constexpr (BF16) {
      uint32_t mx = 0;
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8)
        mx = __vmaxu2(mx, __vmaxu2(__vmaxu2(v[c8].x & 0x7FFF7FFFu, v[c8].y & 0x7FFF7FFFu),
                                   __vmaxu2(v[c8].z & 0x7FFF7FFFu, v[c8].w & 0x7FFF7FFFu)));
      const int sh = bf16_fp16_shift(max(mx & 0xFFFFu, mx >> 16));
      qf = exp2i(sh);
      const float inv = exp2i(-sh);
#pragma unroll
      for (int c8 = 0; c8 < D / 8; ++c8) {
        v[c8].x = bf2_to_h2(v[c8].x, inv);
        v[c8].y = bf2_to_h2(v[c8].y, inv);
        v[c8].z = bf2_to_h2(v[c8].z, inv);
        v[c8].w = bf2_to_h2(v[c8].w, inv);
      }
    }
    // column c holds elements 2c (low half) and 2c + 1 of the row
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
#pragma unroll
    for (int c0 = 0; c0 < D / 2; c0 += 32) {
      uint32_t w[32];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint4 u = v[(c0 + 4 * x) / 4];
        w[4 * x] = u.x;
        w[4 * x + 1] = u.y;
        w[4 * x + 2] = u.z;
        w[4 * x + 3] = u.w;
      }
      tc_st32(tQ(h) + c0 + lanes, w);
    }
    tc_wait_st();
  }
  fence_mbar_init();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  auto fail = [&]() {
    atomicOr(p.err, 0x8u);
    *abort_flag = 1;
  };

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    const int32_t* bt = p.block_tables + (int64_t)b * p.max_blocks;
    const uint32_t raw_u32 = smem_u32(smem + Ly::kRaw);
    const uint32_t rawsc_u32 = smem_u32(smem + Ly::kRawSc);
    int issued = 0;
    // block ids of 32 pages (8 tiles) at a time, one per lane, checked once
    auto load_ids = [&](int base) -> int {
      int id = -1;
      if (base + lane < npages) {
        id = __ldg(&bt[base + lane]);
        if (id < 0 || id >= p.num_blocks) {
          atomicOr(p.err, 0x2u);
          id = -1;
        }
      }
      return id;
    };
    int ids = load_ids(0), ids_next = npages > 32 ? load_ids(32) : -1;
    for (int it = 0; it < n_it; ++it) {
      const int s = it % kTcRaw;
      if (it >= kTcRaw && !mbar_wait_bounded(bar(kBarRawEmpty + s), ((it / kTcRaw) - 1) & 1)) {
        if (lane == 0) fail();
        break;
      }
      if (*abort_flag) break;
      const int chunk_it = it % (32 / kTcPages);
      if (it > 0 && chunk_it == 0) {              // next 32 pages; prefetch the ones after
        ids = ids_next;
        const int nb = (it / (32 / kTcPages) + 1) * 32;
        ids_next = nb < npages ? load_ids(nb) : -1;
      }
      // lanes 4 k + pg: page pg of the tile, copy k (K tile, V tile, K scales, V scales)
      int blk = __shfl_sync(0xFFFFFFFFu, ids, kTcPages * chunk_it + (lane & 3));
      if (lane >= 4 * kTcPages) blk = -1;
      const uint32_t loaded = __ballot_sync(0xFFFFFFFFu, lane < kTcPages && blk >= 0);
      const uint32_t full = bar(kBarRawFull + s);
      if (lane == 0) {
        const uint32_t tx = (uint32_t)__popc(loaded) * (2u * Ly::kTile + 64u);
        if (tx) mbar_arrive_expect_tx(full, tx);
        else mbar_arrive(full);
      }
      __syncwarp();
      if (lane < 4 * kTcPages && blk >= 0) {
        const int k = lane >> 2, pgl = lane & 3;
        const int row = blk * p.Hkv + j;            // (block, KV head) tile index
        const uint32_t stage = raw_u32 + s * Ly::kRawBytes;
        if (k == 0) tma_load_2d(stage + pgl * Ly::kTile, &tmK, 0, row * kBlockSize, full);
        else if (k == 1)
          tma_load_2d(stage + (kTcPages + pgl) * Ly::kTile, &tmV, 0, row * kBlockSize, full);
        else
          bulk_load(rawsc_u32 + (s * kTcPages + pgl) * 64 + (k - 2) * 32,
                    (k == 2 ? p.k_scale : p.v_scale) + (int64_t)row * kBlockSize, 32, full);
      }
      issued = it + 1;
    }
    // copies still in flight (the last stages issued) land before the CTA exits
    for (int it = issued > kTcRaw ? issued - kTcRaw : 0; it < issued; ++it)
      mbar_wait_bounded(bar(kBarRawFull + it % kTcRaw), (it / kTcRaw) & 1);
  } else if (warp >= kWarpCvt) {
    // ---------------------------------------------------------- converters
    const int ct = tid - kWarpCvt * 32;           // 0..127
    int cvt_f = 0;                                // running V exponent F
    for (int it = 0; it < n_it; ++it) {
      const int s = it % kTcRaw, cb = it % kTcConv;
      if (!mbar_wait_bounded(bar(kBarRawFull + s), (it / kTcRaw) & 1) ||
          (it >= kTcConv &&
           !mbar_wait_bounded(bar(kBarCvtEmpty + cb), ((it / kTcConv) - 1) & 1))) {
        if (lane == 0) fail();
        break;
      }
      if (*abort_flag) break;
      const uint8_t* rawK = smem + Ly::kRaw + s * Ly::kRawBytes;
      const uint8_t* rawV = rawK + kTcPages * Ly::kTile;
      uint8_t* kc = smem + Ly::kKc + cb * Ly::kConvBytes;
      uint8_t* vc = smem + Ly::kVc + cb * Ly::kConvBytes;
      const uint16_t* rs =
          reinterpret_cast<const uint16_t*>(smem + Ly::kRawSc) + s * kTcPages * 32;
      // the tile's largest V scale over the tokens that were copied and
      // belong to the sequence (other slots may hold anything), reduced by
      // every converter warp itself; F = its running maximum's FP32 exponent
      // (the softmax tracks the same F from vmax)
      const int vlim = min(L, npages * kBlockSize) - it * kTcKv;   // valid tokens of the tile
      uint32_t vb = 0;
#pragma unroll
      for (int t = lane; t < kTcKv; t += 32)
        if (t < vlim)
          vb = max(vb, __float_as_uint(__half2float(__ushort_as_half(rs[(t >> 4) * 32 + 16 + (t & 15)]))));
      vb = redux_max_u32(vb);
      cvt_f = max(cvt_f, (int)(vb >> 23));
      const float vsf = exp2i(127 - cvt_f);
      if (warp == kWarpCvt && lane == 0) {
        float* vm = reinterpret_cast<float*>(smem + Ly::kVmax) + 2 * cb;
        vm[0] = __uint_as_float(vb);
        vm[1] = 0.f;
      }
      // 16 codes (chunk c of token t) -> FP16 chunks 2c, 2c+1 of row t; K
      // exact, V times its token's s_v 2^(127 - F)
#pragma unroll
      for (int pass = 0; pass < kTcKv * (D / 16) / 128; ++pass) {
        // D = 128: a quarter-warp takes 4 chunks of each of two adjacent
        // tokens, so that its 16-byte reads (raw rows) and writes (converted
        // rows, swizzled) each cover all eight bank groups
        const int e = ct + 128 * pass;
        const int t = D == 128 ? 16 * pass + 4 * (warp - kWarpCvt) + 2 * (lane >> 4) +
                                     (((lane >> 2) ^ (lane >> 3)) & 1)
                               : e / (D / 16);
        const int c = D == 128 ? (lane & 7) : e - t * (D / 16);
        const int src = (t >> 4) * Ly::kTile + tile_off<C>(t & 15, c);
        convert_chunk<D>(rawK + src, kc, t, c);
        const float f =
            t < vlim ? __half2float(__ushort_as_half(rs[(t >> 4) * 32 + 16 + (t & 15)])) * vsf : 0.f;
        convert_chunk_scaled<D>(rawV + src, vc, t, c, __float2half2_rn(f));
      }
      // K scale column (times sm_scale log2 e)
      if (ct < kTcKv) {
        float* cs = reinterpret_cast<float*>(smem + Ly::kColSc) + cb * 2 * kTcKv;
        cs[ct] = __half2float(__ushort_as_half(rs[(ct >> 4) * 32 + (ct & 15)])) * p.scale_log2;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kBarCvtFull + cb));
        mbar_arrive(bar(kBarRawEmpty + s));
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc_idesc_f16(kTcKv, false);
      constexpr uint32_t idO = tc_idesc_f16(D, false, true);
      bool good = true;
      // step it: P V of tile it-1 then S of tile it, for each half in range
      for (int it = 0; it <= n_it && good; ++it) {
        const int cb = it % kTcConv, pcb = (it + kTcConv - 1) % kTcConv;
        if (it < n_it) {
          if (!mbar_wait_bounded(bar(kBarCvtFull + cb), (it / kTcConv) & 1) || *abort_flag) {
            good = false;
            break;
          }
          tc_fence_after();
        }
#pragma unroll
        for (int h = 0; h < kTcHalves; ++h) {
          if (it >= 1 && it <= n_half[h]) {
            const int k = it - 1;
            if (!mbar_wait_bounded(bar(kBarPFull + h), k & 1)) {
              good = false;
              break;
            }
            tc_fence_after();
            const uint32_t vb = smem_u32(smem + Ly::kVc + pcb * Ly::kConvBytes);
#pragma unroll
            for (int ts = 0; ts < kTcKv / 16; ++ts)
              tc_mma_f16_tmem_a(tO(h), tP(h) + 8 * ts,
                                tc_desc_sw128_mn(vb + 16 * 128 * ts, kTcKv * 128), idO,
                                k > 0 || ts > 0);
            if (it == n_half[h]) tc_commit(bar(kBarODone + h));   // the half's O is final
          }
          if (it < n_half[h]) {
            const uint32_t kbase = smem_u32(smem + Ly::kKc + cb * Ly::kConvBytes);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
              tc_mma_f16_tmem_a(tS(h), tQ(h) + 8 * ks,
                                tc_desc_sw128(kbase + (ks >> 2) * (kTcKv * 128) + 32 * (ks & 3)),
                                idS, ks > 0);
            tc_commit(bar(kBarSFull + h));         // also covers the P V above
          }
        }
        if (good && it >= 1) tc_commit(bar(kBarCvtEmpty + pcb));   // tile it-1 fully used
      }
      if (!good) fail();
      tc_commit(bar(kBarFin));                    // every MMA issued has completed
      mbar_wait_bounded(bar(kBarFin), 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- softmax
    const int h = warp >> 2;                      // half
    const int r = 32 * (warp & 3) + lane;         // row = TMEM lane
    const int iq = i_begin + h * TH + r / G;
    const int pos = (r < TH * G && iq < n) ? L - n + iq : -1;   // -1: padding row
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    const int nh = n_half[h];
    float m_use = -INFINITY, l = 0.f;
    // the row's scores are (S * K scale) * qf (BF16 queries entered as q / qf)
    // V scales go onto P: P' = P s_v 2^(127 - vfb) with vfb the FP32 biased
    // exponent of the largest V scale so far (all rows see the same tokens,
    // so it moves for all rows at once); O accumulates in units of
    // 2^(vfb - 127) and is rescaled when vfb grows
    int vfb = 0;
    bool good = true;
    for (int it = 0; it < nh; ++it) {
      const int cb = it % kTcConv;
      // S of this tile has landed (and with it the P V of the previous tile)
      const bool w_ok = mbar_wait_bounded(bar(kBarCvtFull + cb), (it / kTcConv) & 1) &&
                        mbar_wait_bounded(bar(kBarSFull + h), it & 1);
      if (!__all_sync(0xFFFFFFFFu, w_ok)) {
        good = false;
        break;
      }
      tc_fence_after();
      // the tile's K scale column (times sm_scale log2 e)
      const float4* cs4 = reinterpret_cast<const float4*>(smem + Ly::kColSc) + cb * (kTcKv / 2);
      const int t0 = it * kTcKv;
      const bool masked = t0 + kTcKv - 1 > pos;    // some token of the tile is past the row
      float z[kTcKv];
      {
        uint32_t sr[kTcKv];
        tc_ld64(tS(h) + lanes, sr);
#pragma unroll
        for (int x = 0; x < kTcKv; x += 4) {
          const float4 k4 = cs4[x / 4];
          const float2 a = __fmul2_rn(make_float2(__uint_as_float(sr[x]), __uint_as_float(sr[x + 1])),
                                      make_float2(k4.x, k4.y));
          const float2 c = __fmul2_rn(
              make_float2(__uint_as_float(sr[x + 2]), __uint_as_float(sr[x + 3])),
              make_float2(k4.z, k4.w));
          z[x] = a.x;
          z[x + 1] = a.y;
          z[x + 2] = c.x;
          z[x + 3] = c.y;
        }
      }
      if (masked) {
#pragma unroll
        for (int t = 0; t < kTcKv; ++t)
          if (t0 + t > pos) z[t] = -INFINITY;
      }
      float mx;
      {
        // three-way tree (64 -> 22 -> 8 -> 3 -> 1): short dependency chains
        static_assert(kTcKv == 64, "the max tree is laid out for 64 tokens");
        float m1[22], m2[8];
#pragma unroll
        for (int t = 0; t < 21; ++t) m1[t] = fmax3(z[t], z[t + 21], z[t + 42]);
        m1[21] = z[63];
#pragma unroll
        for (int t = 0; t < 7; ++t) m2[t] = fmax3(m1[t], m1[t + 7], m1[t + 14]);
        m2[7] = m1[21];
        mx = fmax3(fmax3(m2[0], m2[1], m2[2]), fmax3(m2[3], m2[4], m2[5]), fmaxf(m2[6], m2[7]));
        mx *= qf;
      }
      const bool grow = mx > m_use + 8.f;
      const float m_new = grow ? mx : m_use;
      const bool resc = grow && m_use != -INFINITY;
      const float alpha = resc ? fast_exp2(m_use - m_new) : 1.f;
      m_use = m_new;
      const float ref = m_use == -INFINITY ? 0.f : m_use;
      float fs = 1.f;                             // O's unit change
      {
        const float* vm = reinterpret_cast<const float*>(smem + Ly::kVmax) + 2 * cb;
        const int eb = (int)(max(__float_as_uint(vm[0]), __float_as_uint(vm[1])) >> 23);
        if (eb > vfb) {
          if (it > 0) fs = exp2i(vfb - eb);       // the first tile starts from O = 0
          vfb = eb;
        }
      }
      // P = 2^(z qf - m): the row sum and the P V operand (the V scales are
      // in the converted V tile; 0 for tokens past the row); FP32 pairs go
      // through the packed (two-lane) FMA instructions
      float lsum;
      {
        const float2 qf2 = make_float2(qf, qf), nref2 = make_float2(-ref, -ref);
        float2 acc[kTcKv / 4];
#pragma unroll
        for (int t = 0; t < kTcKv; t += 2) {
          float2 e = __ffma2_rn(make_float2(z[t], z[t + 1]), qf2, nref2);
          e.x = fast_exp2(e.x);
          e.y = fast_exp2(e.y);
          z[t] = e.x;
          z[t + 1] = e.y;
          acc[t >> 2] = (t & 2) ? __fadd2_rn(acc[t >> 2], e) : e;
        }
#pragma unroll
        for (int w = kTcKv / 8; w >= 1; w >>= 1)
#pragma unroll
          for (int t = 0; t < w; ++t) acc[t] = __fadd2_rn(acc[t], acc[t + w]);
        lsum = acc[0].x + acc[0].y;
      }
      l = fmaf(l, alpha, lsum);
      uint32_t pk[kTcKv / 2];                     // P packed two FP16 per TMEM column
#pragma unroll
      for (int cc = 0; cc < kTcKv / 8; ++cc) {
        float a8[8] = {z[8 * cc],     z[8 * cc + 1], z[8 * cc + 2], z[8 * cc + 3],
                       z[8 * cc + 4], z[8 * cc + 5], z[8 * cc + 6], z[8 * cc + 7]};
        if (masked) {
#pragma unroll
          for (int e2 = 0; e2 < 8; ++e2)
            if (t0 + 8 * cc + e2 > pos) a8[e2] = 0.f;
        }
#pragma unroll
        for (int e2 = 0; e2 < 4; ++e2)
          pk[4 * cc + e2] = h2_as_u32(__floats2half2_rn(a8[2 * e2], a8[2 * e2 + 1]));
      }
      tc_st32(tP(h) + lanes, pk);
      if (__any_sync(0xFFFFFFFFu, resc) || fs != 1.f) {
        // O holds P V of tiles 0..it-1 (complete: S of this tile was
        // committed after them): rescale the rows whose maximum moved, and
        // every row when the unit moved
        const float ra = alpha * fs;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t o[32];
          tc_ld32(tO(h) + c0 + lanes, o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * ra);
          tc_st32(tO(h) + c0 + lanes, o);
        }
      }
      tc_wait_st();                               // P' and any rescaled O are in TMEM
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kBarPFull + h));
    }
    if (good && nh > 0) {
      const bool w_ok = mbar_wait_bounded(bar(kBarODone + h), 0);
      good = __all_sync(0xFFFFFFFFu, w_ok);
    }
    if (!good) {
      if (lane == 0) fail();
    } else if (nh > 0) {
      // ---- epilogue: O / l, rounded to the activation dtype ----
      tc_fence_after();
      const float inv = l > 0.f ? exp2i(vfb - 127) / l : 0.f;
      uint16_t* dst = static_cast<uint16_t*>(p.out) +
                      ((int64_t)(q0 + (pos >= 0 ? iq : 0)) * p.Hq + (int64_t)j * G + r % G) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        tc_ld32(tO(h) + c0 + lanes, o);
        if (pos >= 0) {
#pragma unroll
          for (int x = 0; x < 32; x += 8) {
            uint4 w;
            uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const float a0 = __uint_as_float(o[x + 2 * e2]) * inv;
              const float a1 = __uint_as_float(o[x + 2 * e2 + 1]) * inv;
              if constexpr (BF16) wp[e2] = bf2_as_u32(__floats2bfloat162_rn(a0, a1));
              else wp[e2] = h2_as_u32(__floats2half2_rn(a0, a1));
            }
            *reinterpret_cast<uint4*>(dst + c0 + x) = w;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tc_dealloc(tmem, kTcCols);
  }
}

}  // namespace

size_t prefill_smem_bytes(int D) {
  return D == 128 ? TcLayout<128>::kTotal : TcLayout<64>::kTotal;
}

int prefill_rows_per_cta() { return kTcHalves * kTcRows; }

cudaError_t prefill_configure(int D, bool bf16) {
  const void* f = D == 128 ? (bf16 ? reinterpret_cast<const void*>(&paged_prefill_kernel<128, true>)
                                   : reinterpret_cast<const void*>(&paged_prefill_kernel<128, false>))
                           : (bf16 ? reinterpret_cast<const void*>(&paged_prefill_kernel<64, true>)
                                   : reinterpret_cast<const void*>(&paged_prefill_kernel<64, false>));
  return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)prefill_smem_bytes(D));
}

cudaError_t prefill_launch(int D, bool bf16, const CUtensorMap* maps, const PrefillParams& p,
                           int tiles, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)tiles, (unsigned)p.Hkv, (unsigned)p.B);
  cfg.blockDim = dim3(kTcThreads);
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
