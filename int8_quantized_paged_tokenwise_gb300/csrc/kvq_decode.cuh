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
//  * work distribution: the pages of all sequences form one column stream,
//    cut into ranges of R pages; a unit = (range, KV head) is processed by
//    one warp, units dealt round-robin with the KV head fastest, so that
//    neighbouring warps read neighbouring tiles of the same blocks.  By
//    default there are as many ranges as whole groups of Hkv warps, so every
//    warp gets the same number of pages whatever the mix of context lengths.
//    Inside a unit the warp walks "pieces" (the range's part of one
//    sequence); a piece that holds its whole sequence writes the output, a
//    partial piece writes a normalized partial + log2-sum-exp into one of the
//    unit's two slots for the combine kernel.  Every CTA
//    rebuilds the page prefix over sequences from context_lens in shared
//    memory; warps then run independently (no CTA-wide synchronization after
//    start-up) and no host-side planning is needed.
//  * each warp keeps one continuous stream of page loads across its pieces:
//    lanes 0..5 issue, S pages ahead of the consumer, TMA copies of the
//    (page, KV head) K and V tiles (2-D tensor copies with the 128-/64-byte
//    swizzle so that the ldmatrix reads are bank-conflict free, L2
//    evict-first since each tile is read once per call) and, for INT8,
//    the two 32-byte scale rows (1-D bulk copies), all completing on the
//    stage's mbarrier; a piece's first page also brings its query rows.
//    Block ids come from the block table 32 pages at a time, the next piece's
//    first chunk prefetched.  Waits are bounded (error bit + exit on timeout).
//  * QK^T and PV run on the tensor cores (mma.sync m16n8k16, FP32 accumulate)
//    with the GQA group as the N dimension (padded to 8), so each page is
//    read once for all query heads of its KV head.  INT8 codes become exact
//    FP16 integers with a byte permute and a subtraction; K scales multiply
//    the FP32 scores, V scales multiply the converted V pairs.
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

// STATIC: INT8 codes with one binary32 scale per tensor (no scale planes).
// H: KV heads processed together (a "head group"): the (page, head) tiles of
// H consecutive KV heads of a block are adjacent in the cache, so one copy
// brings the group's H tiles (16 H token rows) and its H scale rows.
// T: pages processed together (a step covers T consecutive pages of the
// group, each brought by its own copies).  H T <= 2.
template <int D, bool INT8, bool STATIC = false, int H = 1, int T = 1>
struct TileCfg {
  static constexpr int kElem = INT8 ? 1 : 2;                 // bytes per cache element
  static constexpr int kRowBytes = D * kElem;                // bytes per token row
  static constexpr int kSubRow = kRowBytes < 128 ? kRowBytes : 128;   // TMA box row bytes
  static constexpr int kSubTiles = kRowBytes / kSubRow;       // TMA copies per page tile
  static constexpr int kPageRows = H * kBlockSize;            // token rows of one page's tiles
  static constexpr int kRows = T * kPageRows;                 // token rows of a step
  static constexpr int kSubBytes = kRows * kSubRow;
  static constexpr int kTile = kRows * kRowBytes;             // bytes of a step's K (or V) tiles
  static constexpr int kStages = INT8 ? KVQ_INT8_STAGES : 2;  // steps in flight per warp
  static constexpr int kStageBytes = 2 * kTile;               // K tiles then V tiles
  static constexpr int kScaleBytes = INT8 && !STATIC ? 2 * kRows * 2 : 0;  // K, V scale rows
  // bytes one page brings: its K and V tiles and scale rows
  static constexpr uint32_t kPageTx = 2 * kPageRows * kRowBytes + kScaleBytes / T;
  static constexpr uint32_t kSwzMask = kSubRow == 128 ? 0x70u : 0x30u;
  static constexpr int kMinCtas = INT8 ? (H * T == 1 ? KVQ_INT8_MIN_CTAS : 3) : 3;
  static_assert(H * T <= 2, "steps of at most two page tiles");
};

// Byte offset inside a (K or V) tile of 16-byte chunk `c` of token row `t`,
// with the TMA swizzle applied (16-byte chunk index XOR row bits).
template <class C>
__device__ __forceinline__ uint32_t tile_off(int t, int c) {
  constexpr int cps = C::kSubRow / 16;  // chunks per sub-tile row
  const uint32_t off = (uint32_t)((c / cps) * C::kSubBytes + t * C::kSubRow + (c % cps) * 16);
  return off ^ ((off >> 3) & C::kSwzMask);
}

// ---------------------------------------------------------- work walk ---
// The pages of all sequences form one column stream (sequence-major; prefix[]
// is its inclusive page prefix over sequences, in shared memory); it is cut
// into ranges of R columns, and unit u = (range u / Hkv, KV head u % Hkv)
// goes to warp u mod (grid warps), so neighbouring warps read the same pages
// of neighbouring KV heads at about the same time.  All counts fit in 32 bits
// (checked on the host).  The walk state lives in shared memory and is only
// touched once per piece, keeping the page loop's registers for the math.

// CTA-wide constants of the walk.
struct WalkConst {
  int B, Hkv, G;
  int R;          // columns per range (0: segment mode, a range = one sequence)
  int T;          // columns in the stream
  int n;          // units
  int stride;     // warps in the grid = unit stride of a warp
  int step_c;     // stride / Hkv
  int step_j;     // stride % Hkv
  int pad[3];
};

// A piece: sequence b, KV head j, pages [pg0, pg0 + npg) of the sequence's L
// tokens, of work unit `unit`; flags bit 0: it covers the whole sequence,
// bit 1: it begins the sequence (partial slot 1, else slot 0).  npg == 0:
// no more pieces.
struct Piece {
  int b, j, pg0, npg, L, unit, flags, pad;
};

// The issuer's position: unit u = (range c, KV head j), the next column x of
// the range (which ends at x_end) and the sequence b holding x.
struct Cursor {
  int u, c, j, b, x, x_end;
};

// Per warp: the issuer's cursor and the descriptors of the pieces it has
// computed, indexed by piece ordinal mod 4 (the consumer reads piece k while
// the issuer holds k + 1 and k + 2).
struct WarpWalk {
  Cursor cur;
  int pad[2];
  Piece ring[4];
};

// Column window of unit (k.u, k.c, k.j) and the sequence at its start (x ==
// x_end when the unit is past the last one or, in segment mode, empty).
__device__ __forceinline__ void unit_window(const WalkConst& w, const int* prefix, Cursor& k) {
  if (k.u >= w.n) {
    k.x = k.x_end = 0;
    return;
  }
  if (w.R == 0) {
    k.b = k.c;
    k.x = k.b > 0 ? prefix[k.b - 1] : 0;
    k.x_end = prefix[k.b];
    return;
  }
  const int64_t x = (int64_t)k.c * w.R;
  k.x = (int)x;
  k.x_end = x + w.R < w.T ? (int)(x + w.R) : w.T;
  int lo = 0, hi = w.B - 1;                   // first b with prefix[b] > x
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] > k.x) hi = mid; else lo = mid + 1;
  }
  k.b = lo;
}

// The piece at the cursor, advancing it (to the warp's following units when
// the current one is used up).
__device__ __forceinline__ Piece next_piece(const WalkConst& w, const int* prefix,
                                            const int* lens, Cursor& k) {
  Piece pc;
  pc.npg = 0;
  while (k.x >= k.x_end) {
    if (k.u >= w.n) return pc;
    k.u += w.stride;
    k.c += w.step_c;
    k.j += w.step_j;
    if (k.j >= w.Hkv) {
      k.j -= w.Hkv;
      ++k.c;
    }
    unit_window(w, prefix, k);
  }
  while (prefix[k.b] <= k.x) ++k.b;           // skip sequences without pages
  const int first = k.b > 0 ? prefix[k.b - 1] : 0;
  const int pages = prefix[k.b] - first;
  pc.b = k.b;
  pc.j = k.j;
  pc.pg0 = k.x - first;
  pc.npg = min(pages - pc.pg0, k.x_end - k.x);
  pc.L = lens[k.b];
  pc.unit = k.c * w.Hkv + k.j;
  pc.flags = (pc.pg0 == 0 && pc.npg == pages ? 1 : 0) | (pc.pg0 == 0 ? 2 : 0);
  k.x += pc.npg;
  return pc;
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base).  Per warp:
// S page stages, one raw query slot (the TMA target, GH*D*2 bytes, GH = query
// heads of the head group) and the query fragments of the MMA B operand:
// per KV head h of the group, [k-step][lane] pairs holding the lane's column
// if that column is one of head h's query heads, else zeros.
template <int D, bool INT8, bool STATIC = false, int H = 1, bool CC = false, int T = 1>
struct SmemLayout {
  using C = TileCfg<D, INT8, STATIC, H, T>;
  // CUDA-core variant (CC): FP32 queries [G][D] and P' [G][16] instead
  static constexpr uint32_t kFragBytes =
      CC ? (uint32_t)kMaxGroup * (D + kBlockSize) * 4 : (uint32_t)H * (D / 16) * 32 * 8;
  size_t tiles, q, qfrag, scales, bars, stage_blk, misc, walk, seq, total_bytes;
  uint32_t q_bytes;  // one piece's query rows: GH * D * 2
  __host__ __device__ SmemLayout(int B, int GH) {
    q_bytes = (uint32_t)(GH * D * 2);
    tiles = 0;
    q = tiles + (size_t)kWarps * C::kStages * C::kStageBytes;
    qfrag = q + (size_t)kWarps * q_bytes;
    scales = qfrag + (size_t)kWarps * kFragBytes;
    bars = (scales + (size_t)kWarps * C::kStages * C::kScaleBytes + 15) & ~(size_t)15;
    stage_blk = bars + (size_t)kWarps * C::kStages * 8;
    misc = stage_blk + (size_t)kWarps * C::kStages * T * 4;   // 4 ints (scan of warp sums)
    walk = (misc + 16 + 15) & ~(size_t)15;                 // WalkConst, then per warp WarpWalk
    seq = walk + sizeof(WalkConst) + (size_t)kWarps * sizeof(WarpWalk);   // page prefix, lengths
    total_bytes = seq + (size_t)B * 8 + 1024;        // + alignment slack of the base
  }
};

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) return bf2_as_u32(__floats2bfloat162_rn(a, b));
  else return h2_as_u32(__floats2half2_rn(a, b));
}

// 16 INT8 codes (offset-binary after the XOR) -> 16 exact floats: each byte
// u = code + 128 goes under the exponent of 2^23 (0x4B000000 + u = 2^23 + u)
// and 2^23 + 128 is subtracted.
__device__ __forceinline__ void i8x16_to_f32(const uint4 w, float (&f)[16]) {
  const uint32_t x[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                         w.w ^ 0x80808080u};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int b = 0; b < 4; ++b)
      f[4 * i + b] = __uint_as_float(__byte_perm(x[i], 0x4B000000u, 0x7540u + b)) - 8388736.f;
  }
}

// The pipeline state one piece's consumer advances.
struct ConsumerState {
  int cs_slot;        // stage read next
  uint32_t cs_phase;  // parity of that wait
  uint32_t n_done;    // pages consumed
  int q_consumed;     // last piece whose query rows were read
};

// One piece on the CUDA cores: the counterpart of the tensor-core path for
// A/B measurements (same pages, same walk, same outputs).  Lane (t, half)
// forms the FP32 dot products of token t over half of the head dims for every
// query head of the group (FFMA over exactly converted codes, the halves
// joined by a shuffle); the online softmax runs per head over the 16 lanes of
// a half; for P V lane l owns head dims [l E, l E + E) of every head and
// reads the page's P' = p s_v (FP32) from shared memory.  Returns false if a
// wait timed out.
template <int D, bool QBF16, class Refill>
__device__ __forceinline__ bool cc_piece(const DecodeParams& p, const Piece& it, int ord,
                                         int lane, const uint16_t* q_raw, float* q32,
                                         float* pbuf, uint32_t tiles_u32,
                                         const uint16_t* scales_w, const int* blk_w,
                                         uint32_t bars_u32, ConsumerState& cs,
                                         Refill&& refill) {
  using C = TileCfg<D, true>;
  constexpr int S = C::kStages;
  constexpr int E = D / 32;           // output dims per lane
  constexpr int QC = D / 32;          // 16-byte K chunks per lane (half a row)
  const int G = p.G;
  const int t = lane & 15, half = lane >> 4;
  float m[kMaxGroup], l[kMaxGroup], o[kMaxGroup][E];
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[g][e] = 0.f;
  }
  for (int pg = 0; pg < it.npg; ++pg) {
    const int s = cs.cs_slot;
    const uint32_t par = cs.cs_phase;
    if (++cs.cs_slot == S) {
      cs.cs_slot = 0;
      cs.cs_phase ^= 1u;
    }
    if (!mbar_wait_bounded(bars_u32 + 8 * s, par)) return false;
    if (pg == 0) {
      for (int i = lane; i < G * D; i += 32) {
        const uint16_t b = q_raw[i];
        q32[i] = QBF16 ? __uint_as_float((uint32_t)b << 16) : __half2float(__ushort_as_half(b));
      }
      __syncwarp();
      cs.q_consumed = ord;
    }
    const int blk = blk_w[s];
    if (blk >= 0) {
      const uint32_t kt = tiles_u32 + s * C::kStageBytes;
      const uint32_t vt = kt + C::kTile;
      const int nvalid = min(kBlockSize, it.L - (it.pg0 + pg) * kBlockSize);
      // ---- scores: token t, all heads (the lane's half row converted once) ----
      float kf[QC * 16];
#pragma unroll
      for (int cc = 0; cc < QC; ++cc) {
        uint4 w;
        asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(w.x), "=r"(w.y), "=r"(w.z), "=r"(w.w)
                     : "r"(kt + tile_off<C>(t, half * QC + cc)));
        i8x16_to_f32(w, *reinterpret_cast<float(*)[16]>(kf + 16 * cc));
      }
      float acc[kMaxGroup];
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        acc[g] = 0.f;
        if (g < G) {
          const float4* qv = reinterpret_cast<const float4*>(q32 + g * D + half * QC * 16);
#pragma unroll
          for (int x = 0; x < QC * 4; ++x) {
            const float4 q4 = qv[x];
            acc[g] = fmaf(kf[4 * x], q4.x, acc[g]);
            acc[g] = fmaf(kf[4 * x + 1], q4.y, acc[g]);
            acc[g] = fmaf(kf[4 * x + 2], q4.z, acc[g]);
            acc[g] = fmaf(kf[4 * x + 3], q4.w, acc[g]);
          }
        }
      }
      const bool valid = t < nvalid;
      const float ks = p.scale_log2 * __half2float(__ushort_as_half(scales_w[s * (C::kScaleBytes / 2) + t]));
      const float sv =
          valid ? __half2float(__ushort_as_half(scales_w[s * (C::kScaleBytes / 2) + kBlockSize + t]))
                : 0.f;
      // ---- online softmax per head over the 16 tokens of a half ----
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g < G) {
          const float a = acc[g] + __shfl_xor_sync(0xFFFFFFFFu, acc[g], 16);
          const float z = valid ? a * ks : -INFINITY;
          float mx = z;
#pragma unroll
          for (int off = 1; off < 16; off <<= 1)
            mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, off));
          const float mn = fmaxf(m[g], mx);
          const float al = fast_exp2(m[g] - mn);
          const float pz = fast_exp2(z - mn);
          float ps = pz;
#pragma unroll
          for (int off = 1; off < 16; off <<= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, off);
          l[g] = l[g] * al + ps;
          m[g] = mn;
          if (al != 1.f) {
#pragma unroll
            for (int e = 0; e < E; ++e) o[g][e] *= al;
          }
          if (half == 0) pbuf[g * kBlockSize + t] = pz * sv;
        }
      }
      __syncwarp();
      // ---- P V: head dims [lane E, lane E + E) of every head ----
      const int d0 = lane * E;
      for (int tt = 0; tt < nvalid; ++tt) {
        const uint32_t a = vt + tile_off<C>(tt, d0 / 16) + (d0 % 16);
        float v[E];
        if constexpr (E == 4) {
          uint32_t w;
          asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(a));
          w ^= 0x80808080u;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            v[b] = __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u + b)) - 8388736.f;
        } else {
          uint16_t w;
          asm volatile("ld.shared.u16 %0, [%1];" : "=h"(w) : "r"(a));
          const uint32_t x = (uint32_t)w ^ 0x8080u;
#pragma unroll
          for (int b = 0; b < 2; ++b)
            v[b] = __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7540u + b)) - 8388736.f;
        }
#pragma unroll
        for (int g = 0; g < kMaxGroup; ++g) {
          if (g < G) {
            const float pp = pbuf[g * kBlockSize + tt];
#pragma unroll
            for (int e = 0; e < E; ++e) o[g][e] = fmaf(pp, v[e], o[g][e]);
          }
        }
      }
      __syncwarp();   // P' is rewritten by the next page
    }
    ++cs.n_done;
    __syncwarp();
    refill();
  }
  // ---- the whole sequence's output, or a partial for the combine ----
#pragma unroll
  for (int g = 0; g < kMaxGroup; ++g) {
    if (g < G) {
      const float inv = l[g] > 0.f ? 1.f / l[g] : 0.f;
      const int64_t hrow = (int64_t)it.b * p.Hq + (int64_t)it.j * G + g;
      if (it.flags & 1) {
        uint16_t* dst = static_cast<uint16_t*>(p.out) + hrow * D + lane * E;
        if constexpr (E == 4)
          *reinterpret_cast<uint2*>(dst) = make_uint2(pack2<QBF16>(o[g][0] * inv, o[g][1] * inv),
                                                       pack2<QBF16>(o[g][2] * inv, o[g][3] * inv));
        else
          *reinterpret_cast<uint32_t*>(dst) = pack2<QBF16>(o[g][0] * inv, o[g][1] * inv);
      } else {
        const int64_t prow = (2 * (int64_t)it.unit + (it.flags >> 1)) * G + g;
        float* dst = p.part_o + prow * D + lane * E;
        if constexpr (E == 4)
          *reinterpret_cast<float4*>(dst) =
              make_float4(o[g][0] * inv, o[g][1] * inv, o[g][2] * inv, o[g][3] * inv);
        else
          *reinterpret_cast<float2*>(dst) = make_float2(o[g][0] * inv, o[g][1] * inv);
        if (lane == 0) p.part_lse[prow] = l[g] > 0.f ? m[g] + __log2f(l[g]) : -INFINITY;
      }
    }
  }
  return true;
}

// INT8: QBF16 = activations are bf16 (converted to FP16 for the tensor cores);
// twin: QBF16 selects the bf16 MMA, otherwise FP16.  H: KV heads per head
// group; the walk sees p.Hkv = Hkv / H groups of p.G = G H query heads each
// (p.Gr = G), the group's query heads being consecutive.
// CC: the page math on the CUDA cores (cc_piece), for A/B measurements.
// T: pages per step (1, or 2 with H = 1).
template <int D, bool INT8, bool QBF16, bool STATIC = false, int H = 1, bool CC = false,
          int T = 1>
__global__ void __launch_bounds__(kThreads, CC ? 2 : TileCfg<D, INT8, STATIC, H, T>::kMinCtas)
    paged_decode_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const DecodeParams p) {
  using C = TileCfg<D, INT8, STATIC, H, T>;
  using Lay = SmemLayout<D, INT8, STATIC, H, CC, T>;
  static_assert(!CC || (INT8 && !STATIC && H == 1 && T == 1),
                "the CUDA-core variant is tokenwise INT8, one page per step");
  const Lay lay(p.B, p.G);
  static_assert(INT8 || H == 1, "head groups are built for the INT8 cache");
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
  WalkConst* wconst = reinterpret_cast<WalkConst*>(smem + lay.walk);
  WarpWalk* wwalk = reinterpret_cast<WarpWalk*>(smem + lay.walk + sizeof(WalkConst));
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
  // Programmatic dependent launch: wait here until the previous kernel in the
  // stream (e.g. the quantize-append that wrote the newest tokens) has
  // completed and its writes are visible, before reading any input; then let
  // the combine kernel be scheduled (it reads context_lens before waiting for
  // this grid).
  griddep_wait();
  griddep_launch_dependents();
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

  // ---- clamped lengths and the inclusive page prefix over sequences ----
  {
    const int per = (B + kThreads - 1) / kThreads;   // consecutive sequences per thread
    const int b0 = tid * per, b1 = min(B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      int L = __ldg(&p.context_lens[b]);
      if (L < 0 || L > max_tok) {
        atomicOr(p.err, 0x4u);
        L = L < 0 ? 0 : max_tok;
      }
      lens[b] = L;
      sum += (L + kBlockSize - 1) / kBlockSize;
    }
    int incl = sum;                                  // block-wide scan of per-thread sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) misc[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += misc[w];
    for (int b = b0; b < b1; ++b) {
      run += (lens[b] + kBlockSize - 1) / kBlockSize;
      prefix[b] = run;
    }
    // ---- constants of the work walk ----
    if (tid == 0) {
      WalkConst wc;
      wc.B = B;
      wc.Hkv = Hkv;
      wc.G = G;
      wc.T = 0;
      for (int w = 0; w < kWarps; ++w) wc.T += misc[w];
      wc.stride = (int)gridDim.x * kWarps;
      wc.step_c = wc.stride / Hkv;
      wc.step_j = wc.stride - wc.step_c * Hkv;
      if (p.R < 0) {
        wc.R = 0;                                  // one range per sequence
        wc.n = B * Hkv;
      } else {
        // balanced: p.groups ranges (about one per group of Hkv warps), so
        // that every warp gets one unit of ceil(columns / groups) pages
        const int64_t even = ((int64_t)wc.T + p.groups - 1) / p.groups;
        wc.R = p.R > 0 ? p.R : (int)(even > kMinRangePages ? even : kMinRangePages);
        const int64_t n = ((int64_t)wc.T + wc.R - 1) / wc.R * Hkv;
        if (n > p.range_cap) {
          // the host sizes the slots for the largest stream its bound
          // allows; refuse rather than write past them
          atomicOr(p.err, 0x4u);
          wc.n = 0;
        } else {
          wc.n = (int)n;
        }
      }
      *wconst = wc;
    }
  }
  fence_mbar_init();
  __syncthreads();

  if (blockIdx.x == 0) {
    // sequences without tokens are in no range: their output is zero
    const int row16 = p.Hq * D / 8;                  // 16-byte stores per sequence
    for (int b = tid; b < B; b += kThreads)
      if (lens[b] == 0) {
        uint4* o = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + (int64_t)b * p.Hq * D);
        for (int i = 0; i < row16; ++i) o[i] = make_uint4(0, 0, 0, 0);
      }
  }
  const int wg = blockIdx.x * kWarps + warp;                   // this warp's first unit

  const uint32_t tiles_u32 = smem_u32(smem + lay.tiles) + warp * S * C::kStageBytes;
  const uint32_t q_u32 = smem_u32(smem + lay.q) + warp * lay.q_bytes;
  uint2* qfrag = reinterpret_cast<uint2*>(smem + lay.qfrag + (size_t)warp * Lay::kFragBytes);
  // this lane's B fragment of (KV head h of the group, k-step ks):
  // qfrag_lane_u32 + qhs * h + qks * ks; columns of other heads (and the
  // padded ones, g >= G H) hold zeros there
  const uint32_t qfrag_lane_u32 = smem_u32(qfrag) + 8 * lane;
  constexpr uint32_t qks = 32u * 8u;                             // bytes per k-step
  constexpr uint32_t qhs = qks * KSTEPS;                         // bytes per KV head
  // KV head (within the group) of this thread's score columns 2c, 2c+1 and
  // of its B column g
  const int Gr = H > 1 ? p.Gr : G;
  const int hc0 = min(2 * c / Gr, H - 1), hc1 = min((2 * c + 1) / Gr, H - 1);
  const int hg = g / Gr;
  const uint32_t scales_u32 = smem_u32(smem + lay.scales) + warp * S * C::kScaleBytes;
  const uint16_t* scales_w =
      reinterpret_cast<const uint16_t*>(smem + lay.scales) + warp * S * (C::kScaleBytes / 2);
  const uint32_t bars_u32 = smem_u32(&bars[warp * S]);
  int* blk_w = stage_blk + warp * S * T;   // per stage: the T pages' block ids

  // Each page arrives as copies issued together by lanes 0..3: 2-D tensor TMA
  // of the K and V tiles (16-bit tiles in 128-byte-wide sub-tiles; a tiled
  // TMA needs a 128-byte aligned shared destination, which the tiles have)
  // and, for INT8, 1-D bulk copies of the K and V scale rows (16-byte aligned
  // destinations).  Per lane: tensor map, x coordinate and destination (+ the
  // per-stage stride), or the scale plane and destination.
  // Lanes [0, T * kTensorCopies): page lane / kTensorCopies, copy lane %
  // kTensorCopies (K sub-tiles, then V sub-tiles); the next 2 T lanes: page
  // (lane - base) / 2, K or V scale row; lane kQLane: the query rows.
  constexpr int kTensorCopies = 2 * C::kSubTiles;
  constexpr int kScaleLanes = INT8 && !STATIC ? 2 * T : 0;
  constexpr int kQLane = T * kTensorCopies + kScaleLanes;
  const int cp_i = lane % kTensorCopies;
  const int cp_page = lane < T * kTensorCopies ? lane / kTensorCopies
                      : (lane - T * kTensorCopies) / 2;       // page of this lane's copy
  const CUtensorMap* cp_map = cp_i < C::kSubTiles ? &tmK : &tmV;
  const int cp_sub = cp_i % C::kSubTiles;               // 128-byte column block
  const int cp_x = cp_sub * (C::kSubRow / C::kElem);
  const uint32_t cp_dst = tiles_u32 + (cp_i < C::kSubTiles ? 0 : C::kTile) + cp_sub * C::kSubBytes +
                          cp_page * C::kPageRows * C::kSubRow;
  const int sc_kind = (lane - T * kTensorCopies) & 1;   // 0: K scales, 1: V scales
  const uint16_t* sc_src = sc_kind == 0 ? p.k_scale : p.v_scale;
  const uint32_t sc_dst =
      scales_u32 + (sc_kind == 0 ? 0 : C::kRows * 2) + cp_page * C::kPageRows * 2;

  // ---------------------------------------------------------------- issuer
  // Warp-uniform state; lanes 0..5 perform the copies.  The block ids of the
  // current 32-page chunk live one per lane (blk_cur); the first chunk of the
  // following piece is prefetched into blk_nxt.
  int is_ord = 0, is_pg = 0, is_chunk = 0;
  int q_issued = -1;                    // ordinal of the last piece whose query was copied
  // consumer side: next stage and its parity, pages consumed, last piece
  // whose query rows were read
  ConsumerState cs{0, 0u, 0u, -1};
  WarpWalk& ww = wwalk[warp];
  // the issuer's piece (the fields the page issue needs); the following
  // piece's descriptor is in ww.ring and its first block-id chunk in blk_nxt
  int is_b = 0, is_j = 0, is_pg0 = 0, is_npg = 0;
  int blk_cur = -1, blk_nxt = -1;
  uint32_t n_issued = 0;
  int is_slot = 0;                       // stage the next issued page goes to

  auto load_chunk = [&](int b, int pg0, int npg, int base) -> int {
    const int pg = base + lane;
    int blk = -1;
    if (pg < npg) {
      blk = __ldg(&p.block_tables[(int64_t)b * p.max_blocks + pg0 + pg]);
      if (blk < 0 || blk >= p.num_blocks) {
        atomicOr(p.err, 0x2u);
        blk = -1;
      }
    }
    return blk;
  };
  // piece `ord` of the walk into ring[ord & 3] (cursor kept in shared
  // memory); returns its first block-id chunk
  auto walk_next = [&](int ord) -> int {
    Cursor k = ww.cur;
    const Piece pc = next_piece(*wconst, prefix, lens, k);
    __syncwarp();
    if (lane == 0) {
      ww.cur = k;
      ww.ring[ord & 3] = pc;
    }
    __syncwarp();
    return load_chunk(pc.b, pc.pg0, pc.npg, 0);
  };
  {
    const WalkConst& wc = *wconst;
    Cursor k;
    k.u = wg;
    k.c = wg / Hkv;
    k.j = wg - k.c * Hkv;
    unit_window(wc, prefix, k);
    if (lane == 0) ww.cur = k;
    __syncwarp();
    blk_cur = walk_next(0);
    const Piece& p0 = ww.ring[0];
    is_b = p0.b;
    is_j = p0.j;
    is_pg0 = p0.pg0;
    is_npg = p0.npg;
    if (is_npg > 0) blk_nxt = walk_next(1);
  }

  // Issue pages while fewer than S are in flight; a piece's first page (which
  // also copies the piece's query rows into the single raw query slot) waits
  // until the previously copied query rows have been read by the consumer.
  auto refill = [&]() {
    while (n_issued - cs.n_done < (uint32_t)S) {
      if (is_npg > 0 && is_pg >= is_npg) {   // next piece (pieces have pages)
        ++is_ord;
        const Piece& nx = ww.ring[is_ord & 3];
        is_b = nx.b;
        is_j = nx.j;
        is_pg0 = nx.pg0;
        is_npg = nx.npg;
        is_pg = 0;
        is_chunk = 0;
        blk_cur = blk_nxt;
        if (is_npg > 0) blk_nxt = walk_next(is_ord + 1);
      }
      if (is_npg == 0 || (is_pg == 0 && q_issued > cs.q_consumed)) return;
      if (is_pg >= is_chunk + 32) {
        is_chunk += 32;
        blk_cur = load_chunk(is_b, is_pg0, is_npg, is_chunk);
      }
      // the step's T pages (T divides 32, so they share the chunk); a page
      // past the piece reads as -1 from load_chunk
      int blk_p[T];
#pragma unroll
      for (int pp = 0; pp < T; ++pp)
        blk_p[pp] = __shfl_sync(0xFFFFFFFFu, blk_cur, is_pg + pp - is_chunk);
      const int s = is_slot;
      is_slot = is_slot + 1 == S ? 0 : is_slot + 1;
      const uint32_t bar = bars_u32 + 8 * s;
      const uint32_t qbytes = is_pg == 0 ? lay.q_bytes : 0u;
      if (lane == 0) {
        uint32_t tx = qbytes;
#pragma unroll
        for (int pp = 0; pp < T; ++pp) {
          blk_w[T * s + pp] = blk_p[pp];
          if (blk_p[pp] >= 0) tx += C::kPageTx;
        }
        if (tx) mbar_arrive_expect_tx(bar, tx);
        else mbar_arrive(bar);
      }
      const int blk = T == 1 || cp_page != 1 ? blk_p[0] : blk_p[T - 1];
      if (blk >= 0) {
        const int row = blk * Hkv + is_j;             // (block, head group) tile index
        if (lane < T * kTensorCopies) {
          tma_load_2d_evict_first(cp_dst + s * C::kStageBytes, cp_map, cp_x, row * C::kPageRows,
                                  bar);
        } else if (lane < kQLane) {
          bulk_load(sc_dst + s * C::kScaleBytes, sc_src + (int64_t)row * C::kPageRows,
                    C::kPageRows * 2, bar);
        }
      }
      if (qbytes && lane == kQLane) {
        const uint16_t* qsrc = static_cast<const uint16_t*>(p.q) +
                               ((int64_t)is_b * p.Hq + (int64_t)is_j * G) * D;
        bulk_load(q_u32, qsrc, qbytes, bar);
      }
      if (is_pg == 0) q_issued = is_ord;
      ++n_issued;
      is_pg += T;
    }
  };
  refill();

  // -------------------------------------------------------------- consumer
  int ord = 0;
  bool aborted = false;
  for (;; ++ord) {
    // the issuer computed this piece's descriptor before issuing its pages
    const int it_npg = ww.ring[ord & 3].npg;
    if (it_npg == 0) break;
    const int it_pg0 = ww.ring[ord & 3].pg0, it_L = ww.ring[ord & 3].L;
    if constexpr (CC) {
      const uint16_t* q_raw =
          reinterpret_cast<const uint16_t*>(smem + lay.q) + (size_t)warp * (lay.q_bytes / 2);
      float* q32 = reinterpret_cast<float*>(smem + lay.qfrag + (size_t)warp * Lay::kFragBytes);
      const Piece piece = ww.ring[ord & 3];
      if (!cc_piece<D, QBF16>(p, piece, ord, lane, q_raw, q32, q32 + kMaxGroup * D, tiles_u32,
                              scales_w, blk_w, bars_u32, cs, refill)) {
        aborted = true;
        break;
      }
      continue;
    }
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
    // BF16 queries enter the FP16 MMAs as q * 2^-sh per head (exact: the
    // head's largest |q| lands in [2^14, 2^15)); qs0/qs1 = 2^sh of the heads
    // 2c, 2c+1 of this thread's score columns multiply their scores.
    float qs0 = 1.f, qs1 = 1.f;
    // INT8 K codes enter the QK MMAs as 1152 + code (no subtraction in the
    // conversion): the score of head column n then carries 1152 * sum_d q[n][d],
    // kb0 / kb1 for this thread's columns 2c / 2c + 1, removed before scaling.
    float kb0 = 0.f, kb1 = 0.f;
    // Tokenwise V scales go onto P: P' = p * s_v * 2^(15 - vfb), vfb the FP16
    // biased exponent of the largest V scale of the piece so far (so P' < 2);
    // O accumulates in units of 2^(vfb - 15) and is rescaled when vfb grows.
    int vfb = 0;

    for (int pg = 0; pg < it_npg; pg += T) {
      const int s = cs.cs_slot;
      const uint32_t par = cs.cs_phase;
      if (++cs.cs_slot == S) {
        cs.cs_slot = 0;
        cs.cs_phase ^= 1u;
      }
      if (!mbar_wait_bounded(bars_u32 + 8 * s, par)) {
        aborted = true;
        break;
      }
      if (pg == 0) {
        // query fragments (the MMA B operand, column g = head g < G), from the
        // raw rows to this lane's slots of the fragment buffer
        const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + lay.q) +
                             (size_t)warp * (lay.q_bytes / 2) + g * D;
        float qinv = 1.f;            // 2^-sh of head g (BF16 queries)
        if constexpr (INT8 && QBF16) {
          // the head's largest |q| over its four lanes' elements
          uint32_t mx = 0;
          if (has_head) {
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
              const uint2 v = *reinterpret_cast<const uint2*>(qs + 16 * ks + 4 * c);
              mx = __vmaxu2(mx, __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu));
            }
          }
          mx = max(mx & 0xFFFFu, mx >> 16);
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
          mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
          const int sh = bf16_fp16_shift(mx);
          qinv = exp2i(-sh);
          const float qsg = exp2i(sh);               // 2^-126 for padded columns
          qs0 = __shfl_sync(0xFFFFFFFFu, qsg, 8 * c);
          qs1 = __shfl_sync(0xFFFFFFFFu, qsg, 8 * c + 4);
        }
        float qsum = 0.f;            // head g's query sum, over this lane's elements
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
          uint2 f = make_uint2(0u, 0u);
          if (has_head) {
            if constexpr (INT8) {
              // logical k {2c,2c+1,2c+8,2c+9} of step ks <-> head-dim 16ks+4c+{0..3}
              const uint2 v = *reinterpret_cast<const uint2*>(qs + 16 * ks + 4 * c);
              if constexpr (QBF16) {
                f.x = h2_as_u32(__floats2half2_rn(__uint_as_float(v.x << 16) * qinv,
                                                  __uint_as_float(v.x & 0xFFFF0000u) * qinv));
                f.y = h2_as_u32(__floats2half2_rn(__uint_as_float(v.y << 16) * qinv,
                                                  __uint_as_float(v.y & 0xFFFF0000u) * qinv));
              } else {
                f = v;
              }
            } else {
              // natural order: k {2c,2c+1} <-> 16ks+2c, k {2c+8,2c+9} <-> 16ks+8+2c
              f.x = *reinterpret_cast<const uint32_t*>(qs + 16 * ks + 2 * c);
              f.y = *reinterpret_cast<const uint32_t*>(qs + 16 * ks + 8 + 2 * c);
            }
          }
          if constexpr (INT8) {
            const float2 a = __half22float2(u32_as_h2(f.x)), b = __half22float2(u32_as_h2(f.y));
            qsum += (a.x + a.y) + (b.x + b.y);
          }
          // the fragment goes to its KV head's MMAs; the others see zeros
#pragma unroll
          for (int h = 0; h < H; ++h)
            qfrag[(h * KSTEPS + ks) * 32 + lane] = h == hg ? f : make_uint2(0u, 0u);
        }
        if constexpr (INT8) {
          qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 1);
          qsum += __shfl_xor_sync(0xFFFFFFFFu, qsum, 2);
          kb0 = 1152.f * __shfl_sync(0xFFFFFFFFu, qsum, 8 * c);
          kb1 = 1152.f * __shfl_sync(0xFFFFFFFFu, qsum, 8 * c + 4);
        }
        __syncwarp();   // the raw query slot may be refilled once every lane is done
        cs.q_consumed = ord;
      }
      // the step's T pages: valid tokens of each (0 when the page is absent)
      int nv[T];
      bool any = false;
#pragma unroll
      for (int pp = 0; pp < T; ++pp) {
        nv[pp] = blk_w[T * s + pp] >= 0
                     ? min(kBlockSize, it_L - (it_pg0 + pg + pp) * kBlockSize) : 0;
        any |= nv[pp] > 0;
      }
      if (any) {
        const uint32_t kt = tiles_u32 + s * C::kStageBytes;
        const uint32_t vt = kt + C::kTile;
        // ldmatrix row address: matrices (tokens 0-7, chunk 2i), (8-15, 2i),
        // (0-7, 2i+1), (8-15, 2i+1) for lanes 0-7, 8-15, 16-23, 24-31
        const int lt = (lane & 7) + ((lane >> 3) & 1) * 8;

        // ---------- S[token][head] = K Q^T: M = 16 tokens, N = 8 heads ----------
        // per page two accumulators (even/odd k-steps) halve the dependent MMA
        // chain; the KV heads of a group add into the same S, each into its own
        // columns (the B fragments of the other columns are zero).  Tile rows:
        // page pp, head h -> rows 16 (pp H + h) ..
        float sa[T][4], sb[T][4];
#pragma unroll
        for (int pp = 0; pp < T; ++pp)
#pragma unroll
          for (int e = 0; e < 4; ++e) sa[pp][e] = sb[pp][e] = 0.f;
#pragma unroll
        for (int pp = 0; pp < T; ++pp) {
#pragma unroll
          for (int hk = 0; hk < (INT8 ? H * (KSTEPS / 2) : 0); ++hk) {
            const int h = hk / (KSTEPS / 2), kk = hk % (KSTEPS / 2);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<C>(16 * (pp * H + h) + lt, 2 * kk + (lane >> 4)), r0, r1, r2,
                    r3);
            const uint2 qa = lds_u2(qfrag_lane_u32 + qhs * h + qks * (2 * kk));
            const uint2 qb = lds_u2(qfrag_lane_u32 + qhs * h + qks * (2 * kk + 1));
            if constexpr (INT8) {
              // r0/r1: tokens g / g+8, head-dim 16(2kk)+4c+{0..3}; r2/r3: next chunk
              uint32_t a0, a2, a1, a3;
              i8x4_to_h2x2_b1152<0x4140u, 0x4342u>(r0, a0, a2);
              i8x4_to_h2x2_b1152<0x4140u, 0x4342u>(r1, a1, a3);
              mma_16816_acc<false>(sa[pp], a0, a1, a2, a3, qa.x, qa.y);
              i8x4_to_h2x2_b1152<0x4140u, 0x4342u>(r2, a0, a2);
              i8x4_to_h2x2_b1152<0x4140u, 0x4342u>(r3, a1, a3);
              mma_16816_acc<false>(sb[pp], a0, a1, a2, a3, qb.x, qb.y);
            }
          }
        }
        if constexpr (!INT8) {
          // 16-bit tiles: one 16-byte chunk holds 8 elements, so k-step ks spans
          // chunks 2ks and 2ks+1 and (r0, r1, r2, r3) is directly its A operand
#pragma unroll
          for (int ks = 0; ks < KSTEPS; ++ks) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kt + tile_off<C>(lt, 2 * ks + (lane >> 4)), r0, r1, r2, r3);
            const uint2 qa = lds_u2(qfrag_lane_u32 + qks * ks);
            // a0: token g, d 16ks+2c..; a1: token g+8; a2: token g, d 16ks+8+2c..; a3: g+8
            if (ks & 1) mma_16816_acc<MMA_BF16>(sb[0], r0, r1, r2, r3, qa.x, qa.y);
            else mma_16816_acc<MMA_BF16>(sa[0], r0, r1, r2, r3, qa.x, qa.y);
          }
        }

        // scores in log2 units, per page: z[pp][0] (token g, head 2c), [1] (g,
        // 2c+1), [2] (g+8, 2c), [3] (g+8, 2c+1) (static scales: the K scale is
        // folded into scale_log2); a column's K scales are those of its KV
        // head hc0 / hc1 (scale slots: page pp, head h, token t -> 16 (pp H + h) + t)
        float z[T][4];
#pragma unroll
        for (int pp = 0; pp < T; ++pp) {
          float ks0 = p.scale_log2, ks1 = p.scale_log2, ks80 = p.scale_log2, ks81 = p.scale_log2;
          if constexpr (INT8 && !STATIC) {
            const uint16_t* ksc = scales_w + s * (C::kScaleBytes / 2) + 16 * pp * H;
            ks0 *= __half2float(__ushort_as_half(ksc[16 * hc0 + g]));
            ks80 *= __half2float(__ushort_as_half(ksc[16 * hc0 + g + 8]));
            if constexpr (H > 1) {
              ks1 *= __half2float(__ushort_as_half(ksc[16 * hc1 + g]));
              ks81 *= __half2float(__ushort_as_half(ksc[16 * hc1 + g + 8]));
            } else {
              ks1 = ks0;
              ks81 = ks80;
            }
          }
          z[pp][0] = ((sa[pp][0] - kb0) + sb[pp][0]) * ks0;
          z[pp][1] = ((sa[pp][1] - kb1) + sb[pp][1]) * ks1;
          z[pp][2] = ((sa[pp][2] - kb0) + sb[pp][2]) * ks80;
          z[pp][3] = ((sa[pp][3] - kb1) + sb[pp][3]) * ks81;
          if (nv[pp] < kBlockSize) {
            if (g >= nv[pp]) z[pp][0] = z[pp][1] = -INFINITY;
            if (g + 8 >= nv[pp]) z[pp][2] = z[pp][3] = -INFINITY;
          }
        }

        // ---------- online softmax per head column (reduce over the 8 g-lanes) ----------
        // true scores are z * qs (BF16 queries); the factor enters the max
        // once and each exponent through an FMA
        float mx0 = fmaxf(z[0][0], z[0][2]), mx1 = fmaxf(z[0][1], z[0][3]);
#pragma unroll
        for (int pp = 1; pp < T; ++pp) {
          mx0 = fmaxf(mx0, fmaxf(z[pp][0], z[pp][2]));
          mx1 = fmaxf(mx1, fmaxf(z[pp][1], z[pp][3]));
        }
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xFFFFFFFFu, mx0, off));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xFFFFFFFFu, mx1, off));
        }
        if constexpr (INT8 && QBF16) {
          mx0 *= qs0;
          mx1 *= qs1;
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = fast_exp2(m0 - mn0), al1 = fast_exp2(m1 - mn1);
        // tokenwise V scales: the step's largest V scale (valid tokens) moves
        // the O unit up when it exceeds the running one; lg = 15 - vfb
        // shifts the exponents so that p' = p * 2^lg, and P' = p' * s_v < 2
        float ra = 1.f;     // O's unit change (power of two)
        int lg = 0;
        float sv[T][4];     // V scales of z[pp][0..3]
#pragma unroll
        for (int pp = 0; pp < T; ++pp)
#pragma unroll
          for (int e = 0; e < 4; ++e) sv[pp][e] = 1.f;
        if constexpr (INT8 && !STATIC) {
          const uint16_t* vsc = scales_w + s * (C::kScaleBytes / 2) + C::kRows;
          uint32_t vb = 0;                       // slots (page, head, token)
#pragma unroll
          for (int i = lane & (C::kRows == 16 ? 15 : 31); i < C::kRows; i += 32)
            if ((i & 15) < (i < 16 * H ? nv[0] : nv[T - 1])) vb = max(vb, (uint32_t)vsc[i]);
          const uint32_t vmax = redux_max_u32(vb);
          const int eb = max((int)(vmax >> 10), 1);
          if (eb > vfb) {
            if (pg > 0) ra = exp2i(vfb - eb);   // the first step starts from O = 0
            vfb = eb;
          }
          lg = 15 - vfb;
#pragma unroll
          for (int pp = 0; pp < T; ++pp) {
            const uint16_t* vp = vsc + 16 * pp * H;
            if (g < nv[pp]) {
              sv[pp][0] = __half2float(__ushort_as_half(vp[16 * hc0 + g]));
              sv[pp][1] = H > 1 ? __half2float(__ushort_as_half(vp[16 * hc1 + g])) : sv[pp][0];
            } else {
              sv[pp][0] = sv[pp][1] = 0.f;
            }
            if (g + 8 < nv[pp]) {
              sv[pp][2] = __half2float(__ushort_as_half(vp[16 * hc0 + g + 8]));
              sv[pp][3] = H > 1 ? __half2float(__ushort_as_half(vp[16 * hc1 + g + 8])) : sv[pp][2];
            } else {
              sv[pp][2] = sv[pp][3] = 0.f;
            }
          }
        }
        const float o0 = (float)lg - mn0, o1 = (float)lg - mn1;
        float pr[T][4];
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int pp = 0; pp < T; ++pp) {
          if constexpr (INT8 && QBF16) {
            pr[pp][0] = fast_exp2(fmaf(z[pp][0], qs0, o0));
            pr[pp][1] = fast_exp2(fmaf(z[pp][1], qs1, o1));
            pr[pp][2] = fast_exp2(fmaf(z[pp][2], qs0, o0));
            pr[pp][3] = fast_exp2(fmaf(z[pp][3], qs1, o1));
          } else {
            pr[pp][0] = fast_exp2(z[pp][0] + o0);
            pr[pp][1] = fast_exp2(z[pp][1] + o1);
            pr[pp][2] = fast_exp2(z[pp][2] + o0);
            pr[pp][3] = fast_exp2(z[pp][3] + o1);
          }
          ps0 += pr[pp][0] + pr[pp][2];
          ps1 += pr[pp][1] + pr[pp][3];
        }
        if constexpr (INT8 && !STATIC) {
          const float ul = exp2i(-lg);
          l0 = fmaf(ps0, ul, l0 * al0);
          l1 = fmaf(ps1, ul, l1 * al1);
#pragma unroll
          for (int pp = 0; pp < T; ++pp)
#pragma unroll
            for (int e = 0; e < 4; ++e) pr[pp][e] *= sv[pp][e];
        } else {
          l0 = l0 * al0 + ps0;
          l1 = l1 * al1 + ps1;
        }
        m0 = mn0;
        m1 = mn1;
        const float ra0 = al0 * ra, ra1 = al1 * ra;
        if (__any_sync(0xFFFFFFFFu, (ra0 != 1.f) || (ra1 != 1.f))) {
#pragma unroll
          for (int cb = 0; cb < D / 16; ++cb) {
            o[4 * cb + 0] *= ra0;
            o[4 * cb + 1] *= ra1;
            o[4 * cb + 2] *= ra0;
            o[4 * cb + 3] *= ra1;
          }
        }

        // ---------- O^T[d][head] += V^T P^T: M = 16 head-dims, N = 8 heads ----------
#pragma unroll
        for (int pp = 0; pp < T; ++pp) {
          // P'^T as the B operand: b0 = P'[tokens 2c, 2c+1][head g], b1 = tokens 2c+8, 2c+9
          const uint32_t pb0 = movmatrix_trans(pack2<MMA_BF16>(pr[pp][0], pr[pp][1]));
          const uint32_t pb1 = movmatrix_trans(pack2<MMA_BF16>(pr[pp][2], pr[pp][3]));
          if constexpr (INT8) {
            // exact codes; the V scales are in P' (tokenwise) or applied once
            // to the output (static).  KV head h of a group multiplies only
            // its own columns of P'^T (the lanes of other columns pass zeros).
#pragma unroll
            for (int hk = 0; hk < H * (KSTEPS / 2); ++hk) {
              const int h = hk / (KSTEPS / 2), kk = hk % (KSTEPS / 2);
              const uint32_t bm0 = H == 1 || hg == h ? pb0 : 0u;
              const uint32_t bm1 = H == 1 || hg == h ? pb1 : 0u;
              uint32_t r[4];
              ldsm_x4_trans(vt + tile_off<C>(16 * (pp * H + h) + lt, 2 * kk + (lane >> 4)), r[0],
                            r[1], r[2], r[3]);
#pragma unroll
              for (int x = 0; x < 2; ++x) {
                // r[2x]: tokens 2c, 2c+1; r[2x+1]: tokens 2c+8, 2c+9; bytes
                // {t0 d0, t0 d1, t1 d0, t1 d1} with d0 = 16cb + 2g (row g), d1 = d0 + 1 (row g+8)
                uint32_t ev0, od0, ev1, od1;
                i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * x], ev0, od0);
                i8x4_to_h2x2<0x4240u, 0x4341u>(r[2 * x + 1], ev1, od1);
                const int cb = 2 * kk + x;
                float* oq = o + 4 * cb;
                mma_16816_acc<false>(*reinterpret_cast<float(*)[4]>(oq), ev0, od0, ev1, od1, bm0,
                                     bm1);
              }
            }
          } else {
            // matrices: (tokens 0-7, chunk 2q), (0-7, 2q+1), (8-15, 2q), (8-15, 2q+1)
            const int vtk = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
            for (int qq = 0; qq < D / 16; ++qq) {
              uint32_t r0, r1, r2, r3;
              ldsm_x4_trans(vt + tile_off<C>(vtk, 2 * qq + ((lane >> 3) & 1)), r0, r1, r2, r3);
              // rows g: d = 16qq + g; rows g+8: d = 16qq + 8 + g
              float* oq = o + 4 * qq;
              mma_16816_acc<MMA_BF16>(*reinterpret_cast<float(*)[4]>(oq), r0, r1, r2, r3, pb0, pb1);
            }
          }
        }
      }
      ++cs.n_done;
      __syncwarp();
      refill();
    }
    if (aborted) break;

    // ---- finalize the piece: the whole sequence, or a partial for the combine ----
    const Piece it = ww.ring[ord & 3];
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
      // O's unit: the static V scale, or 2^(vfb - 15) (tokenwise), or 1 (twin)
      const float unit = STATIC ? p.v_static : (INT8 ? exp2i(vfb - 15) : 1.f);
      const float inv = l > 0.f ? unit / l : 0.f;
      const int64_t hrow = (int64_t)it.b * p.Hq + (int64_t)it.j * G + head;
      if (it.flags & 1) {
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
        const int64_t prow = (2 * (int64_t)it.unit + (it.flags >> 1)) * G + head;
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
    // the failed wait's stage is the one before cs.cs_slot (cs.cs_slot/cs.cs_phase advanced)
    int s = cs.cs_slot == 0 ? S - 1 : cs.cs_slot - 1;
    uint32_t ph = cs.cs_slot == 0 ? (cs.cs_phase ^ 1u) : cs.cs_phase;
    for (; cs.n_done < n_issued; ++cs.n_done) {
      mbar_wait_bounded(bars_u32 + 8 * s, ph);
      if (++s == S) {
        s = 0;
        ph ^= 1u;
      }
    }
  }
}

// Host side of one kernel variant: shared-memory size, attributes,
// occupancy and the launch (programmatic stream serialization, so that the
// launch may overlap the tail of the previous kernel in the stream; the
// kernel waits (griddepcontrol) before reading any input).
template <bool INT8, bool STATIC, int H, bool CC = false, int T = 1>
struct DecodeLaunch {
  template <int D, bool BF16>
  static const void* fn() {
    return reinterpret_cast<const void*>(&paged_decode_kernel<D, INT8, BF16, STATIC, H, CC, T>);
  }
  static const void* pick(int D, bool bf16) {
    if (D == 128) return bf16 ? fn<128, true>() : fn<128, false>();
    return bf16 ? fn<64, true>() : fn<64, false>();
  }
  static size_t smem(int D, int B, int GH) {
    return D == 128 ? SmemLayout<128, INT8, STATIC, H, CC, T>(B, GH).total_bytes
                    : SmemLayout<64, INT8, STATIC, H, CC, T>(B, GH).total_bytes;
  }
  static cudaError_t configure(int D, bool bf16, size_t bytes) {
    // all of the unified L1/shared array as shared memory: the kernel's
    // occupancy is set by its page stages
    cudaError_t e = cudaFuncSetAttribute(pick(D, bf16), cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(pick(D, bf16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)bytes);
  }
  static cudaError_t occupancy(int D, bool bf16, size_t bytes, int* n) {
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, pick(D, bf16), kThreads, bytes);
  }
  static cudaError_t launch(int D, bool bf16, const CUtensorMap* maps, const DecodeParams& p,
                            int grid, size_t bytes, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (D == 128) {
      return bf16 ? cudaLaunchKernelEx(&cfg, paged_decode_kernel<128, INT8, true, STATIC, H, CC, T>,
                                       maps[0], maps[1], p)
                  : cudaLaunchKernelEx(&cfg, paged_decode_kernel<128, INT8, false, STATIC, H, CC, T>,
                                       maps[0], maps[1], p);
    }
    return bf16 ? cudaLaunchKernelEx(&cfg, paged_decode_kernel<64, INT8, true, STATIC, H, CC, T>,
                                     maps[0], maps[1], p)
                : cudaLaunchKernelEx(&cfg, paged_decode_kernel<64, INT8, false, STATIC, H, CC, T>,
                                     maps[0], maps[1], p);
  }
  static constexpr DecodeOps ops() { return DecodeOps{&smem, &configure, &occupancy, &launch}; }
};

}  // namespace kvq
