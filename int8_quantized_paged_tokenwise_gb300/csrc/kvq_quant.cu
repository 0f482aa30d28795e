// Quantize-on-write of new K/V rows into the paged INT8 cache, and the plain
// 16-bit scatter used to fill the A/B twin's cache.
//
// Quantizer ("feat: opt-in INT8 KV-cache quantization", MoE-Infinity PR #183,
// "What landed"; "fix(cuda/kv): correct Int8 KV per-token scale",
// mlxcel PR #717, "The Int8 bug and fix"): per (token, KV head) row,
//   a = max |x|,  s = 1.0 if a == 0 else FP16 round-up of a/127,
//   code = clamp(rint(x / s), -127, 127).
//
// Exactness on the GPU.  a is found on the raw 16-bit magnitudes (integer max
// of the sign-cleared patterns orders finite values by magnitude), then
// decoded exactly to FP32.  a/127 rounded up to FP16 comes from one FP32
// product and a check (row_scale_bits below).
// The code is the exact quotient x / s rounded half to even: for an
// unsaturated row straight from the correctly rounded reciprocal, with an
// exact FMA remainder flagging the exact ties (quantize4_fast below), which
// are recomputed, as are saturated rows, by the remainder-corrected
// quant_code.
// No fast-math and no flush-to-zero: bf16 subnormal rows must keep a > 0.
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

namespace kvq {
namespace {

constexpr int kQuantThreads = 256;

template <bool BF16>
__device__ __forceinline__ float bits_to_float(uint32_t b) {
  if constexpr (BF16) {
    return __uint_as_float(b << 16);
  } else {
    return __half2float(__ushort_as_half((unsigned short)b));
  }
}

// FP16 bits of the row scale for magnitude pattern `amax_bits`: a/127
// rounded up to FP16, without a division.  y = a * fl(1/127) is within
// 2^-23 (relative) of a/127, and a/127 is either an FP16 value or at least
// 2^-17 (relative) away from every FP16 value, so rounding y up gives the
// scale unless a/127 is an FP16 value f and y landed above it; then the
// FP16 value below the result still covers a (127 times it, exact in FP32:
// 11 by 7 bits, is >= a) and is the scale.  The smallest result is 2^-24,
// so a > 0 never gets a zero scale.
template <bool BF16>
__device__ __forceinline__ uint16_t row_scale_bits(uint32_t amax_bits) {
  if (amax_bits == 0u) return 0x3C00u;                   // all-zero token -> 1.0
  const float a = bits_to_float<BF16>(amax_bits);
  unsigned short s = __half_as_ushort(__float2half_ru(__fmul_rn(a, 1.0f / 127.0f)));
  if (s >= 0x7C00u) return 0x7BFFu;                      // saturate at 65504
  if (__fmul_rn(127.0f, __half2float(__ushort_as_half((unsigned short)(s - 1u)))) >= a) --s;
  return s;
}

// The code of x: the exact quotient x / s rounded half to even, clamped to
// +-127, without a division.  x * inv (inv ~ 1/s) is limited to +-256 (only a
// saturated scale lets the quotient leave +-127 by more than rounding) and
// rounded to an integer k by adding M = 1.5 * 2^23, which leaves k in the low
// mantissa bits of t; k is within one of the answer.  The remainder x - k s
// is exact in one FMA (for |k| <= 128, k s has at most 19 significant bits
// and x - k s at most 12), and the quotient is k + r/s: k moves by one when
// |r| > s/2, and on an exact tie |r| = s/2 towards the even neighbour.  For
// |k| > 128 only the clamp to +-127 matters.
// SAT: the scale saturated at 65504, so |x / s| may exceed 127 (else the
// row's largest magnitude maps to at most 127 and neither clamp is needed).
template <bool SAT>
__device__ __forceinline__ int quant_code(float x, float s, float h, float inv) {
  constexpr float kM = 12582912.0f;              // 1.5 * 2^23
  float q = x * inv;
  if constexpr (SAT) q = fminf(fmaxf(q, -256.0f), 256.0f);
  const float t = q + kM;
  const float k = t - kM;
  int ki = (int)(__float_as_uint(t) - 0x4B400000u);   // k as an integer (|k| < 2^22)
  const float r = fmaf(-k, s, x);
  const bool odd = (ki & 1) != 0;
  ki += (r > h || (r == h && odd)) ? 1 : 0;
  ki -= (r < -h || (r == -h && odd)) ? 1 : 0;
  if constexpr (SAT) ki = min(max(ki, -127), 127);
  return ki;
}

template <bool BF16, bool SAT>
__device__ __forceinline__ uint32_t quantize4_as(uint2 x, float s, float inv) {
  const float h = 0.5f * s;
  const uint32_t c0 = (uint32_t)quant_code<SAT>(bits_to_float<BF16>(x.x & 0xFFFFu), s, h, inv);
  const uint32_t c1 = (uint32_t)quant_code<SAT>(bits_to_float<BF16>(x.x >> 16), s, h, inv);
  const uint32_t c2 = (uint32_t)quant_code<SAT>(bits_to_float<BF16>(x.y & 0xFFFFu), s, h, inv);
  const uint32_t c3 = (uint32_t)quant_code<SAT>(bits_to_float<BF16>(x.y >> 16), s, h, inv);
  return __byte_perm(__byte_perm(c0, c1, 0x0040u), __byte_perm(c2, c3, 0x0040u), 0x5410u);
}

// Four codes of an unsaturated row (|x / s| <= 127) from inv ~ 1/s (the
// approximate reciprocal, within 2^-23 relative): k = rint(x * inv), both
// steps rounded, is the round-half-even code of every quotient that is not
// an exact tie.  The product is within 127 * 1.5 * 2^-23 < 2^-15 of x / s,
// while a quotient of a 16-bit x by an FP16 s
// that is not a tie lies at least 2^-14 from every half-integer (near one,
// x / s >= 1/4, and with x = mx 2^e, s = ms 2^(e + d) its distance is a
// nonzero multiple of 1 / (2 ms 2^d), where ms 2^d <= 4 mx <= 2^13).  On an
// exact tie the product may land on either side, so the exact remainder
// x - k s = +-s/2 flags it and `tie` asks for quant_code.  The codes are the low bytes of
// the sums k + 1.5 * 2^23; the FP32 pairs go through the paired instructions.
template <bool BF16>
__device__ __forceinline__ uint32_t quantize4_fast(uint2 x, float s, float inv, bool& tie) {
  constexpr float kM = 12582912.0f;              // 1.5 * 2^23
  const float2 xa = make_float2(bits_to_float<BF16>(x.x & 0xFFFFu), bits_to_float<BF16>(x.x >> 16));
  const float2 xb = make_float2(bits_to_float<BF16>(x.y & 0xFFFFu), bits_to_float<BF16>(x.y >> 16));
  const float2 i2 = make_float2(inv, inv), m2 = make_float2(kM, kM);
  const float2 nm2 = make_float2(-kM, -kM), ns2 = make_float2(-s, -s);
  const float2 ta = __fadd2_rn(__fmul2_rn(xa, i2), m2);
  const float2 tb = __fadd2_rn(__fmul2_rn(xb, i2), m2);
  const float2 ra = __ffma2_rn(__fadd2_rn(ta, nm2), ns2, xa);
  const float2 rb = __ffma2_rn(__fadd2_rn(tb, nm2), ns2, xb);
  const float h = 0.5f * s;
  tie = fabsf(ra.x) == h || fabsf(ra.y) == h || fabsf(rb.x) == h || fabsf(rb.y) == h;
  return __byte_perm(__byte_perm(__float_as_uint(ta.x), __float_as_uint(ta.y), 0x0040u),
                     __byte_perm(__float_as_uint(tb.x), __float_as_uint(tb.y), 0x0040u),
                     0x5410u);
}

// Four 16-bit values -> four int8 codes packed little-endian (scale bits sb,
// inv ~ 1/s).
template <bool BF16>
__device__ __forceinline__ uint32_t quantize4(uint2 x, uint16_t sb, float s, float inv) {
  if (sb == 0x7BFFu) return quantize4_as<BF16, true>(x, s, inv);
  bool tie;
  const uint32_t c = quantize4_fast<BF16>(x, s, inv, tie);
  return tie ? quantize4_as<BF16, false>(x, s, inv) : c;
}

// The approximate reciprocal (relative error within 2^-23) serves both
// paths: quant_code tolerates a few ulp, quantize4_fast one and a half.
__device__ __forceinline__ float approx_rcp(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Largest magnitude pattern (sign cleared) among a lane's 16-bit values.
template <int NW>
__device__ __forceinline__ uint32_t mag_max(const uint32_t (&x)[NW]) {
  uint32_t m = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) m = __vmaxu2(m, x[w] & 0x7FFF7FFFu);
  return max(m & 0xFFFFu, m >> 16);
}

// D / EPL lanes per (token, KV head) row; each lane owns EPL consecutive
// elements (K and V each: one 8-byte load for EPL = 4, two 16-byte loads for
// EPL = 16).  Rows of one warp are adjacent heads of a token, so the 16-bit
// loads and the stores of a warp are contiguous runs.  Each warp takes kPasses
// such passes and issues every load of them (slots, K and V rows) before it
// uses any, so that a warp keeps several rows' loads in flight instead of
// waiting for one row's slot, then its values.  The quantizer takes EPL = 16:
// its per-row work (absmax, scales, addresses) is then shared by four rows
// per warp instruction at D = 128.
template <int D, int EPL>
struct RowTask {
  static constexpr int LPR = D / EPL;             // lanes per row
  static constexpr int RPW = 32 / LPR;            // rows per warp pass
  static constexpr int NW = EPL / 2;              // 32-bit words of K (or V) per lane
  static constexpr int kPasses = EPL == 4 ? 4 : 2;
  static_assert(EPL == 4 || EPL == 16, "8-byte or 32-byte lane slices");
  int64_t row[kPasses], t[kPasses], slot[kPasses];
  int j[kPasses];
  int sub;
  // this thread's rows and their slots, K and V words, all loads in flight
  __device__ __forceinline__ void load(const QuantParams& p, uint32_t (&kx)[kPasses][NW],
                                       uint32_t (&vx)[kPasses][NW]) {
    const int lane = threadIdx.x & 31;
    sub = lane % LPR;
    const int64_t wg = ((int64_t)blockIdx.x * kQuantThreads + threadIdx.x) / 32;
    const int64_t row0 = wg * (kPasses * RPW) + lane / LPR;
    // (token, head) of the first row by one division, the next ones by steps
    int64_t tt = row0 / p.num_kv_heads;
    int jj = (int)(row0 - tt * p.num_kv_heads);
#pragma unroll
    for (int i = 0; i < kPasses; ++i) {
      row[i] = row0 + i * RPW;
      slot[i] = -1;
      t[i] = tt;
      j[i] = jj;
#pragma unroll
      for (int w = 0; w < NW; ++w) kx[i][w] = vx[i][w] = 0u;
      jj += RPW;
      while (jj >= p.num_kv_heads) {              // at most RPW <= 8 turns
        jj -= p.num_kv_heads;
        ++tt;
      }
      if (row[i] < p.num_rows) {
        slot[i] = p.slots[t[i]];
        const uint16_t* kr =
            static_cast<const uint16_t*>(p.k) + t[i] * p.k_stride + (int64_t)j[i] * D + sub * EPL;
        const uint16_t* vr =
            static_cast<const uint16_t*>(p.v) + t[i] * p.v_stride + (int64_t)j[i] * D + sub * EPL;
        if constexpr (EPL == 4) {
          const uint2 a = __ldg(reinterpret_cast<const uint2*>(kr));
          const uint2 b = __ldg(reinterpret_cast<const uint2*>(vr));
          kx[i][0] = a.x; kx[i][1] = a.y;
          vx[i][0] = b.x; vx[i][1] = b.y;
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint4 a = __ldg(reinterpret_cast<const uint4*>(kr) + h);
            const uint4 b = __ldg(reinterpret_cast<const uint4*>(vr) + h);
            kx[i][4 * h] = a.x; kx[i][4 * h + 1] = a.y; kx[i][4 * h + 2] = a.z; kx[i][4 * h + 3] = a.w;
            vx[i][4 * h] = b.x; vx[i][4 * h + 1] = b.y; vx[i][4 * h + 2] = b.z; vx[i][4 * h + 3] = b.w;
          }
        }
      }
    }
  }
  // whether row i is written; a slot past the cache sets the error bit
  __device__ __forceinline__ bool active(const QuantParams& p, int i) const {
    if (row[i] >= p.num_rows || slot[i] < 0) return false;
    if (slot[i] >= p.num_slots) {
      if (sub == 0) atomicOr(p.err, 0x1u);
      return false;
    }
    return true;
  }
  // payload row of row i in the cache [NB][Hkv][bs]
  __device__ __forceinline__ int64_t cache_row(const QuantParams& p, int i) const {
    const int64_t blk = slot[i] / kBlockSize, off = slot[i] % kBlockSize;
    return (blk * p.num_kv_heads + j[i]) * kBlockSize + off;
  }
};

// EPL = 16 when the K and V rows allow 16-byte loads, else 4.
template <int D, bool BF16, int EPL>
__global__ void __launch_bounds__(kQuantThreads) quantize_append_kernel(const QuantParams p) {
  using RT = RowTask<D, EPL>;
  constexpr int NW = RT::NW, LPR = RT::LPR;
  // the next kernel in the stream (a decode launched with programmatic stream
  // serialization) may be scheduled now; it waits for this grid's completion
  griddep_launch_dependents();
  RT rt;
  uint32_t kx[RT::kPasses][NW], vx[RT::kPasses][NW];
  rt.load(p, kx, vx);
#pragma unroll
  for (int i = 0; i < RT::kPasses; ++i) {
    const bool act = rt.active(p, i);
    uint32_t km = mag_max<NW>(kx[i]), vm = mag_max<NW>(vx[i]);
    if constexpr (LPR == 32) {                    // one row per warp: one reduction
      km = __reduce_max_sync(0xFFFFFFFFu, km);
      vm = __reduce_max_sync(0xFFFFFFFFu, vm);
    } else {
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) {
        km = max(km, __shfl_xor_sync(0xFFFFFFFFu, km, off));
        vm = max(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, off));
      }
    }
    if (!act) continue;
    const uint16_t ks = row_scale_bits<BF16>(km);
    const uint16_t vs = row_scale_bits<BF16>(vm);
    const float ksf = __half2float(__ushort_as_half(ks));
    const float vsf = __half2float(__ushort_as_half(vs));
    const float kinv = approx_rcp(ksf), vinv = approx_rcp(vsf);
    uint32_t kc[NW / 2], vc[NW / 2];
#pragma unroll
    for (int g = 0; g < NW / 2; ++g) {
      kc[g] = quantize4<BF16>(make_uint2(kx[i][2 * g], kx[i][2 * g + 1]), ks, ksf, kinv);
      vc[g] = quantize4<BF16>(make_uint2(vx[i][2 * g], vx[i][2 * g + 1]), vs, vsf, vinv);
    }
    const int64_t crow = rt.cache_row(p, i);
    int8_t* kd = static_cast<int8_t*>(p.k_cache) + crow * D + rt.sub * EPL;
    int8_t* vd = static_cast<int8_t*>(p.v_cache) + crow * D + rt.sub * EPL;
    if constexpr (EPL == 16) {
      *reinterpret_cast<uint4*>(kd) = make_uint4(kc[0], kc[1], kc[2], kc[3]);
      *reinterpret_cast<uint4*>(vd) = make_uint4(vc[0], vc[1], vc[2], vc[3]);
    } else {
      *reinterpret_cast<uint32_t*>(kd) = kc[0];
      *reinterpret_cast<uint32_t*>(vd) = vc[0];
    }
    if (rt.sub == 0) {
      p.k_scale[crow] = ks;
      p.v_scale[crow] = vs;
    }
  }
}

// Static (per-tensor, binary32) scales: "fix: #552 int8 kv cache quantization
// cannot be enabled" (InfiniLM PR #553) and "Add calibrated INT8 KV cache to
// PyTorch backend" (TensorRT-LLM PR #18953) -- one scale per tensor applied
// through its reciprocal: code = clamp(rint(fl32(x * inv)), -127, 127) with
// inv = fl32(1 / scale) from the host.  __fmul_rn keeps the product one IEEE
// rounding (no contraction); no scale planes are written.
template <int D, bool BF16>
__global__ void __launch_bounds__(kQuantThreads) quantize_static_kernel(const QuantParams p,
                                                                         float inv_k,
                                                                         float inv_v) {
  griddep_launch_dependents();
  using RT = RowTask<D, 4>;
  RT rt;
  uint32_t kx[RT::kPasses][2], vx[RT::kPasses][2];
  rt.load(p, kx, vx);
#pragma unroll
  for (int i = 0; i < RT::kPasses; ++i) {
    if (!rt.active(p, i)) continue;
    const int64_t crow = rt.cache_row(p, i);
    uint32_t kq = 0, vq = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t kw = kx[i][e >> 1], vw = vx[i][e >> 1];
      const uint32_t kb = (e & 1) ? (kw >> 16) : (kw & 0xFFFFu);
      const uint32_t vb = (e & 1) ? (vw >> 16) : (vw & 0xFFFFu);
      const float kr8 =
          fminf(fmaxf(rintf(__fmul_rn(bits_to_float<BF16>(kb), inv_k)), -127.f), 127.f);
      const float vr8 =
          fminf(fmaxf(rintf(__fmul_rn(bits_to_float<BF16>(vb), inv_v)), -127.f), 127.f);
      kq |= (uint32_t)((int)kr8 & 0xFF) << (8 * e);
      vq |= (uint32_t)((int)vr8 & 0xFF) << (8 * e);
    }
    reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.k_cache) + crow * D)[rt.sub] = kq;
    reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.v_cache) + crow * D)[rt.sub] = vq;
  }
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) append_kv16_kernel(const QuantParams p) {
  using RT = RowTask<D, 4>;
  RT rt;
  uint32_t kx[RT::kPasses][2], vx[RT::kPasses][2];
  rt.load(p, kx, vx);
#pragma unroll
  for (int i = 0; i < RT::kPasses; ++i) {
    if (!rt.active(p, i)) continue;
    const int64_t crow = rt.cache_row(p, i);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.k_cache) + crow * D)[rt.sub] =
        make_uint2(kx[i][0], kx[i][1]);
    reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.v_cache) + crow * D)[rt.sub] =
        make_uint2(vx[i][0], vx[i][1]);
  }
}

// CTAs for `rows` rows: warps of RowTask<D, EPL>::kPasses passes of its
// rows per pass.
template <int D, int EPL>
inline int grid_for(int64_t rows) {
  using RT = RowTask<D, EPL>;
  const int64_t per_warp = (int64_t)RT::kPasses * RT::RPW;
  const int64_t threads = (rows + per_warp - 1) / per_warp * 32;
  return (int)((threads + kQuantThreads - 1) / kQuantThreads);
}

}  // namespace

template <int D, bool BF16, int EPL>
void quantize_append_go(const QuantParams& p, cudaStream_t s) {
  quantize_append_kernel<D, BF16, EPL><<<grid_for<D, EPL>(p.num_rows), kQuantThreads, 0, s>>>(p);
}

cudaError_t quantize_append_launch(int D, bool bf16, const QuantParams& p, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  // 32-byte lane slices need 16-byte aligned rows (pointers and token strides)
  const bool wide = (reinterpret_cast<uintptr_t>(p.k) % 16 == 0) &&
                    (reinterpret_cast<uintptr_t>(p.v) % 16 == 0) && p.k_stride % 8 == 0 &&
                    p.v_stride % 8 == 0;
  if (D == 128) {
    if (wide) bf16 ? quantize_append_go<128, true, 16>(p, s) : quantize_append_go<128, false, 16>(p, s);
    else bf16 ? quantize_append_go<128, true, 4>(p, s) : quantize_append_go<128, false, 4>(p, s);
  } else {
    if (wide) bf16 ? quantize_append_go<64, true, 16>(p, s) : quantize_append_go<64, false, 16>(p, s);
    else bf16 ? quantize_append_go<64, true, 4>(p, s) : quantize_append_go<64, false, 4>(p, s);
  }
  return cudaGetLastError();
}

cudaError_t quantize_static_launch(int D, bool bf16, const QuantParams& p, float inv_k,
                                   float inv_v, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  const int grid = D == 128 ? grid_for<128, 4>(p.num_rows) : grid_for<64, 4>(p.num_rows);
  if (D == 128) {
    if (bf16) quantize_static_kernel<128, true><<<grid, kQuantThreads, 0, s>>>(p, inv_k, inv_v);
    else quantize_static_kernel<128, false><<<grid, kQuantThreads, 0, s>>>(p, inv_k, inv_v);
  } else {
    if (bf16) quantize_static_kernel<64, true><<<grid, kQuantThreads, 0, s>>>(p, inv_k, inv_v);
    else quantize_static_kernel<64, false><<<grid, kQuantThreads, 0, s>>>(p, inv_k, inv_v);
  }
  return cudaGetLastError();
}

cudaError_t append_kv16_launch(int D, const QuantParams& p, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  const int grid = D == 128 ? grid_for<128, 4>(p.num_rows) : grid_for<64, 4>(p.num_rows);
  if (D == 128) append_kv16_kernel<128><<<grid, kQuantThreads, 0, s>>>(p);
  else append_kv16_kernel<64><<<grid, kQuantThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
