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
// decoded exactly to FP32.  a/127 is an IEEE FP32 division (__fdiv_rn): the
// exact quotient of a 16-bit value by 127 is either an FP16 value or at least
// 2^-17 (relative) away from every FP16 value, far above the 2^-24 FP32
// rounding error, so __float2half_ru gives the exact upward rounding.
// x / s is also __fdiv_rn: away from an exact tie the exact quotient is at
// least ~2^-12 from any k + 1/2, and an exact tie is representable, so
// rintf (round half to even) of the FP32 quotient equals the exact rounding.
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

// FP16 bits of the row scale for magnitude pattern `amax_bits`.
template <bool BF16>
__device__ __forceinline__ uint16_t row_scale_bits(uint32_t amax_bits) {
  if (amax_bits == 0u) return 0x3C00u;                   // all-zero token -> 1.0
  const float a = bits_to_float<BF16>(amax_bits);
  unsigned short s = __half_as_ushort(__float2half_ru(__fdiv_rn(a, 127.0f)));
  if (s >= 0x7C00u) s = 0x7BFFu;                         // saturate at 65504
  if (s == 0u) s = 1u;                                   // a > 0 never gets a zero scale
  return s;
}

// Four 16-bit values -> four int8 codes packed little-endian.
template <bool BF16>
__device__ __forceinline__ uint32_t quantize4(uint2 x, float s) {
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t w = (e < 2) ? x.x : x.y;
    const uint32_t b = (e & 1) ? (w >> 16) : (w & 0xFFFFu);
    float r = rintf(__fdiv_rn(bits_to_float<BF16>(b), s));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    out |= (uint32_t)((int)r & 0xFF) << (8 * e);
  }
  return out;
}

__device__ __forceinline__ uint32_t mag_max4(uint2 x) {
  const uint32_t a = max(x.x & 0x7FFFu, (x.x >> 16) & 0x7FFFu);
  const uint32_t b = max(x.y & 0x7FFFu, (x.y >> 16) & 0x7FFFu);
  return max(a, b);
}

// One group of D/4 lanes per (token, KV head) row; each lane owns four
// consecutive elements (one 8-byte load of K and of V, one 4-byte store of
// codes each).  Rows of one warp are adjacent heads of a token, so the
// 16-bit loads and the int8 stores of a warp are contiguous runs.
template <int D, bool BF16>
__global__ void __launch_bounds__(kQuantThreads) quantize_append_kernel(const QuantParams p) {
  constexpr int LPR = D / 4;  // lanes per row
  const int lane = threadIdx.x & 31;
  const int64_t gthread = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x;
  const int64_t row = gthread / LPR;
  const int sub = lane % LPR;
  const bool in_range = row < p.num_rows;
  // the next kernel in the stream (a decode launched with programmatic stream
  // serialization) may be scheduled now; it waits for this grid's completion
  griddep_launch_dependents();

  int64_t t = 0, slot = -1;
  int j = 0;
  if (in_range) {
    t = row / p.num_kv_heads;
    j = (int)(row - t * p.num_kv_heads);
    slot = p.slots[t];
    if (slot >= p.num_slots) {
      if (sub == 0) atomicOr(p.err, 0x1u);
      slot = -1;
    }
  }
  const bool active = slot >= 0;

  uint2 kx = make_uint2(0, 0), vx = make_uint2(0, 0);
  if (active) {
    const uint16_t* kr = static_cast<const uint16_t*>(p.k) + t * p.k_stride + (int64_t)j * D;
    const uint16_t* vr = static_cast<const uint16_t*>(p.v) + t * p.v_stride + (int64_t)j * D;
    kx = __ldg(reinterpret_cast<const uint2*>(kr) + sub);
    vx = __ldg(reinterpret_cast<const uint2*>(vr) + sub);
  }
  uint32_t km = mag_max4(kx), vm = mag_max4(vx);
#pragma unroll
  for (int off = LPR / 2; off > 0; off >>= 1) {
    km = max(km, __shfl_xor_sync(0xFFFFFFFFu, km, off));
    vm = max(vm, __shfl_xor_sync(0xFFFFFFFFu, vm, off));
  }
  if (!active) return;

  const uint16_t ks = row_scale_bits<BF16>(km);
  const uint16_t vs = row_scale_bits<BF16>(vm);
  const float ksf = __half2float(__ushort_as_half(ks));
  const float vsf = __half2float(__ushort_as_half(vs));

  const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
  const int64_t crow = (blk * p.num_kv_heads + j) * kBlockSize + off;  // [NB][Hkv][bs]
  reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.k_cache) + crow * D)[sub] =
      quantize4<BF16>(kx, ksf);
  reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.v_cache) + crow * D)[sub] =
      quantize4<BF16>(vx, vsf);
  if (sub == 0) {
    p.k_scale[crow] = ks;
    p.v_scale[crow] = vs;
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
  constexpr int LPR = D / 4;  // lanes per row
  const int64_t gthread = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x;
  const int64_t row = gthread / LPR;
  const int sub = (threadIdx.x & 31) % LPR;
  griddep_launch_dependents();
  if (row >= p.num_rows) return;
  const int64_t t = row / p.num_kv_heads;
  const int j = (int)(row - t * p.num_kv_heads);
  const int64_t slot = p.slots[t];
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (sub == 0) atomicOr(p.err, 0x1u);
    return;
  }
  const uint16_t* kr = static_cast<const uint16_t*>(p.k) + t * p.k_stride + (int64_t)j * D;
  const uint16_t* vr = static_cast<const uint16_t*>(p.v) + t * p.v_stride + (int64_t)j * D;
  const uint2 kx = __ldg(reinterpret_cast<const uint2*>(kr) + sub);
  const uint2 vx = __ldg(reinterpret_cast<const uint2*>(vr) + sub);
  const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
  const int64_t crow = (blk * p.num_kv_heads + j) * kBlockSize + off;
  uint32_t kq = 0, vq = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t kw = (e < 2) ? kx.x : kx.y, vw = (e < 2) ? vx.x : vx.y;
    const uint32_t kb = (e & 1) ? (kw >> 16) : (kw & 0xFFFFu);
    const uint32_t vb = (e & 1) ? (vw >> 16) : (vw & 0xFFFFu);
    const float kr8 = fminf(fmaxf(rintf(__fmul_rn(bits_to_float<BF16>(kb), inv_k)), -127.f), 127.f);
    const float vr8 = fminf(fmaxf(rintf(__fmul_rn(bits_to_float<BF16>(vb), inv_v)), -127.f), 127.f);
    kq |= (uint32_t)((int)kr8 & 0xFF) << (8 * e);
    vq |= (uint32_t)((int)vr8 & 0xFF) << (8 * e);
  }
  reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.k_cache) + crow * D)[sub] = kq;
  reinterpret_cast<uint32_t*>(static_cast<int8_t*>(p.v_cache) + crow * D)[sub] = vq;
}

template <int D>
__global__ void __launch_bounds__(kQuantThreads) append_kv16_kernel(const QuantParams p) {
  constexpr int LPR = D / 4;
  const int64_t gthread = (int64_t)blockIdx.x * kQuantThreads + threadIdx.x;
  const int64_t row = gthread / LPR;
  const int sub = (threadIdx.x & 31) % LPR;
  if (row >= p.num_rows) return;
  const int64_t t = row / p.num_kv_heads;
  const int j = (int)(row - t * p.num_kv_heads);
  const int64_t slot = p.slots[t];
  if (slot < 0) return;
  if (slot >= p.num_slots) {
    if (sub == 0) atomicOr(p.err, 0x1u);
    return;
  }
  const uint16_t* kr = static_cast<const uint16_t*>(p.k) + t * p.k_stride + (int64_t)j * D;
  const uint16_t* vr = static_cast<const uint16_t*>(p.v) + t * p.v_stride + (int64_t)j * D;
  const int64_t blk = slot / kBlockSize, off = slot % kBlockSize;
  const int64_t crow = (blk * p.num_kv_heads + j) * kBlockSize + off;
  reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.k_cache) + crow * D)[sub] =
      __ldg(reinterpret_cast<const uint2*>(kr) + sub);
  reinterpret_cast<uint2*>(static_cast<uint16_t*>(p.v_cache) + crow * D)[sub] =
      __ldg(reinterpret_cast<const uint2*>(vr) + sub);
}

inline int grid_for(int64_t rows, int D) {
  const int64_t threads = rows * (D / 4);
  return (int)((threads + kQuantThreads - 1) / kQuantThreads);
}

}  // namespace

cudaError_t quantize_append_launch(int D, bool bf16, const QuantParams& p, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  const int grid = grid_for(p.num_rows, D);
  if (D == 128) {
    if (bf16) quantize_append_kernel<128, true><<<grid, kQuantThreads, 0, s>>>(p);
    else quantize_append_kernel<128, false><<<grid, kQuantThreads, 0, s>>>(p);
  } else {
    if (bf16) quantize_append_kernel<64, true><<<grid, kQuantThreads, 0, s>>>(p);
    else quantize_append_kernel<64, false><<<grid, kQuantThreads, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t quantize_static_launch(int D, bool bf16, const QuantParams& p, float inv_k,
                                   float inv_v, cudaStream_t s) {
  if (p.num_rows == 0) return cudaSuccess;
  const int grid = grid_for(p.num_rows, D);
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
  const int grid = grid_for(p.num_rows, D);
  if (D == 128) append_kv16_kernel<128><<<grid, kQuantThreads, 0, s>>>(p);
  else append_kv16_kernel<64><<<grid, kQuantThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace kvq
