// C ABI of libkvq (declared in include/kvq.h): argument validation, the
// decode launcher, TMA descriptor construction, and the device error word.
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>

#include "kvq.h"
#include "kvq_internal.h"
#include "kvq_ptx.cuh"

using namespace kvq;

// Per-device error word: kernels OR KVQ_DEVERR_* bits into it, kvq_get_error
// reads and clears it.
__device__ unsigned int g_kvq_error_word = 0u;

namespace {
// Self-test of the bounded wait every kernel uses: one warp waits on an
// mbarrier that nothing arrives on, gives up after limit_ns, and reports it
// through the error word, as a decode whose copies never landed would.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned int* err) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  __syncwarp();
  const bool ok = mbar_wait_bounded(smem_u32(&bar), 0, limit_ns);
  if (!ok && threadIdx.x == 0) atomicOr(err, KVQ_DEVERR_TIMEOUT);
}
}  // namespace

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxRangePages = 1 << 24;   // forced range length accepted by the _split calls

// Tensor maps of recently used caches, so that repeated calls on the same
// cache skip the driver's encode.
constexpr int kMapCache = 16;
struct MapEntry {
  const void* base = nullptr;
  int64_t rows = 0;
  int D = 0, eb = 0, box_rows = 0;
  CUtensorMap map;
};

struct DeviceState {
  std::atomic<bool> ready{false};
  int sms = 0;
  unsigned int* err = nullptr;
  // occupancy cache: [variant] -> (last smem << 32) | ctas per SM
  std::atomic<uint64_t> occ[32] = {};
  std::mutex map_mu;
  MapEntry maps[kMapCache];
  int map_next = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

kvq_status cuda_fail() { return KVQ_ERR_CUDA; }

// Initializes the current device's state once; returns nullptr on failure.
DeviceState* device_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState& st = g_dev[dev];
  if (st.ready.load(std::memory_order_acquire)) return &st;
  std::lock_guard<std::mutex> lk(g_mu);
  if (st.ready.load(std::memory_order_relaxed)) return &st;
  if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), g_kvq_error_word) != cudaSuccess)
    return nullptr;
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // opt every decode variant into the largest shared-memory footprint it can use
  for (const DecodeOps* ops : {&kDecodeInt8H1, &kDecodeInt8H2, &kDecodeStaticH1,
                               &kDecodeStaticH2, &kDecodeKv16, &kDecodeInt8Cc, &kDecodeInt8T2})
    for (int D : {64, 128})
      for (bool bf : {false, true})
        if (ops->configure(D, bf, ops->smem(D, kMaxSeqs, kMaxGroup)) != cudaSuccess)
          return nullptr;
  for (int D : {64, 128})
    for (bool bf : {false, true})
      if (prefill_configure(D, bf) != cudaSuccess) return nullptr;
  st.ready.store(true, std::memory_order_release);
  return &st;
}

// The decode kernel variants: INT8 with per-token scale planes, INT8 with
// static (per-tensor) scales, the 16-bit twin, and the per-token INT8 decode
// on the CUDA cores (A/B counterpart of the tensor-core one).
enum class Dec { kInt8 = 0, kStatic = 1, kKv16 = 2, kInt8Cc = 3 };

static_assert(kMaxHeadGroup == 1 || kMaxHeadGroup == 2, "head groups of 1 or 2 KV heads");

// KV heads one decode warp processes together: the largest power of two H
// up to kMaxHeadGroup with G H <= 8 (the MMAs' N) that divides Hkv.  The
// 16-bit twin keeps H = 1.
int head_group(Dec var, int32_t G, int32_t Hkv) {
  if (var == Dec::kKv16 || var == Dec::kInt8Cc) return 1;
  int H = 1;
  while (2 * H <= kMaxHeadGroup && 2 * H * G <= kMaxGroup && Hkv % (2 * H) == 0) H *= 2;
  return H;
}

// Pages one decode warp step covers: two for the per-token INT8 decode with
// one KV head per step (G > 4), so that each step's fixed work covers two
// page tiles there too; else one.
int pages_per_step(Dec var, int H) {
  return var == Dec::kInt8 && H == 1 && kMaxPageStep >= 2 ? 2 : 1;
}

// The kernel variant of (cache kind, head group, pages per step), and its
// index among the variants (occupancy cache).
const DecodeOps& ops_of(Dec var, int H, int T, int* vid = nullptr) {
  int v = 4;
  const DecodeOps* o = &kDecodeKv16;
  if (var == Dec::kInt8) {
    v = T == 2 ? 6 : (H == 2 ? 1 : 0);
    o = T == 2 ? &kDecodeInt8T2 : (H == 2 ? &kDecodeInt8H2 : &kDecodeInt8H1);
  } else if (var == Dec::kStatic) {
    v = H == 2 ? 3 : 2;
    o = H == 2 ? &kDecodeStaticH2 : &kDecodeStaticH1;
  } else if (var == Dec::kInt8Cc) {
    v = 5;
    o = &kDecodeInt8Cc;
  }
  if (vid) *vid = v;
  return *o;
}

int ctas_per_sm(DeviceState* st, Dec var, int H, int T, int D, bool bf16, size_t smem) {
  // cache slots: 7 variants x {D128, D64} x {fp16, bf16}
  int vid = 0;
  const DecodeOps& ops = ops_of(var, H, T, &vid);
  const int v = vid * 4 + (D == 128 ? 0 : 2) + (bf16 ? 1 : 0);
  const uint64_t c = st->occ[v].load(std::memory_order_relaxed);
  if ((c >> 32) == (uint64_t)smem && (c & 0xFFFFFFFFu) != 0) return (int)(c & 0xFFFFFFFFu);
  int n = 0;
  if (ops.occupancy(D, bf16, smem, &n) != cudaSuccess || n <= 0) return 0;
  st->occ[v].store(((uint64_t)smem << 32) | (uint32_t)n, std::memory_order_relaxed);
  return n;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Page columns of the stream when every sequence holds max_ctx tokens: the
// bound the host sizes everything for.
int64_t columns_max(int32_t B, int32_t max_ctx) { return (int64_t)B * cdiv(max_ctx, kBlockSize); }

// Workspace: per work unit (range, KV head) two partial slots of G rows:
// log2-sum-exp float [2 * units][G], then normalized partial output float
// [2 * units][G][D].
struct WsLayout {
  size_t lse = 0, o = 0, total = 0;
  int64_t ranges = 0;   // work units the slots hold
};

WsLayout layout_for(int32_t B, int32_t G, int32_t D, int64_t ranges) {
  (void)B;
  WsLayout w;
  w.ranges = ranges;
  w.lse = 0;
  w.o = round_up((size_t)(2 * ranges * G) * 4, 256);
  w.total = w.o + (size_t)(2 * ranges * G * D) * 4;
  return w;
}

// Most work units whose slots fit in `bytes` (0 when not even one does).
int64_t ranges_for_bytes(int32_t B, int32_t G, int32_t D, size_t bytes) {
  int64_t lo = 0, hi = (int64_t)(bytes / ((size_t)2 * G * D * 4)) + 1;   // fits / does not
  if (layout_for(B, G, D, hi).total <= bytes) return hi;
  while (hi - lo > 1) {
    const int64_t mid = lo + (hi - lo) / 2;
    if (layout_for(B, G, D, mid).total <= bytes) lo = mid; else hi = mid;
  }
  return lo;
}

// Warps of a full persistent grid of one decode variant on this device (0
// on failure).
int64_t resident_warps(DeviceState* st, Dec var, int D, bool bf16, int32_t B, int32_t G,
                       int32_t Hkv) {
  const int H = head_group(var, G, Hkv), T = pages_per_step(var, H);
  const size_t smem = ops_of(var, H, T).smem(D, B, G * H);
  return (int64_t)st->sms * ctas_per_sm(st, var, H, T, D, bf16, smem) * kWarps;
}

// Work units of the balanced split for a grid of `warps` warps: one range
// per whole group of Hkv warps (at least one), no more ranges than the stream
// has columns of kMinRangePages.
int64_t balanced_units(int64_t warps, int32_t Hkv, int64_t cols_max) {
  const int64_t groups = warps / Hkv > 0 ? warps / Hkv : 1;
  const int64_t by_cols = cdiv(cols_max, kMinRangePages);
  return (int64_t)Hkv * (groups < by_cols ? groups : by_cols);
}

// Workspace bytes kvq_paged_decode's balanced split uses at most on this
// device: for the full grid of each decode variant (its head group), the
// largest.
size_t balanced_bytes_max(DeviceState* st, int32_t B, int32_t Hkv, int32_t G, int32_t D,
                          int32_t max_ctx) {
  size_t best = 0;
  for (Dec var : {Dec::kInt8, Dec::kStatic, Dec::kKv16, Dec::kInt8Cc})
    for (bool bf : {false, true}) {
      const int H = head_group(var, G, Hkv);
      const int64_t w = resident_warps(st, var, D, bf, B, G, Hkv);
      const size_t x =
          layout_for(B, G * H, D, balanced_units(w, Hkv / H, columns_max(B, max_ctx))).total;
      best = x > best ? x : best;
    }
  return best;
}

// Tensor map over a cache payload seen as `rows` token rows of D elements;
// a box is one 128-byte (or narrower) column block of box_rows rows.
bool encode_map(CUtensorMap* m, const void* base, int elem_bytes, int D, int64_t rows,
                int box_rows) {
  const CUtensorMapDataType dt =
      elem_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const int row_bytes = D * elem_bytes;
  const int sub = row_bytes < 128 ? row_bytes : 128;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(sub / elem_bytes), (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = sub == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tensor map of a cache payload (encoded once per (base, rows, D,
// element size, box rows) and kept among the device's recent ones).
bool make_map(DeviceState* st, CUtensorMap* m, const void* base, int elem_bytes, int D,
              int64_t rows, int box_rows = kBlockSize) {
  std::lock_guard<std::mutex> lk(st->map_mu);
  for (const MapEntry& e : st->maps)
    if (e.base == base && e.rows == rows && e.D == D && e.eb == elem_bytes &&
        e.box_rows == box_rows) {
      *m = e.map;
      return true;
    }
  if (!encode_map(m, base, elem_bytes, D, rows, box_rows)) return false;
  MapEntry& e = st->maps[st->map_next];
  st->map_next = (st->map_next + 1) % kMapCache;
  e.base = base;
  e.rows = rows;
  e.D = D;
  e.eb = elem_bytes;
  e.box_rows = box_rows;
  e.map = *m;
  return true;
}

// Shared validation of the decode arguments (both caches).  `rows`: q and
// out hold at least one row (a prefill without queries passes false, and
// its q and out may be null).
kvq_status check_decode(const void* q, kvq_dtype dtype, int32_t B, int32_t Hq, int32_t Hkv,
                        int32_t D, const void* kc, const void* vc, const void* ks,
                        const void* vs, bool planes, int32_t num_blocks, int32_t bs,
                        const int32_t* bt, int32_t max_blocks, const int32_t* cl,
                        int32_t max_ctx, float sm_scale, const void* out, bool rows = true) {
  if (dtype != KVQ_FP16 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARGUMENT;
  if (B < 0 || Hq <= 0 || Hkv <= 0 || num_blocks <= 0 || max_ctx < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(sm_scale)) return KVQ_ERR_INVALID_ARGUMENT;
  if (bs != kBlockSize) return KVQ_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (Hq % Hkv != 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (Hq / Hkv > kMaxGroup) return KVQ_ERR_UNSUPPORTED;
  if (B > kMaxSeqs) return KVQ_ERR_UNSUPPORTED;
  if ((int64_t)num_blocks * Hkv * kBlockSize > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
  if (B == 0) return KVQ_OK;
  if (max_blocks <= 0) return KVQ_ERR_INVALID_ARGUMENT;
  if ((int64_t)max_ctx > (int64_t)max_blocks * kBlockSize) return KVQ_ERR_INVALID_ARGUMENT;
  if (!kc || !vc || !bt || !cl) return KVQ_ERR_INVALID_ARGUMENT;
  if (rows && (!q || !out || !aligned(q, 16) || !aligned(out, 16)))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (planes && (!ks || !vs)) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(kc, 16) || !aligned(vc, 16) || !aligned(bt, 4) || !aligned(cl, 4))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (planes && (!aligned(ks, 16) || !aligned(vs, 16))) return KVQ_ERR_INVALID_ARGUMENT;
  return KVQ_OK;
}

// R == 0: balanced split (or one range per segment without a workspace, or
// when no sequence can span two pages); R >= 1: ranges of R pages.
kvq_status decode_common(Dec var, const void* q, kvq_dtype dtype, int32_t B, int32_t Hq,
                         int32_t Hkv, int32_t D, const void* kc, const void* vc,
                         const uint16_t* ks, const uint16_t* vs, int32_t num_blocks,
                         int32_t bs, const int32_t* bt, int32_t max_blocks, const int32_t* cl,
                         int32_t max_ctx, float sm_scale, void* out, void* ws, size_t ws_bytes,
                         int32_t R, cudaStream_t stream, float k_static = 1.f,
                         float v_static = 1.f) {
  kvq_status s = check_decode(q, dtype, B, Hq, Hkv, D, kc, vc, ks, vs,
                              var == Dec::kInt8 || var == Dec::kInt8Cc,
                              num_blocks, bs, bt, max_blocks, cl, max_ctx, sm_scale, out);
  if (s != KVQ_OK || B == 0) return s;
  // the page prefix over sequences and token counts are 32-bit in the kernels
  if ((int64_t)B * max_blocks > INT32_MAX || max_blocks > INT32_MAX / kBlockSize)
    return KVQ_ERR_UNSUPPORTED;
  if (R < 0 || R > kMaxRangePages) return KVQ_ERR_INVALID_ARGUMENT;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  const bool bf16 = dtype == KVQ_BF16;
  const int32_t Gr = Hq / Hkv;
  // the kernel walks head groups of H KV heads: HU groups of G = Gr H query
  // heads each (the group's query heads are consecutive)
  const int H = head_group(var, Gr, Hkv), T = pages_per_step(var, H);
  const int32_t HU = Hkv / H, G = Gr * H;
  const DecodeOps& ops = ops_of(var, H, T);
  const size_t smem = ops.smem(D, B, G);
  const int occ = ctas_per_sm(st, var, H, T, D, bf16, smem);
  if (occ <= 0) return cuda_fail();
  const int64_t slots = (int64_t)st->sms * occ;      // CTAs of a full persistent grid
  const int64_t cols = columns_max(B, max_ctx);
  const int64_t pages_max = cdiv(max_ctx, kBlockSize);

  DecodeParams p{};
  WsLayout wl;
  int64_t grid = 0;
  // no split without a workspace, or when no sequence has more pages than the
  // shortest range: such a sequence would gain at most a few pieces, less
  // than the merge launch costs
  if (R == 0 && (ws == nullptr || ws_bytes == 0 || pages_max <= kMinRangePages)) {
    p.R = -1;                                       // one unit per (sequence, head group)
    p.range_cap = 0;
    grid = cdiv((int64_t)B * HU, kWarps);
    if (grid > slots) grid = slots;
  } else if (R == 0) {
    // as many ranges as groups of HU warps of the full grid, within the
    // workspace's slots; with fewer ranges than sequences the per-sequence
    // split (above) keeps more warps busy
    const int64_t cap = ranges_for_bytes(B, G, D, ws_bytes);
    if (cap < HU) return KVQ_ERR_WORKSPACE_TOO_SMALL;
    const int64_t full = balanced_units(slots * kWarps, HU, cols) / HU;
    const int64_t groups = full < cap / HU ? full : cap / HU;
    if (groups < B && groups < full) {
      p.R = -1;
      p.range_cap = 0;
      grid = cdiv((int64_t)B * HU, kWarps);
    } else {
      p.R = 0;
      p.groups = groups;
      p.range_cap = groups * HU;
      wl = layout_for(B, G, D, p.range_cap);
      grid = cdiv(p.range_cap, kWarps);
    }
    if (grid > slots) grid = slots;
  } else {
    p.range_cap = cdiv(cols, R) * HU;
    wl = layout_for(B, G, D, p.range_cap);
    if (ws == nullptr || ws_bytes < wl.total) return KVQ_ERR_WORKSPACE_TOO_SMALL;
    grid = cdiv(p.range_cap, kWarps);
    if (grid > slots) grid = slots;
    p.R = R;
  }
  if (grid < 1) grid = 1;
  // the kernel counts columns and work units in 32 bits
  if (cols > INT32_MAX || p.range_cap > INT32_MAX || (int64_t)B * HU > INT32_MAX)
    return KVQ_ERR_UNSUPPORTED;
  const bool split = p.R >= 0;
  if (split && (!ws || !aligned(ws, 256) || ws_bytes < wl.total))
    return KVQ_ERR_INVALID_ARGUMENT;

  // one box = the adjacent (page, head) tiles of a head group
  CUtensorMap maps[2];
  const int64_t rows = (int64_t)num_blocks * Hkv * kBlockSize;
  const int eb = var == Dec::kKv16 ? 2 : 1;
  if (!make_map(st, &maps[0], kc, eb, D, rows, kBlockSize * H) ||
      !make_map(st, &maps[1], vc, eb, D, rows, kBlockSize * H))
    return cuda_fail();

  p.q = q;
  p.out = out;
  p.k_cache = kc;
  p.v_cache = vc;
  p.k_scale = ks;
  p.v_scale = vs;
  p.block_tables = bt;
  p.context_lens = cl;
  uint8_t* w = static_cast<uint8_t*>(ws);
  p.part_lse = split ? reinterpret_cast<float*>(w + wl.lse) : nullptr;
  p.part_o = split ? reinterpret_cast<float*>(w + wl.o) : nullptr;
  p.err = st->err;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = HU;
  p.G = G;
  p.Gr = Gr;
  p.max_blocks = max_blocks;
  p.max_ctx = max_ctx;
  p.num_blocks = num_blocks;
  p.scale_log2 = (float)((double)sm_scale * (double)k_static * 1.4426950408889634);
  p.v_static = v_static;

  if (ops.launch(D, bf16, maps, p, (int)grid, smem, stream) != cudaSuccess) return cuda_fail();
  if (split) {
    CombineParams cp{};
    cp.part_o = p.part_o;
    cp.part_lse = p.part_lse;
    cp.context_lens = cl;
    cp.out = out;
    cp.B = B;
    cp.Hq = Hq;
    cp.Hkv = HU;
    cp.G = G;
    cp.max_tok = max_blocks * kBlockSize < max_ctx ? max_blocks * kBlockSize : max_ctx;
    cp.R = p.R;
    cp.groups = p.groups;
    // few pairs: their sequences are long and split into many pieces, so a
    // whole CTA per pair shortens the dependent loads
    cp.per_cta = (int64_t)B * Hq <= 2 * (int64_t)st->sms ? 1 : 0;
    if (combine_launch(D, bf16, cp, st->sms, stream) != cudaSuccess) return cuda_fail();
  }
  return KVQ_OK;
}

kvq_status check_append(const void* k, const void* v, int64_t ks, int64_t vs, int32_t T,
                        int32_t Hkv, int32_t D, kvq_dtype dtype, const int64_t* slots,
                        const void* kc, const void* vc, int32_t num_blocks, int32_t bs) {
  if (dtype != KVQ_FP16 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARGUMENT;
  if (T < 0 || Hkv <= 0 || num_blocks <= 0) return KVQ_ERR_INVALID_ARGUMENT;
  if (bs != kBlockSize) return KVQ_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return KVQ_ERR_UNSUPPORTED;
  if (T == 0) return KVQ_OK;
  if (!k || !v || !slots || !kc || !vc) return KVQ_ERR_INVALID_ARGUMENT;
  if (ks < (int64_t)Hkv * D || vs < (int64_t)Hkv * D || ks % 4 || vs % 4)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k, 8) || !aligned(v, 8) || !aligned(slots, 8) || !aligned(kc, 16) ||
      !aligned(vc, 16))
    return KVQ_ERR_INVALID_ARGUMENT;
  return KVQ_OK;
}

}  // namespace

extern "C" {

kvq_status kvq_quantize_append(const void* k, const void* v, int64_t k_token_stride,
                               int64_t v_token_stride, int32_t num_tokens, int32_t num_kv_heads,
                               int32_t head_dim, kvq_dtype dtype, const int64_t* slot_mapping,
                               int8_t* k_cache, int8_t* v_cache, uint16_t* k_scale,
                               uint16_t* v_scale, int32_t num_blocks, int32_t block_size,
                               kvq_stream_t stream) {
  kvq_status s = check_append(k, v, k_token_stride, v_token_stride, num_tokens, num_kv_heads,
                              head_dim, dtype, slot_mapping, k_cache, v_cache, num_blocks,
                              block_size);
  if (s != KVQ_OK || num_tokens == 0) return s;
  if (!k_scale || !v_scale || !aligned(k_scale, 16) || !aligned(v_scale, 16))
    return KVQ_ERR_INVALID_ARGUMENT;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  QuantParams p{};
  p.k = k;
  p.v = v;
  p.k_stride = k_token_stride;
  p.v_stride = v_token_stride;
  p.slots = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.num_rows = (int64_t)num_tokens * num_kv_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_slots = (int64_t)num_blocks * kBlockSize;
  p.err = st->err;
  if (quantize_append_launch(head_dim, dtype == KVQ_BF16, p,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

kvq_status kvq_quantize_append_static(const void* k, const void* v, int64_t k_token_stride,
                                      int64_t v_token_stride, int32_t num_tokens,
                                      int32_t num_kv_heads, int32_t head_dim, kvq_dtype dtype,
                                      const int64_t* slot_mapping, int8_t* k_cache,
                                      int8_t* v_cache, float k_scale, float v_scale,
                                      int32_t num_blocks, int32_t block_size,
                                      kvq_stream_t stream) {
  kvq_status s = check_append(k, v, k_token_stride, v_token_stride, num_tokens, num_kv_heads,
                              head_dim, dtype, slot_mapping, k_cache, v_cache, num_blocks,
                              block_size);
  if (s != KVQ_OK) return s;
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return KVQ_ERR_INVALID_ARGUMENT;
  // the reciprocal each code is computed with: one IEEE binary32 division
  const volatile float one = 1.0f;
  const float inv_k = one / k_scale, inv_v = one / v_scale;
  if (!std::isfinite(inv_k) || !std::isfinite(inv_v)) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return KVQ_OK;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  QuantParams p{};
  p.k = k;
  p.v = v;
  p.k_stride = k_token_stride;
  p.v_stride = v_token_stride;
  p.slots = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.num_rows = (int64_t)num_tokens * num_kv_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_slots = (int64_t)num_blocks * kBlockSize;
  p.err = st->err;
  if (quantize_static_launch(head_dim, dtype == KVQ_BF16, p, inv_k, inv_v,
                             reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

kvq_status kvq_paged_decode_static(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                   int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                   const int8_t* k_cache, const int8_t* v_cache, float k_scale,
                                   float v_scale, int32_t num_blocks, int32_t block_size,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   float sm_scale, void* out, void* workspace,
                                   size_t workspace_bytes, kvq_stream_t stream) {
  if (!(std::isfinite(k_scale) && k_scale > 0.f && std::isfinite(v_scale) && v_scale > 0.f))
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!std::isfinite((double)sm_scale * (double)k_scale * 1.4426950408889634))
    return KVQ_ERR_INVALID_ARGUMENT;
  return decode_common(Dec::kStatic, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       k_cache, v_cache, nullptr, nullptr, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, 0, reinterpret_cast<cudaStream_t>(stream),
                       k_scale, v_scale);
}

kvq_status kvq_cache_append_kv16(const void* k, const void* v, int64_t k_token_stride,
                                 int64_t v_token_stride, int32_t num_tokens,
                                 int32_t num_kv_heads, int32_t head_dim, kvq_dtype dtype,
                                 const int64_t* slot_mapping, void* k_cache, void* v_cache,
                                 int32_t num_blocks, int32_t block_size, kvq_stream_t stream) {
  kvq_status s = check_append(k, v, k_token_stride, v_token_stride, num_tokens, num_kv_heads,
                              head_dim, dtype, slot_mapping, k_cache, v_cache, num_blocks,
                              block_size);
  if (s != KVQ_OK || num_tokens == 0) return s;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  QuantParams p{};
  p.k = k;
  p.v = v;
  p.k_stride = k_token_stride;
  p.v_stride = v_token_stride;
  p.slots = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.num_rows = (int64_t)num_tokens * num_kv_heads;
  p.num_kv_heads = num_kv_heads;
  p.num_slots = (int64_t)num_blocks * kBlockSize;
  p.err = st->err;
  if (append_kv16_launch(head_dim, p, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

kvq_status kvq_paged_decode_split(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  const int8_t* k_cache, const int8_t* v_cache,
                                  const uint16_t* k_scale, const uint16_t* v_scale,
                                  int32_t num_blocks, int32_t block_size,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, int32_t max_context_len,
                                  float sm_scale, void* out, void* workspace,
                                  size_t workspace_bytes, int32_t partition_pages,
                                  kvq_stream_t stream) {
  if (partition_pages <= 0) return KVQ_ERR_INVALID_ARGUMENT;
  return decode_common(Dec::kInt8, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                       v_cache, k_scale, v_scale, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, partition_pages,
                       reinterpret_cast<cudaStream_t>(stream));
}

kvq_status kvq_paged_decode(const void* q, kvq_dtype dtype, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            const int8_t* k_cache, const int8_t* v_cache,
                            const uint16_t* k_scale, const uint16_t* v_scale,
                            int32_t num_blocks, int32_t block_size,
                            const int32_t* block_tables, int32_t max_blocks_per_seq,
                            const int32_t* context_lens, int32_t max_context_len,
                            float sm_scale, void* out, void* workspace, size_t workspace_bytes,
                            kvq_stream_t stream) {
  return decode_common(Dec::kInt8, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                       v_cache, k_scale, v_scale, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, 0, reinterpret_cast<cudaStream_t>(stream));
}

kvq_status kvq_paged_decode_cuda_cores(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, const int8_t* k_cache,
                                       const int8_t* v_cache, const uint16_t* k_scale,
                                       const uint16_t* v_scale, int32_t num_blocks,
                                       int32_t block_size, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float sm_scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       kvq_stream_t stream) {
  return decode_common(Dec::kInt8Cc, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim,
                       k_cache, v_cache, k_scale, v_scale, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, 0, reinterpret_cast<cudaStream_t>(stream));
}

kvq_status kvq_paged_decode_kv16_split(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                       int32_t num_q_heads, int32_t num_kv_heads,
                                       int32_t head_dim, const void* k_cache,
                                       const void* v_cache, int32_t num_blocks,
                                       int32_t block_size, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t max_context_len, float sm_scale, void* out,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t partition_pages, kvq_stream_t stream) {
  if (partition_pages <= 0) return KVQ_ERR_INVALID_ARGUMENT;
  return decode_common(Dec::kKv16, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                       v_cache, nullptr, nullptr, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, partition_pages,
                       reinterpret_cast<cudaStream_t>(stream));
}

kvq_status kvq_paged_decode_kv16(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 const void* k_cache, const void* v_cache, int32_t num_blocks,
                                 int32_t block_size, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* context_lens,
                                 int32_t max_context_len, float sm_scale, void* out,
                                 void* workspace, size_t workspace_bytes, kvq_stream_t stream) {
  return decode_common(Dec::kKv16, q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                       v_cache, nullptr, nullptr, num_blocks, block_size, block_tables,
                       max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                       workspace, workspace_bytes, 0, reinterpret_cast<cudaStream_t>(stream));
}

kvq_status kvq_dequantize_window(const int8_t* k_cache, const int8_t* v_cache,
                                 const uint16_t* k_scale, const uint16_t* v_scale,
                                 int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                 int32_t head_dim, const int32_t* block_tables,
                                 int32_t num_seqs, int32_t max_blocks_per_seq,
                                 const int32_t* context_lens, int32_t max_context_len,
                                 kvq_dtype dtype, void* k_out, void* v_out,
                                 kvq_stream_t stream) {
  if (dtype != KVQ_FP16 && dtype != KVQ_BF16) return KVQ_ERR_INVALID_ARGUMENT;
  if (num_seqs < 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_context_len < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (block_size != kBlockSize) return KVQ_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (num_seqs > kMaxSeqs || (int64_t)num_blocks * num_kv_heads * kBlockSize > INT32_MAX)
    return KVQ_ERR_UNSUPPORTED;
  if (num_seqs == 0) return KVQ_OK;
  if (max_blocks_per_seq <= 0 || max_blocks_per_seq > INT32_MAX / kBlockSize ||
      (int64_t)max_context_len > (int64_t)max_blocks_per_seq * kBlockSize)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !context_lens || !k_out ||
      !v_out)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_out, 16) ||
      !aligned(v_out, 16) || !aligned(k_scale, 2) || !aligned(v_scale, 2) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return KVQ_ERR_INVALID_ARGUMENT;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  DequantParams p{};
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.k_out = k_out;
  p.v_out = v_out;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.err = st->err;
  p.B = num_seqs;
  p.Hkv = num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.max_tok = max_context_len;
  p.num_blocks = num_blocks;
  const int max_pages = (int)cdiv(max_context_len, kBlockSize);
  if (dequant_window_launch(head_dim, dtype == KVQ_BF16, p, max_pages,
                            reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

kvq_status kvq_trim_front_keep_sink(int8_t* k_cache, int8_t* v_cache, uint16_t* k_scale,
                                    uint16_t* v_scale, int32_t num_blocks, int32_t block_size,
                                    int32_t num_kv_heads, int32_t head_dim,
                                    const int32_t* block_tables, int32_t num_seqs,
                                    int32_t max_blocks_per_seq, int32_t* context_lens,
                                    const int32_t* trim, int32_t keep, kvq_stream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_blocks <= 0 || keep < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (block_size != kBlockSize) return KVQ_ERR_UNSUPPORTED;
  if (head_dim != 64 && head_dim != 128) return KVQ_ERR_UNSUPPORTED;
  if (num_kv_heads > 65535 || num_seqs > 65535 ||
      (int64_t)num_blocks * num_kv_heads * kBlockSize > INT32_MAX)
    return KVQ_ERR_UNSUPPORTED;
  if (num_seqs == 0) return KVQ_OK;
  if (max_blocks_per_seq <= 0 || max_blocks_per_seq > INT32_MAX / kBlockSize)
    return KVQ_ERR_INVALID_ARGUMENT;
  if (!k_cache || !v_cache || !block_tables || !context_lens || !trim)
    return KVQ_ERR_INVALID_ARGUMENT;
  if ((k_scale == nullptr) != (v_scale == nullptr)) return KVQ_ERR_INVALID_ARGUMENT;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_tables, 4) ||
      !aligned(context_lens, 4) || !aligned(trim, 4) || (k_scale && !aligned(k_scale, 2)) ||
      (v_scale && !aligned(v_scale, 2)))
    return KVQ_ERR_INVALID_ARGUMENT;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  TrimParams p{};
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.trim = trim;
  p.err = st->err;
  p.B = num_seqs;
  p.Hkv = num_kv_heads;
  p.max_blocks = max_blocks_per_seq;
  p.max_tok = max_blocks_per_seq * kBlockSize;
  p.num_blocks = num_blocks;
  p.keep = keep;
  if (trim_launch(head_dim, p, context_lens, reinterpret_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

kvq_status kvq_paged_prefill(const void* q, kvq_dtype dtype, int32_t num_seqs,
                             int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                             const int8_t* k_cache, const int8_t* v_cache,
                             const uint16_t* k_scale, const uint16_t* v_scale,
                             int32_t num_blocks, int32_t block_size,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len,
                             const int32_t* query_start, int32_t total_q, int32_t max_query_len,
                             float sm_scale, void* out, kvq_stream_t stream) {
  if (max_query_len < 0 || total_q < 0) return KVQ_ERR_INVALID_ARGUMENT;
  kvq_status s = check_decode(q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                              v_cache, k_scale, v_scale, true, num_blocks, block_size,
                              block_tables, max_blocks_per_seq, context_lens, max_context_len,
                              sm_scale, out, total_q > 0);
  if (s != KVQ_OK || num_seqs == 0) return s;
  if (!query_start || !aligned(query_start, 4)) return KVQ_ERR_INVALID_ARGUMENT;
  if (max_query_len == 0 || total_q == 0) return KVQ_OK;
  if (num_kv_heads > 65535 || num_seqs > 65535 || max_blocks_per_seq > INT32_MAX / kBlockSize)
    return KVQ_ERR_UNSUPPORTED;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  const int32_t G = num_q_heads / num_kv_heads;
  const int64_t per_tile = prefill_rows_per_cta() / G;   // queries per CTA tile
  const int64_t tiles = cdiv(max_query_len, per_tile);
  if (tiles > INT32_MAX) return KVQ_ERR_UNSUPPORTED;
  CUtensorMap maps[2];
  const int64_t rows = (int64_t)num_blocks * num_kv_heads * kBlockSize;
  if (!make_map(st, &maps[0], k_cache, 1, head_dim, rows) ||
      !make_map(st, &maps[1], v_cache, 1, head_dim, rows))
    return cuda_fail();
  PrefillParams p{};
  p.q = q;
  p.out = out;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.err = st->err;
  p.B = num_seqs;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.G = G;
  p.max_blocks = max_blocks_per_seq;
  p.max_ctx = max_context_len;
  p.num_blocks = num_blocks;
  p.total_q = total_q;
  p.max_q = max_query_len;
  p.scale_log2 = (float)((double)sm_scale * 1.4426950408889634);
  if (prefill_launch(head_dim, dtype == KVQ_BF16, maps, p, (int)tiles,
                     reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return cuda_fail();
  return KVQ_OK;
}

int32_t kvq_decode_partition_pages(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_context_len) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
      num_q_heads % num_kv_heads || (head_dim != 64 && head_dim != 128) ||
      num_q_heads / num_kv_heads > kMaxGroup || num_seqs > kMaxSeqs)
    return 0;
  DeviceState* st = device_state();
  if (!st) return 0;
  const int32_t G = num_q_heads / num_kv_heads;
  const int64_t w = resident_warps(st, Dec::kInt8, head_dim, true, num_seqs, G, num_kv_heads);
  if (w <= 0) return 0;
  const int64_t HU = num_kv_heads / head_group(Dec::kInt8, G, num_kv_heads);
  const int64_t groups = w / HU > 0 ? w / HU : 1;
  const int64_t r = cdiv(columns_max(num_seqs, max_context_len), groups);
  return (int32_t)(r > kMinRangePages ? (r < INT32_MAX ? r : INT32_MAX) : kMinRangePages);
}

size_t kvq_decode_workspace_bytes_split(int32_t num_seqs, int32_t num_q_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_context_len, int32_t partition_pages) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
      partition_pages < 1 || num_q_heads % num_kv_heads)
    return 0;
  const int32_t G = num_q_heads / num_kv_heads;
  return layout_for(num_seqs, G, head_dim,
                    cdiv(columns_max(num_seqs, max_context_len), partition_pages) * num_kv_heads)
      .total;
}

size_t kvq_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0 ||
      num_q_heads % num_kv_heads || (head_dim != 64 && head_dim != 128) ||
      num_q_heads / num_kv_heads > kMaxGroup || num_seqs > kMaxSeqs)
    return 0;
  if (cdiv(max_context_len, kBlockSize) <= kMinRangePages) return 0;   // never split
  DeviceState* st = device_state();
  if (!st) return 0;
  const int32_t G = num_q_heads / num_kv_heads;
  return balanced_bytes_max(st, num_seqs, num_kv_heads, G, head_dim, max_context_len);
}

kvq_status kvq_selftest_wait_timeout(uint32_t limit_us, kvq_stream_t stream) {
  if (limit_us == 0 || limit_us > 1000000u) return KVQ_ERR_INVALID_ARGUMENT;
  DeviceState* st = device_state();
  if (!st) return cuda_fail();
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      (uint64_t)limit_us * 1000u, st->err);
  return cudaGetLastError() == cudaSuccess ? KVQ_OK : cuda_fail();
}

kvq_status kvq_get_error(kvq_stream_t stream, uint32_t* flags) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KVQ_ERR_CUDA;
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_kvq_error_word, sizeof v) != cudaSuccess) return KVQ_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_kvq_error_word, &zero, sizeof zero) != cudaSuccess)
    return KVQ_ERR_CUDA;
  if (flags) *flags = v;
  if (v == 0) return KVQ_OK;
  return (v & KVQ_DEVERR_TIMEOUT) ? KVQ_ERR_DEVICE_TIMEOUT : KVQ_ERR_DEVICE_INDEX;
}

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported shape or option";
    case KVQ_ERR_CUDA: return "CUDA runtime error";
    case KVQ_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case KVQ_ERR_DEVICE_INDEX: return "device-side index out of range";
    case KVQ_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

int32_t kvq_version(void) { return 100; }

}  // extern "C"
