// kvq_paged_decode_noalloc: the INT8 paged decode for callers that cannot
// allocate device memory.
//
// Who needs it: hosts that own every byte of device memory through their
// own pool (inference servers, framework plugins) and do not let a library
// call cudaMalloc; programs with a fixed memory budget decided at start-up;
// and latency-critical loops that must never trigger the implicit device
// synchronization cudaMalloc/cudaFree can cause.  kvq_paged_decode needs a
// caller-provided split-K workspace; this entry point instead uses a fixed
// scratch array compiled into the library, so the caller passes only inputs
// and outputs.
//
// The scratch is a file-scope __device__ array: every GPU that loads the
// library holds its KVQ_NOALLOC_SCRATCH_BYTES until the process exits.  Host
// code cannot use the array's name as a device address, so its address is
// looked up with cudaGetSymbolAddress once per device, on the first call made
// while that device is current (make that first call before any stream
// capture).  That address belongs to the device's context: after
// cudaDeviceReset (or anything else that destroys and recreates the primary
// context) this entry point must not be called again in the process.  All
// calls on a device share the one array: calls that overlap on the GPU
// (different streams, no ordering between them) race on it.  The split-K
// partials it holds are fully written before they are read, so nothing in it
// needs clearing between calls; it keeps the last call's contents.
//
// The array is handed to kvq_paged_decode as a workspace of exactly
// KVQ_NOALLOC_SCRATCH_BYTES.  That launcher fits its split-K work ranges into
// whatever workspace it is given (fewer, longer ranges when it is smaller
// than kvq_decode_workspace_bytes recommends, or one range per sequence), so
// only shapes for which not even one range per KV head fits are refused, with
// KVQ_ERR_WORKSPACE_TOO_SMALL.
#include <mutex>

#include "kvq.h"

static __device__ __align__(256) unsigned char g_kvq_noalloc_scratch[KVQ_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevicesNoAlloc = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevicesNoAlloc] = {};

// Device address of the scratch array on the current device (looked up once).
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevicesNoAlloc) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_kvq_noalloc_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev] = p;
  }
  return g_scratch_addr[dev];
}

}  // namespace

extern "C" {

kvq_status kvq_paged_decode_noalloc(const void* q, kvq_dtype dtype, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    const int8_t* k_cache, const int8_t* v_cache,
                                    const uint16_t* k_scale, const uint16_t* v_scale,
                                    int32_t num_blocks, int32_t block_size,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t max_context_len,
                                    float sm_scale, void* out, kvq_stream_t stream) {
  // checks that need no device, so that they answer without one
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_context_len < 0)
    return KVQ_ERR_INVALID_ARGUMENT;
  void* scratch = scratch_address();
  if (scratch == nullptr) return KVQ_ERR_CUDA;
  return kvq_paged_decode(q, dtype, num_seqs, num_q_heads, num_kv_heads, head_dim, k_cache,
                          v_cache, k_scale, v_scale, num_blocks, block_size, block_tables,
                          max_blocks_per_seq, context_lens, max_context_len, sm_scale, out,
                          scratch, KVQ_NOALLOC_SCRATCH_BYTES, stream);
}

}  // extern "C"
