// Instantiations of the INT8-cache decode kernel with static (per-tensor,
// binary32) scales -- head_dim 64/128, FP16/BF16 activations -- and their
// host-side launch helpers.
#include "kvq_decode.cuh"

namespace kvq {

namespace {
template <int D, bool BF16>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&paged_decode_kernel<D, true, BF16, true>);
}
const void* pick(int D, bool bf16) {
  if (D == 128) return bf16 ? kernel_ptr<128, true>() : kernel_ptr<128, false>();
  return bf16 ? kernel_ptr<64, true>() : kernel_ptr<64, false>();
}
}  // namespace

size_t decode_smem_bytes_static(int D, int B, int G) {
  return D == 128 ? SmemLayout<128, true, true>(B, G).total_bytes
                  : SmemLayout<64, true, true>(B, G).total_bytes;
}

cudaError_t decode_configure_static(int D, bool bf16, size_t smem) {
  // all of the unified L1/shared array as shared memory: the kernel's
  // occupancy is set by its page stages
  cudaError_t e = cudaFuncSetAttribute(pick(D, bf16), cudaFuncAttributePreferredSharedMemoryCarveout,
                                       (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(pick(D, bf16), cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem);
}

cudaError_t decode_occupancy_static(int D, bool bf16, size_t smem, int* n) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, pick(D, bf16), kThreads, smem);
}

cudaError_t decode_launch_static(int D, bool bf16, const CUtensorMap* maps,
                               const DecodeParams& p, int grid, size_t smem, cudaStream_t s) {
  // programmatic stream serialization: the launch may overlap the tail of the
  // previous kernel in the stream; the kernel waits (griddepcontrol) before
  // reading any input
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (D == 128) {
    return bf16 ? cudaLaunchKernelEx(&cfg, paged_decode_kernel<128, true, true, true>, maps[0],
                                     maps[1], p)
                : cudaLaunchKernelEx(&cfg, paged_decode_kernel<128, true, false, true>, maps[0],
                                     maps[1], p);
  }
  return bf16 ? cudaLaunchKernelEx(&cfg, paged_decode_kernel<64, true, true, true>, maps[0],
                                   maps[1], p)
              : cudaLaunchKernelEx(&cfg, paged_decode_kernel<64, true, false, true>, maps[0],
                                   maps[1], p);
}

}  // namespace kvq
