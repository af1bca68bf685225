// The per-call work-list upload of bip_prefill / bip_append_kv: SM loads of
// the plan's pinned (mapped) host image, stored into the workspace.  A copy
// on the copy engines would share an engine with whatever bulk copies other
// streams have queued (the next batch's inputs, the last batch's outputs)
// and could wait for them to finish; SM loads over the host link do not.

#include "bip_internal.h"

namespace bip {
namespace {

// Plain (coherent) loads: the source is host memory.
__global__ void __launch_bounds__(256) bip_upload_kernel(const uint4* src, uint4* dst, size_t n) {
  for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < n; i += size_t(gridDim.x) * blockDim.x)
    dst[i] = src[i];
}

}  // namespace

cudaError_t launch_upload(const void* src_dev, void* dst, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  if (bytes % 16 != 0 || (reinterpret_cast<uintptr_t>(src_dev) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
    return cudaErrorInvalidValue;
  const size_t n = bytes / 16;
  const size_t blocks = (n + 255) / 256;
  const unsigned grid = unsigned(blocks < 128 ? blocks : 128);
  bip_upload_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(src_dev), static_cast<uint4*>(dst), n);
  return cudaGetLastError();
}

}  // namespace bip
