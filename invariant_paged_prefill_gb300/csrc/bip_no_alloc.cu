// bip_prefill_no_alloc: bip_prefill for callers that cannot allocate device
// memory.  Its workspace is a file-scope device array instead of a buffer
// the caller passes in; everything else (inputs, outputs, stream) is the
// caller's, and the work runs through bip_prefill unchanged.
//
// Who needs this: code that runs where cudaMalloc is not allowed or not
// wanted -- an engine plugin whose host framework owns every byte of device
// memory through its own pool and offers no allocation hook, a real-time
// serving loop that forbids allocation on the request path, or a caller
// without a device allocator at hand.  Such callers still pass q, pages,
// indices, out and lse.
//
// Costs and limits: every GPU that loads this library holds the array
// (BIP_NO_ALLOC_WORKSPACE_BYTES, 32 MiB) until the process exits.  The first
// call on a device looks the array's device address up (cudaGetSymbolAddress,
// with that device current), which may load the module: make that first call
// before any stream capture.  A plan whose workspace
// is larger is rejected with BIP_ERR_WORKSPACE_TOO_SMALL; a smaller split
// budget makes a plan fit.  All calls share the array, which keeps the last
// call's contents: calls whose work overlaps on the GPU race and must be
// ordered.  What must start at zero (the status word in the header) is
// rewritten by every call's work-list upload; every other region is written
// before it is read.

#include <mutex>

#include <cuda_runtime.h>

#include "../../include/bip.h"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = BIP_NO_ALLOC_WORKSPACE_BYTES;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_no_alloc_workspace[kNoAllocWorkspaceBytes];

// Device address of the array per device, looked up once with that device
// current (in host code the array's name is only a stand-in, not an address)
// and kept for the life of the process: after a cudaDeviceReset of that
// device the module may load at another address, so calls made after a
// reset are not supported.
void* g_no_alloc_addr[kMaxDevices] = {};
std::mutex g_no_alloc_mu;

}  // namespace

extern "C" bip_status bip_prefill_no_alloc(bip_plan_t plan, const void* q, int64_t num_q_rows, const void* k_pages,
                                           const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                           const int32_t* kv_indices, float k_scale, float v_scale, void* out,
                                           float* lse, cudaStream_t stream) {
  if (!plan) return BIP_ERR_INVALID_ARG;
  bip_plan_info info;
  bip_status st = bip_plan_get_info(plan, &info);
  if (st != BIP_OK) return st;
  if (info.workspace_bytes > kNoAllocWorkspaceBytes) return BIP_ERR_WORKSPACE_TOO_SMALL;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return BIP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return BIP_ERR_UNSUPPORTED;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_no_alloc_mu);
    if (!g_no_alloc_addr[dev]) {
      void* addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_no_alloc_workspace) != cudaSuccess || !addr) {
        cudaGetLastError();  // the failure is reported through the status, not left pending
        return BIP_ERR_CUDA;
      }
      g_no_alloc_addr[dev] = addr;
    }
    ws = g_no_alloc_addr[dev];
  }
  return bip_prefill(plan, q, num_q_rows, k_pages, v_pages, num_pages, page_stride_elems, kv_indices, k_scale,
                     v_scale, out, lse, ws, kNoAllocWorkspaceBytes, stream);
}
