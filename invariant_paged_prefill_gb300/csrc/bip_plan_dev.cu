// Device-side planner for graph-replayable prefill launches.  One CTA reads
// the batch's indptr arrays from device memory, validates them, and writes
// the work list the attention kernel consumes: for every request with new
// rows, every kv head and every group of tiles_per_unit consecutive absolute
// q tiles that hold rows of the request, one item over all of the group's
// segments (folded in the CTA: no partials, no merge kernel).  The same
// items, field for field, as the host planner's fold-only plan; the order is
// (request, kv head, longest group first), which only affects scheduling.
// Because a row's arithmetic depends on no property of the plan, results are
// the bits of the host-planned launch.

#include <climits>

#include <cuda_runtime.h>

#include "bip_internal.h"

namespace bip {
namespace {

constexpr int kPlanThreads = 1024;

struct ReqGeom {
  int32_t q_len, kv_len, g0, groups;  // groups of tiles holding rows of the request
};

__device__ __forceinline__ bool request_geom(const DevPlanParams& p, int r, ReqGeom& g) {
  const int64_t ql = int64_t(p.qo_indptr[r + 1]) - p.qo_indptr[r];
  const int64_t np = int64_t(p.kv_indptr[r + 1]) - p.kv_indptr[r];
  g.q_len = 0;
  g.kv_len = 0;
  g.g0 = 0;
  g.groups = 0;
  if (ql < 0 || np < 0) return false;
  int64_t kl = 0;
  if (np > 0) {
    const int32_t last = p.kv_last_page_len[r];
    if (last < 1 || last > p.page_size) return false;
    kl = (np - 1) * p.page_size + last;
  }
  if (ql > kl || kl > int64_t(32767) * kSplitLen) return false;
  g.q_len = int32_t(ql);
  g.kv_len = int32_t(kl);
  if (ql > 0) {
    const int32_t t0 = (g.kv_len - g.q_len) / p.tile_pos, t1 = (g.kv_len - 1) / p.tile_pos;
    g.g0 = (t0 / p.tiles_per_unit) * p.tiles_per_unit;
    g.groups = (t1 - g.g0) / p.tiles_per_unit + 1;
  }
  return true;
}

__global__ void __launch_bounds__(kPlanThreads) bip_device_plan_kernel(const DevPlanParams p) {
  __shared__ int32_t s_sum[kPlanThreads];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    p.header->status = 0u;
    p.header->where = 0u;
    p.header->bad_pages = 0u;
    p.header->n_items = 0u;
    s_bad = 0;
    if (p.qo_indptr[0] != 0 || p.kv_indptr[0] != 0 || p.qo_indptr[p.batch] > p.max_total_q) s_bad = 1;
  }
  __syncthreads();
  const int per = (p.batch + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(tid * per, p.batch), r1 = min(r0 + per, p.batch);

  // counts (and validation) per request
  int32_t local = 0;
  bool bad = false;
  for (int r = r0; r < r1; ++r) {
    ReqGeom g;
    if (!request_geom(p, r, g)) bad = true;
    local += g.groups * p.num_kv_heads;
  }
  if (bad) atomicOr(&s_bad, 1);
  s_sum[tid] = local;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {  // inclusive scan
    const int32_t v = tid >= off ? s_sum[tid - off] : 0;
    __syncthreads();
    s_sum[tid] += v;
    __syncthreads();
  }
  const int32_t total = s_sum[kPlanThreads - 1];
  if (s_bad || total > p.capacity) {
    if (tid == 0) p.header->status = s_bad ? 1u /* BIP_ERR_INVALID_ARG */ : 3u /* BIP_ERR_WORKSPACE_TOO_SMALL */;
    return;
  }

  // the items
  int32_t o = s_sum[tid] - local;
  for (int r = r0; r < r1; ++r) {
    ReqGeom g;
    request_geom(p, r, g);
    if (g.groups == 0) continue;
    const int32_t q_lo = g.kv_len - g.q_len;
    const int32_t t0 = q_lo / p.tile_pos, t1 = (g.kv_len - 1) / p.tile_pos;
    for (int h = 0; h < p.num_kv_heads; ++h) {
      for (int gi = g.groups - 1; gi >= 0; --gi) {  // longest group first
        WorkItem w;
        w.kv_len = g.kv_len;
        w.page_base = p.kv_indptr[r];
        w.q_tok0 = p.qo_indptr[r] - q_lo;
        w.q_lo = q_lo;
        w.tile = g.g0 + gi * p.tiles_per_unit;
        w.kv_head = int16_t(h);
        int mask = 0, unit_end = -1, unit_first = INT_MAX;
        w.nseg[0] = w.nseg[1] = 0;
        for (int t = 0; t < p.tiles_per_unit; ++t) {
          const int32_t tile = w.tile + t;
          if (tile < t0 || tile > t1) continue;
          const int32_t tile_end = min(tile * p.tile_pos + p.tile_pos - 1, g.kv_len - 1);
          mask |= 1 << t;
          w.nseg[t] = int16_t(tile_end / kSplitLen + 1);
          unit_end = max(unit_end, tile_end);
          unit_first = min(unit_first, max(tile * p.tile_pos, q_lo));
        }
        // with a sliding window, keys before first - window are skipped
        const int32_t key_lo = p.window_left > 0 ? max(0, unit_first - p.window_left) : 0;
        w.flags = int16_t(mask * kSlotPresent);
        w.seg_lo = int16_t(key_lo / kSplitLen);
        w.seg_hi = int16_t(unit_end / kSplitLen);
        w.part_base[0] = w.part_base[1] = 0;
        w.blk_min = key_lo / p.kv_block;
        w.pad = 0;
        p.items[o++] = w;
      }
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    p.header->n_items = uint32_t(total);
  }
}

}  // namespace

cudaError_t launch_device_plan(const DevPlanParams& p, cudaStream_t stream) {
  bip_device_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bip
