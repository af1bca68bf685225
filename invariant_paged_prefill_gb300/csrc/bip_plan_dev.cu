// Device-side planner for graph-replayable prefill launches.  One CTA reads
// the batch's indptr arrays from device memory, validates them, and writes
// the work list the attention kernel consumes: for every request with new
// rows, every kv head and every group of tiles_per_unit consecutive q tiles
// of the request (counted from its first new row), one unit.  When the batch has few
// units (fewer than 8 per CTA of the launch, the host planner's rule) and
// the capacities allow, every unit with more than one segment is split into
// one item per segment writing partial states, with one merge unit per q
// tile; otherwise each unit is one item folding all its segments in its
// CTA.  Items, partial rows and merge units are laid out exactly as the
// host planner lays out a split or fold unit; the order is (request, kv
// head, longest group first), which only affects scheduling.  Because a
// row's arithmetic depends on no property of the plan (split and fold share
// one merge function), results are the bits of the host-planned launch.

#include <climits>

#include <cuda_runtime.h>

#include "bip_internal.h"

namespace bip {
namespace {

constexpr int kPlanThreads = 1024;
// Batches of up to this many requests keep each request's offsets in shared
// memory and write their items one (request, kv head) pair per thread;
// larger ones write them one request per thread.
constexpr int kPairRequests = 1536;

struct ReqGeom {
  int32_t q_len, kv_len, groups;  // groups of tiles_per_unit tiles holding the request's new rows
};

__device__ __forceinline__ bool request_geom(const DevPlanParams& p, int r, ReqGeom& g) {
  const int64_t ql = int64_t(p.qo_indptr[r + 1]) - p.qo_indptr[r];
  const int64_t np = int64_t(p.kv_indptr[r + 1]) - p.kv_indptr[r];
  g.q_len = 0;
  g.kv_len = 0;
  g.groups = 0;
  if (ql < 0 || np < 0) return false;
  int64_t kl = 0;
  if (np > 0) {
    const int32_t last = p.kv_last_page_len[r];
    if (last < 1 || last > p.page_size) return false;
    kl = (np - 1) * p.page_size + last;
  }
  if (ql > kl || kl > int64_t(32767) * kSplitLen) return false;
  // with a custom mask, every row's keys must lie inside its mask row
  if (p.mask_row_words > 0 && ql > 0 && kl > 32 * p.mask_row_words) return false;
  g.q_len = int32_t(ql);
  g.kv_len = int32_t(kl);
  if (ql > 0) g.groups = ((g.q_len - 1) / p.tile_pos) / p.tiles_per_unit + 1;
  return true;
}

// Group gi of request r (its kv head filled in by the caller): the fold
// item, and per slot the valid rows of its tile.
struct UnitGeom {
  WorkItem w;
  int32_t rows[kMaxTilesPerUnit];
};

__device__ __forceinline__ UnitGeom unit_geom(const DevPlanParams& p, int r, const ReqGeom& g, int gi) {
  UnitGeom u;
  const int32_t q_lo = g.kv_len - g.q_len;
  const int32_t t1 = (g.q_len - 1) / p.tile_pos;  // tile k: positions q_lo + k tile_pos ..
  WorkItem& w = u.w;
  w.kv_len = g.kv_len;
  w.page_base = p.kv_indptr[r];
  w.q_tok0 = p.qo_indptr[r] - q_lo;
  w.q_lo = q_lo;
  w.tile = gi * p.tiles_per_unit;
  w.kv_head = 0;
  int mask = 0, unit_end = -1, unit_first = INT_MAX;
  w.nseg[0] = w.nseg[1] = 0;
  u.rows[0] = u.rows[1] = 0;
  for (int t = 0; t < p.tiles_per_unit; ++t) {
    const int32_t tile = w.tile + t;
    if (tile > t1) continue;
    const int32_t first = q_lo + tile * p.tile_pos;
    const int32_t tile_end = min(first + p.tile_pos - 1, g.kv_len - 1);
    mask |= 1 << t;
    w.nseg[t] = int16_t(tile_end / kSplitLen + 1);
    u.rows[t] = (tile_end - first + 1) * p.group;
    unit_end = max(unit_end, tile_end);
    unit_first = min(unit_first, first);
  }
  // with a sliding window, keys before first - window are skipped
  const int32_t key_lo = p.window_left > 0 ? max(0, unit_first - p.window_left) : 0;
  w.flags = int16_t(mask * kSlotPresent);
  w.seg_lo = int16_t(key_lo / kSplitLen);
  w.seg_hi = int16_t(unit_end / kSplitLen);
  w.part_base[0] = w.part_base[1] = 0;
  w.blk_min = key_lo / p.kv_block;
  w.pad = 0;
  return u;
}

// Items, partial rows and merge units of a unit when split (a one-segment
// unit is never split).
__device__ __forceinline__ void split_counts(const DevPlanParams& p, const UnitGeom& u, int64_t& items,
                                             int64_t& part_rows, int64_t& merges) {
  if (u.w.seg_hi == u.w.seg_lo) {
    items += 1;
    return;
  }
  items += u.w.seg_hi - u.w.seg_lo + 1;
  for (int t = 0; t < p.tiles_per_unit; ++t)
    if (u.w.flags / kSlotPresent >> t & 1) {
      part_rows += int64_t(u.w.nseg[t] - u.w.seg_lo) * u.rows[t];
      merges += 1;
    }
}

// Inclusive block scan of one value per thread; returns the thread's
// exclusive prefix and sets total.
__device__ __forceinline__ int64_t block_scan(int64_t* s, int64_t v, int64_t& total) {
  const int tid = threadIdx.x;
  s[tid] = v;
  __syncthreads();
  for (int off = 1; off < kPlanThreads; off <<= 1) {
    const int64_t x = tid >= off ? s[tid - off] : 0;
    __syncthreads();
    s[tid] += x;
    __syncthreads();
  }
  total = s[kPlanThreads - 1];
  const int64_t excl = s[tid] - v;
  __syncthreads();
  return excl;
}

// Writes the items of unit (r, gi) for kv head h and, split, its merge
// units, starting at the given offsets, and advances them.
__device__ __forceinline__ void write_unit(const DevPlanParams& p, int r, const ReqGeom& g, int gi, int h, bool split,
                                           int64_t& o, int64_t& part, int64_t& mo) {
  UnitGeom u = unit_geom(p, r, g, gi);
  WorkItem w = u.w;
  w.kv_head = int16_t(h);
  if (!split || w.seg_hi == w.seg_lo) {
    p.items[o++] = w;
    return;
  }
  int64_t base[kMaxTilesPerUnit] = {0, 0};
  for (int t = 0; t < p.tiles_per_unit; ++t) {
    if (!(w.flags / kSlotPresent >> t & 1)) continue;
    MergeUnit m;
    m.q_tok0 = w.q_tok0;
    m.q_lo = w.q_lo;
    m.tile = w.tile + t;
    m.part_base = int32_t(part);
    m.rows = u.rows[t];
    m.kv_head = int16_t(h);
    m.nseg = int16_t(w.nseg[t] - w.seg_lo);  // partials of segments seg_lo .. nseg - 1
    m.pad[0] = m.pad[1] = 0;
    p.merges[mo++] = m;
    base[t] = part;
    part += int64_t(w.nseg[t] - w.seg_lo) * u.rows[t];
  }
  for (int sg = w.seg_lo; sg <= w.seg_hi; ++sg) {
    WorkItem ws = w;
    ws.seg_lo = ws.seg_hi = int16_t(sg);
    ws.flags = int16_t(w.flags | kItemSplit);
    for (int t = 0; t < p.tiles_per_unit; ++t) ws.part_base[t] = int32_t(base[t] + int64_t(sg - w.seg_lo) * u.rows[t]);
    p.items[o++] = ws;
  }
}

__global__ void __launch_bounds__(kPlanThreads) bip_device_plan_kernel(const DevPlanParams p) {
  __shared__ int64_t s_sum[kPlanThreads];
  // small batches: each request's first item, partial row and merge unit
  __shared__ int32_t s_item[kPairRequests], s_merge[kPairRequests];
  __shared__ int64_t s_part[kPairRequests];
  __shared__ int s_bad;
  const int tid = threadIdx.x;
  if (tid == 0) {
    p.header->status = 0u;
    p.header->where = 0u;
    p.header->bad_pages = 0u;
    p.header->n_items = 0u;
    p.header->n_merges = 0u;
    s_bad = 0;
    if (p.qo_indptr[0] != 0 || p.kv_indptr[0] != 0 || p.qo_indptr[p.batch] > p.max_total_q) s_bad = 1;
  }
  __syncthreads();
  const int per = (p.batch + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(tid * per, p.batch), r1 = min(r0 + per, p.batch);

  // counts (and validation) per request: fold items, and items, partial
  // rows and merge units if split
  int64_t n_fold = 0, n_split = 0, n_part = 0, n_merge = 0;
  bool bad = false;
  for (int r = r0; r < r1; ++r) {
    ReqGeom g;
    if (!request_geom(p, r, g)) bad = true;
    n_fold += int64_t(g.groups) * p.num_kv_heads;
    for (int gi = 0; gi < g.groups; ++gi) {
      int64_t it = 0, pr = 0, mg = 0;
      split_counts(p, unit_geom(p, r, g, gi), it, pr, mg);
      n_split += it * p.num_kv_heads;
      n_part += pr * p.num_kv_heads;
      n_merge += mg * p.num_kv_heads;
    }
  }
  if (bad) atomicOr(&s_bad, 1);
  int64_t t_fold, t_split, t_part, t_merge;
  const int64_t o_fold = block_scan(s_sum, n_fold, t_fold);
  const int64_t o_split = block_scan(s_sum, n_split, t_split);
  const int64_t o_part = block_scan(s_sum, n_part, t_part);
  const int64_t o_merge = block_scan(s_sum, n_merge, t_merge);
  const bool split = p.merge_capacity > 0 && t_fold < 8 * int64_t(p.grid) && t_split > t_fold &&
                     t_split <= p.capacity && t_part <= p.partial_capacity && t_merge <= p.merge_capacity;
  const int64_t total = split ? t_split : t_fold;
  if (s_bad || total > p.capacity) {
    if (tid == 0) p.header->status = s_bad ? 1u /* BIP_ERR_INVALID_ARG */ : 3u /* BIP_ERR_WORKSPACE_TOO_SMALL */;
    return;
  }

  // the items (and, split, the merge units), in (request, kv head, longest
  // group first) order
  int64_t o = split ? o_split : o_fold, part = o_part, mo = o_merge;
  if (p.batch <= kPairRequests) {
    // each request's offsets, then one (request, kv head) pair per thread:
    // head h of request r starts h shares into the request's range
    for (int r = r0; r < r1; ++r) {
      ReqGeom g;
      request_geom(p, r, g);
      int64_t it = 0, pr = 0, mg = 0;
      for (int gi = 0; gi < g.groups; ++gi) {
        if (split) split_counts(p, unit_geom(p, r, g, gi), it, pr, mg);
        else it += 1;
      }
      s_item[r] = int32_t(o);
      s_part[r] = part;
      s_merge[r] = int32_t(mo);
      o += it * p.num_kv_heads;
      part += pr * p.num_kv_heads;
      mo += mg * p.num_kv_heads;
    }
    __syncthreads();
    for (int i = tid; i < p.batch * p.num_kv_heads; i += kPlanThreads) {
      const int r = i / p.num_kv_heads, h = i - r * p.num_kv_heads;
      ReqGeom g;
      request_geom(p, r, g);
      if (g.groups == 0) continue;
      // this head's share of the request's items, partial rows and merges
      int64_t it = 0, pr = 0, mg = 0;
      for (int gi = 0; gi < g.groups; ++gi) {
        if (split) split_counts(p, unit_geom(p, r, g, gi), it, pr, mg);
        else it += 1;
      }
      int64_t oi = s_item[r] + int64_t(h) * it, pi = s_part[r] + int64_t(h) * pr, mi = s_merge[r] + int64_t(h) * mg;
      for (int gi = g.groups - 1; gi >= 0; --gi) write_unit(p, r, g, gi, h, split, oi, pi, mi);
    }
  } else {
    for (int r = r0; r < r1; ++r) {
      ReqGeom g;
      request_geom(p, r, g);
      for (int h = 0; h < p.num_kv_heads; ++h)
        for (int gi = g.groups - 1; gi >= 0; --gi) write_unit(p, r, g, gi, h, split, o, part, mo);
    }
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    p.header->n_merges = split ? uint32_t(t_merge) : 0u;
    p.header->n_items = uint32_t(total);
  }
}

}  // namespace

cudaError_t launch_device_plan(const DevPlanParams& p, cudaStream_t stream) {
  bip_device_plan_kernel<<<1, kPlanThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bip
