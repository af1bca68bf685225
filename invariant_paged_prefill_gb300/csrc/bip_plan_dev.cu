// Device-side planner for graph-replayable prefill launches.  It reads the
// batch's indptr arrays from device memory, validates them, and writes the
// work list the attention kernel consumes: for every request with new rows,
// every kv head and every group of tiles_per_unit consecutive q tiles of the
// request (counted from its first new row), one unit.  When the batch has
// few units (fewer than 8 per CTA of the attention launch, the host
// planner's rule) and the capacities allow, every unit with more than one
// segment is split into one item per segment writing partial states, with
// one merge unit per q tile; otherwise each unit is one item folding all its
// segments in its CTA.  Items, partial rows and merge units are laid out
// exactly as the host planner lays out a split or fold unit; the order is
// (request, kv head, longest group first), which only affects scheduling.
// Because a row's arithmetic depends on no property of the plan (split and
// fold share one merge function), results are the bits of the host-planned
// launch.
//
// Every CTA of the launch plans the whole batch the same way and writes its
// share of the list.  Batches of up to kSmallBatch requests keep each
// request's geometry and first unit (a scan over requests) in shared
// memory; a thread finds the request of a unit by binary search.  A folded
// unit's item index is its unit index; items are built in shared memory and
// copied out in whole lines.  Split, each unit's first item, partial row and
// merge unit come from scans over the units, and each thread writes one item
// (or one merge unit), finding its unit by binary search over those offsets.
// Larger batches are written by one CTA, one request per thread.

#include <climits>
#include <cstring>

#include <cuda_runtime.h>

#include "bip_internal.h"

namespace bip {
namespace {

constexpr int kPlanThreads = 1024;
static_assert(kPlanThreads == 32 * 32, "the block scan takes one warp of warp totals");
static_assert(sizeof(WorkItem) == 48 && sizeof(MergeUnit) == 32, "16-byte stores");
// Batches of up to this many requests are planned one unit per thread (their
// geometry and first units held in shared memory); larger ones one request
// per thread.
constexpr int kSmallBatch = 1536;
// CTAs of the planner launch: each plans the requests' units (the same in
// every CTA) and writes its share of the items; a large batch is written
// by CTA 0 alone.
constexpr int kPlanCtas = 16;
// Units of a batch that may split: fewer than 8 per CTA of the launch.
constexpr int kSplitUnits = 8 * kMaxCtas;
constexpr int kStageBytes = kPlanThreads * int(sizeof(WorkItem));
static_assert(kSplitUnits * 16 <= kStageBytes, "split unit offsets fit the staging memory");

struct ReqGeom {
  int32_t q_len, kv_len, groups;  // groups of tiles_per_unit tiles holding the request's new rows
  int32_t qo0, page_base;         // the request's first q row and first kv_indices entry
};

__device__ __forceinline__ bool request_geom(const DevPlanParams& p, int r, ReqGeom& g) {
  const int32_t qo0 = p.qo_indptr[r], page_base = p.kv_indptr[r];
  const int64_t ql = int64_t(p.qo_indptr[r + 1]) - qo0;
  const int64_t np = int64_t(p.kv_indptr[r + 1]) - page_base;
  g.q_len = 0;
  g.kv_len = 0;
  g.groups = 0;
  g.qo0 = qo0;
  g.page_base = page_base;
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

__device__ __forceinline__ UnitGeom unit_geom(const DevPlanParams& p, const ReqGeom& g, int gi) {
  UnitGeom u;
  const int32_t q_lo = g.kv_len - g.q_len;
  const int32_t t1 = (g.q_len - 1) / p.tile_pos;  // tile k: positions q_lo + k tile_pos ..
  WorkItem& w = u.w;
  w.kv_len = g.kv_len;
  w.page_base = g.page_base;
  w.q_tok0 = g.qo0 - q_lo;
  w.q_lo = q_lo;
  w.tile = gi * p.tiles_per_unit;
  w.kv_head = 0;
  int mask = 0, unit_end = -1, unit_first = INT_MAX;
  w.nseg[0] = w.nseg[1] = 0;
  u.rows[0] = u.rows[1] = 0;
#pragma unroll
  for (int t = 0; t < kMaxTilesPerUnit; ++t) {
    const int32_t tile = w.tile + t;
    if (t >= p.tiles_per_unit || tile > t1) continue;
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
__device__ __forceinline__ void split_counts(const UnitGeom& u, int64_t& items, int64_t& part_rows,
                                             int64_t& merges) {
  if (u.w.seg_hi == u.w.seg_lo) {
    items += 1;
    return;
  }
  items += u.w.seg_hi - u.w.seg_lo + 1;
#pragma unroll
  for (int t = 0; t < kMaxTilesPerUnit; ++t)
    if (u.w.flags / kSlotPresent >> t & 1) {
      part_rows += int64_t(u.w.nseg[t] - u.w.seg_lo) * u.rows[t];
      merges += 1;
    }
}

// Work items and merge units are written as 16-byte words (both arrays
// start 16-byte aligned in the workspace): narrower stores of a 48-byte item
// cost one L2 write per field and lane.
__device__ __forceinline__ void store_item(WorkItem* dst, const WorkItem& w) {
  int4 v[3];
  memcpy(v, &w, sizeof(v));
  int4* d = reinterpret_cast<int4*>(dst);
  d[0] = v[0];
  d[1] = v[1];
  d[2] = v[2];
}

__device__ __forceinline__ void store_merge(MergeUnit* dst, const MergeUnit& m) {
  int4 v[2];
  memcpy(v, &m, sizeof(v));
  int4* d = reinterpret_cast<int4*>(dst);
  d[0] = v[0];
  d[1] = v[1];
}

// Exclusive block scan of one value per thread (every thread calls it):
// returns the thread's exclusive prefix and sets total.  s_warp holds 32
// values.
__device__ __forceinline__ int64_t block_scan(int64_t* s_warp, int64_t v, int64_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int64_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int64_t w = s_warp[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  total = s_warp[31];
  const int64_t excl = x - v + (warp > 0 ? s_warp[warp - 1] : 0);
  __syncthreads();  // s_warp is free for the next scan
  return excl;
}

// Writes the items of a unit for kv head h and, split, its merge units,
// starting at the given offsets, and advances them.
__device__ __forceinline__ void write_unit(const DevPlanParams& p, const UnitGeom& u, int h, bool split,
                                           int64_t& o, int64_t& part, int64_t& mo) {
  WorkItem w = u.w;
  w.kv_head = int16_t(h);
  if (!split || w.seg_hi == w.seg_lo) {
    store_item(p.items + o++, w);
    return;
  }
  int64_t base[kMaxTilesPerUnit] = {0, 0};
#pragma unroll
  for (int t = 0; t < kMaxTilesPerUnit; ++t) {
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
    store_merge(p.merges + mo++, m);
    base[t] = part;
    part += int64_t(w.nseg[t] - w.seg_lo) * u.rows[t];
  }
  for (int sg = w.seg_lo; sg <= w.seg_hi; ++sg) {
    WorkItem ws = w;
    ws.seg_lo = ws.seg_hi = int16_t(sg);
    ws.flags = int16_t(w.flags | kItemSplit);
#pragma unroll
    for (int t = 0; t < kMaxTilesPerUnit; ++t) ws.part_base[t] = int32_t(base[t] + int64_t(sg - w.seg_lo) * u.rows[t]);
    store_item(p.items + o++, ws);
  }
}

// Small batches: unit u (in (request, kv head, longest group first) order)
// as its request's geometry, kv head and group.  unit0[r] is request r's
// first unit; its units end where the next non-empty request's begin.
__device__ __forceinline__ void locate_unit(const int32_t* unit0, const ReqGeom* geom, int batch, int32_t u,
                                            ReqGeom& g, int& h, int& gi) {
  int lo = 0, hi = batch - 1;  // the last request whose first unit is at or before u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (unit0[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  g = geom[lo];
  const int k = u - unit0[lo];
  h = k / g.groups;
  gi = g.groups - 1 - (k - h * g.groups);
}

__global__ void __launch_bounds__(kPlanThreads) bip_device_plan_kernel(const DevPlanParams p) {
  __shared__ int64_t s_warp[32];
  __shared__ ReqGeom s_geom[kSmallBatch];
  __shared__ int32_t s_unit0[kSmallBatch];
  __shared__ int s_bad;
  // dynamic: kPlanThreads staged work items (fold), or each unit's first
  // item, merge unit and partial row (split candidates)
  extern __shared__ int4 s_dyn[];
  WorkItem* s_stage = reinterpret_cast<WorkItem*>(s_dyn);
  int32_t* s_uitem = reinterpret_cast<int32_t*>(s_dyn);
  int32_t* s_umerge = s_uitem + kSplitUnits;
  int64_t* s_upart = reinterpret_cast<int64_t*>(s_umerge + kSplitUnits);
  const int tid = threadIdx.x, cta = blockIdx.x, ctas = gridDim.x;
  const bool small = p.batch <= kSmallBatch;
  if (tid == 0) {
    if (cta == 0) {
      p.header->status = 0u;
      p.header->where = 0u;
      p.header->bad_pages = 0u;
      p.header->n_items = 0u;
      p.header->n_merges = 0u;
    }
    s_bad = 0;
    if (p.qo_indptr[0] != 0 || p.kv_indptr[0] != 0 || p.qo_indptr[p.batch] > p.max_total_q) s_bad = 1;
  }
  __syncthreads();
  const int per = (p.batch + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(tid * per, p.batch), r1 = min(r0 + per, p.batch);

  // fold units (one per request, kv head and group) and validation
  int64_t n_fold = 0;
  bool bad = false;
  for (int r = r0; r < r1; ++r) {
    ReqGeom g;
    if (!request_geom(p, r, g)) bad = true;
    n_fold += int64_t(g.groups) * p.num_kv_heads;
    if (small) s_geom[r] = g;
  }
  if (bad) atomicOr(&s_bad, 1);
  int64_t t_fold;
  const int64_t o_fold = block_scan(s_warp, n_fold, t_fold);
  if (s_bad || t_fold > p.capacity) {
    if (tid == 0 && cta == 0)
      p.header->status = s_bad ? 1u /* BIP_ERR_INVALID_ARG */ : 3u /* BIP_ERR_WORKSPACE_TOO_SMALL */;
    return;
  }
  if (small) {
    int32_t o = int32_t(o_fold);
    for (int r = r0; r < r1; ++r) {
      s_unit0[r] = o;
      o += s_geom[r].groups * p.num_kv_heads;
    }
  }
  __syncthreads();
  const int32_t n_units = int32_t(t_fold);

  // a batch of few units is split if the capacities hold it
  int64_t t_split = 0, t_part = 0, t_merge = 0;
  int64_t o_split = 0, o_part = 0, o_merge = 0;  // large batches: this thread's first split offsets
  const bool may_split = p.merge_capacity > 0 && t_fold < 8 * int64_t(p.grid);
  if (may_split) {
    if (small) {
      // each unit's first item, partial row and merge unit if split
      for (int32_t c = 0; c < n_units; c += kPlanThreads) {
        int64_t it = 0, pr = 0, mg = 0, ti, tp, tm;
        if (c + tid < n_units) {
          ReqGeom g;
          int h, gi;
          locate_unit(s_unit0, s_geom, p.batch, c + tid, g, h, gi);
          split_counts(unit_geom(p, g, gi), it, pr, mg);
        }
        const int64_t eo = block_scan(s_warp, it, ti);
        const int64_t ep = block_scan(s_warp, pr, tp);
        const int64_t em = block_scan(s_warp, mg, tm);
        if (c + tid < n_units) {
          s_uitem[c + tid] = int32_t(t_split + eo);
          s_upart[c + tid] = t_part + ep;
          s_umerge[c + tid] = int32_t(t_merge + em);
        }
        t_split += ti;
        t_part += tp;
        t_merge += tm;
      }
    } else {
      int64_t it = 0, pr = 0, mg = 0;
      for (int r = r0; r < r1; ++r) {
        ReqGeom g;
        request_geom(p, r, g);
        for (int gi = 0; gi < g.groups; ++gi) split_counts(unit_geom(p, g, gi), it, pr, mg);
      }
      o_split = block_scan(s_warp, it * p.num_kv_heads, t_split);
      o_part = block_scan(s_warp, pr * p.num_kv_heads, t_part);
      o_merge = block_scan(s_warp, mg * p.num_kv_heads, t_merge);
    }
  }
  __syncthreads();  // the unit offsets are written; the fold path reuses their memory
  const bool split = may_split && t_split > t_fold && t_split <= p.capacity && t_part <= p.partial_capacity &&
                     t_merge <= p.merge_capacity;
  const int64_t total = split ? t_split : t_fold;

  // the items (and, split, the merge units), in (request, kv head, longest
  // group first) order
  if (small && !split) {
    // a folded unit's item index is its unit index: chunks of up to
    // kPlanThreads items, spread over the CTAs, are built in shared memory
    // and copied out in whole lines
    const int32_t cs = min(kPlanThreads, (n_units + ctas - 1) / ctas);
    for (int32_t c = cta * cs; c < n_units; c += ctas * cs) {
      const int32_t n = min(cs, n_units - c);
      if (tid < n) {
        ReqGeom g;
        int h, gi;
        locate_unit(s_unit0, s_geom, p.batch, c + tid, g, h, gi);
        WorkItem w = unit_geom(p, g, gi).w;
        w.kv_head = int16_t(h);
        store_item(s_stage + tid, w);
      }
      __syncthreads();
      const int4* src = reinterpret_cast<const int4*>(s_stage);
      int4* dst = reinterpret_cast<int4*>(p.items + c);
      for (int i = tid; i < n * 3; i += kPlanThreads) dst[i] = src[i];
      __syncthreads();
    }
  } else if (small) {
    // split: one item per thread, in unit order (every unit has at least
    // one item, so item i is in the last unit whose first item is at or
    // before i); then one merge unit per thread (slot 0 of a unit is always
    // present, so merge k of a unit is its slot k)
    const int32_t ipc = int32_t((t_split + ctas - 1) / ctas), mpc = int32_t((t_merge + ctas - 1) / ctas);
    const int32_t i1 = int32_t(min(t_split, int64_t(cta + 1) * ipc));
    for (int32_t i = cta * ipc + tid; i < i1; i += kPlanThreads) {
      int lo = 0, hi = n_units - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_uitem[mid] <= i) lo = mid;
        else hi = mid - 1;
      }
      ReqGeom g;
      int h, gi;
      locate_unit(s_unit0, s_geom, p.batch, lo, g, h, gi);
      const UnitGeom ug = unit_geom(p, g, gi);
      WorkItem w = ug.w;
      w.kv_head = int16_t(h);
      if (w.seg_hi != w.seg_lo) {
        const int sg = w.seg_lo + (i - s_uitem[lo]);
        int64_t base = s_upart[lo];
#pragma unroll
        for (int t = 0; t < kMaxTilesPerUnit; ++t) {
          if (!(w.flags / kSlotPresent >> t & 1)) continue;
          w.part_base[t] = int32_t(base + int64_t(sg - w.seg_lo) * ug.rows[t]);
          base += int64_t(w.nseg[t] - w.seg_lo) * ug.rows[t];
        }
        w.seg_lo = w.seg_hi = int16_t(sg);
        w.flags = int16_t(w.flags | kItemSplit);
      }
      store_item(p.items + i, w);
    }
    const int32_t m1 = int32_t(min(t_merge, int64_t(cta + 1) * mpc));
    for (int32_t m = cta * mpc + tid; m < m1; m += kPlanThreads) {
      int lo = 0, hi = n_units - 1;  // the last unit whose first merge unit is at or before m
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_umerge[mid] <= m) lo = mid;
        else hi = mid - 1;
      }
      ReqGeom g;
      int h, gi;
      locate_unit(s_unit0, s_geom, p.batch, lo, g, h, gi);
      const UnitGeom ug = unit_geom(p, g, gi);
      const bool t1 = m - s_umerge[lo] == 1;
      const int32_t rows0 = ug.rows[0], nseg0 = ug.w.nseg[0] - ug.w.seg_lo;
      MergeUnit mu;
      mu.q_tok0 = ug.w.q_tok0;
      mu.q_lo = ug.w.q_lo;
      mu.tile = ug.w.tile + (t1 ? 1 : 0);
      mu.part_base = int32_t(s_upart[lo] + (t1 ? int64_t(nseg0) * rows0 : 0));
      mu.rows = t1 ? ug.rows[1] : rows0;
      mu.kv_head = int16_t(h);
      mu.nseg = int16_t(t1 ? ug.w.nseg[1] - ug.w.seg_lo : nseg0);  // partials of segments seg_lo .. nseg - 1
      mu.pad[0] = mu.pad[1] = 0;
      store_merge(p.merges + m, mu);
    }
  } else if (cta == 0) {
    int64_t o = split ? o_split : o_fold, part = o_part, mo = o_merge;
    for (int r = r0; r < r1; ++r) {
      ReqGeom g;
      request_geom(p, r, g);
      for (int h = 0; h < p.num_kv_heads; ++h)
        for (int gi = g.groups - 1; gi >= 0; --gi) write_unit(p, unit_geom(p, g, gi), h, split, o, part, mo);
    }
  }
  __syncthreads();
  if (tid == 0 && cta == 0) {
    __threadfence();
    p.header->n_merges = split ? uint32_t(t_merge) : 0u;
    p.header->n_items = uint32_t(total);
  }
}

}  // namespace

cudaError_t launch_device_plan(const DevPlanParams& p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e =
        cudaFuncSetAttribute(bip_device_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  bip_device_plan_kernel<<<kPlanCtas, kPlanThreads, kStageBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bip
