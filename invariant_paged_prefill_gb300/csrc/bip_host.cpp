// Host side of the C ABI: validation, the batch-independent tile schedule,
// workspace layout, tensor-map encoding and kernel launches.
//
// The schedule never looks at batch statistics (the failure of the prior
// art: a tile chosen from avg_packed_qo_len, sglang PR 46351 "Root cause").
// Every unit's geometry is a function of its own request's lengths only:
// q tiles are T = floor(128 / group) consecutive positions counted from the
// request's first new row, and keys are cut at absolute multiples of the
// block and segment lengths.  Batch composition, policy and SM count only decide which CTA
// runs a unit and whether its segments are folded or split, which does not
// change any row's arithmetic.

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/bip.h"
#include "bip_internal.h"

using bip::MergeUnit;
using bip::WorkItem;

namespace {

constexpr size_t kDefaultSplitBudget = size_t(256) << 20;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct UnitDesc {
  int32_t request, kv_head, tile;  // tile of slot 0, counted from the request's first new row
  int32_t mask;                    // slots present
  int32_t rows[bip::kMaxTilesPerUnit], nseg[bip::kMaxTilesPerUnit];  // nseg: segments 0 .. tile_end / L
  int32_t blk_min, seg_lo, seg_hi;  // first block, first and last segment the unit visits
  int32_t blocks;                   // blocks visited (union of the slots' keys, window applied)
};

}  // namespace

struct bip_plan_s {
  int32_t batch = 0, hq = 0, hkv = 0, d = 0, page_size = 0, kv_dtype = 0;
  int32_t group = 0, T = 0, bn = 0, nt = 1, total_q = 0;
  int32_t max_kv_q = 0;  // longest kv_len among requests with q rows (custom mask row length)
  bip_plan_options opts{};
  int32_t n_items = 0;               // work items (in the host image, after the header)
  std::vector<MergeUnit> merges;
  std::vector<int32_t> item_desc;  // 8 int32 per item, see bip_plan_get_items
  std::vector<bip::AppendRow> reqs;  // requests with new rows, for bip_append_kv
  int32_t num_units = 0, num_split_units = 0, grid = 0;
  int64_t partial_rows = 0, kv_blocks = 0;
  bool need_scratch = false;
  uint64_t wait_limit_cycles = 0;  // in-kernel wait bound, SM cycles at the peak clock
  int32_t sms = 0;                 // CTAs to fill (the planned device's SM count, capped)
  size_t off_items = 0, off_merges = 0, off_reqs = 0, off_partials = 0, off_scratch = 0, off_keys = 0;
  size_t partial_bytes = 0, scratch_bytes = 0, ws_bytes = 0, upload_bytes = 0;
  uint8_t* upload = nullptr;  // header + items + merges, as copied to the workspace
  const void* upload_dev = nullptr;  // the same pinned buffer as the device sees it (mapped), if it is
  bool pinned = false;
  // One event per stream the plan's calls were enqueued on (eagerly, not
  // under capture), recorded after each call: bip_plan_destroy waits for
  // them before it frees the host image those calls read.
  std::mutex use_mu;
  std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;
};

extern "C" const char* bip_status_string(bip_status s) {
  switch (s) {
    case BIP_OK: return "BIP_OK";
    case BIP_ERR_INVALID_ARG: return "BIP_ERR_INVALID_ARG";
    case BIP_ERR_UNSUPPORTED: return "BIP_ERR_UNSUPPORTED";
    case BIP_ERR_WORKSPACE_TOO_SMALL: return "BIP_ERR_WORKSPACE_TOO_SMALL";
    case BIP_ERR_CUDA: return "BIP_ERR_CUDA";
    case BIP_ERR_DEVICE_TIMEOUT: return "BIP_ERR_DEVICE_TIMEOUT";
    case BIP_ERR_OUT_OF_MEMORY: return "BIP_ERR_OUT_OF_MEMORY";
    case BIP_ERR_BAD_PAGE_INDEX: return "BIP_ERR_BAD_PAGE_INDEX";
  }
  return "BIP_ERR_UNKNOWN";
}

namespace {

bool head_dim_supported(int32_t d) { return d == 128 || d == 256; }

bip_status check_heads(int32_t hq, int32_t hkv, int32_t d) {
  if (hq <= 0 || hkv <= 0 || d <= 0 || hq % hkv != 0) return BIP_ERR_INVALID_ARG;
  if (!head_dim_supported(d) || hq / hkv > bip::kTileRows) return BIP_ERR_UNSUPPORTED;
  return BIP_OK;
}

size_t partial_row_bytes(int32_t d) { return size_t(d + 4) * sizeof(float); }

// Bytes of the custom-mask pass's first-visible-key array: one int32 per q row.
size_t key_bytes_for(int64_t q_rows) { return size_t(q_rows) * sizeof(int32_t); }

size_t layout_bytes(size_t n_items, size_t n_merges, size_t n_reqs, size_t partial_bytes, size_t scratch_bytes,
                    size_t key_bytes, size_t* off_items, size_t* off_merges, size_t* off_reqs, size_t* off_partials,
                    size_t* off_scratch, size_t* off_keys, size_t* upload_bytes) {
  // header | request rows | work items | merge units: the append uploads only
  // the prefix before the work items.
  size_t o = bip::kHeaderBytes;
  *off_reqs = o;
  o += n_reqs * sizeof(bip::AppendRow);
  o = align_up(o, 16);
  *off_items = o;
  o += n_items * sizeof(WorkItem);
  *off_merges = o;
  o += n_merges * sizeof(MergeUnit);
  *upload_bytes = o;
  o = align_up(o, 256);
  *off_partials = o;
  o = align_up(o + partial_bytes, 256);
  *off_scratch = o;
  o = align_up(o + scratch_bytes, 256);
  *off_keys = o;
  o += key_bytes;
  return align_up(o, 256);
}

int query_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 148;
  }
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return 148;
  }
  return n;
}

// Peak SM clock of the current device in kHz (2.07 GHz if it cannot be
// read).  The attribute query is slow (hundreds of microseconds), so each
// device's answer is kept.
uint64_t query_clock_khz() {
  static std::atomic<uint64_t> cache[64];
  int dev = 0, khz = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return 2070000;
  }
  if (dev >= 0 && dev < 64) {
    const uint64_t v = cache[dev].load(std::memory_order_relaxed);
    if (v) return v;
  }
  if (cudaDeviceGetAttribute(&khz, cudaDevAttrClockRate, dev) != cudaSuccess || khz <= 0) {
    cudaGetLastError();
    return 2070000;
  }
  if (dev >= 0 && dev < 64) cache[dev].store(uint64_t(khz), std::memory_order_relaxed);
  return uint64_t(khz);
}

}  // namespace

extern "C" size_t bip_workspace_bound(int32_t max_batch, int32_t max_total_q, int32_t num_qo_heads,
                                      int32_t num_kv_heads, int32_t head_dim, size_t split_budget_bytes) {
  if (max_batch < 0 || max_total_q < 0 || check_heads(num_qo_heads, num_kv_heads, head_dim) != BIP_OK) return 0;
  const int64_t group = num_qo_heads / num_kv_heads;
  const int64_t T = bip::kTileRows / group;
  // A request with q_len rows has ceil(q_len / T) tiles, so at most that
  // many units (a unit holds one or two tiles); the bound allows one more.
  const int64_t units = int64_t(num_kv_heads) * ((int64_t(max_total_q) + T - 1) / T + 2 * int64_t(max_batch));
  // Each extra split item needs at least `group` partial rows of budget.
  const int64_t extra = int64_t(split_budget_bytes / (size_t(group) * partial_row_bytes(head_dim)));
  const size_t scratch =
      size_t(bip::kMaxCtas) * bip::max_tiles_per_unit_for(head_dim) * bip::kTileRows * head_dim * sizeof(float);
  size_t a, b, c, e, k, u, rq;
  return layout_bytes(size_t(units + extra), size_t(units), size_t(max_batch), split_budget_bytes, scratch,
                      key_bytes_for(max_total_q), &a, &b, &rq, &c, &e, &k, &u);
}

extern "C" bip_status bip_plan(bip_plan_t* plan_out, const int32_t* qo_indptr, const int32_t* kv_indptr,
                               const int32_t* kv_last_page_len, int32_t batch, int32_t num_qo_heads,
                               int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                               bip_kv_dtype kv_dtype, const bip_plan_options* opts_in,
                               size_t* workspace_bytes) {
  if (!plan_out) return BIP_ERR_INVALID_ARG;
  *plan_out = nullptr;
  if (batch < 0 || !qo_indptr || !kv_indptr || (batch > 0 && !kv_last_page_len)) return BIP_ERR_INVALID_ARG;
  bip_status st = check_heads(num_qo_heads, num_kv_heads, head_dim);
  if (st != BIP_OK) return st;
  if (kv_dtype != BIP_KV_BF16 && kv_dtype != BIP_KV_FP8_E4M3) return BIP_ERR_INVALID_ARG;
  const int32_t bn = bip::kv_block_for(head_dim);
  if (page_size <= 0) return BIP_ERR_INVALID_ARG;
  if ((page_size & (page_size - 1)) != 0 || page_size > bn) return BIP_ERR_UNSUPPORTED;

  bip_plan_options opts;
  opts.split_policy = BIP_SPLIT_AUTO;
  opts.split_budget_bytes = kDefaultSplitBudget;
  opts.num_sms = 0;
  opts.wait_limit_ns = 0;
  opts.tiles_per_unit = 0;
  opts.window_left = 0;
  if (opts_in) opts = *opts_in;
  if (opts.window_left < 0) return BIP_ERR_INVALID_ARG;
  if (opts.split_policy != BIP_SPLIT_AUTO && opts.split_policy != BIP_SPLIT_NEVER &&
      opts.split_policy != BIP_SPLIT_ALWAYS)
    return BIP_ERR_INVALID_ARG;
  if (opts.num_sms < 0) return BIP_ERR_INVALID_ARG;
  if (opts.tiles_per_unit < 0 || opts.tiles_per_unit > bip::max_tiles_per_unit_for(head_dim))
    return BIP_ERR_INVALID_ARG;
  // FP8 pages and token-granular pages (below 8 slots) run one-tile variants
  // (their dequant and row-gather warpgroups need the room).
  if (page_size < 8 && opts.tiles_per_unit == 2) return BIP_ERR_UNSUPPORTED;
  if (opts.wait_limit_ns == 0) opts.wait_limit_ns = bip::kDefaultWaitNs;

  // ---- lengths and validation
  if (qo_indptr[0] != 0 || kv_indptr[0] != 0) return BIP_ERR_INVALID_ARG;
  const int32_t group = num_qo_heads / num_kv_heads;
  const int32_t T = bip::kTileRows / group;
  std::vector<int32_t> q_len(batch), kv_len(batch);
  for (int32_t r = 0; r < batch; ++r) {
    const int64_t ql = int64_t(qo_indptr[r + 1]) - qo_indptr[r];
    const int64_t np = int64_t(kv_indptr[r + 1]) - kv_indptr[r];
    if (ql < 0 || np < 0) return BIP_ERR_INVALID_ARG;
    int64_t kl = 0;
    if (np > 0) {
      if (kv_last_page_len[r] < 1 || kv_last_page_len[r] > page_size) return BIP_ERR_INVALID_ARG;
      kl = (np - 1) * page_size + kv_last_page_len[r];
    }
    if (ql > kl) return BIP_ERR_INVALID_ARG;
    if (kl > int64_t(32767) * bip::kSplitLen) return BIP_ERR_UNSUPPORTED;  // segment ids are int16
    q_len[r] = int32_t(ql);
    kv_len[r] = int32_t(kl);
  }

  // ---- tiles per unit (numerically neutral).  Two tiles per CTA share every
  // KV block and overlap one tile's softmax with the other's MMAs; one tile
  // per CTA leaves room for a deeper KV ring, which short extends (bound by
  // HBM, one tile per request) need more.
  int32_t NT = opts.tiles_per_unit;
  if (NT == 0) {
    int64_t tiles = 0, active = 0;
    for (int32_t r = 0; r < batch; ++r) {
      if (q_len[r] == 0) continue;
      ++active;
      tiles += (q_len[r] - 1) / T + 1;
    }
    NT = (bip::max_tiles_per_unit_for(head_dim) >= 2 && page_size >= 8 && tiles >= 2 * active) ? 2 : 1;
  }

  // ---- units: (request, kv head, NT consecutive q tiles sharing keys).
  // Tile k of a request holds its new rows at positions q_lo + k T ..
  // q_lo + k T + T - 1: a row's arithmetic does not depend on which rows
  // share its tile, so tiles start at the first new row, and an extend of
  // q_len rows needs ceil(q_len / T) tiles wherever its rows fall.
  std::vector<UnitDesc> units;
  {
    size_t n = 0;
    for (int32_t r = 0; r < batch; ++r)
      if (q_len[r] > 0) n += size_t(((q_len[r] - 1) / T) / NT + 1) * num_kv_heads;
    units.reserve(n);
  }
  for (int32_t r = 0; r < batch; ++r) {
    if (q_len[r] == 0) continue;
    const int32_t q_lo = kv_len[r] - q_len[r];
    const int32_t t1 = (q_len[r] - 1) / T;
    for (int32_t g0 = 0; g0 <= t1; g0 += NT) {
      UnitDesc u;
      u.request = r;
      u.tile = g0;
      u.mask = 0;
      int32_t unit_end = -1, unit_first = INT32_MAX;
      for (int32_t t = 0; t < NT; ++t) {
        const int32_t tile = g0 + t;
        u.rows[t] = 0;
        u.nseg[t] = 0;
        if (tile > t1) continue;
        const int32_t first_valid = q_lo + tile * T;
        const int32_t tile_end = std::min(first_valid + T - 1, kv_len[r] - 1);
        u.mask |= 1 << t;
        u.rows[t] = (tile_end - first_valid + 1) * group;
        u.nseg[t] = tile_end / bip::kSplitLen + 1;
        unit_end = std::max(unit_end, tile_end);
        unit_first = std::min(unit_first, first_valid);
      }
      // With a sliding window the unit's earliest row sees keys from
      // first - window on; blocks and segments before that are skipped.
      const int32_t key_lo = opts.window_left > 0 ? std::max(0, unit_first - opts.window_left) : 0;
      u.blk_min = key_lo / bn;
      u.seg_lo = key_lo / bip::kSplitLen;
      u.seg_hi = unit_end / bip::kSplitLen;
      u.blocks = unit_end / bn + 1 - u.blk_min;
      for (int32_t h = 0; h < num_kv_heads; ++h) {
        u.kv_head = h;
        units.push_back(u);
      }
    }
  }
  auto split_need = [&](const UnitDesc& u) {
    size_t rows = 0;
    for (int t = 0; t < NT; ++t) rows += size_t(std::max(0, u.nseg[t] - u.seg_lo)) * u.rows[t];
    return rows * partial_row_bytes(head_dim);
  };

  // ---- split decision (numerically neutral; see the header)
  int num_sms = opts.num_sms > 0 ? opts.num_sms : query_sm_count();
  num_sms = std::min(num_sms, bip::kMaxCtas);
  // In-kernel waits count SM cycles (the global timer ticks too coarsely for
  // short limits); at any clock up to the peak, the cycle count takes at
  // least the requested time.  The clock query is slow, so it runs here once.
  uint64_t wait_limit_cycles;
  {
    const uint64_t ns = opts.wait_limit_ns, khz = query_clock_khz();
    wait_limit_cycles = ns > (~0ull / khz) ? ~0ull : std::max<uint64_t>(1, ns * khz / 1000000ull);
  }
  std::vector<char> split(units.size(), 0);
  size_t partial_bytes = 0;
  int64_t n_items = int64_t(units.size());
  if (opts.split_policy != BIP_SPLIT_NEVER) {
    std::vector<size_t> cand;
    for (size_t i = 0; i < units.size(); ++i)
      if (units[i].seg_hi > units[i].seg_lo) cand.push_back(i);
    std::stable_sort(cand.begin(), cand.end(),
                     [&](size_t a, size_t b) { return units[a].blocks > units[b].blocks; });
    // AUTO: split by segment when there are too few units to balance a
    // persistent grid (fewer than 8 per SM), or when a unit is longer than
    // half of one CTA's fair share of KV blocks (it would dominate the tail).
    int64_t total_blocks = 0;
    for (const UnitDesc& u : units) total_blocks += u.blocks;
    const int64_t fair_half = total_blocks / (2 * int64_t(num_sms));
    const bool few_units = int64_t(units.size()) < 8 * int64_t(num_sms);
    for (size_t i : cand) {
      if (opts.split_policy == BIP_SPLIT_AUTO && !few_units && units[i].blocks <= fair_half) break;
      const size_t need = split_need(units[i]);
      if (partial_bytes + need > opts.split_budget_bytes) continue;
      split[i] = 1;
      partial_bytes += need;
      n_items += units[i].seg_hi - units[i].seg_lo;
    }
  }

  // ---- items and merge units
  bip_plan_s* p = new (std::nothrow) bip_plan_s;
  if (!p) return BIP_ERR_OUT_OF_MEMORY;
  p->batch = batch;
  p->hq = num_qo_heads;
  p->hkv = num_kv_heads;
  p->d = head_dim;
  p->page_size = page_size;
  p->kv_dtype = kv_dtype;
  p->group = group;
  for (int32_t r = 0; r < batch; ++r)
    if (q_len[r] > 0) p->max_kv_q = std::max(p->max_kv_q, kv_len[r]);
  p->T = T;
  p->bn = bn;
  p->nt = NT;
  p->total_q = qo_indptr[batch];
  p->opts = opts;
  p->num_units = int32_t(units.size());
  for (int32_t r = 0; r < batch; ++r) {
    if (q_len[r] == 0) continue;
    bip::AppendRow row;
    row.tok0 = qo_indptr[r];
    row.q_len = q_len[r];
    row.pos0 = kv_len[r] - q_len[r];
    row.page_base = kv_indptr[r];
    p->reqs.push_back(row);
  }

  // Merge units and partial rows, in unit order; each split unit's first
  // partial row per slot.
  const int32_t bps = bip::kSplitLen / bn;
  int64_t part_rows = 0;
  std::vector<int64_t> ubase;  // [unit][slot], split units only
  for (size_t i = 0; i < units.size(); ++i) {
    if (!split[i]) continue;
    if (ubase.empty()) ubase.assign(units.size() * bip::kMaxTilesPerUnit, 0);
    const UnitDesc& u = units[i];
    const int32_t r = u.request;
    for (int t = 0; t < NT; ++t) {
      if (!(u.mask >> t & 1)) continue;
      MergeUnit m;
      std::memset(&m, 0, sizeof(m));
      m.q_tok0 = qo_indptr[r] - (kv_len[r] - q_len[r]);
      m.q_lo = kv_len[r] - q_len[r];
      m.tile = u.tile + t;
      m.part_base = int32_t(part_rows);
      m.rows = u.rows[t];
      m.kv_head = int16_t(u.kv_head);
      m.nseg = int16_t(u.nseg[t] - u.seg_lo);  // partials of segments seg_lo .. nseg - 1
      p->merges.push_back(m);
      ubase[i * bip::kMaxTilesPerUnit + t] = part_rows;
      part_rows += int64_t(u.nseg[t] - u.seg_lo) * u.rows[t];
    }
    p->num_split_units++;
  }

  // The items in construction order (each unit, or each segment of a split
  // unit), as compact entries; then their launch order: by (request, KV
  // head) group, longest first inside a group, ties in construction order.
  // Concurrent CTAs then stream the same group's pages, so each KV block
  // comes from HBM about once and from L2 for the other q tiles; the short
  // tiles of the last group fill the tail.
  struct Ent {
    uint32_t unit;
    int32_t seg;     // split: the segment; fold: -1
    int32_t blocks;  // KV blocks the item visits
  };
  std::vector<Ent> ents;
  ents.reserve(size_t(n_items));
  for (size_t i = 0; i < units.size(); ++i) {
    const UnitDesc& u = units[i];
    if (!split[i]) {
      ents.push_back({uint32_t(i), -1, u.blocks});
      continue;
    }
    const int32_t blk_end = u.blk_min + u.blocks;  // one past the last block
    for (int32_t sg = u.seg_lo; sg <= u.seg_hi; ++sg)
      ents.push_back({uint32_t(i), sg, std::min(blk_end, (sg + 1) * bps) - std::max(u.blk_min, sg * bps)});
  }
  std::stable_sort(ents.begin(), ents.end(), [&](const Ent& a, const Ent& b) {
    const UnitDesc& ua = units[a.unit];
    const UnitDesc& ub = units[b.unit];
    if (ua.request != ub.request) return ua.request < ub.request;
    if (ua.kv_head != ub.kv_head) return ua.kv_head < ub.kv_head;
    return a.blocks > b.blocks;
  });

  p->n_items = int32_t(ents.size());
  for (const Ent& e : ents)
    if (e.seg < 0 && units[e.unit].seg_hi > units[e.unit].seg_lo) p->need_scratch = true;
  p->partial_rows = part_rows;
  p->partial_bytes = size_t(part_rows) * partial_row_bytes(head_dim);
  p->grid = int32_t(std::min<int64_t>(int64_t(p->n_items), num_sms));
  p->wait_limit_cycles = wait_limit_cycles;
  p->sms = num_sms;
  p->scratch_bytes =
      p->need_scratch ? size_t(p->grid) * NT * bip::kTileRows * head_dim * sizeof(float) : 0;
  p->ws_bytes = layout_bytes(size_t(p->n_items), p->merges.size(), p->reqs.size(), p->partial_bytes,
                             p->scratch_bytes, key_bytes_for(p->total_q), &p->off_items, &p->off_merges, &p->off_reqs,
                             &p->off_partials, &p->off_scratch, &p->off_keys, &p->upload_bytes);

  // ---- host image of what each call uploads: header + items + merge units
  void* buf = nullptr;
  if (cudaHostAlloc(&buf, p->upload_bytes, cudaHostAllocMapped | cudaHostAllocPortable) == cudaSuccess) {
    p->pinned = true;
    void* dev = nullptr;
    if (cudaHostGetDevicePointer(&dev, buf, 0) == cudaSuccess && (reinterpret_cast<uintptr_t>(dev) & 15) == 0)
      p->upload_dev = dev;
    else
      cudaGetLastError();
  } else {
    cudaGetLastError();
    buf = std::malloc(p->upload_bytes);
    if (!buf) {
      delete p;
      return BIP_ERR_OUT_OF_MEMORY;
    }
  }
  p->upload = static_cast<uint8_t*>(buf);
  std::memset(p->upload, 0, bip::kHeaderBytes);

  // the items, in launch order, straight into the image
  WorkItem* out_items = reinterpret_cast<WorkItem*>(p->upload + p->off_items);
  p->item_desc.resize(size_t(p->n_items) * 8);
  for (size_t k = 0; k < ents.size(); ++k) {
    const Ent& e = ents[k];
    const UnitDesc& u = units[e.unit];
    const int32_t r = u.request;
    WorkItem w;
    std::memset(&w, 0, sizeof(w));
    w.kv_len = kv_len[r];
    w.page_base = kv_indptr[r];
    w.q_tok0 = qo_indptr[r] - (kv_len[r] - q_len[r]);
    w.q_lo = kv_len[r] - q_len[r];
    w.tile = u.tile;
    w.kv_head = int16_t(u.kv_head);
    w.flags = int16_t(u.mask * bip::kSlotPresent);
    for (int t = 0; t < NT; ++t) w.nseg[t] = int16_t(u.nseg[t]);
    w.blk_min = u.blk_min;
    int32_t* d = p->item_desc.data() + k * 8;
    if (e.seg < 0) {
      w.seg_lo = int16_t(u.seg_lo);
      w.seg_hi = int16_t(u.seg_hi);
      d[3] = u.seg_lo;
      d[4] = u.seg_hi;
      d[5] = 0;
    } else {
      w.seg_lo = w.seg_hi = int16_t(e.seg);
      w.flags = int16_t(w.flags | bip::kItemSplit);
      for (int t = 0; t < NT; ++t)
        w.part_base[t] =
            int32_t(ubase[size_t(e.unit) * bip::kMaxTilesPerUnit + t] + int64_t(e.seg - u.seg_lo) * u.rows[t]);
      d[3] = d[4] = e.seg;
      d[5] = 1;
    }
    d[0] = r;
    d[1] = u.kv_head;
    d[2] = u.tile;
    d[6] = e.blocks;
    d[7] = u.mask;
    p->kv_blocks += e.blocks;
    std::memcpy(out_items + k, &w, sizeof(w));
  }
  if (!p->merges.empty())
    std::memcpy(p->upload + p->off_merges, p->merges.data(), p->merges.size() * sizeof(MergeUnit));
  if (!p->reqs.empty())
    std::memcpy(p->upload + p->off_reqs, p->reqs.data(), p->reqs.size() * sizeof(bip::AppendRow));

  *plan_out = p;
  if (workspace_bytes) *workspace_bytes = p->ws_bytes;
  return BIP_OK;
}

extern "C" bip_status bip_plan_get_info(bip_plan_t p, bip_plan_info* info) {
  if (!p || !info) return BIP_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  info->batch = p->batch;
  info->total_q = p->total_q;
  info->num_qo_heads = p->hq;
  info->num_kv_heads = p->hkv;
  info->head_dim = p->d;
  info->page_size = p->page_size;
  info->kv_dtype = p->kv_dtype;
  info->gqa_group = p->group;
  info->tile_positions = p->T;
  info->kv_block = p->bn;
  info->split_len = bip::kSplitLen;
  info->num_units = p->num_units;
  info->num_items = p->n_items;
  info->num_split_units = p->num_split_units;
  info->grid = p->grid;
  info->tiles_per_unit = p->nt;
  info->partial_rows = p->partial_rows;
  info->kv_blocks = p->kv_blocks;
  info->workspace_bytes = p->ws_bytes;
  info->partial_bytes = p->partial_bytes;
  info->scratch_bytes = p->scratch_bytes;
  info->upload_bytes = p->upload_bytes;
  return BIP_OK;
}

extern "C" bip_status bip_plan_get_items(bip_plan_t p, int32_t* items, int32_t capacity, int32_t* count) {
  if (!p || capacity < 0 || (capacity > 0 && !items)) return BIP_ERR_INVALID_ARG;
  const int32_t n = p->n_items;
  if (count) *count = n;
  const int32_t m = std::min(n, capacity);
  if (m > 0) std::memcpy(items, p->item_desc.data(), size_t(m) * 8 * sizeof(int32_t));
  return BIP_OK;
}

extern "C" bip_status bip_plan_destroy(bip_plan_t p) {
  if (!p) return BIP_ERR_INVALID_ARG;
  for (auto& u : p->uses) {  // eager work that reads the host image has completed
    cudaEventSynchronize(u.second);
    cudaEventDestroy(u.second);
  }
  p->uses.clear();
  if (p->upload) {
    if (p->pinned)
      cudaFreeHost(p->upload);
    else
      std::free(p->upload);
  }
  delete p;
  return BIP_OK;
}

// ---------------------------------------------------------------- launch

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The pools as plain pointers: page sizes below 8 gather token rows with
// cp.async instead of TMA boxes.
void set_pools(bip::AttnParams& ap, const void* k_pages, const void* v_pages, int64_t page_stride_bytes,
               int32_t slot_bytes) {
  ap.k_pool = static_cast<const uint8_t*>(k_pages);
  ap.v_pool = static_cast<const uint8_t*>(v_pages);
  ap.page_stride_bytes = page_stride_bytes;
  ap.slot_bytes = slot_bytes;
}

}  // namespace

// Record that `stream` has work reading the plan's host image (skipped while
// the stream is being captured: a graph keeps reading the image at every
// replay, so the plan must outlive it).  Streams beyond the first kMaxUses
// reuse the oldest entry after waiting for it.
static void note_use(bip_plan_s* p, cudaStream_t stream) {
  constexpr size_t kMaxUses = 32;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    cudaGetLastError();
    return;
  }
  if (cs != cudaStreamCaptureStatusNone) return;
  std::lock_guard<std::mutex> lk(p->use_mu);
  cudaEvent_t ev = nullptr;
  for (auto& u : p->uses)
    if (u.first == stream) ev = u.second;
  if (!ev) {
    if (p->uses.size() >= kMaxUses) {
      cudaEventSynchronize(p->uses.front().second);
      cudaEventDestroy(p->uses.front().second);
      p->uses.erase(p->uses.begin());
    }
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    p->uses.emplace_back(stream, ev);
  }
  if (cudaEventRecord(ev, stream) != cudaSuccess) cudaGetLastError();
}

// The first `bytes` of the plan's host image into the workspace, on `stream`:
// by the upload kernel when the pinned image is mapped into the device's
// address space, else by one copy-engine copy.
static cudaError_t upload(const bip_plan_s* p, uint8_t* ws, size_t bytes, cudaStream_t stream) {
  if (p->upload_dev) return bip::launch_upload(p->upload_dev, ws, bytes, stream);
  return cudaMemcpyAsync(ws, p->upload, bytes, cudaMemcpyHostToDevice, stream);
}

// TMA descriptors of one launch.  q: [rows, Hq, d] as dims (d, Hq, rows); box
// (64, group, T) = one tile chunk.  pages: [pages, slot, Hkv, d] as dims (d,
// Hkv, slot, page).  bf16: box (64, 1, page_size, 1), one 128-byte-swizzled
// chunk of a page.  FP8: box (d, 1, page_size, 1), a whole page row-major,
// unswizzled (the dequant warps lay out the bf16 operand).
static bool encode_maps(int32_t d, int32_t hq, int32_t hkv, int32_t group, int32_t T, int32_t page_size,
                        bool fp8, const void* q, int64_t q_rows, const void* k_pages, const void* v_pages,
                        int64_t num_pages, int64_t page_stride_elems, CUtensorMap* tm_q, CUtensorMap* tm_k,
                        CUtensorMap* tm_v) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  {
    cuuint64_t dims[3] = {cuuint64_t(d), cuuint64_t(hq), cuuint64_t(q_rows)};
    cuuint64_t strides[2] = {cuuint64_t(d) * 2, cuuint64_t(hq) * d * 2};
    cuuint32_t box[3] = {64, cuuint32_t(group), cuuint32_t(T)};
    cuuint32_t es[3] = {1, 1, 1};
    if (encode(tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  const int64_t elem = fp8 ? 1 : 2;
  for (int which = 0; which < 2; ++which) {
    const void* base = which == 0 ? k_pages : v_pages;
    cuuint64_t dims[4] = {cuuint64_t(d), cuuint64_t(hkv), cuuint64_t(page_size), cuuint64_t(num_pages)};
    cuuint64_t strides[3] = {cuuint64_t(d) * elem, cuuint64_t(hkv) * d * elem, cuuint64_t(page_stride_elems) * elem};
    cuuint32_t box[4] = {fp8 ? cuuint32_t(d) : 64u, 1, cuuint32_t(page_size), 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (encode(which == 0 ? tm_k : tm_v, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
               const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return false;
  }
  return true;
}

// bip_prefill, and bip_prefill_masked with a mask (null: none).
static bip_status prefill(bip_plan_t p, const void* q, int64_t num_q_rows, const void* k_pages, const void* v_pages,
                          int64_t num_pages, int64_t page_stride_elems, const int32_t* kv_indices,
                          const uint32_t* mask, int64_t mask_row_words, float k_scale, float v_scale, void* out,
                          float* lse, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!p) return BIP_ERR_INVALID_ARG;
  if (num_q_rows != p->total_q) return BIP_ERR_INVALID_ARG;
  if (mask && mask_row_words < (int64_t(p->max_kv_q) + 31) / 32) return BIP_ERR_INVALID_ARG;
  if (p->n_items == 0) return BIP_OK;  // nothing to compute (all q_len = 0)
  if (!q || !k_pages || !v_pages || !kv_indices || !out || !lse || !workspace) return BIP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return BIP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return BIP_ERR_INVALID_ARG;
  if (workspace_bytes < p->ws_bytes) return BIP_ERR_WORKSPACE_TOO_SMALL;
  const int64_t page_elems = int64_t(p->page_size) * p->hkv * p->d;
  const int64_t elem = p->kv_dtype == BIP_KV_BF16 ? 2 : 1;
  if (num_pages <= 0 || num_pages > INT32_MAX || page_stride_elems < page_elems ||
      (page_stride_elems * elem) % 16 != 0)
    return BIP_ERR_INVALID_ARG;
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return BIP_ERR_INVALID_ARG;
  if (p->page_size < 8 && page_stride_elems * elem > INT32_MAX) return BIP_ERR_UNSUPPORTED;  // row gather: 32-bit

  const bool fp8 = p->kv_dtype == BIP_KV_FP8_E4M3;
  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_maps(p->d, p->hq, p->hkv, p->group, p->T, p->page_size, fp8, q, num_q_rows, k_pages, v_pages,
                   num_pages, page_stride_elems, &tm_q, &tm_k, &tm_v))
    return BIP_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (upload(p, ws, p->upload_bytes, stream) != cudaSuccess) return BIP_ERR_CUDA;

  bip::AttnParams ap;
  ap.items = reinterpret_cast<const WorkItem*>(ws + p->off_items);
  ap.n_items = p->n_items;
  ap.n_items_dev = nullptr;
  ap.num_qo_heads = p->hq;
  ap.group = p->group;
  ap.tile_pos = p->T;
  ap.page_size = p->page_size;
  ap.num_pages = int32_t(num_pages);
  ap.kv_indices = kv_indices;
  ap.out = static_cast<uint16_t*>(out);
  ap.lse = lse;
  ap.partials = reinterpret_cast<float*>(ws + p->off_partials);
  ap.scratch = reinterpret_cast<float*>(ws + p->off_scratch);
  ap.header = reinterpret_cast<bip::WsHeader*>(ws);
  ap.scale_log2 = float(1.4426950408889634 * double(k_scale) / std::sqrt(double(p->d)));
  ap.v_scale = v_scale;
  ap.wait_limit_cycles = p->wait_limit_cycles;
  ap.window_left = p->opts.window_left;
  set_pools(ap, k_pages, v_pages, page_stride_elems * elem, p->hkv * p->d * int32_t(elem));
  ap.mask = mask;
  ap.mask_row_words = mask ? mask_row_words : 0;
  if (mask) {
    // start every item at the first block one of its rows sees
    bip::MaskSkipParams sp;
    sp.items = reinterpret_cast<WorkItem*>(ws + p->off_items);
    sp.first_key = reinterpret_cast<int32_t*>(ws + p->off_keys);
    sp.n_items = p->n_items;
    sp.n_items_dev = nullptr;
    sp.mask = mask;
    sp.mask_row_words = mask_row_words;
    sp.group = p->group;
    sp.tile_pos = p->T;
    sp.kv_block = bip::kv_block_for(p->d);
    sp.tiles_per_unit = p->nt;
    sp.window_left = p->opts.window_left;
    sp.num_kv_heads = p->hkv;
    if (bip::launch_mask_skip(sp, sp.n_items, stream) != cudaSuccess)
      return BIP_ERR_CUDA;
  }
  const cudaError_t le = mask ? bip::launch_attention_masked(p->d, p->nt, fp8, tm_q, tm_k, tm_v, ap, p->grid, stream)
                              : bip::launch_attention(p->d, p->nt, fp8, tm_q, tm_k, tm_v, ap, p->grid, stream);
  if (le != cudaSuccess) return BIP_ERR_CUDA;

  if (!p->merges.empty()) {
    bip::MergeParams mp;
    mp.units = reinterpret_cast<const MergeUnit*>(ws + p->off_merges);
    mp.n_units = int32_t(p->merges.size());
    mp.n_units_dev = nullptr;
    mp.num_qo_heads = p->hq;
    mp.group = p->group;
    mp.tile_pos = p->T;
    mp.partials = ap.partials;
    mp.out = ap.out;
    mp.lse = lse;
    mp.v_scale = v_scale;
    if (bip::launch_merge(p->d, mp, stream) != cudaSuccess) return BIP_ERR_CUDA;
  }
  note_use(p, stream);
  return BIP_OK;
}

extern "C" bip_status bip_prefill(bip_plan_t p, const void* q, int64_t num_q_rows, const void* k_pages,
                                  const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                  const int32_t* kv_indices, float k_scale, float v_scale, void* out, float* lse,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return prefill(p, q, num_q_rows, k_pages, v_pages, num_pages, page_stride_elems, kv_indices, nullptr, 0, k_scale,
                 v_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" bip_status bip_prefill_masked(bip_plan_t p, const void* q, int64_t num_q_rows, const void* k_pages,
                                         const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                         const int32_t* kv_indices, const uint32_t* mask, int64_t mask_row_words,
                                         float k_scale, float v_scale, void* out, float* lse, void* workspace,
                                         size_t workspace_bytes, cudaStream_t stream) {
  if (!mask || (reinterpret_cast<uintptr_t>(mask) & 3) != 0) return BIP_ERR_INVALID_ARG;
  return prefill(p, q, num_q_rows, k_pages, v_pages, num_pages, page_stride_elems, kv_indices, mask, mask_row_words,
                 k_scale, v_scale, out, lse, workspace, workspace_bytes, stream);
}

extern "C" bip_status bip_append_kv(bip_plan_t p, const void* k_new, const void* v_new, int64_t num_new_rows,
                                    void* k_pages, void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                    const int32_t* kv_indices, float k_scale, float v_scale, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  if (!p) return BIP_ERR_INVALID_ARG;
  if (num_new_rows != p->total_q) return BIP_ERR_INVALID_ARG;
  if (p->total_q == 0) return BIP_OK;
  if (!k_new || !v_new || !k_pages || !v_pages || !kv_indices || !workspace) return BIP_ERR_INVALID_ARG;
  if (num_pages <= 0 || num_pages > INT32_MAX || page_stride_elems <= 0) return BIP_ERR_INVALID_ARG;
  const bool fp8 = p->kv_dtype == BIP_KV_FP8_E4M3;
  const int64_t elem = fp8 ? 1 : 2;
  if (page_stride_elems < int64_t(p->page_size) * p->hkv * p->d) return BIP_ERR_INVALID_ARG;
  if ((page_stride_elems * elem) % 16 != 0) return BIP_ERR_INVALID_ARG;
  auto misaligned = [](const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) != 0; };
  if (misaligned(k_new) || misaligned(v_new) || misaligned(k_pages) || misaligned(v_pages) || misaligned(workspace))
    return BIP_ERR_INVALID_ARG;
  if (fp8) {
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || !std::isfinite(k_scale) || !std::isfinite(v_scale))
      return BIP_ERR_INVALID_ARG;
  } else if (k_scale != 1.f || v_scale != 1.f) {
    return BIP_ERR_INVALID_ARG;  // bf16 pages store the rows unchanged
  }
  if (workspace_bytes < p->off_items) return BIP_ERR_WORKSPACE_TOO_SMALL;

  // header (status word cleared) and request rows only
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (upload(p, ws, p->off_items, stream) != cudaSuccess) return BIP_ERR_CUDA;
  bip::AppendParams ap;
  ap.rows = reinterpret_cast<const bip::AppendRow*>(ws + p->off_reqs);
  ap.n_rows = int32_t(p->reqs.size());
  ap.total_q = p->total_q;
  ap.num_kv_heads = p->hkv;
  ap.page_size = p->page_size;
  ap.num_pages = int32_t(num_pages);
  ap.page_stride = page_stride_elems;
  ap.kv_indices = kv_indices;
  ap.k_new = static_cast<const uint16_t*>(k_new);
  ap.v_new = static_cast<const uint16_t*>(v_new);
  ap.k_pages = k_pages;
  ap.v_pages = v_pages;
  ap.k_scale = k_scale;
  ap.v_scale = v_scale;
  ap.header = reinterpret_cast<bip::WsHeader*>(ws);
  if (bip::launch_append(p->d, fp8, ap, p->sms, stream) != cudaSuccess) return BIP_ERR_CUDA;
  note_use(p, stream);
  return BIP_OK;
}

// ------------------------------------------------------------ graph plans

struct bip_graph_plan_s {
  int32_t max_batch = 0, max_total_q = 0, hq = 0, hkv = 0, d = 0, page_size = 0, group = 0, T = 0, nt = 1;
  int32_t grid = 0, capacity = 0, merge_capacity = 0;
  int64_t partial_capacity = 0;  // partial rows
  bip_kv_dtype kv_dtype = BIP_KV_BF16;
  uint64_t wait_limit_cycles = 0;
  int32_t window_left = 0;
  size_t off_items = 0, off_merges = 0, off_partials = 0, off_scratch = 0, off_keys = 0, ws_bytes = 0;
};

// Split budget of a graph plan when the caller gives no options: batches
// with few units split their segments within it (short extends behind long
// prefixes need a few MB).
constexpr size_t kDefaultGraphSplitBudget = size_t(64) << 20;
// Items a graph plan holds beyond one per unit, for split segments.
constexpr int64_t kGraphSplitItems = 65536;

extern "C" bip_status bip_graph_plan(bip_graph_plan_t* plan_out, int32_t max_batch, int32_t max_total_q,
                                     int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                     bip_kv_dtype kv_dtype, const bip_plan_options* opts_in,
                                     size_t* workspace_bytes) {
  if (!plan_out) return BIP_ERR_INVALID_ARG;
  *plan_out = nullptr;
  if (max_batch < 0 || max_total_q < 0) return BIP_ERR_INVALID_ARG;
  bip_status st = check_heads(num_qo_heads, num_kv_heads, head_dim);
  if (st != BIP_OK) return st;
  if (kv_dtype != BIP_KV_BF16 && kv_dtype != BIP_KV_FP8_E4M3) return BIP_ERR_INVALID_ARG;
  const int32_t bn = bip::kv_block_for(head_dim);
  if (page_size <= 0) return BIP_ERR_INVALID_ARG;
  if ((page_size & (page_size - 1)) != 0 || page_size > bn) return BIP_ERR_UNSUPPORTED;
  bip_plan_options opts;
  opts.split_policy = BIP_SPLIT_AUTO;
  opts.split_budget_bytes = kDefaultGraphSplitBudget;
  opts.num_sms = 0;
  opts.wait_limit_ns = 0;
  opts.tiles_per_unit = 0;
  opts.window_left = 0;
  if (opts_in) opts = *opts_in;
  if (opts.window_left < 0) return BIP_ERR_INVALID_ARG;
  if (opts.split_policy == BIP_SPLIT_ALWAYS) return BIP_ERR_UNSUPPORTED;  // the batch decides, on the device
  if (opts.split_policy != BIP_SPLIT_AUTO && opts.split_policy != BIP_SPLIT_NEVER) return BIP_ERR_INVALID_ARG;
  if (opts.num_sms < 0) return BIP_ERR_INVALID_ARG;
  if (opts.tiles_per_unit < 0 || opts.tiles_per_unit > bip::max_tiles_per_unit_for(head_dim))
    return BIP_ERR_INVALID_ARG;
  if (page_size < 8 && opts.tiles_per_unit == 2) return BIP_ERR_UNSUPPORTED;
  if (opts.wait_limit_ns == 0) opts.wait_limit_ns = bip::kDefaultWaitNs;

  bip_graph_plan_s* p = new (std::nothrow) bip_graph_plan_s;
  if (!p) return BIP_ERR_OUT_OF_MEMORY;
  p->max_batch = max_batch;
  p->max_total_q = max_total_q;
  p->window_left = opts.window_left;
  p->hq = num_qo_heads;
  p->hkv = num_kv_heads;
  p->d = head_dim;
  p->page_size = page_size;
  p->kv_dtype = kv_dtype;
  p->group = num_qo_heads / num_kv_heads;
  p->T = bip::kTileRows / p->group;
  // No batch statistics at capture time: the host planner's rule (two
  // tiles per CTA when requests average at least two q tiles) applied to
  // the bucket's capacities, where the variant exists (numerically neutral,
  // like every plan choice).
  p->nt = opts.tiles_per_unit ? opts.tiles_per_unit
                              : (bip::max_tiles_per_unit_for(head_dim) >= 2 && page_size >= 8 &&
                                         int64_t(max_total_q) >= 2 * int64_t(p->T) * max_batch
                                     ? 2 : 1);
  int num_sms = opts.num_sms > 0 ? opts.num_sms : query_sm_count();
  p->grid = std::min(num_sms, bip::kMaxCtas);
  {
    const uint64_t ns = opts.wait_limit_ns, khz = query_clock_khz();
    p->wait_limit_cycles = ns > (~0ull / khz) ? ~0ull : std::max<uint64_t>(1, ns * khz / 1000000ull);
  }
  // A request with q_len rows has ceil(q_len / T) tiles (the bound allows one more).
  const int64_t cap = int64_t(num_kv_heads) * ((int64_t(max_total_q) + p->T - 1) / p->T + 2 * int64_t(max_batch));
  if (cap > INT32_MAX) {
    delete p;
    return BIP_ERR_UNSUPPORTED;
  }
  // Split segments (policy AUTO): up to kGraphSplitItems more items, one
  // merge unit per q tile of a unit, and partial rows within the budget.
  const bool may_split = opts.split_policy == BIP_SPLIT_AUTO && opts.split_budget_bytes >= partial_row_bytes(head_dim);
  const int64_t item_cap = cap + (may_split ? kGraphSplitItems : 0);
  const int64_t merge_cap = may_split ? cap * p->nt : 0;
  const int64_t part_cap =
      may_split ? std::min<int64_t>(int64_t(opts.split_budget_bytes / partial_row_bytes(head_dim)), INT32_MAX) : 0;
  if (item_cap > INT32_MAX || merge_cap > INT32_MAX) {
    delete p;
    return BIP_ERR_UNSUPPORTED;
  }
  p->capacity = int32_t(item_cap);
  p->merge_capacity = int32_t(merge_cap);
  p->partial_capacity = part_cap;
  p->off_items = bip::kHeaderBytes;
  p->off_merges = align_up(p->off_items + size_t(item_cap) * sizeof(WorkItem), 256);
  p->off_partials = align_up(p->off_merges + size_t(merge_cap) * sizeof(MergeUnit), 256);
  p->off_scratch = align_up(p->off_partials + size_t(part_cap) * partial_row_bytes(head_dim), 256);
  p->off_keys = align_up(p->off_scratch + size_t(p->grid) * p->nt * bip::kTileRows * head_dim * sizeof(float), 256);
  p->ws_bytes = align_up(p->off_keys + key_bytes_for(max_total_q), 256);
  *plan_out = p;
  if (workspace_bytes) *workspace_bytes = p->ws_bytes;
  return BIP_OK;
}

extern "C" bip_status bip_graph_plan_destroy(bip_graph_plan_t p) {
  delete p;
  return BIP_OK;
}

// bip_prefill_graph, and bip_prefill_graph_masked with a mask (null: none).
static bip_status prefill_graph(bip_graph_plan_t p, int32_t batch, const int32_t* qo_indptr,
                                const int32_t* kv_indptr, const int32_t* kv_last_page_len, const void* q,
                                const void* k_pages, const void* v_pages, int64_t num_pages, int64_t page_stride_elems,
                                const int32_t* kv_indices, const uint32_t* mask, int64_t mask_row_words,
                                float k_scale, float v_scale, void* out, float* lse, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream) {
  if (!p) return BIP_ERR_INVALID_ARG;
  if (batch < 0 || batch > p->max_batch) return BIP_ERR_INVALID_ARG;
  if (!qo_indptr || !kv_indptr || !kv_last_page_len || !q || !k_pages || !v_pages || !kv_indices || !out || !lse ||
      !workspace)
    return BIP_ERR_INVALID_ARG;
  if (mask && mask_row_words <= 0) return BIP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(out)) return BIP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return BIP_ERR_INVALID_ARG;
  if (workspace_bytes < p->ws_bytes) return BIP_ERR_WORKSPACE_TOO_SMALL;
  const int64_t page_elems = int64_t(p->page_size) * p->hkv * p->d;
  const bool fp8 = p->kv_dtype == BIP_KV_FP8_E4M3;
  const int64_t elem = fp8 ? 1 : 2;
  if (num_pages <= 0 || num_pages > INT32_MAX || page_stride_elems < page_elems ||
      (page_stride_elems * elem) % 16 != 0)
    return BIP_ERR_INVALID_ARG;
  if (!std::isfinite(k_scale) || !std::isfinite(v_scale)) return BIP_ERR_INVALID_ARG;
  if (p->page_size < 8 && page_stride_elems * elem > INT32_MAX) return BIP_ERR_UNSUPPORTED;  // row gather: 32-bit
  if (p->max_total_q == 0) return BIP_OK;  // no buffer rows: nothing can ever run

  CUtensorMap tm_q, tm_k, tm_v;
  if (!encode_maps(p->d, p->hq, p->hkv, p->group, p->T, p->page_size, fp8, q, p->max_total_q, k_pages, v_pages,
                   num_pages, page_stride_elems, &tm_q, &tm_k, &tm_v))
    return BIP_ERR_CUDA;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  bip::WsHeader* header = reinterpret_cast<bip::WsHeader*>(ws);
  bip::DevPlanParams dp;
  dp.batch = batch;
  dp.max_total_q = p->max_total_q;
  dp.page_size = p->page_size;
  dp.group = p->group;
  dp.tile_pos = p->T;
  dp.tiles_per_unit = p->nt;
  dp.num_kv_heads = p->hkv;
  dp.kv_block = bip::kv_block_for(p->d);
  dp.capacity = p->capacity;
  dp.window_left = p->window_left;
  dp.grid = p->grid;
  dp.merge_capacity = p->merge_capacity;
  dp.partial_capacity = p->partial_capacity;
  dp.mask_row_words = mask ? mask_row_words : 0;
  dp.qo_indptr = qo_indptr;
  dp.kv_indptr = kv_indptr;
  dp.kv_last_page_len = kv_last_page_len;
  dp.items = reinterpret_cast<WorkItem*>(ws + p->off_items);
  dp.merges = reinterpret_cast<MergeUnit*>(ws + p->off_merges);
  dp.header = header;
  if (bip::launch_device_plan(dp, stream) != cudaSuccess) return BIP_ERR_CUDA;

  bip::AttnParams ap;
  ap.items = dp.items;
  ap.n_items = p->capacity;
  ap.n_items_dev = &header->n_items;
  ap.num_qo_heads = p->hq;
  ap.group = p->group;
  ap.tile_pos = p->T;
  ap.page_size = p->page_size;
  ap.num_pages = int32_t(num_pages);
  ap.kv_indices = kv_indices;
  ap.out = static_cast<uint16_t*>(out);
  ap.lse = lse;
  ap.partials = reinterpret_cast<float*>(ws + p->off_partials);
  ap.scratch = reinterpret_cast<float*>(ws + p->off_scratch);
  ap.header = header;
  ap.scale_log2 = float(1.4426950408889634 * double(k_scale) / std::sqrt(double(p->d)));
  ap.v_scale = v_scale;
  ap.wait_limit_cycles = p->wait_limit_cycles;
  ap.window_left = p->window_left;
  ap.mask = mask;
  ap.mask_row_words = mask ? mask_row_words : 0;
  set_pools(ap, k_pages, v_pages, page_stride_elems * elem, p->hkv * p->d * int32_t(elem));
  if (mask) {
    // start every item the planner wrote at the first block one of its rows sees
    bip::MaskSkipParams sp;
    sp.items = dp.items;
    sp.first_key = reinterpret_cast<int32_t*>(ws + p->off_keys);
    sp.n_items = p->capacity;
    sp.n_items_dev = &header->n_items;
    sp.mask = mask;
    sp.mask_row_words = mask_row_words;
    sp.group = p->group;
    sp.tile_pos = p->T;
    sp.kv_block = bip::kv_block_for(p->d);
    sp.tiles_per_unit = p->nt;
    sp.window_left = p->window_left;
    sp.num_kv_heads = p->hkv;
    if (bip::launch_mask_skip(sp, p->capacity, stream) != cudaSuccess)
      return BIP_ERR_CUDA;
  }
  const cudaError_t le = mask ? bip::launch_attention_masked(p->d, p->nt, fp8, tm_q, tm_k, tm_v, ap, p->grid, stream)
                              : bip::launch_attention(p->d, p->nt, fp8, tm_q, tm_k, tm_v, ap, p->grid, stream);
  if (le != cudaSuccess) return BIP_ERR_CUDA;
  if (p->merge_capacity > 0) {
    // the merge units the planner wrote (none when the batch folded)
    bip::MergeParams mp;
    mp.units = dp.merges;
    mp.n_units = std::min(p->merge_capacity, 4 * p->grid);
    mp.n_units_dev = &header->n_merges;
    mp.num_qo_heads = p->hq;
    mp.group = p->group;
    mp.tile_pos = p->T;
    mp.partials = ap.partials;
    mp.out = ap.out;
    mp.lse = lse;
    mp.v_scale = v_scale;
    if (bip::launch_merge(p->d, mp, stream) != cudaSuccess) return BIP_ERR_CUDA;
  }
  return BIP_OK;
}

extern "C" bip_status bip_prefill_graph(bip_graph_plan_t p, int32_t batch, const int32_t* qo_indptr,
                                        const int32_t* kv_indptr, const int32_t* kv_last_page_len, const void* q,
                                        const void* k_pages, const void* v_pages, int64_t num_pages,
                                        int64_t page_stride_elems, const int32_t* kv_indices, float k_scale,
                                        float v_scale, void* out, float* lse, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  return prefill_graph(p, batch, qo_indptr, kv_indptr, kv_last_page_len, q, k_pages, v_pages, num_pages,
                       page_stride_elems, kv_indices, nullptr, 0, k_scale, v_scale, out, lse, workspace,
                       workspace_bytes, stream);
}

extern "C" bip_status bip_prefill_graph_masked(bip_graph_plan_t p, int32_t batch, const int32_t* qo_indptr,
                                               const int32_t* kv_indptr, const int32_t* kv_last_page_len,
                                               const void* q, const void* k_pages, const void* v_pages,
                                               int64_t num_pages, int64_t page_stride_elems,
                                               const int32_t* kv_indices, const uint32_t* mask,
                                               int64_t mask_row_words, float k_scale, float v_scale, void* out,
                                               float* lse, void* workspace, size_t workspace_bytes,
                                               cudaStream_t stream) {
  if (!mask || (reinterpret_cast<uintptr_t>(mask) & 3) != 0) return BIP_ERR_INVALID_ARG;
  return prefill_graph(p, batch, qo_indptr, kv_indptr, kv_last_page_len, q, k_pages, v_pages, num_pages,
                       page_stride_elems, kv_indices, mask, mask_row_words, k_scale, v_scale, out, lse, workspace,
                       workspace_bytes, stream);
}

extern "C" bip_status bip_read_device_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return BIP_ERR_INVALID_ARG;
  bip::WsHeader h;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return BIP_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return BIP_ERR_CUDA;
  if (h.status != 0) return static_cast<bip_status>(h.status);
  if (h.bad_pages != 0) return BIP_ERR_BAD_PAGE_INDEX;
  return BIP_OK;
}
