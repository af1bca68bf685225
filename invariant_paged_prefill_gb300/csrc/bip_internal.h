// Contract between the host planner (bip_host.cpp) and the kernels
// (attention, merge, KV append, device planner): work-list records, workspace header and
// launch parameters.  Host and device code include it.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda.h>
#include <cuda_runtime_api.h>

namespace bip {

constexpr int kTileRows = 128;      // M of every tcgen05 MMA: packed (position, head) rows
constexpr int kSplitLen = 4096;     // keys per segment (absolute positions)
constexpr int kMaxCtas = 256;       // cap on the persistent grid (sizes the fold scratch)
constexpr int kHeaderBytes = 256;   // workspace header
constexpr uint64_t kDefaultWaitNs = 4000000000ull;

constexpr int kv_block_for(int head_dim) { return head_dim == 128 ? 128 : 64; }

// Workspace header, written by the host upload, updated by kernels.
struct WsHeader {
  uint32_t status;          // 0 = ok, else a bip_status code
  uint32_t where;           // which wait expired (diagnostics)
  uint32_t bad_pages;       // count of out-of-range page ids seen
  uint32_t n_items;         // work items, when the device planner wrote them
  uint32_t n_merges;        // merge units, when the device planner wrote them
  uint32_t reserved[59];
};
static_assert(sizeof(WsHeader) == kHeaderBytes, "header size");

// One attention work item: a unit (request x KV head x up to two q tiles
// that share the same keys) over a range of its segments.  48 bytes.
struct WorkItem {
  int32_t kv_len;
  int32_t page_base;   // first entry of the request in kv_indices
  int32_t q_tok0;      // q row of sequence position 0 (may be negative)
  int32_t q_lo;        // first position that has a q row (kv_len - q_len)
  int32_t tile;        // tile of slot 0; slot t covers positions q_lo + (tile+t)*T .. +T-1
  int16_t kv_head;
  int16_t seg_lo;      // inclusive segment range
  int16_t seg_hi;
  int16_t flags;       // kItemSplit | tile-present bits (kSlotPresent << t)
  int32_t part_base[2];  // split: partial row of slot t's first valid row in this segment
  int16_t nseg[2];       // segments that hold slot t's rows (tile_end / 4096 + 1)
  int32_t blk_min;       // first KV block any row of the item sees (0 without a sliding window)
  int32_t pad;
};
static_assert(sizeof(WorkItem) == 48, "work item size");
constexpr int16_t kItemSplit = 1;
constexpr int16_t kSlotPresent = 1 << 8;
constexpr int kMaxTilesPerUnit = 2;

// Most q tiles a CTA carries at once: two for head_dim 128 (TMEM holds S and
// O of both), one for head_dim 256 (O alone takes 256 of the 512 columns).
constexpr int max_tiles_per_unit_for(int head_dim) { return head_dim == 128 ? 2 : 1; }

// One merge unit: the partials of a split unit, folded in segment order.
struct MergeUnit {
  int32_t q_tok0;
  int32_t q_lo;
  int32_t tile;
  int32_t part_base;   // partial row of (segment 0, first valid row)
  int32_t rows;        // valid rows of the tile; segment s starts at part_base + s*rows
  int16_t kv_head;
  int16_t nseg;
  int32_t pad[2];
};
static_assert(sizeof(MergeUnit) == 32, "merge unit size");

struct AttnParams {
  const WorkItem* items;
  int32_t n_items;
  const uint32_t* n_items_dev;  // if set, the item count is read here (device-planned launches)
  int32_t num_qo_heads;
  int32_t group;        // q heads per kv head
  int32_t tile_pos;     // T = floor(128 / group)
  int32_t page_size;
  int32_t num_pages;
  const int32_t* kv_indices;
  uint16_t* out;        // bf16 bits
  float* lse;
  float* partials;      // [rows][head_dim + 4]: m, l, 0, 0, o[head_dim]
  float* scratch;       // [grid][tiles per CTA][head_dim / 4][128] float4: fold state, row-fastest
  WsHeader* header;
  float scale_log2;     // log2(e) * k_scale / sqrt(head_dim)
  float v_scale;
  uint64_t wait_limit_cycles;  // wait bound in SM clock cycles (the limit in ns at the peak clock)
  int32_t window_left;         // > 0: a row at position p sees keys p - window_left .. p only
  // Pools as plain pointers, for page sizes below 8 (rows gathered with
  // cp.async instead of TMA boxes).
  const uint8_t* k_pool;
  const uint8_t* v_pool;
  int64_t page_stride_bytes;
  int32_t slot_bytes;          // one token slot: num_kv_heads * head_dim * element size
  // Custom mask (null: none): q row r's bits start at mask + r * mask_row_words;
  // bit j % 32 of word j / 32 set = key j of the request visible to the row
  // (within the causal and window rule).
  const uint32_t* mask;
  int64_t mask_row_words;
};

struct MergeParams {
  const MergeUnit* units;
  int32_t n_units;                 // merge CTAs launched (the count, or a capacity)
  const uint32_t* n_units_dev;     // if set, the unit count is read here (device-planned launches)
  int32_t num_qo_heads;
  int32_t group;
  int32_t tile_pos;
  const float* partials;
  uint16_t* out;
  float* lse;
  float v_scale;
};

// One request with new rows, for the KV append: its rows of k_new / v_new
// are [tok0, tok0 + q_len) and go to positions pos0 .. pos0 + q_len - 1
// (pos0 = kv_len - q_len) of the page table starting at kv_indices[page_base].
// Only requests with q_len > 0, in row order.  16 bytes.
struct AppendRow {
  int32_t tok0;
  int32_t q_len;
  int32_t pos0;
  int32_t page_base;
};
static_assert(sizeof(AppendRow) == 16, "append row size");

struct AppendParams {
  const AppendRow* rows;
  int32_t n_rows;           // entries of rows
  int32_t total_q;          // new rows
  int32_t num_kv_heads;
  int32_t page_size;
  int32_t num_pages;
  int64_t page_stride;      // elements (bf16) or bytes (E4M3) between pages
  const int32_t* kv_indices;
  const uint16_t* k_new;    // bf16 [total_q, num_kv_heads, head_dim]
  const uint16_t* v_new;
  void* k_pages;
  void* v_pages;
  float k_scale, v_scale;   // E4M3 pages store e4m3(x / scale)
  WsHeader* header;
};

// Device-side planner for graph-replayable launches: reads the batch's
// indptr arrays on the device and writes the work list and its count into
// the workspace header.  A batch of few units (fewer than 8 per CTA) has
// every multi-segment unit split by segment, with partials and merge units
// (count in the header), when they fit the capacities; otherwise every unit
// folds its segments in one CTA.  Validation failures set the header status
// and leave zero items.
// Custom masks: the first KV block any row of each work item sees
// (bip_mask_skip.cu), written into the items before the attention launch.
struct MaskSkipParams {
  WorkItem* items;
  int32_t* first_key;  // [q rows]: each row's first visible key (INT32_MAX: none), in the workspace
  int32_t n_items;
  const uint32_t* n_items_dev;  // if set, the item count is read here (device-planned launches)
  const uint32_t* mask;
  int64_t mask_row_words;
  int32_t group;
  int32_t tile_pos;
  int32_t kv_block;
  int32_t tiles_per_unit;
  int32_t window_left;
  int32_t num_kv_heads;
};

struct DevPlanParams {
  int32_t batch;
  int32_t max_total_q;   // q rows the buffers hold
  int32_t page_size;
  int32_t group;         // q heads per kv head
  int32_t tile_pos;      // T
  int32_t tiles_per_unit;
  int32_t num_kv_heads;
  int32_t kv_block;      // BN
  int32_t capacity;      // work items the workspace holds
  int32_t window_left;   // > 0: sliding window of this many keys left of the diagonal
  int32_t grid;          // CTAs of the attention launch
  int32_t merge_capacity;  // merge units the workspace holds (0: never split)
  int64_t partial_capacity;  // partial rows the workspace holds
  int64_t mask_row_words;  // > 0: a custom mask of this many words per row (each request's keys must fit)
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_last_page_len;
  WorkItem* items;      // 16-byte aligned
  MergeUnit* merges;    // 16-byte aligned
  WsHeader* header;
};

// Kernel launchers (bip_attn.cu / bip_attn_gather.cu / bip_attn_mask.cu / bip_merge.cu /
// bip_append.cu / bip_plan_dev.cu / bip_mask_skip.cu / bip_upload.cu).  launch_attention hands page sizes below
// 8 to launch_attention_gather.
cudaError_t launch_attention(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                             cudaStream_t stream);
cudaError_t launch_attention_gather(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                                    const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                    cudaStream_t stream);
// The custom-mask variants of both (bip_attn_mask.cu): p.mask is set.
cudaError_t launch_attention_masked(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                                    const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                    cudaStream_t stream);
cudaError_t launch_merge(int head_dim, const MergeParams& p, cudaStream_t stream);
cudaError_t launch_append(int head_dim, bool kv_fp8, const AppendParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_device_plan(const DevPlanParams& p, cudaStream_t stream);
cudaError_t launch_mask_skip(const MaskSkipParams& p, int max_items, cudaStream_t stream);  // max_items: the count or a bound
// bytes (a multiple of 16) from a device-visible pinned host buffer to the
// workspace, by SM loads (bip_upload.cu).
cudaError_t launch_upload(const void* src_dev, void* dst, size_t bytes, cudaStream_t stream);

}  // namespace bip
