// Contract between the host planner (bip_host.cpp) and the kernels
// (bip_attn.cu, bip_merge.cu): work-list records, workspace header and
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
  uint32_t reserved[61];
};
static_assert(sizeof(WsHeader) == kHeaderBytes, "header size");

// One attention work item: a (request, kv head, q tile) unit over a range
// of its segments.  32 bytes.
struct WorkItem {
  int32_t kv_len;
  int32_t page_base;   // first entry of the request in kv_indices
  int32_t q_tok0;      // q row of sequence position 0 (may be negative)
  int32_t q_lo;        // first position that has a q row (kv_len - q_len)
  int32_t tile;        // absolute tile: positions [tile*T, tile*T + T)
  int16_t kv_head;
  int16_t seg_lo;      // inclusive segment range
  int16_t seg_hi;
  int16_t flags;       // kItemSplit: write fp32 partials instead of out/lse
  int32_t part_base;   // split: partial row of this item's first valid row
};
static_assert(sizeof(WorkItem) == 32, "work item size");
constexpr int16_t kItemSplit = 1;

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
  int32_t num_qo_heads;
  int32_t group;        // q heads per kv head
  int32_t tile_pos;     // T = floor(128 / group)
  int32_t page_size;
  int32_t num_pages;
  const int32_t* kv_indices;
  uint16_t* out;        // bf16 bits
  float* lse;
  float* partials;      // [rows][head_dim + 4]: m, l, 0, 0, o[head_dim]
  float* scratch;       // [grid][128][head_dim]
  WsHeader* header;
  float scale_log2;     // log2(e) * k_scale / sqrt(head_dim)
  float v_scale;
  uint64_t wait_limit_ns;
};

struct MergeParams {
  const MergeUnit* units;
  int32_t n_units;
  int32_t num_qo_heads;
  int32_t group;
  int32_t tile_pos;
  const float* partials;
  uint16_t* out;
  float* lse;
  float v_scale;
};

// Kernel launchers (bip_attn.cu / bip_merge.cu).
cudaError_t launch_attention(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const AttnParams& p, int grid, cudaStream_t stream);
cudaError_t launch_merge(int head_dim, const MergeParams& p, cudaStream_t stream);

}  // namespace bip
