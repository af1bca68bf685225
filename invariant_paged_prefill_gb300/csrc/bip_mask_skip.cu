// Custom masks: skip the KV blocks before the first key any row of a work
// item sees.  The pages name custom masks among the cases the batch-invariant
// path must cover (sglang PR 46351, "Fix"); a block that no row of an item
// sees contributes exact zeros to every row, so the work list may start each
// item at the first block some row sees, as a sliding window does.
//
// Runs after the work list is in the workspace (uploaded, or written by the
// device planner) and before the attention launch, in two launches.  First, the
// items of one kv head per unit (every q row of the batch lies in one of them;
// the other kv heads' items hold the same rows) find each of their rows' first
// visible key, from the first key the causal and window rules allow up to the
// row's own position, into a per-row array in the workspace: the rows are
// spread over the CTA's warps, four at a time per warp; lane i loads words i,
// 32 + i, 64 + i and 96 + i of a 128-word window of each of the four rows
// (sixteen independent, coalesced loads), ballots find a row's first nonzero
// word, and the window moves on until every row has its key.  Then every item
// (one warp each) takes the smallest key over its rows and starts at that key's
// block.  A folded item also starts at that block's segment (the segments
// before it hold no visible key for any row and are not visited, as under a
// window); a split item keeps its segment.  An item none of whose rows sees a
// key in its range keeps only its last block, which still writes the rows'
// empty state (m = -inf, l = 0).
//
// Whether a block is visited changes no bit of any row: a row that sees no
// key of a block gets p = 0 for all of its columns, an unchanged running
// max and row sum, and exact zeros added to O; a segment with no visible key
// merges as the empty state.  So the rows of an extend still equal the rows
// of the full prefill, whose items group other rows.

#include <climits>

#include <cuda_runtime.h>

#include "bip_internal.h"

namespace bip {
namespace {

constexpr int kSkipThreads = 256;
constexpr int kSkipWarps = kSkipThreads / 32;
constexpr int kKeyRows = 4;  // rows a warp scans together
constexpr int kKeyWins = 4;  // 32-word windows of each row loaded at once

// Position of row r (slot-major over the item's tiles), and whether the
// item holds it.
__device__ __forceinline__ bool item_row(const MaskSkipParams& p, const WorkItem& w, int r, int& pos) {
  const int t = r / p.tile_pos;
  pos = w.q_lo + (w.tile + t) * p.tile_pos + (r - t * p.tile_pos);
  const int present = (w.flags / kSlotPresent) & ((1 << kMaxTilesPerUnit) - 1);
  return r < p.tiles_per_unit * p.tile_pos && (present >> t & 1) && pos < w.kv_len;
}

__global__ void __launch_bounds__(kSkipThreads, 2) bip_mask_keys_kernel(const MaskSkipParams p) {
  const int n_items = p.n_items_dev ? int(*p.n_items_dev) : p.n_items;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int npos = p.tiles_per_unit * p.tile_pos;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkItem w = p.items[it];
    // One kv head's items per unit scan its rows (the others hold the same
    // rows); which head depends on the unit, so that a work list that keeps
    // a unit's heads together does not leave the scans to every
    // num_kv_heads-th CTA.
    const uint32_t pick = (uint32_t(w.tile) * 2654435761u + uint32_t(w.page_base)) % uint32_t(p.num_kv_heads);
    if (uint32_t(w.kv_head) != pick) continue;  // uniform over the CTA
    for (int r0 = warp; r0 < npos; r0 += kSkipWarps * kKeyRows) {
      int lo_w[kKeyRows], hi_w[kKeyRows], lo[kKeyRows], pos[kKeyRows], key[kKeyRows];
      const uint32_t* mrow[kKeyRows];
      bool act[kKeyRows], has[kKeyRows];
#pragma unroll
      for (int i = 0; i < kKeyRows; ++i) {
        has[i] = item_row(p, w, r0 + i * kSkipWarps, pos[i]);
        act[i] = has[i];
        key[i] = INT_MAX;
        lo[i] = p.window_left > 0 ? max(0, pos[i] - p.window_left) : 0;
        lo_w[i] = lo[i] >> 5;
        hi_w[i] = pos[i] >> 5;
        mrow[i] = has[i] ? p.mask + int64_t(w.q_tok0 + pos[i]) * p.mask_row_words : p.mask;
      }
      for (int cw = 0;; cw += 32 * kKeyWins) {
        uint32_t bits[kKeyRows][kKeyWins];
#pragma unroll
        for (int i = 0; i < kKeyRows; ++i)
#pragma unroll
          for (int h = 0; h < kKeyWins; ++h) {
            const int wd = lo_w[i] + cw + 32 * h + lane;
            uint32_t v = (act[i] && wd <= hi_w[i]) ? __ldg(mrow[i] + wd) : 0u;
            if (wd == lo_w[i]) v &= ~0u << (lo[i] & 31);                                      // keys from lo on
            if (wd == hi_w[i]) v &= (pos[i] & 31) == 31 ? ~0u : (2u << (pos[i] & 31)) - 1u;  // up to pos
            bits[i][h] = v;
          }
        bool more = false;
#pragma unroll
        for (int i = 0; i < kKeyRows; ++i) {
          if (!act[i]) continue;  // uniform over the warp
          bool found = false;
          int k = 0;
#pragma unroll
          for (int h = 0; h < kKeyWins; ++h) {
            const unsigned ball = __ballot_sync(0xffffffffu, bits[i][h] != 0u);
            if (!found && ball) {  // uniform over the warp
              const int src = __ffs(int(ball)) - 1;
              const uint32_t b = __shfl_sync(0xffffffffu, bits[i][h], src);
              k = (lo_w[i] + cw + 32 * h + src) * 32 + __ffs(int(b)) - 1;
              found = true;
            }
          }
          if (found) {
            key[i] = k;
            act[i] = false;
          } else if (lo_w[i] + cw + 32 * kKeyWins > hi_w[i]) {
            act[i] = false;  // no visible key
          } else {
            more = true;
          }
        }
        if (!more) break;
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kKeyRows; ++i)
          if (has[i]) p.first_key[w.q_tok0 + pos[i]] = key[i];
      }
    }
  }
}

__global__ void __launch_bounds__(kSkipThreads) bip_mask_skip_kernel(const MaskSkipParams p) {
  // one warp per item
  const int n_items = p.n_items_dev ? int(*p.n_items_dev) : p.n_items;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int npos = p.tiles_per_unit * p.tile_pos;
  for (int it = blockIdx.x * kSkipWarps + warp; it < n_items; it += gridDim.x * kSkipWarps) {
    const WorkItem w = p.items[it];
    int m = INT_MAX;
    for (int r = lane; r < npos; r += 32) {
      int pos;
      if (item_row(p, w, r, pos)) m = min(m, p.first_key[w.q_tok0 + pos]);
    }
    m = __reduce_min_sync(0xffffffffu, m);
    if (lane == 0) {
      // the item's block range, as the attention kernel derives it
      const int present = (w.flags / kSlotPresent) & ((1 << kMaxTilesPerUnit) - 1);
      int unit_end = 0;
      for (int s = 0; s < p.tiles_per_unit; ++s)
        if (present >> s & 1) unit_end = min(w.q_lo + (w.tile + s + 1) * p.tile_pos - 1, w.kv_len - 1);
      const int bps = kSplitLen / p.kv_block;
      const int blk_lo = max(int(w.seg_lo) * bps, w.blk_min);
      const int blk_hi = min((int(w.seg_hi) + 1) * kSplitLen - 1, unit_end) / p.kv_block;
      const int blk = min(m == INT_MAX ? blk_hi : m / p.kv_block, blk_hi);
      if (blk > blk_lo) {
        p.items[it].blk_min = blk;
        if (!(w.flags & kItemSplit)) p.items[it].seg_lo = int16_t(blk / bps);
      }
    }
  }
}

}  // namespace

cudaError_t launch_mask_skip(const MaskSkipParams& p, int max_items, cudaStream_t stream) {
  if (max_items <= 0) return cudaSuccess;
  constexpr int kMaxCtas = 1024;
  bip_mask_keys_kernel<<<min(max_items, kMaxCtas), kSkipThreads, 0, stream>>>(p);  // a CTA per item
  bip_mask_skip_kernel<<<min((max_items + kSkipWarps - 1) / kSkipWarps, kMaxCtas), kSkipThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bip
