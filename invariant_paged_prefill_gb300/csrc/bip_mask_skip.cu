// Custom masks: skip the KV blocks before the first key any row of a work
// item sees.  The pages name custom masks among the cases the batch-invariant
// path must cover (sglang PR 46351, "Fix"); a block that no row of an item
// sees contributes exact zeros to every row, so the work list may start each
// item at the first block some row sees, as a sliding window does.
//
// Runs after the work list is in the workspace (uploaded, or written by the
// device planner) and before the attention launch.  For each item, one
// thread per tile row (the first q head of each position: the heads of a
// position share its mask row) scans the row's mask words from the first key
// the causal and window rules allow up to the row's own position and stops
// at the first visible key; the item's first block becomes the block of the
// smallest such key over its rows.  A folded item also starts at that
// block's segment (the segments before it hold no visible key for any row
// and are not visited, as under a window); a split item keeps its segment.
// An item none of whose rows sees a key in its range keeps only its last
// block, which still writes the rows' empty state (m = -inf, l = 0).
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

constexpr int kSkipThreads = kMaxTilesPerUnit * kTileRows;  // one thread per row of each tile slot

__global__ void __launch_bounds__(kSkipThreads) bip_mask_skip_kernel(const MaskSkipParams p) {
  __shared__ int s_min[kSkipThreads / 32];
  const int n_items = p.n_items_dev ? int(*p.n_items_dev) : p.n_items;
  const int tid = threadIdx.x, t = tid / kTileRows, row = tid % kTileRows;
  const int local_pos = row / p.group, hg = row - local_pos * p.group;
  for (int it = blockIdx.x; it < n_items; it += gridDim.x) {
    const WorkItem w = p.items[it];
    const int present = (w.flags / kSlotPresent) & ((1 << kMaxTilesPerUnit) - 1);
    int first = INT_MAX;
    if (t < p.tiles_per_unit && (present >> t & 1) && hg == 0 && local_pos < p.tile_pos) {
      const int tile_start = w.q_lo + (w.tile + t) * p.tile_pos;
      const int pos = tile_start + local_pos;
      if (pos < w.kv_len) {
        const uint32_t* mrow = p.mask + int64_t(w.q_tok0 + pos) * p.mask_row_words;
        const int lo = p.window_left > 0 ? max(0, pos - p.window_left) : 0;
        for (int wd = lo >> 5; wd <= (pos >> 5); ++wd) {
          uint32_t bits = __ldg(mrow + wd);
          if (wd == (lo >> 5)) bits &= ~0u << (lo & 31);                            // keys from lo on
          if (wd == (pos >> 5)) bits &= (pos & 31) == 31 ? ~0u : (2u << (pos & 31)) - 1u;  // up to pos
          if (bits) {
            first = wd * 32 + __ffs(int(bits)) - 1;
            break;
          }
        }
      }
    }
    first = __reduce_min_sync(0xffffffffu, first);
    if ((tid & 31) == 0) s_min[tid / 32] = first;
    __syncthreads();
    if (tid == 0) {
      int m = INT_MAX;
#pragma unroll
      for (int i = 0; i < kSkipThreads / 32; ++i) m = min(m, s_min[i]);
      // the item's block range, as the attention kernel derives it
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
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_mask_skip(const MaskSkipParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  bip_mask_skip_kernel<<<grid, kSkipThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace bip
