// Persistent paged prefill attention for sm_103a: TMA page loads, tcgen05
// MMAs with TMEM accumulators, an fp32 online softmax with one thread per
// row, P kept in TMEM, and a fixed-order segment merge.  Kernel templates;
// bip_attn.cu instantiates the variants that load whole pages with TMA,
// bip_attn_gather.cu those that gather token rows (page sizes below 8).
//
// One CTA (one per SM) walks work items: a unit = (request, KV head, NT
// consecutive q tiles that share the same keys; tiles are counted from the
// request's first new row) over some of its 4096-key segments.  Roles,
// whole warpgroups each:
//   softmax warps   one warpgroup per q tile slot t: thread i owns packed
//                   row i (TMEM lane i); masks, keeps the row's running max
//                   and sum, writes P_t (bf16) over S_t in TMEM, rescales
//                   O_t when needed, and at each segment end folds or
//                   writes the segment.
//   (FP8 pages)     dequant warpgroups (two with one q-tile slot and whole
//                   pages, one per K/V stream) convert staged E4M3 blocks
//                   to f16.
//   (token pages)   row-gather warps copy K and V rows with cp.async (bf16:
//                   two warpgroups; FP8: one).
//   control         warp 0: spare; warp 1: the tcgen05 issuer,
//                   S_t = Q_t K^T into TMEM, then O_t += P_t V with P_t read
//                   from TMEM; warp 2: V blocks by TMA (its own ring),
//                   zeroing V rows past kv_len before they enter a product;
//                   warp 3: q tiles and K blocks by TMA through an ST-deep
//                   ring (q only when rows are gathered).
// With two slots (head_dim 128) the softmax of one tile overlaps the MMAs of
// the other.  Slots, ring depth and the way pages are fetched only decide
// scheduling; every row's arithmetic is the same in every variant.
//
// Packed rows (GQA group inside the 128-row tile, sglang PR 46351 "Root
// cause": packed q length = q_len * group): row = local_pos * group + head
// within the KV head's group, local_pos in [0, T), T = floor(128 / group).
//
// Invariance: a row's arithmetic depends only on its own q row, on keys at
// positions <= its own, and on the compile-time block/segment lengths.  MMA
// rows never mix; blocks beyond a row's position contribute exact zeros
// (p = 0 against finite V: rows of V past kv_len are zeroed in shared
// memory), and segments wholly beyond it are empty and skipped by the merge.
// The running max is moved (and O rescaled) only when a row's block max
// exceeds it by more than kLazyRescale in log2 units: a per-row decision.
//
// Mask kinds (template MK): 0 causal; 1 causal with a sliding window; 2
// causal narrowed by a per-row custom mask (and by the window when
// window_left > 0).  A custom mask row is read one block of bits at a time,
// and a row that ends with no visible key is written as zeros with lse -inf.

#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <climits>
#include <type_traits>

#include "bip_internal.h"
#include "bip_numerics.cuh"
#include "bip_ptx.cuh"

namespace bip {
namespace {

// A row keeps a stale running max until a block raises it by more than this
// (log2 units): probabilities then stay below 2^8 and O is rescaled rarely.
constexpr float kLazyRescale = 8.0f;

// Bytes at the end of shared memory for the mbarriers, the TMEM address,
// the abort mark and (FP8 pages) the q rows' scale exponents.
constexpr int kBarArea = 1024;

template <int D, int NT, int ST, bool KV8 = false, bool GATHER = false>
struct Cfg {
  static constexpr int BN = kv_block_for(D);        // keys per block
  static constexpr int NS = NT == 1 ? 2 : 1;        // S buffers per tile slot
  // FP8 pages, 128-key blocks: the softmax publishes the first 64 columns of
  // P early (B_P_HALF) and the PV of those keys starts while it computes the
  // rest.  Measured on GB300: +2 % (long prefill) and +4.5 % (short extend)
  // with E4M3 pages; bf16 pages ran 2 % (long prefill) to 7 % (document
  // masks) slower, so they keep one PV per block.
  static constexpr bool HALF_P = KV8 && BN == 128;
  static constexpr int DCH = D / 64;                // 64-column (128-byte) chunks of a d-row
  static constexpr int Q_CHUNK = kTileRows * 128;   // bytes of one q chunk (128 rows)
  static constexpr int Q_BYTES = DCH * Q_CHUNK;     // one tile slot
  static constexpr int KV_CHUNK = BN * 128;         // bytes of one K/V chunk (BN rows)
  static constexpr int KV_BYTES = DCH * KV_CHUNK;   // one K or V block
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NT * Q_BYTES;
  static constexpr int OFF_V = OFF_K + ST * KV_BYTES;
  // FP8 pages land raw (BN rows x D bytes, unswizzled) in a staging ring and
  // are converted to the bf16 operand layout by the dequant warpgroups.
  // (two q-tile slots leave room for one)
  static constexpr int SS = KV8 ? ((D == 128 && NT == 1) ? 2 : 1) : 0;  // staging stages
  static constexpr int KV8_BYTES = BN * D;
  static constexpr int OFF_K8 = OFF_V + ST * KV_BYTES;
  static constexpr int OFF_V8 = OFF_K8 + SS * KV8_BYTES;
  static constexpr int OFF_BAR = OFF_V8 + SS * KV8_BYTES;
  static constexpr int SMEM = OFF_BAR + kBarArea + 1024;  // + room to align the base to 1024
  // Custom-mask kernels with bf16 pages, where shared memory has room,
  // stage the output: each softmax warp writes its 32 rows' bf16 output 64
  // columns at a time here, then the warp stores whole 128-byte lines (a
  // row-per-lane store puts 32 rows' 16-byte pieces in 32 different
  // lines).  Measured on GB300: +2 % under custom masks, -3 % on the plain
  // causal long prefill, which keeps row-per-lane stores.
  static constexpr int OUT_STAGE_WARP = 32 * 128;
  static constexpr int OFF_OSTG = OFF_BAR + kBarArea;
  static constexpr int SMEM_OSTG = OFF_OSTG + 4 * NT * OUT_STAGE_WARP + 1024;  // 4 NT softmax warps
  static constexpr bool OUT_STAGE = !KV8 && SMEM_OSTG <= 227 * 1024;
  // Warp roles, whole warpgroups each: softmax warps 0 .. 4 NT - 1 (slot
  // t = warp / 4, TMEM lane quarter = warp % 4), then the FP8 dequant
  // warpgroups, then (GATHER) the row-gather warps, half for K and half for
  // V (bf16: two warpgroups; FP8: one, next to a single dequant warpgroup),
  // then the control warpgroup: a spare warp, the MMA issuer, the V
  // producer and the q/K producer.
  static constexpr int SM_WARPS = 4 * NT;
  static constexpr int DQ_WARP0 = SM_WARPS;
  // FP8 dequant warpgroups.  With two, one converts every K block and the
  // other every V block, so a K stage is released as soon as its codes are
  // in registers even while a V block waits for its ring slot; each walks
  // its stream's stages and slots in order, so its parity waits never run
  // two phases ahead of a barrier (at head_dim 256 each stream has one
  // staging stage).  One warpgroup converts both next to the row-gather
  // warpgroup.  Two give up registers (setmaxnreg); one keeps its launch
  // count.
  static constexpr int DQ_WGS = KV8 ? ((NT == 1 && !GATHER) ? 2 : 1) : 0;
  static constexpr int DQ_REGS = D == 256 ? 104 : 80;  // head_dim 256: its q-tile conversion spilled at 80
  static constexpr int GA_WARP0 = SM_WARPS + 4 * DQ_WGS;
  static constexpr int GA_WARPS = GATHER ? (KV8 ? 4 : 8) : 0;
  static constexpr int GW = GATHER ? (KV8 ? 2 : 4) : 0;  // gather warps per stream (K or V)
  static constexpr int CTL_WARP0 = GA_WARP0 + GA_WARPS;
  static constexpr int THREADS = 32 * (CTL_WARP0 + 4);
  // Register split: launches of more than 256 threads start at LAUNCH_REGS
  // a thread; the control and gather warpgroups then give registers back
  // (setmaxnreg) and the softmax warpgroups take them.  The dequant
  // warpgroup keeps its launch count.  The sum never exceeds what the
  // launch holds.
  static constexpr int LAUNCH_REGS = (65536 / THREADS) & ~7;
  static constexpr bool SPLIT_REGS = THREADS > 256;
  static constexpr int CTL_REGS = KV8 ? 80 : (GATHER ? 72 : 56);  // FP8: softmax is capped at 240 anyway
  static constexpr int GA_REGS = 56;
  static constexpr int FIXED_REGS = CTL_REGS * 128 + GA_REGS * 32 * GA_WARPS +
                                   (DQ_WGS == 2 ? DQ_REGS * 256 : DQ_WGS * LAUNCH_REGS * 128);
  static constexpr int SM_REGS_FREE = ((LAUNCH_REGS * THREADS - FIXED_REGS) / (32 * SM_WARPS)) & ~7;
  static constexpr int SM_REGS = SPLIT_REGS ? (SM_REGS_FREE < 240 ? SM_REGS_FREE : 240) : 255;
  static_assert(!SPLIT_REGS || SM_REGS * 32 * SM_WARPS + FIXED_REGS <= LAUNCH_REGS * THREADS,
                "register split exceeds the launch's registers");
  static_assert(!SPLIT_REGS || SM_REGS >= LAUNCH_REGS, "softmax warps must not lose registers");
  static constexpr int TM_COLS = 512;
  // Unroll factor of the MMA issue loops.  The tensor pipe queues only a few
  // MMAs, so the issuing thread's per-MMA instructions show up as pipe time;
  // measured on GB300, full unrolling is best with one q-tile slot and 4
  // with two (whose larger issue path slows down when fully unrolled).
  static constexpr int ISSUE_UNROLL = NT == 1 ? 16 : 4;
  static constexpr int BPS = kSplitLen / BN;         // blocks per segment
  // TMEM columns: two slots use [0,256) and [256,512), each S (BN) then O (D);
  // one slot keeps two S buffers at [0, 2 BN) and O at [256, 256 + D).
  __host__ __device__ static constexpr uint32_t tm_s(int t, int s) {
    return NT == 2 ? uint32_t(t * 256) : uint32_t(s * BN);
  }
  __host__ __device__ static constexpr uint32_t tm_o(int t) { return NT == 2 ? uint32_t(t * 256 + BN) : 256u; }
  // One q-tile slot: the q tile also lives in TMEM (D / 2 columns, copied
  // once per item), so that S = Q K^T reads only K from shared memory.
  // Two slots fill TMEM with S and O and read q from shared memory.
  static constexpr bool QT = NT == 1;
  static constexpr uint32_t TQ = (2 * BN + D / 2 <= 256) ? 2 * BN : 256 + D;
  static_assert(!QT || (TQ + D / 2 <= TM_COLS && (TQ >= 2 * BN) && (TQ + D / 2 <= 256 || TQ >= 256 + D)),
                "q tile columns clash with S or O");
  static_assert(NT == 1 || (BN + D <= 256), "two slots need S and O in 256 columns each");
  static_assert(NT == 2 || (2 * BN <= 256 && 256 + D <= TM_COLS), "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(!KV8 || NT == 1 || D == 128, "two FP8 q-tile slots exist at head_dim 128");
};

// Barrier slots (8 bytes each) at OFF_BAR.
enum Bar {
  B_Q_FULL = 0, B_Q_FREE = 1,
  B_K_FULL = 2, B_K_FREE = 6, B_V_FULL = 10, B_V_FREE = 14,  // up to 4 ring stages
  // Per slot and per S buffer (index 2 slot + buffer).  P_FULL and O_DONE
  // are kept per buffer too: with two S buffers the softmax may finish two
  // blocks before the issuer waits on the first, and a single barrier two
  // phases ahead of its waiter reads as zero under a parity wait.
  B_S_FULL = 18, B_P_FULL = 22, B_O_DONE = 26,
  B_DRAIN = 30,
  B_K8_FULL = 31, B_K8_FREE = 33, B_V8_FULL = 35, B_V8_FREE = 37,  // FP8 staging, up to 2 stages
  B_V_TX = 39,  // bf16 V blocks that end past kv_len land here first (the V producer zeroes the tail)
  // FP8 pages: the q tile has been converted to f16 (Q_READY, 128 dequant
  // threads) / the softmax has read the tile's row scales (QS_FREE, 128
  // softmax threads).
  B_Q_READY = 40, B_QS_FREE = 41,
  // FP8 pages with 128-key blocks: P's first 64 columns are in TMEM (and O
  // rescaled), per slot and S buffer like P_FULL; the PV of those keys
  // starts while the softmax computes the other half.
  B_P_HALF = 42,
  B_COUNT = 46
};
constexpr int OFF_TMEM_SLOT = 8 * B_COUNT;    // u32: TMEM base address
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;  // u32: a wait expired somewhere in this CTA
constexpr int OFF_QSCALE = 512;               // int8 [NT][128]: FP8 pages, each q row's scale exponent
static_assert(OFF_ABORT + 4 <= OFF_QSCALE && OFF_QSCALE + kMaxTilesPerUnit * kTileRows <= kBarArea,
              "barrier area");

struct Ctx {
  uint32_t bar0;
  volatile uint32_t* abort;
  WsHeader* header;
  uint64_t limit_cycles;
};

__device__ __forceinline__ uint32_t bar(const Ctx& c, int i) { return c.bar0 + 8u * i; }

// Bounded wait on an mbarrier phase.  On expiry the CTA is marked aborted,
// the workspace status records a timeout, and false is returned; any wait
// that sees the abort mark also returns false.  The first probe answers at
// once; after it the clock is checked before every (suspending) probe, so a
// wait that is not already complete always meets the limit check.  (Inlined:
// an out-of-line call cannot be shared by warpgroups running with different
// register budgets.)
__device__ __forceinline__ bool wait_phase(const Ctx& c, uint32_t b, uint32_t parity, uint32_t where) {
  const uint64_t t0 = clock64();
  if (mbar_ready(b, parity)) return true;
  while (true) {
    if (uint64_t(clock64()) - t0 > c.limit_cycles) {
      *c.abort = 1u;
      atomicCAS(&c.header->status, 0u, 5u /* BIP_ERR_DEVICE_TIMEOUT */);
      atomicExch(&c.header->where, where);
      return false;
    }
    if (mbar_test(b, parity)) return true;
    if (*c.abort) return false;
  }
}

// Same, with the result made uniform across the warp.
__device__ __forceinline__ bool wait_warp(const Ctx& c, uint32_t b, uint32_t parity, uint32_t where) {
  const bool ok = wait_phase(c, b, parity, where);
  return __all_sync(0xffffffffu, ok);
}

// Bounded wait used only while draining at exit (ignores the abort mark).
__device__ __forceinline__ void drain_wait(uint32_t b, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test(b, parity))
    if (globaltimer_ns() - t0 > 2000000000ull) break;
}

struct Geom {
  int tile_start[kMaxTilesPerUnit];  // first position of each slot's tile
  int tile_end[kMaxTilesPerUnit];    // last position with a q row or key in each slot's tile
  int first_valid[kMaxTilesPerUnit];
  int mask, last_slot;
  int blk_lo, blk_hi;  // inclusive block range of the item (union of the slots' keys)
};

template <int NT, int BN>
__device__ __forceinline__ Geom geom_of(const WorkItem& w, int T) {
  Geom g;
  g.mask = (w.flags / kSlotPresent) & ((1 << NT) - 1);
  g.last_slot = 0;
  int unit_end = 0;
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    g.tile_start[t] = w.q_lo + (w.tile + t) * T;  // tiles count from the request's first new row
    g.tile_end[t] = min(g.tile_start[t] + T - 1, w.kv_len - 1);
    g.first_valid[t] = g.tile_start[t];
    if (g.mask >> t & 1) {
      g.last_slot = t;
      unit_end = g.tile_end[t];
    }
  }
  g.blk_lo = max(int(w.seg_lo) * (kSplitLen / BN), w.blk_min);  // a sliding window starts mid-segment
  g.blk_hi = min((int(w.seg_hi) + 1) * kSplitLen - 1, unit_end) / BN;
  return g;
}

// Work items of this launch: fixed by the host plan, or counted on the
// device by the planner kernel that ran before (graph-replayable launches).
__device__ __forceinline__ int item_count(const AttnParams& p) {
  return p.n_items_dev ? int(*p.n_items_dev) : p.n_items;
}

// ------------------------------------------------------------------ roles

// Page id of page `lane` of KV block `blk` (0 for lanes past the block's
// pages), and the block's page count.  Pages per block <= 16 <= warp size.
__device__ __forceinline__ int lane_page_id(const AttnParams& p, const WorkItem& w, int blk, int pages_per_blk,
                                            int npages_req, int lane, int& n) {
  const int p0 = blk * pages_per_blk;
  n = min(p0 + pages_per_blk, npages_req) - p0;
  return lane < n ? __ldg(p.kv_indices + w.page_base + p0 + lane) : 0;
}

// Token-granular pages (page_size below 8) hold fewer than the eight
// 128-byte rows of one swizzle atom, so no TMA box lands a page in place;
// the block is gathered row by row instead.  row_ids: the page ids of rows
// r0 .. r0 + RW - 1 of block blk, lane l holding row r0 + l + 32 k (0 at or
// past kv_len, and for an out-of-range id, which the K stream counts once,
// at the page's first row).
template <int BN, int RW>
__device__ __forceinline__ void row_ids(const Ctx& c, const AttnParams& p, const WorkItem& w, int blk, int r0,
                                        int lg_page, bool count_bad, int lane, int (&ids)[(RW + 31) / 32]) {
#pragma unroll
  for (int k = 0; k < (RW + 31) / 32; ++k) {
    const int rr = 32 * k + lane;
    const int t = blk * BN + r0 + rr;
    int id = 0;
    if (rr < RW && t < w.kv_len) {
      id = __ldg(p.kv_indices + w.page_base + (t >> lg_page));
      if (uint32_t(id) >= uint32_t(p.num_pages)) {
        if (count_bad && (t & ((1 << lg_page) - 1)) == 0) atomicAdd(&c.header->bad_pages, 1u);
        id = 0;
      }
    }
    ids[k] = id;
  }
}

// Issue rows r0 .. r0 + RW - 1 of the block as 16-byte cp.async copies: each
// warp instruction covers 32 / UPR whole rows (UPR 16-byte units a row),
// lanes along a row, so every row is read as one contiguous run.  bf16: row
// r, unit u of 64-column chunk ch goes to
// ch * KV_CHUNK + r * 128 + ((u ^ (r & 7)) * 16), the 128-byte swizzle the
// MMA descriptors read.  FP8: rows land row-major in the staging slot, as
// the TMA box would put them.  Rows at or past kv_len are zero-filled.
// Then one arrival per lane on `land` once its copies have landed.
template <int D, int BN, bool KV8, int RW>
__device__ __forceinline__ void gather_rows(const AttnParams& p, const WorkItem& w, int blk, int r0, int lg_page,
                                            const uint8_t* pool, uint32_t dst, uint32_t land, int lane,
                                            const int (&ids)[(RW + 31) / 32]) {
  constexpr int ES = KV8 ? 1 : 2;
  constexpr int UPR = D * ES / 16;  // 8, 16 or 32
  constexpr int RPI = 32 / UPR;     // rows per warp instruction
  constexpr int RK = RW < 32 ? RW : 32;  // rows per page-id register
  static_assert(RK % RPI == 0, "whole instructions per page-id register");
  const int u = lane % UPR;
  const uint8_t* base = pool + int64_t(w.kv_head) * (D * ES) + u * 16;
  const int smask = (1 << lg_page) - 1;
  const int32_t stride = int32_t(p.page_stride_bytes);  // below 2^31 (checked on the host)
#pragma unroll
  for (int k = 0; k < (RW + 31) / 32; ++k) {
#pragma unroll 4
    for (int i = 0; i < RK / RPI; ++i) {
      const int rl = i * RPI + lane / UPR;  // row within this register's rows = the lane holding its page id
      const int r = r0 + 32 * k + rl;
      const int t = blk * BN + r;
      const int id = __shfl_sync(0xffffffffu, ids[k], rl);
      const uint8_t* src = base + int64_t(id) * stride + (t & smask) * p.slot_bytes;
      uint32_t d;
      if constexpr (KV8) {
        d = dst + r * D + u * 16;
      } else {
        d = dst + (u >> 3) * (BN * 128) + r * 128 + (((u & 7) ^ (r & 7)) << 4);
      }
      cp_async_16(d, src, t < w.kv_len ? 16u : 0u);
    }
  }
  cp_async_arrive_noinc(land);
}

// One TMA stream, run by a whole warp: the control warpgroup's first warp
// loads the q tiles and K, its third warp loads V, so a V slot still in use
// never holds back K loads (or the reverse).  Lane i holds the page id of
// page i of the next block (fetched one block ahead) and issues that page's
// loads; lane 0 posts the expected bytes first.  Each item's first
// ring-depth K blocks are issued before its q tiles, whose load waits for
// the previous item's last S, so the ring keeps streaming across item
// boundaries.  GATHER (token-granular pages): K and V rows are gathered by
// the row-gather warps; this warp loads the q tiles only.
template <int D, int NT, int ST, bool KV8, bool GATHER>
__device__ void producer(const Ctx& c, uint32_t sbase, const CUtensorMap* tq, const CUtensorMap* tkv,
                         const AttnParams& p, const bool is_v) {
  using C = Cfg<D, NT, ST, KV8>;
  static_assert(C::BN / 8 <= 32, "one lane per page");
  const int lane = threadIdx.x & 31;
  const uint32_t sQ = sbase + C::OFF_Q;
  const int pages_per_blk = C::BN / p.page_size;
  const uint32_t q_slot_bytes = uint32_t(C::DCH * 128 * p.group * p.tile_pos);
  // bf16: TMA fills the ring slot; FP8: TMA fills the staging ring, the
  // dequant warps fill the slot.
  constexpr int RING = KV8 ? C::SS : ST;
  const int full0 = KV8 ? (is_v ? B_V8_FULL : B_K8_FULL) : (is_v ? B_V_FULL : B_K_FULL);
  const int free0 = KV8 ? (is_v ? B_V8_FREE : B_K8_FREE) : (is_v ? B_V_FREE : B_K_FREE);
  const uint32_t ring0 = sbase + (KV8 ? (is_v ? C::OFF_V8 : C::OFF_K8) : (is_v ? C::OFF_V : C::OFF_K));
  const uint32_t ring_bytes = KV8 ? uint32_t(C::KV8_BYTES) : uint32_t(C::KV_BYTES);
  const uint32_t page_bytes = uint32_t(p.page_size * D * (KV8 ? 1 : 2));
  uint32_t b = 0;      // blocks started by this CTA
  int n = 0;           // items started by this CTA
  uint32_t n_tail = 0;  // bf16 V blocks routed through B_V_TX (issued)
  uint32_t n_q = 0;     // q tile loads issued
  bool ok = true;

  auto load_q = [&](const WorkItem& w, const Geom& g) -> bool {
    if (n > 0 && !wait_warp(c, bar(c, B_Q_FREE), (n - 1) & 1, 1)) return false;
    ++n_q;
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(c, B_Q_FULL), q_slot_bytes * __popc(g.mask));
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (!(g.mask >> t & 1)) continue;
        for (int ch = 0; ch < C::DCH; ++ch)
          tma_load_3d(sQ + t * C::Q_BYTES + ch * C::Q_CHUNK, tq, bar(c, B_Q_FULL), ch * 64, w.kv_head * p.group,
                      w.q_tok0 + g.tile_start[t]);
      }
    }
    __syncwarp();
    return true;
  };

  if constexpr (GATHER) {
    for (int it = blockIdx.x; it < item_count(p) && ok; it += gridDim.x, ++n) {
      const WorkItem w = p.items[it];
      if (!load_q(w, geom_of<NT, C::BN>(w, p.tile_pos))) ok = false;
    }
  }
  for (int it = blockIdx.x; !GATHER && it < item_count(p) && ok; it += gridDim.x, ++n) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<NT, C::BN>(w, p.tile_pos);
    const int npages_req = (w.kv_len + p.page_size - 1) / p.page_size;
    int nid;
    int id_next = lane_page_id(p, w, g.blk_lo, pages_per_blk, npages_req, lane, nid);
    bool q_done = is_v;
    for (int blk = g.blk_lo; blk <= g.blk_hi; ++blk, ++b) {
      if (!q_done && blk - g.blk_lo == min(RING, g.blk_hi - g.blk_lo + 1)) {
        if (!load_q(w, g)) { ok = false; break; }
        q_done = true;
      }
      const int slot = b % RING;
      const uint32_t use = b / RING;
      const int ncur = nid;
      int id = id_next;
      if (lane < ncur && (id < 0 || id >= p.num_pages)) {  // counted once, by the K stream
        if (!is_v) atomicAdd(&c.header->bad_pages, 1u);
        id = 0;
      }
      if (blk < g.blk_hi) id_next = lane_page_id(p, w, blk + 1, pages_per_blk, npages_req, lane, nid);
      if (use > 0 && !wait_warp(c, bar(c, free0 + slot), (use - 1) & 1, is_v ? 3 : 2)) { ok = false; break; }
      // A bf16 V block that ends past kv_len lands on B_V_TX; once it is in,
      // this warp zeroes the rows at or past kv_len (the tail of the last
      // page, and pages the request does not have) so that p = 0 meets a
      // finite value, then completes the slot's V_FULL phase itself.  (FP8:
      // the dequant warps write those zeros.)
      const int valid_rows = w.kv_len - blk * C::BN;
      const bool tail = !KV8 && is_v && valid_rows < C::BN;
      const uint32_t land = tail ? bar(c, B_V_TX) : bar(c, full0 + slot);
      if (lane == 0) mbar_arrive_expect_tx(land, uint32_t(ncur) * page_bytes);
      n_tail += tail ? 1u : 0u;
      __syncwarp();
      if (lane < ncur) {
        if constexpr (KV8) {
          tma_load_4d(ring0 + slot * ring_bytes + lane * page_bytes, tkv, land, 0, w.kv_head, 0, id);
        } else {
          for (int ch = 0; ch < C::DCH; ++ch)
            tma_load_4d(ring0 + slot * ring_bytes + ch * C::KV_CHUNK + lane * p.page_size * 128, tkv, land,
                        ch * 64, w.kv_head, 0, id);
        }
      }
      if (tail) {
        if (!wait_warp(c, land, (n_tail - 1) & 1, 4)) { ok = false; break; }
        const uint32_t vbase = ring0 + slot * ring_bytes;
        const int per_chunk = (C::BN - valid_rows) * 8;  // 16-byte units per chunk
        for (int u = lane; u < per_chunk * C::DCH; u += 32) {
          const int ch = u / per_chunk, rem = u % per_chunk;
          const uint32_t addr = vbase + ch * C::KV_CHUNK + (valid_rows + rem / 8) * 128 + (rem % 8) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(c, full0 + slot));
        __syncwarp();
      }
    }
    if (ok && !q_done && !load_q(w, g)) ok = false;  // items shorter than the ring
  }
  // Drain: the last load on every barrier must have landed before exit (on
  // the normal path these phases completed long ago).  Phases issued: one
  // per q load (K stream only), and blocks started / RING per slot.
  if (lane == 0) {
    if (n_q) drain_wait(bar(c, B_Q_FULL), (n_q - 1) & 1);
    if (n_tail) drain_wait(bar(c, B_V_TX), (n_tail - 1) & 1);
#pragma unroll
    for (int slot = 0; slot < RING; ++slot) {
      const uint32_t issued = b / RING + (uint32_t(slot) < b % RING ? 1u : 0u);
      if (issued) drain_wait(bar(c, full0 + slot), (issued - 1) & 1);
    }
  }
  __syncwarp();
}

// Token-granular pages: the row-gather warps, GW per stream (gw < GW: K,
// else V), each owning a fixed range of BN / GW rows of every block, walk the
// same block schedule as the TMA producers and gather their rows into the
// ring slot.  A slot's landing phase completes when every gather lane of its
// stream has seen its own copies land.
template <int D, int NT, int ST, bool KV8, int GW>
__device__ void row_gatherer(const Ctx& c, uint32_t sbase, const AttnParams& p, const int gw) {
  using C = Cfg<D, NT, ST, KV8>;
  constexpr int RW = C::BN / GW;  // rows per warp
  static_assert(C::BN % GW == 0 && RW % 4 == 0, "row ranges");
  const int lane = threadIdx.x & 31;
  const bool is_v = gw >= GW;
  const int r0 = (gw % GW) * RW;
  constexpr int RING = KV8 ? C::SS : ST;
  const int full0 = KV8 ? (is_v ? B_V8_FULL : B_K8_FULL) : (is_v ? B_V_FULL : B_K_FULL);
  const int free0 = KV8 ? (is_v ? B_V8_FREE : B_K8_FREE) : (is_v ? B_V_FREE : B_K_FREE);
  const uint32_t ring0 = sbase + (KV8 ? (is_v ? C::OFF_V8 : C::OFF_K8) : (is_v ? C::OFF_V : C::OFF_K));
  const uint32_t ring_bytes = KV8 ? uint32_t(C::KV8_BYTES) : uint32_t(C::KV_BYTES);
  const int lg_page = __ffs(p.page_size) - 1;  // page_size is a power of two
  const uint8_t* pool = is_v ? p.v_pool : p.k_pool;
  uint32_t b = 0;  // blocks started by this CTA
  bool ok = true;
  for (int it = blockIdx.x; it < item_count(p) && ok; it += gridDim.x) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<NT, C::BN>(w, p.tile_pos);
    for (int blk = g.blk_lo; blk <= g.blk_hi; ++blk, ++b) {
      const int slot = b % RING;
      const uint32_t use = b / RING;
      int ids[(RW + 31) / 32];
      row_ids<C::BN, RW>(c, p, w, blk, r0, lg_page, !is_v, lane, ids);
      if (use > 0 && !wait_warp(c, bar(c, free0 + slot), (use - 1) & 1, is_v ? 3 : 2)) { ok = false; break; }
      gather_rows<D, C::BN, KV8, RW>(p, w, blk, r0, lg_page, pool, ring0 + slot * ring_bytes,
                                     bar(c, full0 + slot), lane, ids);
    }
  }
  // Drain: every copy issued has landed before exit.
  if (lane == 0) {
#pragma unroll
    for (int slot = 0; slot < RING; ++slot) {
      const uint32_t issued = b / RING + (uint32_t(slot) < b % RING ? 1u : 0u);
      if (issued) drain_wait(bar(c, full0 + slot), (issued - 1) & 1);
    }
  }
  __syncwarp();
}

// The tcgen05 issuer: one thread.  The tensor pipe queues only a few MMAs,
// so every cycle spent between two groups of MMAs (barrier probes, warp
// votes) shows up as pipe idle time; a single thread with plain probes keeps
// that gap short.
template <int D, int NT, int ST, bool KV8, bool GATHER>
__device__ void mma_issuer(const Ctx& c, uint32_t sbase, uint32_t tmem, const AttnParams& p) {
  using C = Cfg<D, NT, ST, KV8>;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  // bf16 operands; with FP8 pages every operand is f16 (q rows converted
  // exactly with a per-row power-of-two scale, K and V decoded from E4M3,
  // P rounded to f16).
  constexpr uint32_t kIdescS = idesc_f32acc(128, C::BN, false, false, KV8);  // S = Q K^T, both K-major
  constexpr uint32_t kIdescO = idesc_f32acc(128, D, false, true, KV8);       // O += P V, V MN-major
  // bf16 token rows gathered with cp.async are generic-proxy writes: once
  // their landing phase is seen, a proxy fence orders them before the MMAs'
  // operand reads.  (TMA writes, and FP8 slots the dequant warps fenced,
  // need none.)
  constexpr bool gathered = GATHER && !KV8;
  uint32_t gb = 0;                       // KV blocks consumed by this CTA (ring position)
  uint32_t k_seen = 0;                   // K blocks known to have landed
  uint32_t s_cnt[NT] = {}, pv_cnt[NT] = {};  // blocks whose S / PV was issued, per slot
  int n = 0;
  bool ok = true;
  for (int it = blockIdx.x; it < item_count(p) && ok; it += gridDim.x, ++n) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<NT, C::BN>(w, p.tile_pos);
    const int nb = g.blk_hi - g.blk_lo + 1;
    // FP8 pages: the q tile once the dequant warps have converted it to f16
    if (!wait_phase(c, bar(c, KV8 ? B_Q_READY : B_Q_FULL), n & 1, 10)) { ok = false; break; }
    tc_fence_after();
    if constexpr (C::QT) {
      // The previous item's S MMAs read the q columns: wait for its last one
      // (later PVs stay queued meanwhile), then copy this tile in, one
      // 32-byte K slice per 8 columns, and free the shared q tile.
      if (n > 0) {
        const uint32_t last_s = s_cnt[0] - 1;
        if (!wait_phase(c, bar(c, B_S_FULL + last_s % C::NS), (last_s / C::NS) & 1, 12)) { ok = false; break; }
        tc_fence_after();
      }
      const uint64_t dq = sdesc_sw128(sQ, 16, 1024);
#pragma unroll 1
      for (int k = 0; k < D / 16; ++k)
        tc_cp_128x256b(tmem + C::TQ + k * 8, dq + uint32_t(((k >> 2) * C::Q_CHUNK + (k & 3) * 32) >> 4));
      tc_commit(bar(c, B_Q_FREE));
    }

    // S_t for item-local block j into the slot's next S buffer.
    auto issue_s = [&](int t, int j) -> bool {
      const uint32_t kb = gb + j;
      const int kslot = kb % ST;
      if (kb >= k_seen) {  // the other slot's S may already have seen this K block land
        if (!wait_phase(c, bar(c, B_K_FULL + kslot), (kb / ST) & 1, 11)) return false;
        k_seen = kb + 1;
        tc_fence_after();
        if constexpr (gathered) fence_proxy_async_smem();
      }
      const int sbuf = s_cnt[t] % C::NS;
      const uint32_t d_tmem = tmem + C::tm_s(t, sbuf);
      // K step k: 32 bytes along a 128-byte row, 64 columns per chunk.  The
      // start address sits in the descriptor's low bits (16-byte units), so
      // a step is an add.
      const uint64_t dq = sdesc_sw128(sQ + t * C::Q_BYTES, 16, 1024);
      const uint64_t dk = sdesc_sw128(sK + kslot * C::KV_BYTES, 16, 1024);
#pragma unroll (C::ISSUE_UNROLL)
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t cq = ((k >> 2) * C::Q_CHUNK + (k & 3) * 32) >> 4;
        const uint32_t ck = ((k >> 2) * C::KV_CHUNK + (k & 3) * 32) >> 4;
        if constexpr (C::QT) tc_mma_ts(d_tmem, tmem + C::TQ + k * 8, dk + ck, kIdescS, k > 0 ? 1u : 0u);
        else tc_mma_ss(d_tmem, dq + cq, dk + ck, kIdescS, k > 0 ? 1u : 0u);
      }
      tc_commit(bar(c, B_S_FULL + 2 * t + sbuf));
      if (t == g.last_slot) {
        tc_commit(bar(c, B_K_FREE + kslot));                // last reader of this K block
        if (!C::QT && j == nb - 1) tc_commit(bar(c, B_Q_FREE));  // last reader of the q tiles
      }
      ++s_cnt[t];
      return true;
    };

    for (int j = 0; j < C::NS && j < nb && ok; ++j)
#pragma unroll
      for (int t = 0; t < NT; ++t)
        if ((g.mask >> t & 1) && !issue_s(t, j)) { ok = false; break; }
    if (!ok) break;

    for (int j = 0; j < nb && ok; ++j) {
      const uint32_t vb = gb + j;
      const int vslot = vb % ST;
      const int blk = g.blk_lo + j;
      // O starts afresh at a segment's first visited block (a block boundary
      // of the segment grid, or the item's first block under a window)
      const bool first_in_seg = (blk % C::BPS) == 0 || j == 0;
      bool v_ready = false;
#pragma unroll
      for (int t = 0; t < NT; ++t) {
        if (!(g.mask >> t & 1)) continue;
        const int pbuf = pv_cnt[t] % C::NS;
        const uint32_t ppar = (pv_cnt[t] / C::NS) & 1;
        // HALF_P: the PV of the first 64 keys starts once their P is in
        // TMEM, the rest once all of P is.  The MMAs and their order are
        // those of one 128-key PV.
        constexpr bool kHalfP = C::HALF_P;
        constexpr int KH = kHalfP ? C::BN / 32 : C::BN / 16;  // K steps issued before P is complete
        if (!wait_phase(c, bar(c, (kHalfP ? B_P_HALF : B_P_FULL) + 2 * t + pbuf), ppar, kHalfP ? 15 : 13)) {
          ok = false;
          break;
        }
        if (!v_ready) {
          // V rows at or past kv_len were zeroed before this phase completed.
          if (!wait_phase(c, bar(c, B_V_FULL + vslot), (vb / ST) & 1, 14)) { ok = false; break; }
          v_ready = true;
          if constexpr (gathered) fence_proxy_async_smem();
        }
        tc_fence_after();
        const uint32_t p_tmem = tmem + C::tm_s(t, pbuf);  // P_t (bf16) over its S buffer
        const uint64_t dv = sdesc_sw128(sV + vslot * C::KV_BYTES, C::KV_CHUNK, 1024);
        // K step k: 16 V rows (2048 bytes), 8 TMEM columns of P
#pragma unroll (kHalfP ? C::ISSUE_UNROLL / 2 : C::ISSUE_UNROLL)
        for (int k = 0; k < KH; ++k)
          tc_mma_ts(tmem + C::tm_o(t), p_tmem + k * 8, dv + uint32_t(k * 128), kIdescO,
                    (k > 0 || !first_in_seg) ? 1u : 0u);
        if constexpr (kHalfP) {
          if (!wait_phase(c, bar(c, B_P_FULL + 2 * t + pbuf), ppar, 13)) { ok = false; break; }
          tc_fence_after();
#pragma unroll (C::ISSUE_UNROLL / 2)
          for (int k = KH; k < C::BN / 16; ++k)
            tc_mma_ts(tmem + C::tm_o(t), p_tmem + k * 8, dv + uint32_t(k * 128), kIdescO, 1u);
        }
        tc_commit(bar(c, B_O_DONE + 2 * t + pbuf));
        ++pv_cnt[t];
        // The slot's next S goes into the buffer this PV has just been queued
        // to read; tcgen05 MMAs of one thread execute in issue order.
        if (j + C::NS < nb && !issue_s(t, j + C::NS)) { ok = false; break; }
      }
      if (!ok) break;
      tc_commit(bar(c, B_V_FREE + vslot));
    }
    gb += nb;
  }
  // Drain: every MMA this thread issued has completed before TMEM is freed.
  tc_commit(bar(c, B_DRAIN));
  drain_wait(bar(c, B_DRAIN), 0);
}

// Column j of a block is visible to a row when lo <= j <= lim and, with a
// custom mask, bit j of the row's mask bits for the block is set.
template <int MK, int NB>
__device__ __forceinline__ bool col_visible(int j, int lim, int lo, const uint32_t (&mb)[NB]) {
  return j <= lim && (MK == 0 || j >= lo) && (MK != 2 || ((mb[j >> 5] >> (j & 31)) & 1u));
}

template <int D, int NT, int ST, bool KV8, int MK, bool NARROW_LD>
__device__ void softmax_role(const Ctx& c, uint32_t tmem, const AttnParams& p, const int t,
                             const int8_t* p_qscale) {
  using C = Cfg<D, NT, ST, KV8>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;          // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;   // packed tile row == TMEM lane
  const uint32_t t_lane = tmem + (uint32_t(quarter * 32) << 16);
  float scale = p.scale_log2;     // log2(e) k_scale / sqrt(d), per logit of the MMA's S
  uint32_t cnt = 0, pv_seen = 0;  // blocks of this slot processed / PVs known complete
  uint32_t n_items = 0;           // items of this CTA started
  bool ok = true;

  // PV of this slot's block x has completed.  PVs complete in order, so
  // pv_seen only skips waits already satisfied.
  auto wait_pv = [&](uint32_t x) -> bool {
    if (pv_seen > x) return true;
    if (!wait_warp(c, bar(c, B_O_DONE + 2 * t + x % C::NS), (x / C::NS) & 1, 20)) return false;
    pv_seen = x + 1;
    return true;
  };

  for (int it = blockIdx.x; it < item_count(p) && ok; it += gridDim.x, ++n_items) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<NT, C::BN>(w, p.tile_pos);
    if constexpr (KV8) {
      // This row's q values were multiplied by 2^e (e from the row's largest
      // magnitude) when the tile became f16, so its S is 2^e times the
      // logits: the scale takes 2^-e back out, exactly.
      if (!wait_warp(c, bar(c, B_Q_READY), n_items & 1, 22)) { ok = false; break; }
      const int e = *reinterpret_cast<const volatile int8_t*>(p_qscale + t * kTileRows + row);
      scale = __fmul_rn(p.scale_log2, __int_as_float((127 - e) << 23));
      mbar_arrive(bar(c, B_QS_FREE));
    }
    if (!(g.mask >> t & 1)) continue;
    const int local_pos = row / p.group;
    const int hg = row - local_pos * p.group;
    const int pos = g.tile_start[t] + local_pos;
    const bool valid = row < p.tile_pos * p.group && pos >= g.first_valid[t] && pos <= g.tile_end[t];
    const bool split = (w.flags & kItemSplit) != 0;
    float Mrun = -INFINITY, Lrun = 0.f;  // merged state of the segments before this one
    // The fold state of this CTA and slot, 16-byte word j of every row
    // together (row-fastest): a warp's 32 rows load and store 512
    // contiguous bytes per instruction.
    float4* scratch_row = reinterpret_cast<float4*>(p.scratch) + (size_t(blockIdx.x) * NT + t) * kTileRows * (D / 4) + row;
    const uint32_t o_addr = t_lane + C::tm_o(t);
    // this warp's output staging (OUT_STAGE, custom masks)
    const uint32_t ostage = c.bar0 - C::OFF_BAR + C::OFF_OSTG + uint32_t(warp) * C::OUT_STAGE_WARP;
    // Custom mask: the row's bits for block blk (bit j of word j / 32 =
    // column j).  Only words holding a column at or before the row's
    // position are read (they lie inside the row, below its kv_len); the
    // next block's words are loaded one block ahead, so that their latency
    // hides behind a whole block.
    const uint32_t* mrow = MK == 2 ? p.mask + int64_t(w.q_tok0 + pos) * p.mask_row_words : nullptr;
    auto load_words = [&](int blk, uint32_t (&dst)[C::BN / 32]) {
#pragma unroll
      for (int k = 0; k < C::BN / 32; ++k)
        dst[k] = (valid && blk <= g.blk_hi && 32 * k <= pos - blk * C::BN)
                     ? __ldg(mrow + int64_t(blk) * (C::BN / 32) + k) : 0u;
    };
    uint32_t mb_next[C::BN / 32];
    if constexpr (MK == 2) load_words(g.blk_lo, mb_next);

    for (int s = w.seg_lo; s <= w.seg_hi && ok; ++s) {
      const int sb_lo = max(s * C::BPS, g.blk_lo);
      const int sb_hi = min((s + 1) * C::BPS - 1, g.blk_hi);
      float m = -INFINITY, l = 0.f;  // running raw-score max (possibly stale) and sum over this segment
      bool seg_first = true;  // first block of this segment: O is overwritten, never rescaled
      for (int blk = sb_lo; blk <= sb_hi; ++blk, ++cnt, seg_first = false) {
        const int sbuf = cnt % C::NS;
        // Columns lo..lim are visible: keys up to the row's position, and
        // with a sliding window none before position - window_left.
        const int lim = valid ? pos - blk * C::BN : -1;
        const int lo = (MK == 0 || (MK == 2 && p.window_left <= 0)) ? INT_MIN / 2
                                                                    : pos - p.window_left - blk * C::BN;
        // Custom mask: this block's visible columns as bits, vis = mask
        // words & the causal limit & the window (one bit test per column in
        // the masked loops); the next block's words are requested now.
        uint32_t mb[C::BN / 32], vis[C::BN / 32];
#pragma unroll
        for (int k = 0; k < C::BN / 32; ++k) mb[k] = vis[k] = 0u;
        if constexpr (MK == 2) {
#pragma unroll
          for (int k = 0; k < C::BN / 32; ++k) mb[k] = mb_next[k];
          load_words(blk + 1, mb_next);
#pragma unroll
          for (int k = 0; k < C::BN / 32; ++k) {
            const int base = 32 * k;
            const uint32_t cw = lim >= base + 31 ? ~0u : (lim < base ? 0u : (~0u >> (31 - (lim - base))));
            const uint32_t ww = lo <= base ? ~0u : (lo > base + 31 ? 0u : (~0u << (lo - base)));
            vis[k] = mb[k] & cw & ww;
          }
        }
        if (!wait_warp(c, bar(c, B_S_FULL + 2 * t + sbuf), (cnt / C::NS) & 1, 21)) { ok = false; break; }
        tc_fence_after();
        const uint32_t sa = t_lane + C::tm_s(t, sbuf);

        // Blocks wholly visible to every valid row of the warp skip the
        // per-column mask (same values for those rows, fewer instructions).
        // Rows that are not valid (before the first q row of an extend, past
        // the tile's end) are never written out; on the whole-block path they
        // compute on whatever scores their q rows give, which touches no other
        // row (each row of P V depends only on that row of P) and never asks
        // for a rescale.  A warp with no visible column in this block skips
        // the arithmetic but still stores P = 0: its rows may be valid rows
        // past whose position the block lies, and their O keeps accumulating
        // P V.
        bool whole, live;
        if constexpr (MK == 2) {
          uint32_t a = ~0u, o = 0u;
#pragma unroll
          for (int k = 0; k < C::BN / 32; ++k) {
            a &= vis[k];
            o |= vis[k];
          }
          whole = __all_sync(0xffffffffu, !valid || a == ~0u);
          live = __any_sync(0xffffffffu, o != 0u);  // the mask may leave a warp no column at all
        } else {
          whole = __all_sync(0xffffffffu, !valid || (lim >= C::BN - 1 && (MK == 0 || lo <= 0)));
          live = __any_sync(0xffffffffu, lim >= 0 && (MK == 0 || lo < C::BN));
        }
        // column j visible (blocks that are not whole)
        auto seen = [&](int j) -> bool {
          if constexpr (MK == 2) return (vis[j >> 5] >> (j & 31)) & 1u;
          else return col_visible<MK>(j, lim, lo, mb);
        };

        // Block max: one TMEM round trip for the whole S row in the bf16
        // two-slot kernel and under custom masks, one per 64-column half
        // elsewhere; a 128-column row is then reread in halves for the
        // exponentials instead of being kept live (which spills even at 255
        // registers a thread).
        constexpr bool kHalves = C::BN == 128;
        constexpr int HW = kHalves ? C::BN / 2 : C::BN;  // columns per exp pass
        float mx = -INFINITY;
        uint32_t sv[C::BN];
        // eight independent partial maxima over column pairs (max is exact in
        // any order); masked columns enter as -inf.  Whole blocks and masked
        // blocks get separately compiled loops.
        // Blocks that are not whole: all kernels but the bf16 two-slot kernel
        // without a custom mask set the hidden columns of S to -inf first
        // (below) and then run the unmasked loops; that kernel (224 registers
        // a thread, where the fold measured 1 % slower) keeps masked copies of
        // the loops.
        constexpr bool kFold = MK == 2 || KV8 || NT == 1 || NARROW_LD;
        auto block_max = [&](auto whole_c) {
          constexpr bool kWhole = decltype(whole_c)::value;
          float m8[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll
          for (int j = 0; j < C::BN; j += 2) {
            float a = __uint_as_float(sv[j]), b = __uint_as_float(sv[j + 1]);
            if (!kWhole) {
              a = seen(j) ? a : -INFINITY;
              b = seen(j + 1) ? b : -INFINITY;
            }
            m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], a, b);
          }
          return fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
        };
        if constexpr (MK != 2 && kHalves && ((NARROW_LD && NT == 2) || NT == 1)) {
          // The one-slot kernels and the two-slot kernel of 128 registers a
          // thread (E4M3 pages), without a custom mask: 64 columns at a time
          // (a loop, not unrolled) into the same eight partial maxima, which
          // keeps 64 fewer registers live and the code smaller (measured 1-4 %
          // faster there; 6 % slower in the bf16 two-slot kernel).
          if (live) {
            float m8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) m8[k] = -INFINITY;
#pragma unroll 1
            for (int h = 0; h < 2; ++h) {
              tmem_ld_x64(sa + h * 64, *reinterpret_cast<uint32_t(*)[64]>(sv));
              if (!whole) {  // hidden columns become -inf in S itself (see below)
#pragma unroll
                for (int j = 0; j < 64; ++j) sv[j] = seen(h * 64 + j) ? sv[j] : 0xff800000u;
                tmem_st_x64(sa + h * 64, sv);
              }
#pragma unroll
              for (int j = 0; j < 64; j += 2)
                m8[(j >> 1) & 7] = fmax3(m8[(j >> 1) & 7], __uint_as_float(sv[j]), __uint_as_float(sv[j + 1]));
            }
            mx = fmax3(fmax3(m8[0], m8[1], m8[2]), fmax3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
          }
        } else if (live) {
          if constexpr (C::BN == 128 && !NARROW_LD) {
            tmem_ld_x128(sa, sv);
          } else if constexpr (C::BN == 128) {  // launches of 128 registers a thread: no 128-wide load
            tmem_ld_x64(sa, *reinterpret_cast<uint32_t(*)[64]>(sv));
            tmem_ld_x64(sa + 64, *reinterpret_cast<uint32_t(*)[64]>(sv + 64));
          } else {
            tmem_ld_x64(sa, sv);
          }
          // A block that is not whole for the warp: hidden columns become
          // -inf in S itself (written back to TMEM), so the max and
          // exponential passes run one unmasked loop each: one visibility
          // test per column instead of two, and no masked copies of the
          // loops.  2^(-inf) is exactly the zero a masked loop substitutes.
          if constexpr (kFold) {
            if (!whole) {
#pragma unroll
              for (int j = 0; j < C::BN; ++j) sv[j] = seen(j) ? sv[j] : 0xff800000u;
              if constexpr (C::BN == 128) {
                tmem_st_x64(sa, sv);
                tmem_st_x64(sa + 64, sv + 64);
              } else {
                tmem_st_x64(sa, sv);
              }
            }
            mx = block_max(std::true_type{});
          } else {
            mx = whole ? block_max(std::true_type{}) : block_max(std::false_type{});
          }
        }
        float alpha = 1.f;
        if (mx != -INFINITY) {
          if (m == -INFINITY) {
            m = mx;  // first visible block of the segment: O starts fresh
          } else {
            const float ms_old = __fmul_rn(m, scale), ms_new = __fmul_rn(mx, scale);
            if (__fsub_rn(ms_new, ms_old) > kLazyRescale) {
              alpha = ex2(__fsub_rn(ms_old, ms_new));
              m = mx;
            }
          }
        }
        const float ms = (m == -INFINITY) ? 0.f : __fmul_rn(m, scale);

        // O must be rescaled (rarely) where the running max moved: a warp that
        // has to publishes its first half of P (HALF_P) only after the
        // rescale.
        bool rescale = false;
        if constexpr (C::HALF_P) rescale = !seg_first && __any_sync(0xffffffffu, valid && alpha != 1.f);

        // Probabilities, the row sum and P (bf16 pairs, packed in place)
        // written back over the S columns already read; 2^x on MUFU.  Hidden
        // columns hold -inf (or, in the masked loops, are computed and then
        // replaced), so their probabilities are exact zeros, which add
        // nothing to the row sum: a row gets the same bits either way.
        // Row-sum partials: acc[i] holds columns 2i, 2i + 1 (mod 8), each
        // pair summed with one packed add (four chains, so that the adds do
        // not wait on each other); they are combined pairwise at the end.
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        const uint64_t sc2 = f2_splat(scale), nm2 = f2_splat(-ms);
        // One loop body for both halves, not unrolled: half the code, measured
        // faster (the softmax's instruction footprint).  Unrolled under a
        // custom mask (its visibility words are indexed by column) and in the
        // bf16 row-gather kernel (measured 4 % slower looped).
#pragma unroll ((MK == 2 || (NARROW_LD && !KV8)) ? C::BN / HW : 1)
        for (int h = 0; h < C::BN / HW; ++h) {
          uint32_t* hv = kHalves ? sv : sv + h * HW;
          if (live) {
            if constexpr (kHalves) tmem_ld_x64(sa + h * HW, *reinterpret_cast<uint32_t(*)[64]>(hv));
            auto exp_pass = [&](auto whole_c) {
              constexpr bool kWhole = decltype(whole_c)::value;
#pragma unroll
              for (int j = 0; j < HW; j += 2) {
                const int cu = h * HW + j;
                const uint64_t x =
                    ffma2(f2_bits(__uint_as_float(hv[j]), __uint_as_float(hv[j + 1])), sc2, nm2);
                const int pair = (cu >> 1) & 7;
                uint64_t e = f2_bits(ex2(f2_lo(x)), ex2(f2_hi(x)));
                if (!kWhole)
                  e = f2_bits(seen(cu) ? f2_lo(e) : 0.f, seen(cu + 1) ? f2_hi(e) : 0.f);
                acc[pair & 3] = fadd2(acc[pair & 3], e);
                hv[j / 2] = KV8 ? pack_f16x2(f2_lo(e), f2_hi(e)) : pack_bf16x2(f2_lo(e), f2_hi(e));
              }
            };
            if constexpr (kFold) {
              exp_pass(std::true_type{});
            } else {
              if (whole) exp_pass(std::true_type{});
              else exp_pass(std::false_type{});
            }
          } else {
#pragma unroll
            for (int k = 0; k < HW / 2; ++k) hv[k] = 0u;
          }
          if constexpr (HW == 128) tmem_st_x64(sa, hv);
          else tmem_st_x32_p(sa + h * (HW / 2), hv);
          if (C::HALF_P && h == 0 && !rescale) {  // the first half of P is out: its PV may start
            tc_fence_before();
            mbar_arrive(bar(c, B_P_HALF + 2 * t + sbuf));
          }
        }
        if (valid) {
          const uint64_t a = fadd2(fadd2(acc[0], acc[1]), fadd2(acc[2], acc[3]));
          const float rowsum = __fadd_rn(f2_lo(a), f2_hi(a));
          l = __fadd_rn(__fmul_rn(l, alpha), rowsum);
        }
        // Rescale O where the running max moved (alpha is exactly 1 elsewhere);
        // the first block of a segment overwrites O instead.  With one S
        // buffer the S_FULL phase already implies the previous PV completed.
        if constexpr (!C::HALF_P) rescale = !seg_first && __any_sync(0xffffffffu, valid && alpha != 1.f);
        if (rescale) {
          if (C::NS == 2 && !wait_pv(cnt - 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t ov[32];
            tmem_ld_x32(o_addr + c0, ov);
#pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__fmul_rn(__uint_as_float(ov[j]), alpha));
            tmem_st_x32(o_addr + c0, ov);
          }
        }
        tc_fence_before();
        if (C::HALF_P && rescale) mbar_arrive(bar(c, B_P_HALF + 2 * t + sbuf));
        mbar_arrive(bar(c, B_P_FULL + 2 * t + sbuf));
      }
      if (!ok) break;

      // ---- segment end: O of this segment is complete after the last PV
      if (!wait_pv(cnt - 1)) { ok = false; break; }
      tc_fence_after();
      const float m_seg = (m == -INFINITY) ? -INFINITY : __fmul_rn(m, scale);
      const int vr = (pos - g.first_valid[t]) * p.group + hg;  // row among the tile's valid rows
      if (split) {
        const bool write = valid && s < w.nseg[t];
        float* prow = p.partials + (size_t(w.part_base[t]) + vr) * (D + 4);
        if (write) *reinterpret_cast<float4*>(prow) = make_float4(m_seg, l, 0.f, 0.f);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_x32(o_addr + c0, ov);
          if (write) {
            float4* dst = reinterpret_cast<float4*>(prow + 4 + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_float4(__uint_as_float(ov[4 * j]), __uint_as_float(ov[4 * j + 1]),
                                   __uint_as_float(ov[4 * j + 2]), __uint_as_float(ov[4 * j + 3]));
          }
        }
      } else {
        const MergeStep st = merge_step(Mrun, Lrun, m_seg, l);
        const bool last = (s == w.seg_hi);
        const bool use_scratch = (w.seg_hi > w.seg_lo);
        // A row with no visible key at all (possible only under a custom
        // mask) is written as zeros, with lse = -inf.
        const bool empty = MK == 2 && st.m == -INFINITY;
        const float osc = (last && !empty) ? out_scale(st.l, p.v_scale) : 0.f;
        const int tok = w.q_tok0 + pos;
        const int head = w.kv_head * p.group + hg;
        uint16_t* orow = p.out + (size_t(tok) * p.num_qo_heads + head) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_x32(o_addr + c0, ov);
          if (valid) {
            float o[32];
            if (use_scratch && st.kind != 1) {
              const float4* src = scratch_row + (c0 / 4) * kTileRows;
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 v = src[j * kTileRows];
                o[4 * j] = v.x; o[4 * j + 1] = v.y; o[4 * j + 2] = v.z; o[4 * j + 3] = v.w;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = merge_elem(st, o[j], __uint_as_float(ov[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(ov[j]);
            }
            if (empty) {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = 0.f;
            }
            if (!last) {
              float4* dst = scratch_row + (c0 / 4) * kTileRows;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j * kTileRows] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
              uint4 packed[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                packed[j] = make_uint4(pack_bf16x2(__fmul_rn(o[8 * j + 0], osc), __fmul_rn(o[8 * j + 1], osc)),
                                       pack_bf16x2(__fmul_rn(o[8 * j + 2], osc), __fmul_rn(o[8 * j + 3], osc)),
                                       pack_bf16x2(__fmul_rn(o[8 * j + 4], osc), __fmul_rn(o[8 * j + 5], osc)),
                                       pack_bf16x2(__fmul_rn(o[8 * j + 6], osc), __fmul_rn(o[8 * j + 7], osc)));
              if constexpr (C::OUT_STAGE && MK == 2) {
                // 16-byte piece u of this row's 64-column half at the
                // row's 128 bytes, pieces XOR-swizzled by the row
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const int u = ((c0 & 32) >> 3) + j;
                  st_shared_v4(ostage + lane * 128 + ((u ^ (lane & 7)) << 4), packed[j]);
                }
              } else {
                uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
                for (int j = 0; j < 4; ++j) dst[j] = packed[j];
              }
            }
          }
          if constexpr (C::OUT_STAGE && MK == 2) {
            if (last && (c0 & 32)) {
              // the warp's 32 rows x 64 columns are staged: store them as
              // 4 rows (whole lines) per instruction, valid rows only
              __syncwarp();
              const uint64_t my_row = reinterpret_cast<uint64_t>(orow + (c0 - 32));
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const int r = 4 * i + (lane >> 3), u = lane & 7;
                const uint64_t base = __shfl_sync(0xffffffffu, my_row, r);
                const bool rv = __shfl_sync(0xffffffffu, valid, r);
                const uint4 v = ld_shared_v4(ostage + r * 128 + ((u ^ (r & 7)) << 4));
                if (rv) reinterpret_cast<uint4*>(base)[u] = v;
              }
              __syncwarp();
            }
          }
        }
        if (last && valid) p.lse[size_t(tok) * p.num_qo_heads + head] = final_lse(st.m, st.l);
        Mrun = st.m;
        Lrun = st.l;
      }
      tc_fence_before();
    }
  }
}

// Four E4M3 codes (the bytes of w, lowest first) -> four f16 (two pairs,
// lo: bytes 0 and 1, hi: bytes 2 and 3, low half first), one conversion
// instruction per pair, each reading a 16-bit half of w's register in place
// (no shift or mask to isolate the pair: measured 6-23 % faster kernels than
// the same conversions on separately extracted halves).  Exact: every E4M3
// value, subnormals included, is an f16 normal number or zero; the NaN codes
// give NaN.
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 c01, c23;\n\t"
      "mov.b32 {c01, c23}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c01;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, c23;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// FP8 pages: the q tile (bf16, 128-byte swizzled rows of 64-column chunks)
// becomes f16 in place, thread `row` taking one packed row.  The row is
// multiplied by 2^e, e = 141 - (biased exponent of its largest magnitude),
// clamped to [-64, 64], so that its largest value lands in [2^14, 2^15):
// every bf16 value within 2^29 of the row's largest is then exact in f16
// (8 significant bits, inside f16's normal range), smaller ones round to
// f16's subnormal grid, which holds them to 2^-39 of the row's largest.
// e goes to `qscale[row]`; the softmax multiplies its logit scale by 2^-e.
// A row of zeros (or NaN/inf) keeps e at a clamp end.
template <int D>
__device__ __forceinline__ void q_tile_to_f16(uint32_t sQ, int row, int8_t* qscale) {
  constexpr int DCH = D / 64;
  const uint32_t rbase = sQ + row * 128;
  // Units are visited at their swizzled positions (u ^ row % 8), so that the
  // eight rows of a quarter-warp touch eight different bank groups.
  uint32_t mx = 0;  // largest |q| as bf16 magnitude bits, in both halves
#pragma unroll 1
  for (int ch = 0; ch < DCH; ++ch)
#pragma unroll 4
    for (int u = 0; u < 8; ++u) {
      uint32_t w[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(rbase + ch * kTileRows * 128 + ((u ^ (row & 7)) << 4))
                   : "memory");
#pragma unroll
      for (int j = 0; j < 4; ++j) asm("max.u16x2 %0, %0, %1;" : "+r"(mx) : "r"(w[j] & 0x7FFF7FFFu));
    }
  const uint32_t m16 = max(mx & 0xFFFFu, mx >> 16);  // bf16 bits: exponent field at [7, 15)
  const int e = min(64, max(-64, 141 - int(m16 >> 7)));
  qscale[row] = int8_t(e);
  const uint64_t s2 = f2_splat(__int_as_float((127 + e) << 23));
#pragma unroll 1
  for (int ch = 0; ch < DCH; ++ch)
#pragma unroll 4
    for (int u = 0; u < 8; ++u) {
      const uint32_t a = rbase + ch * kTileRows * 128 + ((u ^ (row & 7)) << 4);
      uint32_t w[4];
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                   : "r"(a)
                   : "memory");
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint64_t x = fmul2(f2_bits(__uint_as_float(w[j] << 16), __uint_as_float(w[j] & 0xFFFF0000u)), s2);
        w[j] = pack_f16x2(f2_lo(x), f2_hi(x));
      }
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
                   : "memory");
    }
}

// FP8 pages (with NWG = 2 warpgroups, wg 0 converts the K blocks and wg 1
// the V blocks; with one, it converts K then V of every block; NWG is the
// launching kernel's count, passed explicitly): convert each staged block
// (BN rows x D codes, row-major) into the f16, 128-byte-swizzled K/V ring
// slot the MMAs read; V rows at or past kv_len are written as zeros.  The
// staging stage is released once the codes are in registers; the ring slot
// is taken once the MMA that last read it has completed.
template <int D, int NT, int ST, bool KV8, int NWG>
__device__ void dequant_role(const Ctx& c, uint32_t sbase, const AttnParams& p, const int wg, int8_t* qscale) {
  if constexpr (KV8) {
    using C = Cfg<D, NT, ST, KV8>;
    const int tid = (int(threadIdx.x) - C::DQ_WARP0 * 32) & 127;  // 0..127 within the warpgroup
    uint32_t b = 0, n = 0;  // blocks / items started by this CTA
    bool ok = true;
    for (int it = blockIdx.x; it < item_count(p) && ok; it += gridDim.x, ++n) {
      const WorkItem w = p.items[it];
      const Geom g = geom_of<NT, C::BN>(w, p.tile_pos);
      // Warpgroup 0 turns each item's q tile into f16 (thread = packed row)
      // once it has landed and the softmax has read the previous tile's row
      // scales; the tile is ready for the MMAs after the proxy fence.
      if (wg == 0) {
        if (n > 0 && !wait_warp(c, bar(c, B_QS_FREE), (n - 1) & 1, 34)) { ok = false; break; }
        if (!wait_warp(c, bar(c, B_Q_FULL), n & 1, 35)) { ok = false; break; }
#pragma unroll
        for (int t = 0; t < NT; ++t) q_tile_to_f16<D>(sbase + C::OFF_Q + t * C::Q_BYTES, tid, qscale + t * kTileRows);
        fence_proxy_async_smem();
        mbar_arrive(bar(c, B_Q_READY));
      }
      for (int blk = g.blk_lo; blk <= g.blk_hi && ok; ++blk, ++b) {
        const int ss = b % C::SS, slot = b % ST;
        const uint32_t suse = b / C::SS, use = b / ST;
        const int valid_rows = w.kv_len - blk * C::BN;
#pragma unroll 1
        for (int which = NWG == 2 ? wg : 0; which < (NWG == 2 ? wg + 1 : 2); ++which) {
          const int full8 = which ? B_V8_FULL : B_K8_FULL, free8 = which ? B_V8_FREE : B_K8_FREE;
          const int full = which ? B_V_FULL : B_K_FULL, freeb = which ? B_V_FREE : B_K_FREE;
          if (!wait_warp(c, bar(c, full8 + ss), suse & 1, 30 + which)) { ok = false; break; }
          const uint32_t src = sbase + (which ? C::OFF_V8 : C::OFF_K8) + ss * C::KV8_BYTES;
          const uint32_t dst = sbase + (which ? C::OFF_V : C::OFF_K) + slot * C::KV_BYTES;
          // Thread unit: 8 codes (8 staged bytes) -> one 16-byte f16 unit.
          // Unit u of a block is row u / UPR, unit ui = u % UPR of the row;
          // 16 consecutive lanes read a 128-byte staged run (conflict-free
          // 8-byte loads) and each quarter-warp stores the 8 units of one
          // 64-column chunk row, which the 128-byte swizzle spreads over all
          // eight 16-byte bank groups (conflict-free stores).  All of this
          // thread's staged units are loaded before any is converted: each
          // load and store is an ordered asm statement, so a
          // load-convert-store loop would pay the shared-memory latency once
          // per unit.
          constexpr int UPR = D / 8;                     // f16 units (8 codes) per row
          constexpr int ITER = C::BN * UPR / 128;
          constexpr int RSTEP = 128 / UPR;               // rows between a thread's units
          static_assert(128 % UPR == 0 && C::BN % RSTEP == 0, "whole units per thread");
          const int r0 = tid / UPR, ui = tid % UPR;
          const uint32_t src0 = src + r0 * D + ui * 8;
          uint32_t raw[ITER][2];
#pragma unroll
          for (int k = 0; k < ITER; ++k)
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];"
                         : "=r"(raw[k][0]), "=r"(raw[k][1])
                         : "r"(src0 + k * RSTEP * D)
                         : "memory");
          // The staged codes are in registers: the stage may take the next
          // load while this block waits for its bf16 slot.  The next load is
          // an async-proxy (TMA or cp.async) write, so a proxy fence orders
          // the generic-proxy reads above before the arrival releases the
          // stage to it.
          fence_proxy_async_smem();
          mbar_arrive(bar(c, free8 + ss));
          if (use > 0 && !wait_warp(c, bar(c, freeb + slot), (use - 1) & 1, 32 + which)) { ok = false; break; }
          const int ch = ui >> 3, pos = ui & 7;
          const uint32_t dst0 = dst + ch * C::KV_CHUNK + r0 * 128;
#pragma unroll
          for (int k = 0; k < ITER; ++k) {
            const int r = r0 + k * RSTEP;
            uint32_t o[4];
#pragma unroll
            for (int j = 0; j < 2; ++j) e4m3x4_to_f16x4(raw[k][j], o[2 * j], o[2 * j + 1]);
            if (which == 1 && r >= valid_rows) {
#pragma unroll
              for (int j = 0; j < 4; ++j) o[j] = 0u;
            }
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         ::"r"(dst0 + k * RSTEP * 128 + ((pos ^ (r & 7)) << 4)), "r"(o[0]), "r"(o[1]), "r"(o[2]),
                         "r"(o[3])
                         : "memory");
          }
          fence_proxy_async_smem();
          mbar_arrive(bar(c, full + slot));
        }
      }
    }
  }
}

template <int D, int NT, int ST, bool KV8, int MK, bool GATHER>
__global__ void __launch_bounds__(Cfg<D, NT, ST, KV8, GATHER>::THREADS, 1)
    bip_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D, NT, ST, KV8, GATHER>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw + pad;
  const int warp = threadIdx.x >> 5;

  Ctx c;
  c.bar0 = sbase + C::OFF_BAR;
  c.abort = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_BAR + OFF_ABORT);
  c.header = p.header;
  c.limit_cycles = p.wait_limit_cycles;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + OFF_TMEM_SLOT);
  int8_t* qscale = reinterpret_cast<int8_t*>(smem + C::OFF_BAR + OFF_QSCALE);

  if (threadIdx.x == 0) {
    mbar_init(bar(c, B_Q_FULL), 1);
    mbar_init(bar(c, B_Q_FREE), 1);
    // Landing barriers: one arrival (the TMA byte count completes the
    // phase), or one per gather lane of the stream when token rows are
    // gathered with cp.async; FP8 bf16 slots: one per dequant thread.
    constexpr uint32_t land = GATHER ? 32u * C::GW : 1u;
    for (int s = 0; s < ST; ++s) {
      mbar_init(bar(c, B_K_FULL + s), KV8 ? 128u : land);
      mbar_init(bar(c, B_K_FREE + s), 1);
      mbar_init(bar(c, B_V_FULL + s), KV8 ? 128u : land);
      mbar_init(bar(c, B_V_FREE + s), 1);
    }
    for (int s = 0; s < C::SS; ++s) {
      mbar_init(bar(c, B_K8_FULL + s), land);
      mbar_init(bar(c, B_K8_FREE + s), 128);
      mbar_init(bar(c, B_V8_FULL + s), land);
      mbar_init(bar(c, B_V8_FREE + s), 128);
    }
    for (int t = 0; t < NT; ++t)
      for (int s = 0; s < C::NS; ++s) {
        mbar_init(bar(c, B_S_FULL + 2 * t + s), 1);
        mbar_init(bar(c, B_P_FULL + 2 * t + s), 128);
        mbar_init(bar(c, B_P_HALF + 2 * t + s), 128);
        mbar_init(bar(c, B_O_DONE + 2 * t + s), 1);
      }
    mbar_init(bar(c, B_DRAIN), 1);
    mbar_init(bar(c, B_V_TX), 1);
    mbar_init(bar(c, B_Q_READY), 128);             // one dequant warpgroup
    mbar_init(bar(c, B_QS_FREE), 32 * C::SM_WARPS);  // every softmax thread
    *c.abort = 0u;
    fence_mbar_init();
  }
  if (warp == C::CTL_WARP0 + 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  const int lane = threadIdx.x & 31;
  if (warp < C::SM_WARPS) {
    if constexpr (C::SPLIT_REGS) reg_alloc<C::SM_REGS>();
    softmax_role<D, NT, ST, KV8, MK, (C::LAUNCH_REGS < 160)>(c, tmem, p, warp / 4, qscale);
  } else if (warp < C::GA_WARP0) {
    if constexpr (C::DQ_WGS == 2) reg_dealloc<C::DQ_REGS>();
    dequant_role<D, NT, ST, KV8, C::DQ_WGS>(c, sbase, p, (warp - C::DQ_WARP0) / 4, qscale);
  } else if (warp < C::CTL_WARP0) {
    if constexpr (C::GA_WARPS > 0) {
      reg_dealloc<C::GA_REGS>();
      row_gatherer<D, NT, ST, KV8, C::GW>(c, sbase, p, warp - C::GA_WARP0);
    }
  } else {
    if constexpr (C::SPLIT_REGS) reg_dealloc<C::CTL_REGS>();
    // Warp w runs on the scheduler w % 4.  The q/K producer takes the
    // control group's last warp and the spare its first, so that the
    // scheduler of softmax warp 0 (the rows of a short extend, which sit at
    // the start of their tile) has one busy warp fewer.
    const int role = warp - C::CTL_WARP0;
    if (role == 3) {
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        if (!GATHER) prefetch_tmap(&tm_k);
      }
      producer<D, NT, ST, KV8, GATHER>(c, sbase, &tm_q, &tm_k, p, false);
    } else if (role == 1) {
      if (lane == 0) mma_issuer<D, NT, ST, KV8, GATHER>(c, sbase, tmem, p);
    } else if (!GATHER) {
      if (role == 2) {
        if (lane == 0) prefetch_tmap(&tm_v);
        producer<D, NT, ST, KV8, GATHER>(c, sbase, &tm_q, &tm_v, p, true);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::CTL_WARP0 + 1) tmem_dealloc(tmem, C::TM_COLS);
}

// Each mask kind is a separate instantiation, so that the plain causal
// kernel carries none of the window or custom-mask arithmetic; so is the row
// gather of token-granular pages.
template <int D, int NT, int ST, bool KV8, int MK, bool GATHER>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                       int grid, cudaStream_t stream) {
  using C = Cfg<D, NT, ST, KV8, GATHER>;
  constexpr int smem = (MK == 2 && C::OUT_STAGE) ? C::SMEM_OSTG : C::SMEM;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bip_attn_kernel<D, NT, ST, KV8, MK, GATHER>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  bip_attn_kernel<D, NT, ST, KV8, MK, GATHER><<<grid, C::THREADS, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

template <int D, int NT, int ST, bool KV8, bool GATHER>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                   int grid, cudaStream_t stream) {
  return p.window_left > 0 ? launch_one<D, NT, ST, KV8, 1, GATHER>(tq, tk, tv, p, grid, stream)
                           : launch_one<D, NT, ST, KV8, 0, GATHER>(tq, tk, tv, p, grid, stream);
}

}  // namespace
}  // namespace bip
