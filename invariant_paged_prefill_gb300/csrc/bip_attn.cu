// Persistent paged prefill attention for sm_103a: TMA page loads, tcgen05
// MMAs with TMEM accumulators, an fp32 online softmax with one thread per
// row, and a fixed-order segment merge.
//
// One CTA (192 threads, one per SM) walks work items (a request x KV head
// x absolute q tile, over some of its 4096-key segments):
//   warp 0      TMA producer: the q tile once per item, then K and V blocks
//               page by page through a 2-deep ring of each.
//   warp 1      tcgen05 issuer: S = Q K^T into one of two TMEM S buffers,
//               O += P V into the TMEM O accumulator; zeroes V rows past
//               kv_len before they enter a product.
//   warps 2-5   softmax: thread i owns packed row i (TMEM lane i); masks,
//               keeps m and l, writes P (bf16) to shared memory, rescales
//               O, and at each segment end folds or writes the segment.
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

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bip_internal.h"
#include "bip_numerics.cuh"
#include "bip_ptx.cuh"

namespace bip {
namespace {

template <int D>
struct Cfg {
  static constexpr int BN = kv_block_for(D);        // keys per block
  static constexpr int DCH = D / 64;                // 64-column (128-byte) chunks of a d-row
  static constexpr int Q_CHUNK = kTileRows * 128;   // bytes of one q chunk (128 rows)
  static constexpr int Q_BYTES = DCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;         // bytes of one K/V chunk (BN rows)
  static constexpr int KV_BYTES = DCH * KV_CHUNK;   // one K or V block
  static constexpr int PCH = BN / 64;               // chunks of a P row
  static constexpr int P_BYTES = PCH * Q_CHUNK;
  static constexpr int STAGES = 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + Q_BYTES;
  static constexpr int OFF_V = OFF_K + STAGES * KV_BYTES;
  static constexpr int OFF_P = OFF_V + STAGES * KV_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int SMEM = OFF_BAR + 256 + 1024;  // + room to align the base to 1024
  static constexpr int TM_S = 0;                     // S buffers: columns [0, BN) and [BN, 2 BN)
  static constexpr int TM_O = 256;                   // O accumulator: columns [256, 256 + D)
  static constexpr int TM_COLS = 512;
  static constexpr int BPS = kSplitLen / BN;         // blocks per segment
  static_assert(2 * BN <= TM_O && TM_O + D <= TM_COLS, "TMEM budget");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
};

// Barrier slots (8 bytes each) at OFF_BAR.
enum Bar {
  B_Q_FULL = 0, B_Q_FREE = 1, B_K_FULL = 2, B_K_FREE = 4, B_V_FULL = 6, B_V_FREE = 8,
  B_S_FULL = 10, B_S_FREE = 12, B_P_FULL = 14, B_O_DONE = 15, B_DRAIN = 16, B_COUNT = 17
};
constexpr int OFF_TMEM_SLOT = 8 * B_COUNT;    // u32: TMEM base address
constexpr int OFF_ABORT = OFF_TMEM_SLOT + 4;  // u32: a wait expired somewhere in this CTA

constexpr int kThreads = 192;

struct Ctx {
  uint32_t bar0;
  volatile uint32_t* abort;
  WsHeader* header;
  uint64_t limit_ns;
};

__device__ __forceinline__ uint32_t bar(const Ctx& c, int i) { return c.bar0 + 8u * i; }

// Bounded wait on an mbarrier phase.  On expiry the CTA is marked aborted,
// the workspace status records a timeout, and false is returned; any wait
// that sees the abort mark also returns false.
__device__ __noinline__ bool wait_phase(const Ctx& c, uint32_t b, uint32_t parity, uint32_t where) {
  if (mbar_test(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    for (int i = 0; i < 32; ++i)
      if (mbar_test(b, parity)) return true;
    if (*c.abort) return false;
    if (globaltimer_ns() - t0 > c.limit_ns) {
      *c.abort = 1u;
      atomicCAS(&c.header->status, 0u, 5u /* BIP_ERR_DEVICE_TIMEOUT */);
      atomicExch(&c.header->where, where);
      return false;
    }
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
  int kv_len, tile_start, tile_end, first_valid;
  int blk_lo, blk_hi;  // inclusive block range of the item
};

template <int D>
__device__ __forceinline__ Geom geom_of(const WorkItem& w, int T) {
  using C = Cfg<D>;
  Geom g;
  g.kv_len = w.kv_len;
  g.tile_start = w.tile * T;
  g.tile_end = min(g.tile_start + T - 1, w.kv_len - 1);
  g.first_valid = max(g.tile_start, w.q_lo);
  g.blk_lo = w.seg_lo * C::BPS;
  g.blk_hi = min((int(w.seg_hi) + 1) * kSplitLen - 1, g.tile_end) / C::BN;
  return g;
}

// ------------------------------------------------------------------ roles

template <int D>
__device__ void producer(const Ctx& c, uint32_t sbase, const CUtensorMap* tq, const CUtensorMap* tk,
                         const CUtensorMap* tv, const AttnParams& p) {
  using C = Cfg<D>;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const int pages_per_blk = C::BN / p.page_size;
  uint32_t b = 0;  // blocks started by this CTA
  int n = 0;       // items started by this CTA
  uint32_t k_issued[2] = {0u, 0u}, v_issued[2] = {0u, 0u}, q_issued = 0u;  // loads per barrier
  for (int it = blockIdx.x; it < p.n_items; it += gridDim.x, ++n) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<D>(w, p.tile_pos);
    if (n > 0 && !wait_phase(c, bar(c, B_Q_FREE), (n - 1) & 1, 1)) break;
    mbar_arrive_expect_tx(bar(c, B_Q_FULL), uint32_t(C::DCH * 128 * p.group * p.tile_pos));
    ++q_issued;
    for (int ch = 0; ch < C::DCH; ++ch)
      tma_load_3d(sQ + ch * C::Q_CHUNK, tq, bar(c, B_Q_FULL), ch * 64, w.kv_head * p.group,
                  w.q_tok0 + g.tile_start);
    const int npages_req = (w.kv_len + p.page_size - 1) / p.page_size;
    bool ok = true;
    for (int blk = g.blk_lo; blk <= g.blk_hi && ok; ++blk, ++b) {
      const int slot = b & 1;
      const uint32_t use = b >> 1;
      const int p0 = blk * pages_per_blk;
      const int p1 = min(p0 + pages_per_blk, npages_req);
      int ids[C::BN / 8];
#pragma unroll
      for (int i = 0; i < C::BN / 8; ++i) {
        int id = 0;
        if (i < p1 - p0) {
          id = __ldg(p.kv_indices + w.page_base + p0 + i);
          if (id < 0 || id >= p.num_pages) {
            atomicAdd(&c.header->bad_pages, 1u);
            id = 0;
          }
        }
        ids[i] = id;
      }
      const uint32_t bytes = uint32_t((p1 - p0) * p.page_size * D * 2);
      // K block
      if (use > 0 && !wait_phase(c, bar(c, B_K_FREE + slot), (use - 1) & 1, 2)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(c, B_K_FULL + slot), bytes);
      ++k_issued[slot];
      for (int i = 0; i < p1 - p0; ++i)
        for (int ch = 0; ch < C::DCH; ++ch)
          tma_load_4d(sK + slot * C::KV_BYTES + ch * C::KV_CHUNK + i * p.page_size * 128, tk,
                      bar(c, B_K_FULL + slot), ch * 64, w.kv_head, 0, ids[i]);
      // V block
      if (use > 0 && !wait_phase(c, bar(c, B_V_FREE + slot), (use - 1) & 1, 3)) { ok = false; break; }
      mbar_arrive_expect_tx(bar(c, B_V_FULL + slot), bytes);
      ++v_issued[slot];
      for (int i = 0; i < p1 - p0; ++i)
        for (int ch = 0; ch < C::DCH; ++ch)
          tma_load_4d(sV + slot * C::KV_BYTES + ch * C::KV_CHUNK + i * p.page_size * 128, tv,
                      bar(c, B_V_FULL + slot), ch * 64, w.kv_head, 0, ids[i]);
    }
    if (!ok) break;
  }
  // Drain: the last load on every barrier must have landed before exit
  // (on the normal path these phases completed long ago).
  if (q_issued) drain_wait(bar(c, B_Q_FULL), (q_issued - 1) & 1);
  for (int slot = 0; slot < 2; ++slot) {
    if (k_issued[slot]) drain_wait(bar(c, B_K_FULL + slot), (k_issued[slot] - 1) & 1);
    if (v_issued[slot]) drain_wait(bar(c, B_V_FULL + slot), (v_issued[slot] - 1) & 1);
  }
}

template <int D>
__device__ void mma_issuer(const Ctx& c, uint32_t sbase, uint32_t tmem, const AttnParams& p) {
  using C = Cfg<D>;
  const int lane = threadIdx.x & 31;
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V, sP = sbase + C::OFF_P;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, C::BN, false, false);  // S = Q K^T, both K-major
  constexpr uint32_t kIdescO = idesc_bf16_f32(128, D, false, true);       // O += P V, V MN-major
  uint32_t b = 0;
  int n = 0;
  bool ok = true;
  for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++n) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<D>(w, p.tile_pos);
    const int nb = g.blk_hi - g.blk_lo + 1;
    if (!wait_warp(c, bar(c, B_Q_FULL), n & 1, 10)) { ok = false; break; }
    tc_fence_after();

    // Issue S for block i of this item (global block counter bb).
    auto issue_s = [&](uint32_t bb, bool last_of_item) -> bool {
      const int slot = bb & 1;
      if (!wait_warp(c, bar(c, B_K_FULL + slot), (bb >> 1) & 1, 11)) return false;
      if (bb >= 2 && !wait_warp(c, bar(c, B_S_FREE + slot), ((bb >> 1) - 1) & 1, 12)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t d_tmem = tmem + C::TM_S + slot * C::BN;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t off_q = (k >> 2) * C::Q_CHUNK + (k & 3) * 32;
          const uint32_t off_k = slot * C::KV_BYTES + (k >> 2) * C::KV_CHUNK + (k & 3) * 32;
          tc_mma_ss(d_tmem, sdesc_sw128(sQ + off_q, 16, 1024), sdesc_sw128(sK + off_k, 16, 1024), kIdescS,
                    k > 0 ? 1u : 0u);
        }
        tc_commit(bar(c, B_S_FULL + slot));
        tc_commit(bar(c, B_K_FREE + slot));
        if (last_of_item) tc_commit(bar(c, B_Q_FREE));
      }
      __syncwarp();
      return true;
    };

    if (!issue_s(b, nb == 1)) { ok = false; break; }
    for (int i = 0; i < nb; ++i) {
      const uint32_t bb = b + i;
      const int blk = g.blk_lo + i;
      const int slot = bb & 1;
      if (i + 1 < nb && !issue_s(bb + 1, i + 2 == nb)) { ok = false; break; }
      if (!wait_warp(c, bar(c, B_P_FULL), bb & 1, 13)) { ok = false; break; }
      if (!wait_warp(c, bar(c, B_V_FULL + slot), (bb >> 1) & 1, 14)) { ok = false; break; }
      tc_fence_after();
      // Rows of V at or past kv_len (the tail of the last page, and pages the
      // request does not have) are zeroed so that p = 0 meets a finite value.
      const int valid_rows = g.kv_len - blk * C::BN;
      if (valid_rows < C::BN) {
        const uint32_t vbase = sV + slot * C::KV_BYTES;
        const int nz = (C::BN - valid_rows) * C::DCH * 8;  // 16-byte units to clear
        for (int u = lane; u < nz; u += 32) {
          const int ch = u / ((C::BN - valid_rows) * 8);
          const int rem = u % ((C::BN - valid_rows) * 8);
          const int row = valid_rows + rem / 8;
          const uint32_t addr = vbase + ch * C::KV_CHUNK + row * 128 + (rem % 8) * 16;
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        const bool first_in_seg = (blk % C::BPS) == 0;
#pragma unroll
        for (int k = 0; k < C::BN / 16; ++k) {
          const uint32_t off_p = (k >> 2) * C::Q_CHUNK + (k & 3) * 32;
          const uint32_t off_v = slot * C::KV_BYTES + k * 16 * 128;
          tc_mma_ss(tmem + C::TM_O, sdesc_sw128(sP + off_p, 16, 1024),
                    sdesc_sw128(sV + off_v, C::KV_CHUNK, 1024), kIdescO, (k > 0 || !first_in_seg) ? 1u : 0u);
        }
        tc_commit(bar(c, B_O_DONE));
        tc_commit(bar(c, B_V_FREE + slot));
      }
      __syncwarp();
    }
    b += nb;
  }
  // Drain: every MMA this thread issued has completed before TMEM is freed.
  if (lane == 0) {
    tc_commit(bar(c, B_DRAIN));
    drain_wait(bar(c, B_DRAIN), 0);
  }
  __syncwarp();
}

template <int D>
__device__ void softmax_role(const Ctx& c, uint32_t sbase, uint32_t tmem, const AttnParams& p) {
  using C = Cfg<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int quarter = warp & 3;          // TMEM lanes this warp may access
  const int row = quarter * 32 + lane;   // packed tile row == TMEM lane
  const uint32_t t_lane = tmem + (uint32_t(quarter * 32) << 16);
  const uint32_t sP = sbase + C::OFF_P;
  const float scale = p.scale_log2;
  uint32_t b = 0, pv_seen = 0;
  int n = 0;
  bool ok = true;

  // PV of global block x has completed (its o_done phase observed).
  auto wait_pv = [&](uint32_t x) -> bool {
    if (pv_seen > x) return true;
    if (!wait_warp(c, bar(c, B_O_DONE), x & 1, 20)) return false;
    pv_seen = x + 1;
    return true;
  };

  for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++n) {
    const WorkItem w = p.items[it];
    const Geom g = geom_of<D>(w, p.tile_pos);
    const int local_pos = row / p.group;
    const int hg = row - local_pos * p.group;
    const int pos = g.tile_start + local_pos;
    const bool valid = row < p.tile_pos * p.group && pos >= g.first_valid && pos <= g.tile_end;
    const bool split = (w.flags & kItemSplit) != 0;
    float Mrun = -INFINITY, Lrun = 0.f;  // merged state of the segments before this one
    float* scratch_row = p.scratch + (size_t(blockIdx.x) * kTileRows + row) * D;

    for (int s = w.seg_lo; s <= w.seg_hi && ok; ++s) {
      const int sb_lo = max(s * C::BPS, g.blk_lo);
      const int sb_hi = min((s + 1) * C::BPS - 1, g.blk_hi);
      float m = -INFINITY, l = 0.f;  // raw-score max and sum over this segment
      for (int blk = sb_lo; blk <= sb_hi; ++blk, ++b) {
        const int slot = b & 1;
        if (!wait_warp(c, bar(c, B_S_FULL + slot), (b >> 1) & 1, 21)) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[C::BN];
        if constexpr (C::BN == 128) tmem_ld_x128(t_lane + C::TM_S + slot * C::BN, sv);
        else tmem_ld_x64(t_lane + C::TM_S + slot * C::BN, sv);
        tc_fence_before();
        mbar_arrive(bar(c, B_S_FREE + slot));

        float alpha = 1.f;
        if (valid) {
          const int lim = pos - blk * C::BN;  // columns 0..lim are visible
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < C::BN; ++j)
            if (j <= lim) mx = fmaxf(mx, __uint_as_float(sv[j]));
          const float m_new = fmaxf(m, mx);
          if (m_new != -INFINITY) {
            const float ms = __fmul_rn(m_new, scale);
            if (m_new != m) alpha = ex2(__fsub_rn(__fmul_rn(m, scale), ms));  // m = -inf gives 0
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int j = 0; j < C::BN; ++j) {
              const float pj = (j <= lim) ? ex2(__fmaf_rn(__uint_as_float(sv[j]), scale, -ms)) : 0.f;
              acc[j & 3] = __fadd_rn(acc[j & 3], pj);
              sv[j] = __float_as_uint(pj);
            }
            const float rowsum = __fadd_rn(__fadd_rn(acc[0], acc[1]), __fadd_rn(acc[2], acc[3]));
            l = __fadd_rn(__fmul_rn(l, alpha), rowsum);
            m = m_new;
          } else {
#pragma unroll
            for (int j = 0; j < C::BN; ++j) sv[j] = 0u;
          }
        }
        // P buffer and O are free once PV of the previous block completed.
        if (b > 0 && !wait_pv(b - 1)) { ok = false; break; }
        tc_fence_after();
        if ((blk % C::BPS) != 0) {  // the first block of a segment overwrites O instead
          // Rescale O where the running max moved (alpha is exactly 1 elsewhere).
          if (__any_sync(0xffffffffu, valid && alpha != 1.f)) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 32) {
              uint32_t ov[32];
              tmem_ld_x32(t_lane + C::TM_O + c0, ov);
#pragma unroll
              for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__fmul_rn(__uint_as_float(ov[j]), alpha));
              tmem_st_x32(t_lane + C::TM_O + c0, ov);
            }
          }
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < C::BN / 8; ++u) {
            const uint32_t w0 = pack_bf16x2(__uint_as_float(sv[8 * u + 0]), __uint_as_float(sv[8 * u + 1]));
            const uint32_t w1 = pack_bf16x2(__uint_as_float(sv[8 * u + 2]), __uint_as_float(sv[8 * u + 3]));
            const uint32_t w2 = pack_bf16x2(__uint_as_float(sv[8 * u + 4]), __uint_as_float(sv[8 * u + 5]));
            const uint32_t w3 = pack_bf16x2(__uint_as_float(sv[8 * u + 6]), __uint_as_float(sv[8 * u + 7]));
            const uint32_t addr = sP + (u >> 3) * C::Q_CHUNK + row * 128 + (((u & 7) ^ (row & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w0), "r"(w1), "r"(w2),
                         "r"(w3)
                         : "memory");
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(c, B_P_FULL));
      }
      if (!ok) break;

      // ---- segment end: O of this segment is complete after the last PV
      if (!wait_pv(b - 1)) { ok = false; break; }
      tc_fence_after();
      const float m_seg = (m == -INFINITY) ? -INFINITY : __fmul_rn(m, scale);
      const int vr = (pos - g.first_valid) * p.group + hg;  // row among the tile's valid rows
      if (split) {
        float* prow = p.partials + (size_t(w.part_base) + vr) * (D + 4);
        if (valid) *reinterpret_cast<float4*>(prow) = make_float4(m_seg, l, 0.f, 0.f);
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_x32(t_lane + C::TM_O + c0, ov);
          if (valid) {
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
        const float osc = last ? out_scale(st.l, p.v_scale) : 0.f;
        const int tok = w.q_tok0 + pos;
        const int head = w.kv_head * p.group + hg;
        uint16_t* orow = p.out + (size_t(tok) * p.num_qo_heads + head) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_x32(t_lane + C::TM_O + c0, ov);
          if (valid) {
            float o[32];
            if (use_scratch && st.kind != 1) {
              const float4* src = reinterpret_cast<const float4*>(scratch_row + c0);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float4 v = src[j];
                o[4 * j] = v.x; o[4 * j + 1] = v.y; o[4 * j + 2] = v.z; o[4 * j + 3] = v.w;
              }
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = merge_elem(st, o[j], __uint_as_float(ov[j]));
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __uint_as_float(ov[j]);
            }
            if (!last) {
              float4* dst = reinterpret_cast<float4*>(scratch_row + c0);
#pragma unroll
              for (int j = 0; j < 8; ++j) dst[j] = make_float4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                dst[j] = make_uint4(pack_bf16x2(__fmul_rn(o[8 * j + 0], osc), __fmul_rn(o[8 * j + 1], osc)),
                                    pack_bf16x2(__fmul_rn(o[8 * j + 2], osc), __fmul_rn(o[8 * j + 3], osc)),
                                    pack_bf16x2(__fmul_rn(o[8 * j + 4], osc), __fmul_rn(o[8 * j + 5], osc)),
                                    pack_bf16x2(__fmul_rn(o[8 * j + 6], osc), __fmul_rn(o[8 * j + 7], osc)));
              }
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

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bip_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnParams p) {
  using C = Cfg<D>;
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
  c.limit_ns = p.wait_limit_ns;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_BAR + OFF_TMEM_SLOT);

  if (threadIdx.x == 0) {
    mbar_init(bar(c, B_Q_FULL), 1);
    mbar_init(bar(c, B_Q_FREE), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar(c, B_K_FULL + s), 1);
      mbar_init(bar(c, B_K_FREE + s), 1);
      mbar_init(bar(c, B_V_FULL + s), 1);
      mbar_init(bar(c, B_V_FREE + s), 1);
      mbar_init(bar(c, B_S_FULL + s), 1);
      mbar_init(bar(c, B_S_FREE + s), 128);
    }
    mbar_init(bar(c, B_P_FULL), 128);
    mbar_init(bar(c, B_O_DONE), 1);
    mbar_init(bar(c, B_DRAIN), 1);
    *c.abort = 0u;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), C::TM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(tmem_slot);

  if (warp == 0) {
    if ((threadIdx.x & 31) == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      producer<D>(c, sbase, &tm_q, &tm_k, &tm_v, p);
    }
  } else if (warp == 1) {
    mma_issuer<D>(c, sbase, tmem, p);
  } else {
    softmax_role<D>(c, sbase, tmem, p);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::TM_COLS);
}

template <int D>
cudaError_t launch(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const AttnParams& p,
                   int grid, cudaStream_t stream) {
  using C = Cfg<D>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(bip_attn_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  bip_attn_kernel<D><<<grid, kThreads, C::SMEM, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(int head_dim, const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                             const CUtensorMap& tm_v, const AttnParams& p, int grid, cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (head_dim == 128) return launch<128>(tm_q, tm_k, tm_v, p, grid, stream);
  if (head_dim == 256) return launch<256>(tm_q, tm_k, tm_v, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bip
