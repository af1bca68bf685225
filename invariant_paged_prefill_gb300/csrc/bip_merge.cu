// Split-merge: fold the per-segment partial states of split units in
// ascending segment order with the same merge and normalisation the
// attention kernel uses when it folds segments itself, so a split unit and a
// folded one give identical bits.  The pages describe split partial buffers
// for 4096-token KV splits (model-serving-minefield issue 73 correction:
// fixed 4096-token splits, batch_prefill_tmp_v); here their number is
// bounded by the plan's split budget.
//
// One CTA (8 warps) per merge unit at a time; one warp per valid row; lane L holds
// columns {c * 128 + 4 L .. +3}.  Element arithmetic is per column, so the
// distribution over lanes does not change any bit.

#include <cuda_runtime.h>

#include "bip_internal.h"
#include "bip_numerics.cuh"

namespace bip {
namespace {

constexpr int kMergeThreads = 256;  // one warp per valid row, eight rows at a time

template <int D>
__global__ void __launch_bounds__(kMergeThreads) bip_merge_kernel(const MergeParams p) {
  constexpr int E = D / 128;  // float4 groups per lane
  constexpr int G = 4;        // segments whose partials are loaded before any is folded
  constexpr int W = kMergeThreads / 32;
  // Units by stride over the grid; device-planned launches read the count.
  const int n_units = p.n_units_dev ? int(*p.n_units_dev) : p.n_units;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int ui = blockIdx.x; ui < n_units; ui += gridDim.x) {
    const MergeUnit u = p.units[ui];
    const int first_valid = u.q_lo + u.tile * p.tile_pos;  // the tile's first position
    for (int vr = warp; vr < u.rows; vr += W) {
      float o[E][4];
#pragma unroll
      for (int e = 0; e < E; ++e) o[e][0] = o[e][1] = o[e][2] = o[e][3] = 0.f;
      float M = -INFINITY, L = 0.f;
      for (int s0 = 0; s0 < u.nseg; s0 += G) {
        // The loads of a group do not depend on the folds before them, so
        // they are all issued first: one memory latency per group of
        // segments instead of one per segment.  The fold order is unchanged.
        float2 ml[G];
        float4 v[G][E];
#pragma unroll
        for (int k = 0; k < G; ++k) {
          if (s0 + k < u.nseg) {
            const float* prow = p.partials + (size_t(u.part_base) + size_t(s0 + k) * u.rows + vr) * (D + 4);
            ml[k] = *reinterpret_cast<const float2*>(prow);
#pragma unroll
            for (int e = 0; e < E; ++e) v[k][e] = *reinterpret_cast<const float4*>(prow + 4 + e * 128 + lane * 4);
          }
        }
#pragma unroll
        for (int k = 0; k < G; ++k) {
          if (s0 + k < u.nseg) {
            const MergeStep st = merge_step(M, L, ml[k].x, ml[k].y);
#pragma unroll
            for (int e = 0; e < E; ++e) {
              o[e][0] = merge_elem(st, o[e][0], v[k][e].x);
              o[e][1] = merge_elem(st, o[e][1], v[k][e].y);
              o[e][2] = merge_elem(st, o[e][2], v[k][e].z);
              o[e][3] = merge_elem(st, o[e][3], v[k][e].w);
            }
            M = st.m;
            L = st.l;
          }
        }
      }
      const int pos = first_valid + vr / p.group;
      const int hg = vr % p.group;
      const size_t tok = size_t(u.q_tok0 + pos);
      const int head = u.kv_head * p.group + hg;
      // A row with no visible key in any segment (only under a custom mask)
      // has L = 0 and o = 0: written as zeros, with lse = -inf.
      const float osc = L > 0.f ? out_scale(L, p.v_scale) : 0.f;
      uint16_t* orow = p.out + (tok * p.num_qo_heads + head) * D;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        uint2 packed = make_uint2(pack_bf16x2(__fmul_rn(o[e][0], osc), __fmul_rn(o[e][1], osc)),
                                  pack_bf16x2(__fmul_rn(o[e][2], osc), __fmul_rn(o[e][3], osc)));
        *reinterpret_cast<uint2*>(orow + e * 128 + lane * 4) = packed;
      }
      if (lane == 0) p.lse[tok * p.num_qo_heads + head] = final_lse(M, L);
    }
  }
}

}  // namespace

// grid: p.n_units CTAs (host-planned: one per unit; device-planned: the
// grid given, units by stride).
cudaError_t launch_merge(int head_dim, const MergeParams& p, cudaStream_t stream) {
  if (p.n_units <= 0) return cudaSuccess;
  if (head_dim == 128)
    bip_merge_kernel<128><<<p.n_units, kMergeThreads, 0, stream>>>(p);
  else if (head_dim == 256)
    bip_merge_kernel<256><<<p.n_units, kMergeThreads, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace bip
