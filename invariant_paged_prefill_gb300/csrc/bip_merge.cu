// Split-merge: fold the per-segment partial states of split units in
// ascending segment order with the same merge and normalisation the
// attention kernel uses when it folds segments itself, so a split unit and a
// folded one give identical bits.  The pages describe split partial buffers
// for 4096-token KV splits (model-serving-minefield issue 73 correction:
// fixed 4096-token splits, batch_prefill_tmp_v); here their number is
// bounded by the plan's split budget.
//
// One CTA (4 warps) per merge unit; one warp per valid row; lane L holds
// columns {c * 128 + 4 L .. +3}.  Element arithmetic is per column, so the
// distribution over lanes does not change any bit.

#include <cuda_runtime.h>

#include "bip_internal.h"
#include "bip_numerics.cuh"

namespace bip {
namespace {

template <int D>
__global__ void __launch_bounds__(128) bip_merge_kernel(const MergeParams p) {
  constexpr int E = D / 128;  // float4 groups per lane
  const MergeUnit u = p.units[blockIdx.x];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int first_valid = max(u.tile * p.tile_pos, u.q_lo);
  for (int vr = warp; vr < u.rows; vr += 4) {
    float o[E][4];
#pragma unroll
    for (int e = 0; e < E; ++e) o[e][0] = o[e][1] = o[e][2] = o[e][3] = 0.f;
    float M = -INFINITY, L = 0.f;
    for (int s = 0; s < u.nseg; ++s) {
      const float* prow = p.partials + (size_t(u.part_base) + size_t(s) * u.rows + vr) * (D + 4);
      const float2 ml = *reinterpret_cast<const float2*>(prow);
      const MergeStep st = merge_step(M, L, ml.x, ml.y);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float4 v = *reinterpret_cast<const float4*>(prow + 4 + e * 128 + lane * 4);
        o[e][0] = merge_elem(st, o[e][0], v.x);
        o[e][1] = merge_elem(st, o[e][1], v.y);
        o[e][2] = merge_elem(st, o[e][2], v.z);
        o[e][3] = merge_elem(st, o[e][3], v.w);
      }
      M = st.m;
      L = st.l;
    }
    const int pos = first_valid + vr / p.group;
    const int hg = vr % p.group;
    const size_t tok = size_t(u.q_tok0 + pos);
    const int head = u.kv_head * p.group + hg;
    const float osc = out_scale(L, p.v_scale);
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

}  // namespace

cudaError_t launch_merge(int head_dim, const MergeParams& p, cudaStream_t stream) {
  if (p.n_units <= 0) return cudaSuccess;
  if (head_dim == 128)
    bip_merge_kernel<128><<<p.n_units, 128, 0, stream>>>(p);
  else if (head_dim == 256)
    bip_merge_kernel<256><<<p.n_units, 128, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace bip
