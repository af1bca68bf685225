// Attention launches under a per-row custom mask, for every pool layout the
// unmasked launches cover: whole pages by TMA (8 or more slots) and token
// rows gathered with cp.async (1, 2 or 4 slots).  Kernel templates in
// bip_attn_impl.cuh (mask kind 2).

#include "bip_attn_impl.cuh"

namespace bip {

cudaError_t launch_attention_masked(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                                    const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                    cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (!p.mask) return cudaErrorInvalidValue;
  if (p.page_size < 8) {
    if (tiles_per_unit != 1) return cudaErrorInvalidValue;
    if (!kv_fp8) {
      if (head_dim == 128) return launch_one<128, 1, 3, false, 2, true>(tm_q, tm_k, tm_v, p, grid, stream);
      if (head_dim == 256) return launch_one<256, 1, 2, false, 2, true>(tm_q, tm_k, tm_v, p, grid, stream);
    } else {
      if (head_dim == 128) return launch_one<128, 1, 2, true, 2, true>(tm_q, tm_k, tm_v, p, grid, stream);
      if (head_dim == 256) return launch_one<256, 1, 2, true, 2, true>(tm_q, tm_k, tm_v, p, grid, stream);
    }
    return cudaErrorInvalidValue;
  }
  if (!kv_fp8) {
    if (head_dim == 128 && tiles_per_unit == 2)
      return launch_one<128, 2, 2, false, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 128 && tiles_per_unit == 1)
      return launch_one<128, 1, 3, false, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256 && tiles_per_unit == 1)
      return launch_one<256, 1, 2, false, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
  } else if (tiles_per_unit == 1) {
    if (head_dim == 128) return launch_one<128, 1, 2, true, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256) return launch_one<256, 1, 2, true, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
  } else if (head_dim == 128 && tiles_per_unit == 2) {
    return launch_one<128, 2, 2, true, 2, false>(tm_q, tm_k, tm_v, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bip
