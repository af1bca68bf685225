// Attention launches for token-granular pools (pages of 1, 2 or 4 slots):
// K and V rows are gathered with cp.async by dedicated warps; one q tile
// per CTA (the gather warps take the room a second tile would need).
// Kernel templates in bip_attn_impl.cuh.

#include "bip_attn_impl.cuh"

namespace bip {

cudaError_t launch_attention_gather(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                                    const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                                    cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (tiles_per_unit != 1) return cudaErrorInvalidValue;
  if (!kv_fp8) {
    if (head_dim == 128) return launch<128, 1, 3, false, true>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256) return launch<256, 1, 2, false, true>(tm_q, tm_k, tm_v, p, grid, stream);
  } else {
    if (head_dim == 128) return launch<128, 1, 2, true, true>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256) return launch<256, 1, 2, true, true>(tm_q, tm_k, tm_v, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bip
