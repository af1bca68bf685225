// Attention launches for pools whose pages hold 8 or more token slots:
// every page lands in shared memory as TMA boxes (kernel templates in
// bip_attn_impl.cuh).  Smaller pages go to the row-gather variants.

#include "bip_attn_impl.cuh"

namespace bip {

cudaError_t launch_attention(int head_dim, int tiles_per_unit, bool kv_fp8, const CUtensorMap& tm_q,
                             const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnParams& p, int grid,
                             cudaStream_t stream) {
  if (grid <= 0) return cudaSuccess;
  if (p.page_size < 8) return launch_attention_gather(head_dim, tiles_per_unit, kv_fp8, tm_q, tm_k, tm_v, p, grid,
                                                      stream);
  if (!kv_fp8) {
    if (head_dim == 128 && tiles_per_unit == 2)
      return launch<128, 2, 2, false, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 128 && tiles_per_unit == 1)
      return launch<128, 1, 3, false, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256 && tiles_per_unit == 1)
      return launch<256, 1, 2, false, false>(tm_q, tm_k, tm_v, p, grid, stream);
  } else if (tiles_per_unit == 1) {
    if (head_dim == 128) return launch<128, 1, 2, true, false>(tm_q, tm_k, tm_v, p, grid, stream);
    if (head_dim == 256) return launch<256, 1, 2, true, false>(tm_q, tm_k, tm_v, p, grid, stream);
  } else if (head_dim == 128 && tiles_per_unit == 2) {
    return launch<128, 2, 2, true, false>(tm_q, tm_k, tm_v, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace bip
