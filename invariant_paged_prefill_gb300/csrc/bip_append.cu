// Paged KV append: write each request's new K/V rows (bf16, one per new
// token and kv head) into its pages, the step before the attention of an
// extend.  A request's new rows take positions kv_len - q_len .. kv_len - 1
// (the tail alignment of the extend rows); position p lives in page
// kv_indices[page_base + p / page_size] at slot p % page_size.  bf16 pages
// get the bits unchanged; FP8 E4M3 pages get e4m3(x / scale): the bf16
// value widened to float32, divided by the scale with IEEE rounding, then
// converted with round-to-nearest-even and saturation at +-448.
//
// One warp per new row (all kv heads), K and V in the same pass.  Pure
// streaming: each byte is read once and written once.

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "bip_internal.h"

namespace bip {
namespace {

constexpr int kAppendThreads = 256;

// Request holding new row `tok`: the last entry whose tok0 <= tok.
__device__ __forceinline__ int find_request(const AppendRow* rows, int n, int tok) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(&rows[mid].tok0) <= tok) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// N bf16 (packed two per 32-bit word) -> N E4M3 codes (packed four per
// word), each x / scale first.
template <int N>
__device__ __forceinline__ void quantize(const uint32_t (&in)[N / 2], float scale, uint32_t (&out)[N / 4]) {
#pragma unroll
  for (int i = 0; i < N / 4; ++i) out[i] = 0u;
#pragma unroll
  for (int i = 0; i < N / 2; ++i) {
    const float lo = __fdiv_rn(__uint_as_float(in[i] << 16), scale);
    const float hi = __fdiv_rn(__uint_as_float(in[i] & 0xFFFF0000u), scale);
    const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    out[i >> 1] |= uint32_t(c) << (16 * (i & 1));
  }
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kAppendThreads) bip_append_kernel(const AppendParams p) {
  // A token's K (or V) row for all kv heads, [Hkv, D] bf16, is contiguous in
  // k_new and lands contiguously in its slot (slots are [Hkv, D] in NHD
  // pages): one warp copies a token, 16-byte chunks per lane, every load of
  // a batch of chunks issued before its stores.
  constexpr int kBatch = 4;  // chunks per lane per batch, K and V each
  const int lane = threadIdx.x & 31;
  const int chunks = p.num_kv_heads * D / 8;  // 16-byte chunks of bf16 per row
  const int64_t warps = int64_t(gridDim.x) * (kAppendThreads / 32);
  for (int64_t tok = int64_t(blockIdx.x) * (kAppendThreads / 32) + (threadIdx.x >> 5); tok < p.total_q;
       tok += warps) {
    const AppendRow rq = p.rows[find_request(p.rows, p.n_rows, int(tok))];
    const int pos = rq.pos0 + (int(tok) - rq.tok0);
    const int page = __ldg(p.kv_indices + rq.page_base + pos / p.page_size);
    if (page < 0 || page >= p.num_pages) {  // counted, and the row is skipped
      if (lane == 0) atomicAdd(&p.header->bad_pages, 1u);
      continue;
    }
    const int slot = pos % p.page_size;
    const uint4* ksrc = reinterpret_cast<const uint4*>(p.k_new + tok * p.num_kv_heads * D);
    const uint4* vsrc = reinterpret_cast<const uint4*>(p.v_new + tok * p.num_kv_heads * D);
    const int64_t dst_elem = int64_t(page) * p.page_stride + int64_t(slot) * p.num_kv_heads * D;
    for (int c0 = 0; c0 < chunks; c0 += 32 * kBatch) {
      uint4 kv[kBatch], vv[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c < chunks) {
          kv[i] = __ldg(ksrc + c);
          vv[i] = __ldg(vsrc + c);
        }
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        const int c = c0 + i * 32 + lane;
        if (c >= chunks) continue;
        if constexpr (FP8) {
          const uint32_t kw[4] = {kv[i].x, kv[i].y, kv[i].z, kv[i].w};
          const uint32_t vw[4] = {vv[i].x, vv[i].y, vv[i].z, vv[i].w};
          uint32_t kq[2], vq[2];
          quantize<8>(kw, p.k_scale, kq);
          quantize<8>(vw, p.v_scale, vq);
          reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.k_pages) + dst_elem)[c] = make_uint2(kq[0], kq[1]);
          reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.v_pages) + dst_elem)[c] = make_uint2(vq[0], vq[1]);
        } else {
          reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pages) + dst_elem)[c] = kv[i];
          reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pages) + dst_elem)[c] = vv[i];
        }
      }
    }
  }
}

template <int D, bool FP8>
cudaError_t launch(const AppendParams& p, int num_sms, cudaStream_t stream) {
  const int64_t blocks_needed = (int64_t(p.total_q) + kAppendThreads / 32 - 1) / (kAppendThreads / 32);
  const int grid = int(blocks_needed < int64_t(num_sms) * 8 ? blocks_needed : int64_t(num_sms) * 8);
  if (grid <= 0) return cudaSuccess;
  bip_append_kernel<D, FP8><<<grid, kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(int head_dim, bool kv_fp8, const AppendParams& p, int num_sms, cudaStream_t stream) {
  if (head_dim == 128) return kv_fp8 ? launch<128, true>(p, num_sms, stream) : launch<128, false>(p, num_sms, stream);
  if (head_dim == 256) return kv_fp8 ? launch<256, true>(p, num_sms, stream) : launch<256, false>(p, num_sms, stream);
  return cudaErrorInvalidValue;
}

}  // namespace bip
