// The arithmetic every output row goes through, shared by the attention
// kernel (segments folded in one CTA) and the merge kernel (segments written
// as partials by several CTAs).  Using one definition, with explicitly
// rounded operations and no contraction, is what makes folding and splitting
// give identical bits.
//
// State of a row over some keys, in the log2 domain:
//   m  = max_j s_j * log2(e)        (the softmax scale folded in)
//   l  = sum_j 2^(s_j log2 e - m)
//   o  = sum_j 2^(s_j log2 e - m) v_j     (unnormalised)
// Merging R (running) with P (next segment, in ascending order):
//   P empty (m = -inf): R unchanged.     R empty: R := P (exact copy).
//   else m' = max(mR, mP), a = 2^(mR - m'), b = 2^(mP - m'),
//        l' = lR a + lP b,  o' = oR a + oP b.
// Output: out = o * (1 / l) * v_scale rounded to bf16 (nearest even),
//         lse = (m + log2 l) * ln 2   (natural log).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

namespace bip {

constexpr float kLn2 = 0.693147180559945309f;

// Hardware base-2 exponential / logarithm (ex2.approx / lg2.approx, flush
// to zero).  Deterministic for a given input; ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs: one instruction for two round-to-nearest operations,
// each lane exactly the scalar __fmaf_rn / __fmul_rn / __fadd_rn.
__device__ __forceinline__ uint64_t f2_bits(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t f2_splat(float c) {
  return uint64_t(__float_as_uint(c)) * 0x100000001ull;
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float(uint32_t(v)); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float(uint32_t(v >> 32)); }
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// max(a, b, c), exact.
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

struct MergeStep {
  int kind;  // 0: keep R, 1: take P, 2: combine
  float m, l, a, b;
};

__device__ __forceinline__ MergeStep merge_step(float mR, float lR, float mP, float lP) {
  MergeStep s;
  if (mP == -INFINITY) {
    s.kind = 0; s.m = mR; s.l = lR; s.a = 1.f; s.b = 0.f;
  } else if (mR == -INFINITY) {
    s.kind = 1; s.m = mP; s.l = lP; s.a = 0.f; s.b = 1.f;
  } else {
    s.kind = 2;
    s.m = fmaxf(mR, mP);
    s.a = ex2(__fsub_rn(mR, s.m));
    s.b = ex2(__fsub_rn(mP, s.m));
    s.l = __fadd_rn(__fmul_rn(lR, s.a), __fmul_rn(lP, s.b));
  }
  return s;
}

__device__ __forceinline__ float merge_elem(const MergeStep& s, float oR, float oP) {
  if (s.kind == 2) return __fadd_rn(__fmul_rn(oR, s.a), __fmul_rn(oP, s.b));
  return s.kind == 1 ? oP : oR;
}

__device__ __forceinline__ float out_scale(float l, float v_scale) { return __fmul_rn(__frcp_rn(l), v_scale); }

__device__ __forceinline__ float final_lse(float m, float l) { return __fmul_rn(__fadd_rn(m, lg2(l)), kLn2); }

// Two fp32 -> a bf16 (or f16) pair, each rounded to nearest even, lo in
// the low half: one conversion instruction (the second source lands in
// the low half).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

}  // namespace bip
