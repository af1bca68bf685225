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

// 2^x on the FMA pipe, to take load off MUFU for a fixed subset of columns.
// Method (Cody-Waite style range reduction, base 2): x = n + f with n the
// nearest integer (adding and subtracting 1.5 * 2^23), 2^f from a degree-4
// polynomial fitted by relative-error weighted least squares on [-1/2, 1/2]
// (fit_exp2_poly.py; worst relative error 2.7e-6 in float32), and 2^n added
// to the exponent field.  x is clamped to >= -126: smaller terms vanish
// against a row sum that is at least 1.  Deterministic for a given input.
__device__ __forceinline__ float ex2_fma(float x) {
  x = fmaxf(x, -126.f);
  const float t = __fadd_rn(x, 12582912.f);
  const float r = __fsub_rn(t, 12582912.f);
  const float f = __fsub_rn(x, r);
  float q = 0.009560510516166687f;
  q = __fmaf_rn(q, f, 0.05591703951358795f);
  q = __fmaf_rn(q, f, 0.24024981260299683f);
  q = __fmaf_rn(q, f, 0.6931219696998596f);
  q = __fmaf_rn(q, f, 0.9999991655349731f);
  const uint32_t n = uint32_t(__float_as_int(t) - 0x4B400000);
  return __uint_as_float(__float_as_uint(q) + (n << 23));
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

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace bip
