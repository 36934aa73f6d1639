// quant_common.cuh — the E4M3 group quantiser shared by the quantisation
// kernels (quant.cu, backward.cu): exact per-group scale s = fl32(amax / 448)
// and codes E4M3_RNE_satfinite(fl32(x / s)) ("The Definitive Information To
// Deepseek", paragraph 2: per-group online scaling; "Figure 7 (a)": the
// groups).
#pragma once

#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

// fl32(1 / 448), the float32 nearest to 1/448.
constexpr float kInv448 = 0x1.24924ap-9f;

// s = fl32(amax / 448) without a division: q = fl32(amax * fl32(1/448)), then
// one correction with the exact FMA residual amax - 448 q.  amax is always a
// BF16 value (the largest |x| of BF16 inputs), and this sequence returns the
// correctly rounded quotient for every non-negative finite BF16 value,
// subnormals included (verified exhaustively against exact rational
// arithmetic, and on the GPU by a test that feeds every BF16 magnitude).
__device__ __forceinline__ float scale_of(float amax) {
  const float q = __fmul_rn(amax, kInv448);
  const float r = __fmaf_rn(-q, 448.0f, amax);
  return __fmaf_rn(r, kInv448, q);
}

__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

// Per-group constants of the quantiser.
//
// The codes are E4M3_RNE_satfinite(fl32(x / s)).  Each element is first coded
// from the two bracketing products x * r_lo and x * r_hi, where r approximates
// 1 / s to within a few float32 ulps (rcp.approx) and r_lo / r_hi = r * (1 -/+
// 2^-19), rounded.  With every rounding counted, x * r_lo < fl32(x / s) <
// x * r_hi for x > 0 (reversed for x < 0) with a margin of more than 2^-21
// relative.  E4M3 rounding with saturation is monotonic, so when both ends
// give the same code the quotient gives it too.  Only pairs whose bracket
// straddles a rounding boundary (about 2^-14 of random data) are recomputed
// with the IEEE division.  Products that underflow keep the sign of x and
// code to +-0 at both ends, as the quotient does.  Subnormal scales, whose
// reciprocal may overflow, take the division for the whole group.
struct GroupScale {
  float s;
  float2 r_lo;
  float2 r_hi;
  bool bracket_ok;  // s is a normal float32: the bracketing products are valid
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
  GroupScale g;
  g.s = scale_of(amax);
  g.bracket_ok = g.s >= 1.17549435e-38f;  // smallest normal float32
  const float r = rcp_approx(g.s);
  const float lo = __fmul_rn(r, 1.0f - 0x1p-19f);
  const float hi = __fmul_rn(r, 1.0f + 0x1p-19f);
  g.r_lo = make_float2(lo, lo);
  g.r_hi = make_float2(hi, hi);
  return g;
}

// Four E4M3 codes (x0 in the low byte) from four float32 values.
__device__ __forceinline__ uint32_t cvt_e4m3x4(float x0, float x1, float x2, float x3) {
  uint32_t out;
  asm("{\n\t.reg .b16 l, h;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 l, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 h, %4, %3;\n\t"
      "mov.b32 %0, {l, h};\n\t}"
      : "=r"(out)
      : "f"(x0), "f"(x1), "f"(x2), "f"(x3));
  return out;
}

__device__ __forceinline__ float2 bf16x2_to_f32x2(uint32_t u) {
  return make_float2(bf16lo_to_f32(u), bf16hi_to_f32(u));
}

// Codes of 8 values by correctly rounded division (the rare fallback).
static __device__ __noinline__ uint2 quantise8_div(uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  float f[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __fdiv_rn(bf16lo_to_f32(w[i]), s);
    f[2 * i + 1] = __fdiv_rn(bf16hi_to_f32(w[i]), s);
  }
  return make_uint2(cvt_e4m3x4(f[0], f[1], f[2], f[3]), cvt_e4m3x4(f[4], f[5], f[6], f[7]));
}

// Quantise 8 BF16 values (one 16-byte vector) of a group into 8 codes.
__device__ __forceinline__ uint2 quantise8(const uint4 v, const GroupScale& g) {
  if (g.s == 0.0f) return make_uint2(0u, 0u);  // all-zero group
  const float2 a = bf16x2_to_f32x2(v.x), b = bf16x2_to_f32x2(v.y);
  const float2 c = bf16x2_to_f32x2(v.z), d = bf16x2_to_f32x2(v.w);
  const float2 al = __fmul2_rn(a, g.r_lo), ah = __fmul2_rn(a, g.r_hi);
  const float2 bl = __fmul2_rn(b, g.r_lo), bh = __fmul2_rn(b, g.r_hi);
  const float2 cl = __fmul2_rn(c, g.r_lo), ch = __fmul2_rn(c, g.r_hi);
  const float2 dl = __fmul2_rn(d, g.r_lo), dh = __fmul2_rn(d, g.r_hi);
  const uint32_t lo0 = cvt_e4m3x4(al.x, al.y, bl.x, bl.y), hi0 = cvt_e4m3x4(ah.x, ah.y, bh.x, bh.y);
  const uint32_t lo1 = cvt_e4m3x4(cl.x, cl.y, dl.x, dl.y), hi1 = cvt_e4m3x4(ch.x, ch.y, dh.x, dh.y);
  if (lo0 == hi0 && lo1 == hi1 && g.bracket_ok) return make_uint2(lo0, lo1);
  return quantise8_div(v, g.s);
}

__device__ __forceinline__ __nv_bfloat162 as_bf162(uint32_t u) {
  __nv_bfloat162 h;
  *reinterpret_cast<uint32_t*>(&h) = u;
  return h;
}
__device__ __forceinline__ uint32_t as_u32(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Pairwise maxima of |x| over one 16-byte vector (two BF16 lanes).  Clearing
// the sign bits gives |x|, and the max of non-negative values is exact.
__device__ __forceinline__ uint32_t absmax8_pairs(const uint4 v) {
  constexpr uint32_t kMag = 0x7FFF7FFFu;
  const __nv_bfloat162 m01 = __hmax2(as_bf162(v.x & kMag), as_bf162(v.y & kMag));
  const __nv_bfloat162 m23 = __hmax2(as_bf162(v.z & kMag), as_bf162(v.w & kMag));
  return as_u32(__hmax2(m01, m23));
}
__device__ __forceinline__ uint32_t max_pairs(uint32_t a, uint32_t b) {
  return as_u32(__hmax2(as_bf162(a), as_bf162(b)));
}
// float32 value of the larger of the two BF16 lanes.
__device__ __forceinline__ float pairs_to_max(uint32_t m) {
  return fmaxf(bf16lo_to_f32(m), bf16hi_to_f32(m));
}

}  // namespace fp8bs
