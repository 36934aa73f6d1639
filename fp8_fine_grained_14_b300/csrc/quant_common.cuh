// quant_common.cuh — the E4M3 group quantiser shared by the quantisation
// kernels (quant.cu, backward.cu): exact per-group scale s = fl32(amax / 448)
// and codes E4M3_RNE_satfinite(fl32(x / s)) ("The Definitive Information To
// Deepseek", paragraph 2: per-group online scaling; "Figure 7 (a)": the
// groups).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fp8bs {

// Two E4M3 codes (the low 16 bits; the lower byte is the first value) ->
// their exact values in FP32: E4M3 values are exact in FP16, so the pair is
// widened with the hardware e4m3x2 -> f16x2 conversion.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_codes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 c;\n\t"
      "cvt.u16.u32 c, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
      : "=r"(h2)
      : "r"(two_codes));
  const __half2 h = *reinterpret_cast<const __half2*>(&h2);
  return __half22float2(h);
}

// Two FP32 values -> a packed BF16 pair, each rounded to nearest even.
__device__ __forceinline__ uint32_t bf16x2_rn(float2 v) {
  const __nv_bfloat162 b = __float22bfloat162_rn(v);
  return *reinterpret_cast<const uint32_t*>(&b);
}

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

// Per-group constants of the quantiser.
//
// The codes are E4M3_RNE_satfinite(fl32(x / s)).  The quotient is formed
// without a division by Markstein's FMA correction (P. Markstein, "Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = fl32(1 / s) correctly rounded,
//   q0 = fl32(x r),  e = x - q0 s (exact, one FMA),  q1 = fl32(q0 + e r) (one FMA),
// and q1 == fl32(x / s).  Every step is invariant under scaling x and s by
// powers of two while the values stay in the normal float32 range, so an
// exhaustive check over all 128 BF16 significands x all 2^23 float32
// significands of s covers every case that matters here; it found no
// mismatch.  Groups with s < 2^-64 (where e could fall below the normal range
// for quotients large enough to give a non-zero code) take the IEEE division.
// x = -0 makes the chain return +0, so the sign of x is put back on the code.
struct GroupScale {
  float s;
  float2 r;      // fl32(1 / s) in both halves
  float2 s_neg;  // -s in both halves
  bool fast;     // s >= 2^-64: the FMA correction is exact
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
  GroupScale g;
  g.s = scale_of(amax);
  g.fast = g.s >= 0x1p-64f;
  const float r = __frcp_rn(g.s);
  g.r = make_float2(r, r);
  g.s_neg = make_float2(-g.s, -g.s);
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

// fl32(x / s) for two values (see GroupScale), with packed FP32 arithmetic.
__device__ __forceinline__ float2 quotient2(float2 x, float2 r, float2 s_neg) {
  const float2 q0 = __fmul2_rn(x, r);
  const float2 e = __ffma2_rn(q0, s_neg, x);
  return __ffma2_rn(e, r, q0);
}

// The sign bits of four BF16 values (two 32-bit words) placed on the sign
// bits of their four code bytes.
__device__ __forceinline__ uint32_t sign_bytes(uint32_t w0, uint32_t w1) {
  return __byte_perm(w0, w1, 0x7531) & 0x80808080u;
}

// Codes of 8 values by correctly rounded division (groups with tiny scales).
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
  if (!g.fast) return quantise8_div(v, g.s);
  const float2 a = quotient2(bf16x2_to_f32x2(v.x), g.r, g.s_neg);
  const float2 b = quotient2(bf16x2_to_f32x2(v.y), g.r, g.s_neg);
  const float2 c = quotient2(bf16x2_to_f32x2(v.z), g.r, g.s_neg);
  const float2 d = quotient2(bf16x2_to_f32x2(v.w), g.r, g.s_neg);
  return make_uint2(cvt_e4m3x4(a.x, a.y, b.x, b.y) | sign_bytes(v.x, v.y),
                    cvt_e4m3x4(c.x, c.y, d.x, d.y) | sign_bytes(v.z, v.w));
}

// Quantise 8 BF16 values that belong to 8 different groups (one scale per
// column, e.g. per-channel groups).  special0 / special1 mark (0xFF per byte)
// the elements whose scale is zero or below the fast range; those are coded
// one by one (code 0 for a zero scale, else the IEEE division).
__device__ __forceinline__ uint32_t fix_word_cols(uint32_t code, uint32_t special, uint32_t w0, uint32_t w1,
                                                  float s0, float s1, float s2, float s3) {
  while (special != 0u) {
    const int byte = (__ffs(special) - 1) >> 3;
    const uint32_t word = byte < 2 ? w0 : w1;
    const float x = (byte & 1) ? bf16hi_to_f32(word) : bf16lo_to_f32(word);
    const float sc = byte == 0 ? s0 : byte == 1 ? s1 : byte == 2 ? s2 : s3;
    const uint32_t c = sc == 0.0f ? 0u : (cvt_e4m3x4(__fdiv_rn(x, sc), 0.0f, 0.0f, 0.0f) & 0xFFu);
    code = (code & ~(0xFFu << (8 * byte))) | (c << (8 * byte));
    special &= ~(0xFFu << (8 * byte));
  }
  return code;
}

// quantise8_cols with the per-column constants already paired as the packed
// arithmetic takes them: r2[i] = (r of column 2i, r of column 2i + 1), and
// likewise sn2 for -s (pairs built once per thread, not once per vector).
__device__ __forceinline__ uint2 quantise8_cols_paired(const uint4 v, const float2 (&r2)[4], const float2 (&sn2)[4],
                                                       const GroupScale (&g)[8], uint32_t special0,
                                                       uint32_t special1) {
  const float2 a = quotient2(bf16x2_to_f32x2(v.x), r2[0], sn2[0]);
  const float2 b = quotient2(bf16x2_to_f32x2(v.y), r2[1], sn2[1]);
  const float2 c = quotient2(bf16x2_to_f32x2(v.z), r2[2], sn2[2]);
  const float2 d = quotient2(bf16x2_to_f32x2(v.w), r2[3], sn2[3]);
  uint32_t lo = cvt_e4m3x4(a.x, a.y, b.x, b.y) | sign_bytes(v.x, v.y);
  uint32_t hi = cvt_e4m3x4(c.x, c.y, d.x, d.y) | sign_bytes(v.z, v.w);
  if ((special0 | special1) != 0u) {
    lo = fix_word_cols(lo, special0, v.x, v.y, g[0].s, g[1].s, g[2].s, g[3].s);
    hi = fix_word_cols(hi, special1, v.z, v.w, g[4].s, g[5].s, g[6].s, g[7].s);
  }
  return make_uint2(lo, hi);
}

__device__ __forceinline__ uint2 quantise8_cols(const uint4 v, const GroupScale (&g)[8], uint32_t special0,
                                                uint32_t special1) {
  const float2 a = quotient2(bf16x2_to_f32x2(v.x), make_float2(g[0].r.x, g[1].r.x),
                             make_float2(g[0].s_neg.x, g[1].s_neg.x));
  const float2 b = quotient2(bf16x2_to_f32x2(v.y), make_float2(g[2].r.x, g[3].r.x),
                             make_float2(g[2].s_neg.x, g[3].s_neg.x));
  const float2 c = quotient2(bf16x2_to_f32x2(v.z), make_float2(g[4].r.x, g[5].r.x),
                             make_float2(g[4].s_neg.x, g[5].s_neg.x));
  const float2 d = quotient2(bf16x2_to_f32x2(v.w), make_float2(g[6].r.x, g[7].r.x),
                             make_float2(g[6].s_neg.x, g[7].s_neg.x));
  uint32_t lo = cvt_e4m3x4(a.x, a.y, b.x, b.y) | sign_bytes(v.x, v.y);
  uint32_t hi = cvt_e4m3x4(c.x, c.y, d.x, d.y) | sign_bytes(v.z, v.w);
  if ((special0 | special1) != 0u) {
    lo = fix_word_cols(lo, special0, v.x, v.y, g[0].s, g[1].s, g[2].s, g[3].s);
    hi = fix_word_cols(hi, special1, v.z, v.w, g[4].s, g[5].s, g[6].s, g[7].s);
  }
  return make_uint2(lo, hi);
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
