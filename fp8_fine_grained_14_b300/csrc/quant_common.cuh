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
// give the same code the quotient gives it too.  Elements whose bracket holds
// a rounding boundary -- for BF16 data about 0.5 %, almost all exact E4M3
// ties, since BF16 values and their group scale are short binary numbers --
// are decided exactly by straddle_code.  Products that underflow keep the sign
// of x and code to +-0 at both ends, as the quotient does.  Subnormal scales,
// whose reciprocal may overflow, take the IEEE division for the whole group.
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

// Magnitude of an E4M3 code 0x00 .. 0x7E as a float32 (exact).
__device__ __forceinline__ float e4m3_magnitude(uint32_t m) {
  const uint32_t e = m >> 3, f = m & 7u;
  return e == 0 ? static_cast<float>(f) * 0x1p-9f : __uint_as_float(((e + 120u) << 23) | (f << 20));
}

// Exact code of one element whose bracketing products fell on different
// codes m_lo < m_hi (magnitudes; the bracket holds the rounding boundary mu,
// their midpoint).  fl32(x / s) is above mu, equal to it, or below it as
// x / s lies above mu + h+, inside [mu - h-, mu + h+], or below mu - h-, with
// h+- half a float32 ulp of mu above / below (ties of the float32 rounding go
// to mu, whose significand is even).  The comparisons are done exactly in
// 64-bit integers: |x| = X 2^a (X <= 8 bits, BF16), s = S 2^b (S 24 bits),
// mu +- h = T 2^u with u = e(mu) - 25 (T < 2^26), so |x| > (mu + h+) s is
// X 2^(a - u - b) > T S, a comparison of numbers below 2^56.  For BF16 inputs
// these elements are nearly all exact E4M3 ties, which take the even code.
// Anything outside the expected magnitudes falls back to the IEEE division.
static __device__ __noinline__ uint32_t straddle_code(float x, uint32_t c_lo, uint32_t c_hi, float s) {
  const uint32_t m_lo = c_lo & 0x7Fu, m_hi = c_hi & 0x7Fu;
  const uint32_t sign = (__float_as_uint(x) >> 31) << 7;
  const uint32_t xa = __float_as_uint(x) & 0x7FFFFFFFu;
  const uint32_t sb = __float_as_uint(s);
  const float mu = 0.5f * (e4m3_magnitude(m_lo) + e4m3_magnitude(m_hi));
  const uint32_t mb = __float_as_uint(mu);
  // |x| = X 2^a
  const int xe = static_cast<int>(xa >> 23);
  const uint64_t X = xe ? ((xa & 0x7FFFFFu) | 0x800000u) >> 16 : (xa & 0x7FFFFFu) >> 16;
  const int a = (xe ? xe : 1) - 127 - 7;
  // s = S 2^b (normal: the caller guarantees it)
  const uint64_t S = (sb & 0x7FFFFFu) | 0x800000u;
  const int b = static_cast<int>((sb >> 23) & 0xFFu) - 150;
  // mu = P 2^u, u = e(mu) - 25, P in [2^25, 2^26)
  const int mexp = static_cast<int>((mb >> 23) & 0xFFu) - 127;
  const uint64_t P = static_cast<uint64_t>((mb & 0x7FFFFFu) | 0x800000u) << 2;
  const int u = mexp - 25;
  const bool pow2 = (mb & 0x7FFFFFu) == 0u;
  const int shift = a - u - b;
  if (m_hi != m_lo + 1u || m_hi > 0x7Eu || xa == 0u || shift < 0 || shift > 63 - 8) {
    uint32_t code;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(code)
        : "f"(__fdiv_rn(x, s)));
    return code & 0xFFu;
  }
  const uint64_t lhs = X << shift;
  const uint64_t upper = (P + 2u) * S;               // (mu + h+) s in units of 2^(u + b)
  const uint64_t lower = (P - (pow2 ? 1u : 2u)) * S;  // (mu - h-) s
  uint32_t m;
  if (lhs > upper)
    m = m_hi;
  else if (lhs < lower)
    m = m_lo;
  else
    m = (m_lo & 1u) ? m_hi : m_lo;  // fl32(x / s) == mu: E4M3 tie, even code
  return m | sign;
}

// Replace the codes of the straddling elements (bytes where lo and hi
// differ) of one 4-element word by the code of the IEEE quotient.
__device__ __forceinline__ uint32_t fix_word(uint32_t lo, uint32_t hi, uint32_t w0, uint32_t w1, float s) {
  uint32_t diff = lo ^ hi;
  while (diff != 0u) {
    const int byte = (__ffs(diff) - 1) >> 3;
    const uint32_t word = byte < 2 ? w0 : w1;
    const float x = (byte & 1) ? bf16hi_to_f32(word) : bf16lo_to_f32(word);
    const uint32_t code = cvt_e4m3x4(__fdiv_rn(x, s), 0.0f, 0.0f, 0.0f) & 0xFFu;
    lo = (lo & ~(0xFFu << (8 * byte))) | (code << (8 * byte));
    diff &= ~(0xFFu << (8 * byte));
  }
  return lo;
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
  uint32_t lo0 = cvt_e4m3x4(al.x, al.y, bl.x, bl.y);
  const uint32_t hi0 = cvt_e4m3x4(ah.x, ah.y, bh.x, bh.y);
  uint32_t lo1 = cvt_e4m3x4(cl.x, cl.y, dl.x, dl.y);
  const uint32_t hi1 = cvt_e4m3x4(ch.x, ch.y, dh.x, dh.y);
  if (!g.bracket_ok) return quantise8_div(v, g.s);
  if (((lo0 ^ hi0) | (lo1 ^ hi1)) != 0u) {
    lo0 = fix_word(lo0, hi0, v.x, v.y, g.s);
    lo1 = fix_word(lo1, hi1, v.z, v.w, g.s);
  }
  return make_uint2(lo0, lo1);
}

// Quantise 8 BF16 values that belong to 8 different groups (one scale per
// column, e.g. per-channel groups): g points at the 8 groups' constants and
// special0 / special1 mark (0xFF per byte) the elements whose scale is zero
// or subnormal.  Straddling and special elements are fixed one by one.
__device__ __forceinline__ uint32_t fix_word_cols(uint32_t lo, uint32_t diff, uint32_t w0, uint32_t w1, float s0,
                                                  float s1, float s2, float s3) {
  while (diff != 0u) {
    const int byte = (__ffs(diff) - 1) >> 3;
    const uint32_t word = byte < 2 ? w0 : w1;
    const float x = (byte & 1) ? bf16hi_to_f32(word) : bf16lo_to_f32(word);
    const float sc = byte == 0 ? s0 : byte == 1 ? s1 : byte == 2 ? s2 : s3;
    const uint32_t code = sc == 0.0f ? 0u : (cvt_e4m3x4(__fdiv_rn(x, sc), 0.0f, 0.0f, 0.0f) & 0xFFu);
    lo = (lo & ~(0xFFu << (8 * byte))) | (code << (8 * byte));
    diff &= ~(0xFFu << (8 * byte));
  }
  return lo;
}

__device__ __forceinline__ uint2 quantise8_cols(const uint4 v, const GroupScale (&g)[8], uint32_t special0,
                                                uint32_t special1) {
  const float2 a = bf16x2_to_f32x2(v.x), b = bf16x2_to_f32x2(v.y);
  const float2 c = bf16x2_to_f32x2(v.z), d = bf16x2_to_f32x2(v.w);
  const float2 al = __fmul2_rn(a, make_float2(g[0].r_lo.x, g[1].r_lo.x));
  const float2 ah = __fmul2_rn(a, make_float2(g[0].r_hi.x, g[1].r_hi.x));
  const float2 bl = __fmul2_rn(b, make_float2(g[2].r_lo.x, g[3].r_lo.x));
  const float2 bh = __fmul2_rn(b, make_float2(g[2].r_hi.x, g[3].r_hi.x));
  const float2 cl = __fmul2_rn(c, make_float2(g[4].r_lo.x, g[5].r_lo.x));
  const float2 ch = __fmul2_rn(c, make_float2(g[4].r_hi.x, g[5].r_hi.x));
  const float2 dl = __fmul2_rn(d, make_float2(g[6].r_lo.x, g[7].r_lo.x));
  const float2 dh = __fmul2_rn(d, make_float2(g[6].r_hi.x, g[7].r_hi.x));
  uint32_t lo0 = cvt_e4m3x4(al.x, al.y, bl.x, bl.y);
  const uint32_t hi0 = cvt_e4m3x4(ah.x, ah.y, bh.x, bh.y);
  uint32_t lo1 = cvt_e4m3x4(cl.x, cl.y, dl.x, dl.y);
  const uint32_t hi1 = cvt_e4m3x4(ch.x, ch.y, dh.x, dh.y);
  const uint32_t diff0 = (lo0 ^ hi0) | special0, diff1 = (lo1 ^ hi1) | special1;
  if ((diff0 | diff1) != 0u) {
    lo0 = fix_word_cols(lo0, diff0, v.x, v.y, g[0].s, g[1].s, g[2].s, g[3].s);
    lo1 = fix_word_cols(lo1, diff1, v.z, v.w, g[4].s, g[5].s, g[6].s, g[7].s);
  }
  return make_uint2(lo0, lo1);
}

// Code of a single value with its own group's scale (the per-element form of
// quantise8, for groups that run across vectors).
__device__ __forceinline__ uint32_t quantise1(float x, const GroupScale& g) {
  if (g.s == 0.0f) return 0u;
  if (!g.bracket_ok) {
    uint32_t code;
    asm("{\n\t.reg .b16 t;\n\tcvt.rn.satfinite.e4m3x2.f32 t, %1, %1;\n\tcvt.u32.u16 %0, t;\n\t}"
        : "=r"(code)
        : "f"(__fdiv_rn(x, g.s)));
    return code & 0xFFu;
  }
  const uint32_t lo = cvt_e4m3x4(__fmul_rn(x, g.r_lo.x), 0.0f, 0.0f, 0.0f) & 0xFFu;
  const uint32_t hi = cvt_e4m3x4(__fmul_rn(x, g.r_hi.x), 0.0f, 0.0f, 0.0f) & 0xFFu;
  return lo == hi ? lo : straddle_code(x, lo, hi, g.s);
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
