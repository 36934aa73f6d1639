// quant.cu — online FP8 (E4M3) quantisation kernels for sm_103a.
//
// Method ("The Definitive Information To Deepseek", paragraph 3,
// "Figure 7 (a)"; paragraph 2 for the online scale): activations are grouped
// per token per 128 channels (1x128 tiles), weights per 128x128 block.  Each
// group's scale is s = amax / 448 in IEEE float32 and every element is coded
// as E4M3(x / s), round-to-nearest-even, saturating.  An all-zero group gets
// s = 0 and codes 0x00.
//
// Both kernels are HBM-bound (2 bytes read, 1 byte + 4/group written per
// element): 16-byte vector loads, shuffle reductions, packed 8-byte code
// stores.  Scales use the correctly rounded __fdiv_rn; codes come from a
// bracketing reciprocal product with an exact-division fallback (see
// GroupScale).  The build never enables fast math or flush-to-zero, so codes
// and scales are bit-identical to the float32 definition.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr float kE4M3Max = 448.0f;

// Per-group constants of the quantiser.
//
// The codes are defined as E4M3_RNE_satfinite(fl32(x / s)).  Dividing every
// element is the slowest part of the kernel, so each element is first coded
// from the two bracketing products x * r_lo and x * r_hi, with
// r = fl32(1 / s) and r_lo / r_hi = r * (1 -/+ 2^-20) rounded.  Each product
// rounds at most three times by 2^-24 relative, so the pair brackets the
// correctly rounded quotient with a margin of more than 12 float32 ulps:
// x * r_lo <= fl32(x / s) <= x * r_hi (order reversed for x < 0).  E4M3
// rounding with saturation is monotonic, so when both ends give the same code
// the quotient gives it too.  Only pairs whose bracket straddles a rounding
// boundary (about 2^-16 of random data) fall back to the IEEE division.
// Products that underflow keep the sign of x and code to +-0 on both ends,
// as the quotient does.  Subnormal scales (1 / s would overflow) take the
// division for the whole group.
struct GroupScale {
  float s;
  float r_lo;
  float r_hi;
  bool bracket_ok;  // s is a normal float: the bracketing products are valid
};

__device__ __forceinline__ GroupScale group_scale(float amax) {
  GroupScale g;
  g.s = __fdiv_rn(amax, kE4M3Max);
  g.bracket_ok = g.s >= 1.17549435e-38f;  // smallest normal float32
  const float r = __frcp_rn(g.s);
  g.r_lo = __fmul_rn(r, 1.0f - 0x1p-20f);
  g.r_hi = __fmul_rn(r, 1.0f + 0x1p-20f);
  return g;
}

// Codes of two values (a in the low byte) by correctly rounded division.
__device__ __forceinline__ uint32_t quant_pair_div(float a, float b, float s) {
  return cvt_e4m3x2(__fdiv_rn(a, s), __fdiv_rn(b, s));
}

// Quantise 8 BF16 values (one 16-byte vector) of a group into 8 codes.
__device__ __forceinline__ uint2 quantise8(const uint4 v, const GroupScale& g) {
  if (g.s == 0.0f) return make_uint2(0u, 0u);  // all-zero group
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t pair[4];
  bool same = true;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float a = bf16lo_to_f32(w[i]);
    const float b = bf16hi_to_f32(w[i]);
    const uint32_t lo = cvt_e4m3x2(__fmul_rn(a, g.r_lo), __fmul_rn(b, g.r_lo));
    const uint32_t hi = cvt_e4m3x2(__fmul_rn(a, g.r_hi), __fmul_rn(b, g.r_hi));
    pair[i] = lo;
    same = same && (lo == hi);
  }
  if (!(same && g.bracket_ok)) {
#pragma unroll
    for (int i = 0; i < 4; ++i) pair[i] = quant_pair_div(bf16lo_to_f32(w[i]), bf16hi_to_f32(w[i]), g.s);
  }
  return make_uint2(pair[0] | (pair[1] << 16), pair[2] | (pair[3] << 16));
}

__device__ __forceinline__ float absmax8(const uint4 v) {
  float m = 0.0f;
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m = fmaxf(m, fabsf(bf16lo_to_f32(w[i])));
    m = fmaxf(m, fabsf(bf16hi_to_f32(w[i])));
  }
  return m;
}

// ---------------------------------------------------------------------------
// 1x128 activation tiles.
//
// A CTA of 256 threads = 16 half-warps works on a tile of 16 rows x UNROLL
// groups: half-warp h owns row (16*tm + h) and walks UNROLL consecutive
// 128-channel groups; each of its 16 lanes holds 8 channels of a group.  The
// UNROLL loads of a thread are issued before any arithmetic.  For a given
// group, the 16 scales of the tile's rows are 64 contiguous bytes of sa.
// ---------------------------------------------------------------------------
template <int UNROLL>
__global__ void __launch_bounds__(256) quant_act_1x128_kernel(const uint4* __restrict__ x, int64_t M, int64_t KB,
                                                              int64_t ldx_v, uint2* __restrict__ q, int64_t ldq_v,
                                                              float* __restrict__ sa, int64_t ld_sa) {
  const int lane16 = threadIdx.x & 15;
  const int h = threadIdx.x >> 4;
  const int64_t tiles_m = (M + 15) / 16;
  const int64_t tiles_k = (KB + UNROLL - 1) / UNROLL;
  const int64_t total = tiles_m * tiles_k;
  for (int64_t t = blockIdx.x; t < total; t += gridDim.x) {
    const int64_t tm = t / tiles_k;
    const int64_t kb0 = (t - tm * tiles_k) * UNROLL;
    const int64_t row = tm * 16 + h;
    const bool row_ok = row < M;
    uint4 v[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && kb0 + u < KB) v[u] = ld_nc_v4(x + row * ldx_v + (kb0 + u) * 16 + lane16);
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float amax = absmax8(v[u]);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      const GroupScale g = group_scale(amax);
      const int64_t kb = kb0 + u;
      if (row_ok && kb < KB) {
        q[row * ldq_v + kb * 16 + lane16] = quantise8(v[u], g);
        if (lane16 == 0) sa[kb * ld_sa + row] = g.s;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block.  Thread t holds the 16-byte
// column slice (t % 16) of rows (t / 16) + 16 i, i = 0..7, i.e. the whole
// block sits in registers, so the block is read from HBM exactly once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) quant_weight_128x128_kernel(const uint4* __restrict__ w, int64_t NB,
                                                                   int64_t KB, int64_t ldw_v, uint2* __restrict__ q,
                                                                   int64_t ldq_v, float* __restrict__ sw) {
  __shared__ float warp_max[8];
  const int c = threadIdx.x & 15;
  const int r0 = threadIdx.x >> 4;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t total = NB * KB;
  for (int64_t b = blockIdx.x; b < total; b += gridDim.x) {
    const int64_t nb = b / KB;
    const int64_t kb = b - nb * KB;
    const int64_t row0 = nb * 128 + r0;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_nc_v4(w + (row0 + 16 * i) * ldw_v + kb * 16 + c);
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, absmax8(v[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if (lane == 0) warp_max[warp] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    __syncthreads();  // warp_max is reused by the next block of this CTA
    const GroupScale g = group_scale(amax);
    if (threadIdx.x == 0) sw[nb * KB + kb] = g.s;
#pragma unroll
    for (int i = 0; i < 8; ++i) q[(row0 + 16 * i) * ldq_v + kb * 16 + c] = quantise8(v[i], g);
  }
}

}  // namespace

cudaError_t launch_quant_act_1x128(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                   int64_t ldq, float* sa, int64_t ld_sa, cudaStream_t stream) {
  constexpr int kUnroll = 4;
  const int64_t KB = K / 128;
  const int64_t tiles = ((M + 15) / 16) * ((KB + kUnroll - 1) / kUnroll);
  const int64_t resident = static_cast<int64_t>(dev.num_sms) * 8;  // 8 CTAs of 256 threads per SM
  const int grid = static_cast<int>(tiles < resident ? tiles : resident);
  quant_act_1x128_kernel<kUnroll><<<grid, 256, 0, stream>>>(static_cast<const uint4*>(x), M, KB, ldx / 8,
                                                            static_cast<uint2*>(q), ldq / 8, sa, ld_sa);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight_128x128(const DeviceInfo& dev, const void* w, int64_t N, int64_t K, int64_t ldw,
                                        void* q, int64_t ldq, float* sw, cudaStream_t stream) {
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t blocks = NB * KB;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 64;  // grid-stride beyond this
  const int grid = static_cast<int>(blocks < cap ? blocks : cap);
  quant_weight_128x128_kernel<<<grid, 256, 0, stream>>>(static_cast<const uint4*>(w), NB, KB, ldw / 8,
                                                        static_cast<uint2*>(q), ldq / 8, sw);
  return cudaGetLastError();
}

}  // namespace fp8bs
