// variants.cu — quantisation variants for sm_103a: FP8 per token and per
// channel, the E5M6 activation format, and SwiGLU fused with the 1x128
// quantiser.
//
// Method: the TileKernels release ("DeepSeek starts updating frequently",
// the tile kernels' features, item "Quantification") converts to FP8 / FP4 /
// E5M6 per token, per block and per channel and fuses SwiGLU with the
// quantisation; the V3 excerpt ("The Definitive Information To Deepseek",
// paragraph 3) keeps certain activations in a custom E5M6 format.  Every FP8
// variant uses the same exact group quantiser as the 1x128 / 128x128 kernels
// (quant_common.cuh): s = fl32(amax / 448), codes E4M3_RNE_satfinite(x / s).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_common.cuh"

namespace fp8bs {
namespace {

// ---------------------------------------------------------------------------
// Per token: one CTA (256 threads) per row, the row held in registers (U
// 16-byte vectors per thread, K <= 2048 U), amax reduced across the CTA.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(256) quant_per_token_kernel(const uint4* __restrict__ x, int64_t M, int64_t KV,
                                                              int64_t ldx_v, uint2* __restrict__ q, int64_t ldq_v,
                                                              float* __restrict__ s) {
  pdl_wait();
  __shared__ uint32_t warp_max[8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const uint4* src = x + row * ldx_v;
    uint4 v[U];
    uint32_t m = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = threadIdx.x + 256 * u;
      v[u] = i < KV ? ld_nc_v4(src + i) : make_uint4(0u, 0u, 0u, 0u);
      m = max_pairs(m, absmax8_pairs(v[u]));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max_pairs(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    m = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max_pairs(m, warp_max[i]);
    __syncthreads();  // warp_max is reused by the next row
    const GroupScale g = group_scale(pairs_to_max(m));
    if (threadIdx.x == 0) s[row] = g.s;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = threadIdx.x + 256 * u;
      if (i < KV) q[row * ldq_v + i] = quantise8(v[u], g);
    }
  }
}

// ---------------------------------------------------------------------------
// Per channel, two passes (inputs taller than the one-pass cluster kernel
// below takes): (1) column maxima of |x| as BF16 bit patterns (non-negative
// values order like their patterns), reduced across a CTA in shared memory
// and merged into s with atomicMax, (2) every element quantised with its
// column's scale, (3) s turned from maxima into scales.  A CTA covers 256
// columns (thread t: the 8 columns of vector t % 32) and walks row tiles of 64
// (thread t: rows t / 32 + 8 i).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) channel_absmax_kernel(const uint4* __restrict__ x, int64_t M, int64_t KV,
                                                             int64_t ldx_v, uint32_t* __restrict__ amax_bits) {
  pdl_wait();
  __shared__ uint32_t part[8][32 * 4];  // [row slot][packed column pairs]
  const int lane = threadIdx.x & 31, r8 = threadIdx.x >> 5;
  const int64_t col_v = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  const int64_t row_tiles = (M + 63) / 64;
  uint32_t mm[4] = {0u, 0u, 0u, 0u};
  if (col_v < KV) {
    for (int64_t tile = blockIdx.y; tile < row_tiles; tile += gridDim.y) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t row = tile * 64 + r8 + 8 * i;
        if (row < M) {
          const uint4 v = ld_nc_v4(x + row * ldx_v + col_v);
          constexpr uint32_t kMag = 0x7FFF7FFFu;
          mm[0] = max_pairs(mm[0], v.x & kMag);
          mm[1] = max_pairs(mm[1], v.y & kMag);
          mm[2] = max_pairs(mm[2], v.z & kMag);
          mm[3] = max_pairs(mm[3], v.w & kMag);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) part[r8][lane * 4 + i] = mm[i];
  __syncthreads();
  if (r8 == 0 && col_v < KV) {
    uint32_t* dst = amax_bits + col_v * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t m = part[0][lane * 4 + i];
#pragma unroll
      for (int k = 1; k < 8; ++k) m = max_pairs(m, part[k][lane * 4 + i]);
      atomicMax(dst + 2 * i, m & 0xFFFFu);
      atomicMax(dst + 2 * i + 1, m >> 16);
    }
  }
}

__global__ void __launch_bounds__(256) quant_per_channel_kernel(const uint4* __restrict__ x, int64_t M, int64_t KV,
                                                                int64_t ldx_v, const uint32_t* __restrict__ amax_bits,
                                                                uint2* __restrict__ q, int64_t ldq_v) {
  pdl_wait();
  const int lane = threadIdx.x & 31, r8 = threadIdx.x >> 5;
  const int64_t col_v = static_cast<int64_t>(blockIdx.x) * 32 + lane;
  if (col_v >= KV) return;
  GroupScale g[8];  // the scales of this thread's 8 columns
  uint32_t special0 = 0u, special1 = 0u;  // zero scales or scales below 2^-64, 0xFF per element
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    g[c] = group_scale(__uint_as_float(__ldg(amax_bits + col_v * 8 + c) << 16));
    const uint32_t mark = (g[c].s == 0.0f || !g[c].fast) ? 0xFFu : 0u;
    if (c < 4)
      special0 |= mark << (8 * c);
    else
      special1 |= mark << (8 * (c - 4));
  }
  const int64_t row_tiles = (M + 63) / 64;
  for (int64_t tile = blockIdx.y; tile < row_tiles; tile += gridDim.y) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int64_t row = tile * 64 + r8 + 8 * i;
      if (row < M) q[row * ldq_v + col_v] = quantise8_cols(ld_nc_v4(x + row * ldx_v + col_v), g, special0, special1);
    }
  }
}

// Per channel in one pass, for M <= kPcCluster * 32 * 16 rows: a cluster of
// kPcCluster CTAs covers 64 channels and all rows (CTA rank r: rows 32 R r ..
// 32 R r + 32 R - 1), each thread holding R 16-byte vectors (8 channels of R
// rows, row phase t / 8) in registers.  Column maxima combine per thread,
// across the warp's four row phases (shuffles), across the eight warps
// (shared memory) and across the cluster (each CTA reads every rank's maxima
// through distributed shared memory after a cluster barrier); then every CTA
// codes its rows from registers, so X is read once and no atomics are needed.
constexpr int kPcCluster = 8;

__device__ __forceinline__ uint4 ld_shared_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

template <int R>
__global__ void __launch_bounds__(256) quant_per_channel_cluster_kernel(const uint4* __restrict__ x, int64_t M,
                                                                        int64_t KV, int64_t ldx_v,
                                                                        uint2* __restrict__ q, int64_t ldq_v,
                                                                        float* __restrict__ s) {
  pdl_wait();
  __shared__ uint32_t warp_max[8][8][4];            // [warp][channel group][BF16 pair]
  __shared__ __align__(16) uint32_t cta_max[8][4];  // [channel group][BF16 pair]: this CTA's maxima
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cg = t & 7, rp = t >> 3;
  const uint32_t rank = cluster_ctarank();
  const int64_t cb = blockIdx.x / kPcCluster;
  const int64_t col_v = cb * 8 + cg;
  const bool col_ok = col_v < KV;
  const int64_t row0 = static_cast<int64_t>(rank) * (32 * R) + rp;
  uint4 v[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int64_t row = row0 + 32 * i;
    v[i] = (col_ok && row < M) ? ld_nc_v4(x + row * ldx_v + col_v) : make_uint4(0u, 0u, 0u, 0u);
  }
  constexpr uint32_t kMag = 0x7FFF7FFFu;
  uint32_t m0 = 0u, m1 = 0u, m2 = 0u, m3 = 0u;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    m0 = max_pairs(m0, v[i].x & kMag);
    m1 = max_pairs(m1, v[i].y & kMag);
    m2 = max_pairs(m2, v[i].z & kMag);
    m3 = max_pairs(m3, v[i].w & kMag);
  }
#pragma unroll
  for (int off = 8; off <= 16; off <<= 1) {
    m0 = max_pairs(m0, __shfl_xor_sync(0xffffffffu, m0, off));
    m1 = max_pairs(m1, __shfl_xor_sync(0xffffffffu, m1, off));
    m2 = max_pairs(m2, __shfl_xor_sync(0xffffffffu, m2, off));
    m3 = max_pairs(m3, __shfl_xor_sync(0xffffffffu, m3, off));
  }
  if (lane < 8) {
    warp_max[warp][lane][0] = m0;
    warp_max[warp][lane][1] = m1;
    warp_max[warp][lane][2] = m2;
    warp_max[warp][lane][3] = m3;
  }
  __syncthreads();
  if (t < 32) {
    const int c = t >> 2, w = t & 3;
    uint32_t mm = warp_max[0][c][w];
#pragma unroll
    for (int k = 1; k < 8; ++k) mm = max_pairs(mm, warp_max[k][c][w]);
    cta_max[c][w] = mm;
  }
  cluster_sync_all();  // every CTA's maxima visible to the cluster
  uint32_t a0 = 0u, a1 = 0u, a2 = 0u, a3 = 0u;
  const uint32_t local = smem_u32(&cta_max[cg][0]);
#pragma unroll
  for (int r = 0; r < kPcCluster; ++r) {
    const uint4 o = ld_shared_cluster_v4(map_shared_rank(local, r));
    a0 = max_pairs(a0, o.x);
    a1 = max_pairs(a1, o.y);
    a2 = max_pairs(a2, o.z);
    a3 = max_pairs(a3, o.w);
  }
  cluster_sync_all();  // no CTA leaves while another may still read its maxima
  const uint32_t a[4] = {a0, a1, a2, a3};
  GroupScale g[8];
  uint32_t special0 = 0u, special1 = 0u;  // zero scales or scales below 2^-64, 0xFF per element
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    g[c] = group_scale((c & 1) ? bf16hi_to_f32(a[c >> 1]) : bf16lo_to_f32(a[c >> 1]));
    const uint32_t mark = (g[c].s == 0.0f || !g[c].fast) ? 0xFFu : 0u;
    if (c < 4)
      special0 |= mark << (8 * c);
    else
      special1 |= mark << (8 * (c - 4));
  }
  if (col_ok) {
#pragma unroll
    for (int i = 0; i < R; ++i) {
      const int64_t row = row0 + 32 * i;
      if (row < M) q[row * ldq_v + col_v] = quantise8_cols(v[i], g, special0, special1);
    }
    if (rank == 0 && rp == 0) {
#pragma unroll
      for (int c = 0; c < 8; ++c) s[col_v * 8 + c] = g[c].s;
    }
  }
}

__global__ void channel_scales_kernel(uint32_t* __restrict__ amax_bits_to_scales, int64_t K) {
  pdl_wait();
  const int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (k < K) {
    const float amax = __uint_as_float(amax_bits_to_scales[k] << 16);
    amax_bits_to_scales[k] = __float_as_uint(group_scale(amax).s);
  }
}

__global__ void zero_words_kernel(uint32_t* __restrict__ p, int64_t n) {
  pdl_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i < n) p[i] = 0u;
}

// ---------------------------------------------------------------------------
// E5M6: sign, 5 exponent bits (bias 15), 6 mantissa bits in the low 12 bits
// of a 16-bit word; subnormals 2^-14 * m / 64; round to nearest even,
// magnitudes above 65024 saturate (no scale).  Encoding rounds the float32
// bit pattern directly: adding 0xFFFF plus the kept LSB to the pattern and
// dropping 17 bits rounds the significand to 6 bits with ties to even and
// carries into the exponent; re-biasing 127 -> 15 gives the code.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t e5m6_encode(float f) {
  const uint32_t bits = __float_as_uint(f);
  const uint32_t sign = (bits >> 31) << 11;
  const uint32_t a = bits & 0x7FFFFFFFu;
  uint32_t code;
  if (a > 0x477E0000u) {                 // |f| > 65024
    code = 0x7BFu;
  } else if (a >= 0x38800000u) {         // |f| >= 2^-14: normal E5M6
    code = ((a + 0xFFFFu + ((a >> 17) & 1u)) >> 17) - (112u << 6);
  } else {                               // subnormal E5M6: multiples of 2^-20
    code = __float2uint_rn(__uint_as_float(a) * 0x1p20f);
  }
  return code | sign;
}

__device__ __forceinline__ uint32_t e5m6_to_bf16(uint32_t c) {
  const uint32_t sign = (c & 0x800u) << 4;
  const uint32_t e = (c >> 6) & 0x1Fu, m = c & 0x3Fu;
  uint32_t f;
  if (e == 0)
    f = __float_as_uint(static_cast<float>(m) * 0x1p-20f);
  else if (e == 31)
    f = m == 0 ? 0x7F800000u : 0x7FC00000u;
  else
    f = ((e + 112u) << 23) | (m << 17);
  return sign | (f >> 16);  // exact: the low 16 bits are zero
}

// Two E5M6 codes (in the two 16-bit halves) from two BF16 values (one 32-bit
// word), with integer arithmetic on the bit patterns: dropping BF16's last
// mantissa bit with round-to-nearest-even is (a + kept LSB) >> 1, and the
// exponent is re-biased from 127 to 15 by subtracting 112 << 6.  Halves above
// 65024 saturate to 0x7BF; halves below 2^-14 (E5M6 subnormals) go through
// e5m6_encode one by one.  Per-half flags come from additions that cannot
// carry into the other half.
__device__ __forceinline__ uint32_t e5m6_encode2(uint32_t w) {
  const uint32_t a = w & 0x7FFF7FFFu;
  const uint32_t rounded = ((a + ((a >> 1) & 0x00010001u)) >> 1) & 0x7FFF7FFFu;
  uint32_t code = rounded - 0x1C001C00u;
  const uint32_t small = ~(a + 0x47804780u) & 0x80008000u;  // half < 0x3880 (2^-14)
  const uint32_t big = (a + 0x38813881u) & 0x80008000u;     // half > 0x477E (65024)
  const uint32_t big_mask = (big >> 15) * 0xFFFFu;
  code = (code & ~big_mask) | (0x07BF07BFu & big_mask);
  if (small != 0u) {
    // (rare) recompute both halves: the subnormal half's subtraction above
    // may have borrowed from its neighbour
    code = e5m6_encode(bf16lo_to_f32(w & 0x7FFF7FFFu)) | (e5m6_encode(bf16hi_to_f32(w & 0x7FFF7FFFu)) << 16);
  }
  return code | ((w >> 4) & 0x08000800u);
}

// Grid-stride over blocks of 1024 vectors: each thread loads its 4 vectors
// (t, t + 256, ..) of a block before coding any of them.
__global__ void __launch_bounds__(256) cast_e5m6_kernel(const uint4* __restrict__ x, int64_t nv,
                                                        uint4* __restrict__ out) {
  pdl_wait();
  for (int64_t b = static_cast<int64_t>(blockIdx.x) * 1024; b < nv; b += static_cast<int64_t>(gridDim.x) * 1024) {
    uint4 v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = b + threadIdx.x + 256 * j;
      v[j] = i < nv ? ld_nc_v4(x + i) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t i = b + threadIdx.x + 256 * j;
      if (i < nv)
        out[i] = make_uint4(e5m6_encode2(v[j].x), e5m6_encode2(v[j].y), e5m6_encode2(v[j].z), e5m6_encode2(v[j].w));
    }
  }
}

__global__ void __launch_bounds__(256) e5m6_to_bf16_kernel(const uint4* __restrict__ c, int64_t nv,
                                                           uint4* __restrict__ out) {
  pdl_wait();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < nv;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 v = ld_nc_v4(c + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) o[k] = e5m6_to_bf16(w[k] & 0xFFFFu) | (e5m6_to_bf16(w[k] >> 16) << 16);
    out[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// ---------------------------------------------------------------------------
// SwiGLU + 1x128 quantisation: h = bf16(silu(g) * u) with silu(g) = g / (1 +
// exp(-g)) = g * sigmoid(g), evaluated in float32 from t = expf(-|g|), which
// never overflows: sigmoid(g) = r for g >= 0 and t * r for g < 0, with r the
// hardware reciprocal approximation of 1 + t in [1, 2] (rcp.approx, within
// one float32 ulp).  The product is a few float32 ulps from the exact value
// wherever it is a normal float32.  Then the 1x128 quantiser on the BF16 h,
// bit for bit.  Layout and tiling as the activation quantiser:
// grid x over pairs of 128-channel groups of h, y over 32-row tiles; an
// eight-lane team per row and group, 16 channels per lane.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
  const float t = expf(-fabsf(g));
  const float r = rcp_approx(__fadd_rn(1.0f, t));
  const float sig = g >= 0.0f ? r : __fmul_rn(t, r);
  return __fmul_rn(__fmul_rn(g, sig), u);
}

__device__ __forceinline__ uint32_t swiglu_pair(uint32_t g2, uint32_t u2) {
  const __nv_bfloat162 b = __floats2bfloat162_rn(silu_mul(bf16lo_to_f32(g2), bf16lo_to_f32(u2)),
                                                 silu_mul(bf16hi_to_f32(g2), bf16hi_to_f32(u2)));
  return *reinterpret_cast<const uint32_t*>(&b);
}

__device__ __forceinline__ uint4 swiglu8(uint4 g, uint4 u) {
  return make_uint4(swiglu_pair(g.x, u.x), swiglu_pair(g.y, u.y), swiglu_pair(g.z, u.z), swiglu_pair(g.w, u.w));
}

template <int U>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(const uint4* __restrict__ gu, int64_t M, int64_t FB,
                                                           int64_t ld_v, uint4* __restrict__ q, int64_t ldq_v,
                                                           float* __restrict__ sa, int64_t ld_sa,
                                                           uint4* __restrict__ h_out, int64_t ldh_v) {
  pdl_wait();
  const int lane8 = threadIdx.x & 7;
  const int r = threadIdx.x >> 3;  // 32 rows per CTA
  const int64_t fb0 = static_cast<int64_t>(blockIdx.x) * U;
  const int64_t tiles_m = (M + 31) / 32;
  const int64_t up_off = FB * 16;  // the up half starts F channels (FB * 16 vectors) in
  for (int64_t tm = blockIdx.y; tm < tiles_m; tm += gridDim.y) {
    const int64_t row = tm * 32 + r;
    const bool row_ok = row < M;
    const uint4* src = gu + row * ld_v + fb0 * 16 + lane8 * 2;
    uint4 gv[U][2], uv[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      gv[u][0] = gv[u][1] = uv[u][0] = uv[u][1] = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && fb0 + u < FB) {
        gv[u][0] = ld_nc_v4(src + u * 16);
        gv[u][1] = ld_nc_v4(src + u * 16 + 1);
        uv[u][0] = ld_nc_v4(src + up_off + u * 16);
        uv[u][1] = ld_nc_v4(src + up_off + u * 16 + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 h0 = swiglu8(gv[u][0], uv[u][0]), h1 = swiglu8(gv[u][1], uv[u][1]);
      uint32_t m = max_pairs(absmax8_pairs(h0), absmax8_pairs(h1));
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) m = max_pairs(m, __shfl_xor_sync(0xffffffffu, m, off));
      const GroupScale g = group_scale(pairs_to_max(m));
      const int64_t fb = fb0 + u;
      if (row_ok && fb < FB) {
        const uint2 c0 = quantise8(h0, g), c1 = quantise8(h1, g);
        q[row * ldq_v + fb * 8 + lane8] = make_uint4(c0.x, c0.y, c1.x, c1.y);
        if (lane8 == 0) sa[fb * ld_sa + row] = g.s;
        if (h_out != nullptr) {
          uint4* hd = h_out + row * ldh_v + fb * 16 + lane8 * 2;
          hd[0] = h0;
          hd[1] = h1;
        }
      }
    }
  }
}

constexpr int64_t kMaxGridY = 65535;

}  // namespace

cudaError_t launch_quant_per_token(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                   int64_t ldq, float* s, cudaStream_t stream) {
  const int64_t KV = K / 8;
  const int64_t grid_cap = static_cast<int64_t>(dev.num_sms) * 8;
  const int grid = static_cast<int>(M < grid_cap ? M : grid_cap);
  const uint4* xv = static_cast<const uint4*>(x);
  uint2* qv = static_cast<uint2*>(q);
if (KV <= 256)
    (void)launch_pdl(quant_per_token_kernel<1>, grid, 256, 0, stream, xv, M, KV, ldx / 8, qv, ldq / 8, s);
  else if (KV <= 512)
    (void)launch_pdl(quant_per_token_kernel<2>, grid, 256, 0, stream, xv, M, KV, ldx / 8, qv, ldq / 8, s);
  else if (KV <= 1024)
    (void)launch_pdl(quant_per_token_kernel<4>, grid, 256, 0, stream, xv, M, KV, ldx / 8, qv, ldq / 8, s);
  else if (KV <= 2048)
    (void)launch_pdl(quant_per_token_kernel<8>, grid, 256, 0, stream, xv, M, KV, ldx / 8, qv, ldq / 8, s);
  else
    (void)launch_pdl(quant_per_token_kernel<16>, grid, 256, 0, stream, xv, M, KV, ldx / 8, qv, ldq / 8, s);
  return cudaGetLastError();
}

template <int R>
cudaError_t launch_per_channel_cluster(const void* x, int64_t M, int64_t KV, int64_t ldx, void* q, int64_t ldq,
                                       float* s, cudaStream_t stream) {
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kPcCluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((KV + 7) / 8 * kPcCluster), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, quant_per_channel_cluster_kernel<R>, static_cast<const uint4*>(x), M, KV, ldx / 8,
                            static_cast<uint2*>(q), ldq / 8, s);
}

cudaError_t launch_quant_per_channel(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* q, int64_t ldq, float* s, cudaStream_t stream) {
  (void)dev;
  const int64_t KV = K / 8;
  // One pass on clusters when every row fits a cluster's registers.
  cudaError_t e = cudaErrorNotSupported;
  if (M <= kPcCluster * 32 * 1)
    e = launch_per_channel_cluster<1>(x, M, KV, ldx, q, ldq, s, stream);
  else if (M <= kPcCluster * 32 * 2)
    e = launch_per_channel_cluster<2>(x, M, KV, ldx, q, ldq, s, stream);
  else if (M <= kPcCluster * 32 * 4)
    e = launch_per_channel_cluster<4>(x, M, KV, ldx, q, ldq, s, stream);
  else if (M <= kPcCluster * 32 * 8)
    e = launch_per_channel_cluster<8>(x, M, KV, ldx, q, ldq, s, stream);
  else if (M <= kPcCluster * 32 * 16)
    e = launch_per_channel_cluster<16>(x, M, KV, ldx, q, ldq, s, stream);
  if (e != cudaErrorNotSupported) return e == cudaSuccess ? cudaGetLastError() : e;
  uint32_t* bits = reinterpret_cast<uint32_t*>(s);
  (void)launch_pdl(zero_words_kernel, static_cast<unsigned>((K + 255) / 256), 256, 0, stream, bits, K);
  const int64_t row_tiles = (M + 63) / 64;
  const dim3 grid(static_cast<unsigned>((KV + 31) / 32),
                  static_cast<unsigned>(row_tiles < kMaxGridY ? row_tiles : kMaxGridY));
  (void)launch_pdl(channel_absmax_kernel, grid, 256, 0, stream, static_cast<const uint4*>(x), M, KV, ldx / 8, bits);
  (void)launch_pdl(quant_per_channel_kernel, grid, 256, 0, stream, static_cast<const uint4*>(x), M, KV, ldx / 8, bits,
                                                     static_cast<uint2*>(q), ldq / 8);
  (void)launch_pdl(channel_scales_kernel, static_cast<unsigned>((K + 255) / 256), 256, 0, stream, bits, K);
  return cudaGetLastError();
}

cudaError_t launch_cast_e5m6(const DeviceInfo& dev, const void* x, int64_t n, void* codes, cudaStream_t stream) {
  const int64_t nv = n / 8;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  const int64_t blocks = (nv + 1023) / 1024;
  (void)launch_pdl(cast_e5m6_kernel, static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, stream,
      static_cast<const uint4*>(x), nv, static_cast<uint4*>(codes));
  return cudaGetLastError();
}

cudaError_t launch_e5m6_to_bf16(const DeviceInfo& dev, const void* codes, int64_t n, void* y, cudaStream_t stream) {
  const int64_t nv = n / 8;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  const int64_t blocks = (nv + 255) / 256;
  (void)launch_pdl(e5m6_to_bf16_kernel, static_cast<unsigned>(blocks < cap ? blocks : cap), 256, 0, stream,
      static_cast<const uint4*>(codes), nv, static_cast<uint4*>(y));
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quant_act_1x128(const DeviceInfo& dev, const void* gate_up, int64_t M, int64_t F,
                                          int64_t ld, void* q, int64_t ldq, float* sa, int64_t ld_sa, void* h,
                                          int64_t ldh, cudaStream_t stream) {
  (void)dev;
  constexpr int kUnroll = 2;
  const int64_t FB = F / 128;
  const int64_t tiles_m = (M + 31) / 32;
  const dim3 grid(static_cast<unsigned>((FB + kUnroll - 1) / kUnroll),
                  static_cast<unsigned>(tiles_m < kMaxGridY ? tiles_m : kMaxGridY));
  (void)launch_pdl(swiglu_quant_kernel<kUnroll>, grid, 256, 0, stream, static_cast<const uint4*>(gate_up), M, FB, ld / 8,
                                                         static_cast<uint4*>(q), ldq / 16, sa, ld_sa,
                                                         static_cast<uint4*>(h), ldh / 8);
  return cudaGetLastError();
}

}  // namespace fp8bs
