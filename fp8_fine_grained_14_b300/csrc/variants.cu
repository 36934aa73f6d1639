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
// Per channel: a cluster of kPcCluster CTAs covers a strip of SV vectors of 8
// channels and all M rows, CTA rank r the r-th of kPcCluster equal row
// ranges.  Thread t takes vector t % SV of the strip and rows t / SV +
// (T / SV) i of its range, so a warp reads 32 / SV rows of 16 SV contiguous
// bytes per instruction.  Pass 1 streams those rows for the column maxima of
// |x| (BF16 bit patterns: non-negative values order like their patterns),
// combined across the warp's row phases (shuffles), the CTA's warps (shared
// memory) and the cluster (each CTA reads every rank's maxima through
// distributed shared memory).  Pass 2 reads the same rows again and codes
// them: all of X was read a moment before (with an evict-last L2 policy), so
// while X fits in L2 (58.7 MB for 4096 x 7168 against 126 MB) the second
// read comes from L2 and HBM sees X once.  Nothing stays in registers between
// the passes.
// ---------------------------------------------------------------------------
constexpr int kPcCluster = 8;
// 8 vectors (64 channels, 128 bytes of a row) per strip and 128-thread CTAs:
// seven CTAs per SM, so a 4096 x 7168 input's 896 CTAs run in one wave.
// (Strips of 16 or 32 vectors, with fewer, larger CTAs, measured slower.)
constexpr int kPcSV = 8;           // vectors (of 8 channels) per strip
constexpr int kPcThreads = 128;    // threads per CTA
constexpr int kPcMinBlocks = 7;    // CTAs per SM (72 registers a thread)
constexpr int kPcUnroll = 8;       // loads in flight per thread
static_assert(kPcSV <= 32 && 32 % kPcSV == 0 && kPcThreads % 32 == 0, "strip layout");

__device__ __forceinline__ uint4 ld_shared_cluster_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

template <int SV, int T>
__global__ void __launch_bounds__(T, kPcMinBlocks) quant_per_channel_kernel(const uint4* __restrict__ x, int64_t M,
                                                                     int64_t KV, int64_t ldx_v,
                                                                     int64_t rows_per_cta, uint2* __restrict__ q,
                                                                     int64_t ldq_v, float* __restrict__ s) {
  constexpr int kWarps = T / 32;
  constexpr int kPhases = T / SV;  // row phases of a CTA
  constexpr int kStep = kPhases * kPcUnroll;
  pdl_wait();
  __shared__ uint32_t warp_max[kWarps][SV][4];       // [warp][vector][BF16 pair]
  __shared__ __align__(16) uint32_t cta_max[SV][4];  // [vector][BF16 pair]: this CTA's maxima
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int cg = t % SV, rp = t / SV;
  const uint32_t rank = cluster_ctarank();
  const int64_t col_v = static_cast<int64_t>(blockIdx.x / kPcCluster) * SV + cg;
  const bool col_ok = col_v < KV;
  const int64_t r_begin = static_cast<int64_t>(rank) * rows_per_cta;
  const int64_t r_end = r_begin + rows_per_cta < M ? r_begin + rows_per_cta : M;
  const uint4* xc = x + col_v;
  constexpr uint32_t kMag = 0x7FFF7FFFu;

  // pass 1: column maxima of this CTA's rows, which stay in L2 for pass 2
  // (evict-last; pass 2 reads them evict-first and stores the codes so)
  const uint64_t keep = l2_evict_last_policy(), drop = l2_evict_first_policy();
  uint32_t m0 = 0u, m1 = 0u, m2 = 0u, m3 = 0u;
  if (col_ok) {
    const uint4* xp = xc + (r_begin + rp) * ldx_v;
    const int64_t xstep = kPhases * ldx_v;
    int64_t r = r_begin + rp;
    for (; r + kPhases * (kPcUnroll - 1) < r_end; r += kStep) {
      uint4 v[kPcUnroll];
#pragma unroll
      for (int i = 0; i < kPcUnroll; ++i) v[i] = ld_nc_v4_hint(xp + i * xstep, keep);
#pragma unroll
      for (int i = 0; i < kPcUnroll; ++i) {
        m0 = max_pairs(m0, v[i].x & kMag);
        m1 = max_pairs(m1, v[i].y & kMag);
        m2 = max_pairs(m2, v[i].z & kMag);
        m3 = max_pairs(m3, v[i].w & kMag);
      }
      xp += kPcUnroll * xstep;
    }
    for (; r < r_end; r += kPhases) {
      const uint4 v = ld_nc_v4_hint(xp, keep);
      m0 = max_pairs(m0, v.x & kMag);
      m1 = max_pairs(m1, v.y & kMag);
      m2 = max_pairs(m2, v.z & kMag);
      m3 = max_pairs(m3, v.w & kMag);
      xp += xstep;
    }
  }
  // lanes SV p + cg of a warp hold the same vector for its row phases p
#pragma unroll
  for (int off = SV; off < 32; off <<= 1) {
    m0 = max_pairs(m0, __shfl_xor_sync(0xffffffffu, m0, off));
    m1 = max_pairs(m1, __shfl_xor_sync(0xffffffffu, m1, off));
    m2 = max_pairs(m2, __shfl_xor_sync(0xffffffffu, m2, off));
    m3 = max_pairs(m3, __shfl_xor_sync(0xffffffffu, m3, off));
  }
  if (lane < SV) {
    warp_max[warp][lane][0] = m0;
    warp_max[warp][lane][1] = m1;
    warp_max[warp][lane][2] = m2;
    warp_max[warp][lane][3] = m3;
  }
  __syncthreads();
  if (t < 4 * SV) {
    const int c = t >> 2, w = t & 3;
    uint32_t mm = warp_max[0][c][w];
#pragma unroll
    for (int k = 1; k < kWarps; ++k) mm = max_pairs(mm, warp_max[k][c][w]);
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
  if (!col_ok) return;
  if (rank == 0 && rp == 0) {
#pragma unroll
    for (int c = 0; c < 8; ++c) s[col_v * 8 + c] = g[c].s;
  }
  float2 r2[4], sn2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    r2[i] = make_float2(g[2 * i].r.x, g[2 * i + 1].r.x);
    sn2[i] = make_float2(g[2 * i].s_neg.x, g[2 * i + 1].s_neg.x);
  }
  // pass 2: the same rows again (from L2 while X fits there), coded; whole
  // groups of kPcUnroll rows without per-row checks, then the ragged rest
  const uint4* xp = xc + (r_begin + rp) * ldx_v;
  uint2* qp = q + (r_begin + rp) * ldq_v + col_v;
  const int64_t xstep = kPhases * ldx_v, qstep = kPhases * ldq_v;
  int64_t r = r_begin + rp;
  for (; r + kPhases * (kPcUnroll - 1) < r_end; r += kStep) {
    uint4 v[kPcUnroll];
#pragma unroll
    for (int i = 0; i < kPcUnroll; ++i) v[i] = ld_nc_v4_hint(xp + i * xstep, drop);
#pragma unroll
    for (int i = 0; i < kPcUnroll; ++i)
      st_global_v2_hint(qp + i * qstep, quantise8_cols_paired(v[i], r2, sn2, g, special0, special1), drop);
    xp += kPcUnroll * xstep;
    qp += kPcUnroll * qstep;
  }
  for (; r < r_end; r += kPhases) {
    st_global_v2_hint(qp, quantise8_cols_paired(ld_nc_v4_hint(xp, drop), r2, sn2, g, special0, special1), drop);
    xp += xstep;
    qp += qstep;
  }
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

cudaError_t launch_quant_per_channel(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* q, int64_t ldq, float* s, cudaStream_t stream) {
  (void)dev;
  const int64_t KV = K / 8;
  constexpr int kPhases = kPcThreads / kPcSV;
  int64_t rows_per_cta = (M + kPcCluster - 1) / kPcCluster;
  rows_per_cta = (rows_per_cta + kPhases - 1) / kPhases * kPhases;
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = kPcCluster;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((KV + kPcSV - 1) / kPcSV * kPcCluster), 1, 1);
  cfg.blockDim = dim3(kPcThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, quant_per_channel_kernel<kPcSV, kPcThreads>, static_cast<const uint4*>(x), M, KV,
                                           ldx / 8, rows_per_cta, static_cast<uint2*>(q), ldq / 8, s);
  return e == cudaSuccess ? cudaGetLastError() : e;
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
