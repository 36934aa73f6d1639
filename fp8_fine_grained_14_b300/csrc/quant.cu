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
// element), so the arithmetic per element is kept to a handful of
// instructions: packed BF16 abs-max, a division-free exact scale, the exact
// quotient from a correctly rounded reciprocal and one packed FMA correction,
// and the hardware E4M3 pair conversion.  The build never enables fast math or flush-to-zero; codes and
// scales are bit-identical to the float32 definition (see group_scale and
// quantise8 for why).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_common.cuh"

namespace fp8bs {
namespace {

// ---------------------------------------------------------------------------
// 1x128 activation tiles.
//
// Grid: x over groups of U consecutive 128-channel groups, y over tiles of 32
// rows.  A CTA of 256 threads = 32 eight-lane teams; team r owns row
// (32 * tile + r) and each of its 8 lanes holds 16 channels (two 16-byte
// vectors) of a group, so the codes leave as one 16-byte store per lane.  The
// 2U loads of a thread are issued before any arithmetic.
// ---------------------------------------------------------------------------
template <int U>
__global__ void __launch_bounds__(256, 6) quant_act_1x128_kernel(const uint4* __restrict__ x, int64_t M, int64_t KB,
                                                              int64_t ldx_v, uint4* __restrict__ q, int64_t ldq_v,
                                                              float* __restrict__ sa, int64_t ld_sa) {
  pdl_wait();
  // The codes usually feed the GEMM next: let it set up (and pull its first
  // weight stages into L2) while this kernel finishes.
  pdl_launch_dependents();
  const int lane8 = threadIdx.x & 7;
  const int r = threadIdx.x >> 3;  // 32 rows per CTA
  const int64_t kb0 = static_cast<int64_t>(blockIdx.x) * U;
  const int64_t tiles_m = (M + 31) / 32;
  for (int64_t tm = blockIdx.y; tm < tiles_m; tm += gridDim.y) {
    const int64_t row = tm * 32 + r;
    const bool row_ok = row < M;
    const uint4* src = x + row * ldx_v + kb0 * 16 + lane8 * 2;
    uint4 v[U][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      v[u][0] = v[u][1] = make_uint4(0u, 0u, 0u, 0u);
      if (row_ok && kb0 + u < KB) {
        v[u][0] = ld_nc_v4(src + u * 16);
        v[u][1] = ld_nc_v4(src + u * 16 + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      uint32_t m = max_pairs(absmax8_pairs(v[u][0]), absmax8_pairs(v[u][1]));
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) m = max_pairs(m, __shfl_xor_sync(0xffffffffu, m, off));
      const GroupScale g = group_scale(pairs_to_max(m));
      const int64_t kb = kb0 + u;
      if (row_ok && kb < KB) {
        const uint2 c0 = quantise8(v[u][0], g), c1 = quantise8(v[u][1], g);
        q[row * ldq_v + kb * 8 + lane8] = make_uint4(c0.x, c0.y, c1.x, c1.y);
        if (lane8 == 0) sa[kb * ld_sa + row] = g.s;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// 128x128 weight blocks: one CTA per block (grid x over K blocks, y over N
// blocks).  Thread t holds the 16-byte column slice (t % 16) of rows
// (t / 16) + 16 i, i = 0..7, i.e. the whole block sits in registers and is
// read from HBM exactly once.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 3) quant_weight_128x128_kernel(const uint4* __restrict__ w, int64_t NB,
                                                                      int64_t KB, int64_t ldw_v,
                                                                      uint2* __restrict__ q, int64_t ldq_v,
                                                                      float* __restrict__ sw) {
  pdl_wait();
  __shared__ uint32_t warp_max[8];
  const int c = threadIdx.x & 15;
  const int r0 = threadIdx.x >> 4;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t kb = blockIdx.x;
  for (int64_t nb = blockIdx.y; nb < NB; nb += gridDim.y) {
    const uint4* src = w + (nb * 128 + r0) * ldw_v + kb * 16 + c;
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = ld_nc_v4(src + 16 * i * ldw_v);
    uint32_t m = absmax8_pairs(v[0]);
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max_pairs(m, absmax8_pairs(v[i]));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = max_pairs(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (lane == 0) warp_max[warp] = m;
    __syncthreads();
    m = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) m = max_pairs(m, warp_max[i]);
    __syncthreads();  // warp_max is reused by the next block of this CTA
    const GroupScale g = group_scale(pairs_to_max(m));
    if (threadIdx.x == 0) sw[nb * KB + kb] = g.s;
    // The codes leave with an evict-first L2 policy: a weight matrix is larger
    // than L2 and is not read back by this kernel, so its lines should not
    // displace other data (in a layer step, the activation that is quantised
    // next saw its time drop by about 0.8 us on X [4096, 7168]).
    uint2* dst = q + (nb * 128 + r0) * ldq_v + kb * 16 + c;
    const uint64_t policy = l2_evict_first_policy();
#pragma unroll
    for (int i = 0; i < 8; ++i) st_global_v2_hint(dst + 16 * i * ldq_v, quantise8(v[i], g), policy);
  }
}

// ---------------------------------------------------------------------------
// 128x128 block dequantisation (FP8 codes + block scale -> BF16), the
// inverse of the weight quantiser: y = bf16_rn(fl32(dec(q) * s)).  E4M3
// values are exact in FP16, so each code pair is widened with the hardware
// e4m3x2 -> f16x2 conversion, then to FP32, multiplied by the block scale
// (one rounding) and rounded to BF16.  One CTA per block (grid x over K
// blocks, y over N blocks); thread t handles 16 codes (one 16-byte chunk) of
// rows (t / 8) + 32 i, i = 0..3.
// ---------------------------------------------------------------------------
// 4 codes (one 32-bit word) -> 4 BF16 values (two 32-bit words).
__device__ __forceinline__ uint2 dequant4(uint32_t codes, float2 s2) {
  const float2 lo = __fmul2_rn(e4m3x2_to_f32x2(codes & 0xFFFFu), s2);
  const float2 hi = __fmul2_rn(e4m3x2_to_f32x2(codes >> 16), s2);
  return make_uint2(bf16x2_rn(lo), bf16x2_rn(hi));
}

// Each CTA takes the K block blockIdx.x of a pair of N blocks (2 blockIdx.y,
// 2 blockIdx.y + 1) and issues the loads of both before converting either.
__global__ void __launch_bounds__(256) dequant_weight_128x128_kernel(const uint4* __restrict__ q, int64_t NB,
                                                                     int64_t KB, int64_t ldq_v,
                                                                     const float* __restrict__ sw,
                                                                     uint4* __restrict__ y, int64_t ldy_v) {
  pdl_wait();
  const int c = threadIdx.x & 7;
  const int r0 = threadIdx.x >> 3;
  const int64_t kb = blockIdx.x;
  for (int64_t nb0 = 2 * static_cast<int64_t>(blockIdx.y); nb0 < NB; nb0 += 2 * static_cast<int64_t>(gridDim.y)) {
    const int nblk = nb0 + 1 < NB ? 2 : 1;
    uint4 v[2][4];
    float s[2];
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (b < nblk) {
        const int64_t nb = nb0 + b;
        s[b] = __ldg(sw + nb * KB + kb);
        const uint4* src = q + (nb * 128 + r0) * ldq_v + kb * 8 + c;
#pragma unroll
        for (int i = 0; i < 4; ++i) v[b][i] = ld_nc_v4(src + 32 * i * ldq_v);
      }
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      if (b < nblk) {
        const float2 s2 = make_float2(s[b], s[b]);
        uint4* dst = y + ((nb0 + b) * 128 + r0) * ldy_v + kb * 16 + 2 * c;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint2 a = dequant4(v[b][i].x, s2), bb = dequant4(v[b][i].y, s2);
          const uint2 d = dequant4(v[b][i].z, s2), e = dequant4(v[b][i].w, s2);
          dst[32 * i * ldy_v] = make_uint4(a.x, a.y, bb.x, bb.y);
          dst[32 * i * ldy_v + 1] = make_uint4(d.x, d.y, e.x, e.y);
        }
      }
    }
  }
}

constexpr int64_t kMaxGridY = 65535;

}  // namespace

cudaError_t launch_quant_act_1x128(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                   int64_t ldq, float* sa, int64_t ld_sa, cudaStream_t stream) {
  (void)dev;
  // Two 128-channel groups per thread: small work units keep the last wave of
  // CTAs short (the grid is several waves of 8 resident CTAs per SM).
  constexpr int kUnroll = 2;
  const int64_t KB = K / 128;
  const int64_t tiles_m = (M + 31) / 32;
  const dim3 grid(static_cast<unsigned>((KB + kUnroll - 1) / kUnroll),
                  static_cast<unsigned>(tiles_m < kMaxGridY ? tiles_m : kMaxGridY));
  (void)launch_pdl(quant_act_1x128_kernel<kUnroll>, grid, 256, 0, stream, static_cast<const uint4*>(x), M, KB, ldx / 8,
                                                            static_cast<uint4*>(q), ldq / 16, sa, ld_sa);
  return cudaGetLastError();
}

cudaError_t launch_quant_weight_128x128(const DeviceInfo& dev, const void* w, int64_t N, int64_t K, int64_t ldw,
                                        void* q, int64_t ldq, float* sw, cudaStream_t stream) {
  (void)dev;
  const int64_t NB = N / 128, KB = K / 128;
  const dim3 grid(static_cast<unsigned>(KB), static_cast<unsigned>(NB < kMaxGridY ? NB : kMaxGridY));
  (void)launch_pdl(quant_weight_128x128_kernel, grid, 256, 0, stream, static_cast<const uint4*>(w), NB, KB, ldw / 8,
                                                        static_cast<uint2*>(q), ldq / 8, sw);
  return cudaGetLastError();
}

cudaError_t launch_dequant_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                          const float* sw, void* y, int64_t ldy, cudaStream_t stream) {
  (void)dev;
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t pairs = (NB + 1) / 2;
  const dim3 grid(static_cast<unsigned>(KB), static_cast<unsigned>(pairs < kMaxGridY ? pairs : kMaxGridY));
  (void)launch_pdl(dequant_weight_128x128_kernel, grid, 256, 0, stream, static_cast<const uint4*>(q), NB, KB, ldq / 16, sw,
                                                          static_cast<uint4*>(y), ldy / 8);
  return cudaGetLastError();
}

}  // namespace fp8bs
