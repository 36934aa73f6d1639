// backward.cu — operand preparation for the backward GEMMs of the FP8 linear
// layer on sm_103a.
//
// Method ("The Definitive Information To Deepseek"): the activation is kept in
// FP8 for the backward pass of the linear layer (paragraph 2) and the backward
// is split into its input-gradient and weight-gradient parts (paragraph 3),
// both run as FP8 GEMMs with the 1x128 / 128x128 grouping of "Figure 7 (a)".
//   dX = dY . W     needs W^T: a 128x128 block is a block either way round,
//                   so the codes and scales of W are transposed, not requantised
//                   (transpose_weight_128x128_kernel);
//   dW = dY^T . X   reduces over tokens, so dY and X are quantised on 1x128
//                   tiles of their transposes, i.e. per channel per 128 tokens
//                   (quant_act_1x128_t_kernel), and multiplied by the row-scaled
//                   GEMM (gemm.cu).  X may also come from its FP8 cache, the
//                   forward's 1x128 codes and scales: each value is dequantised
//                   to BF16 (bf16_rn(fl32(dec(q) * s))) in registers and then
//                   quantised the same way, without a BF16 copy of X in HBM.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_common.cuh"

namespace fp8bs {
namespace {

// ---------------------------------------------------------------------------
// 1x128 quantisation of X^T.  Tiles of 128 rows (tokens) x 128 columns
// (channels) of X arrive by TMA in a two-stage ring (persistent CTAs, three
// per SM): 64 KB of BF16 tiles, or 32 KB of FP8 code tiles when X comes from
// its FP8 cache.  Thread t owns the column pair cp = t % 64 (channels 2cp, 2cp+1)
// over the 32 rows 32 * (t / 64) ..; cached codes are dequantised to BF16 with
// their rows' scales as they are read (the tile's 128 row scales travel with
// it: a 512-byte bulk copy on the same barrier).  Per-column maxima combine across the
// four row quarters through shared memory; each thread then codes its 2 x 32
// values and writes them as two 32-byte runs of X^T's rows.  Scales go to
// s[m / 128][k] (the activation-scale layout of X^T).
// ---------------------------------------------------------------------------
template <bool FROM_FP8>
struct TQuant {
  // three CTAs per SM of two stages each: measured 4-5% faster than two
  // CTAs of three BF16 stages (or three of four code stages)
  static constexpr int kCtasPerSm = 3;
  static constexpr int kRingBytes = (FROM_FP8 ? 32 : 64) * 1024;
  static constexpr int kTileBytes = 128 * 128 * (FROM_FP8 ? 1 : 2);
  static constexpr int kStages = kRingBytes / kTileBytes;
  static constexpr int kScaleBytes = FROM_FP8 ? 128 * 4 : 0;  // per stage: the tile's row scales
  static constexpr int kOffBars = kRingBytes + kStages * kScaleBytes;
  static constexpr int kSmem = kOffBars + kStages * 8 + 4 * 64 * 4 + 1024;
};

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Gather 8 BF16 values of one column (low or high halves of 8 packed pairs).
__device__ __forceinline__ uint4 column8(const uint32_t* r, bool high) {
  const uint32_t sel = high ? 0x7632u : 0x5410u;
  return make_uint4(__byte_perm(r[0], r[1], sel), __byte_perm(r[2], r[3], sel), __byte_perm(r[4], r[5], sel),
                    __byte_perm(r[6], r[7], sel));
}

template <bool FROM_FP8>
__global__ void __launch_bounds__(256, TQuant<FROM_FP8>::kCtasPerSm) quant_act_1x128_t_kernel(const __grid_constant__ CUtensorMap tmX,
                                                                   int64_t MB, int64_t KB, uint4* __restrict__ q,
                                                                   int64_t ldq_v, float* __restrict__ s,
                                                                   int64_t ld_s, const float* __restrict__ sa,
                                                                   int64_t ld_sa, unsigned* status,
                                                                   uint64_t timeout_ns) {
  pdl_wait();
  constexpr int kTStages = TQuant<FROM_FP8>::kStages;
  constexpr int kTTileBytes = TQuant<FROM_FP8>::kTileBytes;
  constexpr int kScaleBytes = TQuant<FROM_FP8>::kScaleBytes;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw_addr);
  const uint32_t bar_full = base + TQuant<FROM_FP8>::kOffBars;
  uint32_t* quarter_max = reinterpret_cast<uint32_t*>(smem + TQuant<FROM_FP8>::kOffBars + kTStages * 8);  // [4][64]
  // load of tile t into stage st: the tile by TMA, plus (cached input) its
  // 128 row scales sa[kb][128 mb ..] by a bulk copy, on one barrier
  auto issue = [&](int st, int64_t t) {
    mbar_arrive_expect_tx(bar_full + 8 * st, kTTileBytes + kScaleBytes);
    tma_load_2d(base + st * kTTileBytes, &tmX, bar_full + 8 * st, static_cast<int32_t>((t % KB) * 128),
                static_cast<int32_t>((t / KB) * 128));
    if constexpr (FROM_FP8)
      bulk_load_1d(base + TQuant<FROM_FP8>::kRingBytes + st * kScaleBytes, sa + (t % KB) * ld_sa + (t / KB) * 128, kScaleBytes,
                   bar_full + 8 * st);
  };

  const int64_t tiles = MB * KB;
  const int64_t first = blockIdx.x, stride = gridDim.x;
  const int cp = threadIdx.x & 63;
  const int rq = threadIdx.x >> 6;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kTStages; ++st) mbar_init(bar_full + 8 * st, 1);
    fence_mbar_init();
    prefetch_tmap(&tmX);
    for (int st = 0; st < kTStages; ++st) {
      const int64_t t = first + st * stride;
      if (t >= tiles) break;
      issue(st, t);
    }
  }
  __syncthreads();

  int64_t i = 0;
  for (int64_t t = first; t < tiles; t += stride, ++i) {
    const int st = static_cast<int>(i % kTStages);
    const uint32_t parity = static_cast<uint32_t>((i / kTStages) & 1);
    const int64_t mb = t / KB, kb = t % KB;
    const bool landed = mbar_wait(bar_full + 8 * st, parity, nullptr, timeout_ns);
    if (!__syncthreads_and(landed)) {
      if (threadIdx.x == 0) {
        record_status(status, kStatusTimeout);
        for (int k = 0; k < kTStages; ++k) {
          const int64_t j = i + k;
          if (first + j * stride >= tiles) break;
          (void)mbar_wait(bar_full + 8 * (j % kTStages), static_cast<uint32_t>((j / kTStages) & 1), nullptr,
                          timeout_ns);
        }
      }
      return;
    }
    const uint8_t* tile = smem + st * kTTileBytes;
    uint32_t r[32];  // BF16 pairs of rows 32 rq + j, columns 2cp (low half) and 2cp + 1 (high half)
    if constexpr (FROM_FP8) {
      const float* row_s = reinterpret_cast<const float*>(smem + TQuant<FROM_FP8>::kRingBytes + st * kScaleBytes) + 32 * rq;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t c2 = *reinterpret_cast<const uint16_t*>(tile + (32 * rq + j) * 128 + cp * 2);
        const float sj = row_s[j];
        r[j] = bf16x2_rn(__fmul2_rn(e4m3x2_to_f32x2(c2), make_float2(sj, sj)));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) r[j] = *reinterpret_cast<const uint32_t*>(tile + (32 * rq + j) * 256 + cp * 4);
    }
    uint32_t m = r[0] & 0x7FFF7FFFu;
#pragma unroll
    for (int j = 1; j < 32; ++j) m = max_pairs(m, r[j] & 0x7FFF7FFFu);
    quarter_max[rq * 64 + cp] = m;
    __syncthreads();  // quarter maxima visible; stage st fully read into registers
    if (threadIdx.x == 0) {
      const int64_t tn = t + kTStages * stride;
      if (tn < tiles) issue(st, tn);
    }
    m = max_pairs(max_pairs(quarter_max[cp], quarter_max[64 + cp]),
                  max_pairs(quarter_max[128 + cp], quarter_max[192 + cp]));
    const GroupScale g_lo = group_scale(bf16lo_to_f32(m));
    const GroupScale g_hi = group_scale(bf16hi_to_f32(m));
    const int64_t k0 = kb * 128 + 2 * cp;
    // X^T rows k0 and k0 + 1, tokens mb * 128 + 32 rq .. + 31: two 16-byte stores each
    uint4* dst_lo = q + k0 * ldq_v + mb * 8 + rq * 2;
    uint4* dst_hi = dst_lo + ldq_v;
    const uint2 a0 = quantise8(column8(r + 0, false), g_lo), a1 = quantise8(column8(r + 8, false), g_lo);
    const uint2 a2 = quantise8(column8(r + 16, false), g_lo), a3 = quantise8(column8(r + 24, false), g_lo);
    dst_lo[0] = make_uint4(a0.x, a0.y, a1.x, a1.y);
    dst_lo[1] = make_uint4(a2.x, a2.y, a3.x, a3.y);
    const uint2 b0 = quantise8(column8(r + 0, true), g_hi), b1 = quantise8(column8(r + 8, true), g_hi);
    const uint2 b2 = quantise8(column8(r + 16, true), g_hi), b3 = quantise8(column8(r + 24, true), g_hi);
    dst_hi[0] = make_uint4(b0.x, b0.y, b1.x, b1.y);
    dst_hi[1] = make_uint4(b2.x, b2.y, b3.x, b3.y);
    if (rq == 0) *reinterpret_cast<float2*>(s + mb * ld_s + k0) = make_float2(g_lo.s, g_hi.s);
    // quarter_max is rewritten only after the next tile's __syncthreads_and,
    // which every thread reaches after its reads above
  }
}

// ---------------------------------------------------------------------------
// 128x128 code blocks of W [N, K] -> W^T [K, N], and the block-scale matrix
// transposed.  One CTA per block, N blocks fastest in the grid (concurrent
// CTAs then write adjacent 128-byte pieces of the same W^T rows, which
// measured faster than reading adjacent pieces of the same W rows): the block
// arrives in shared memory by one TMA copy, then thread t takes the input
// columns 4 (t % 32) .. + 3 over the 16 rows 16 (t / 32) .., reading 4x4 byte
// squares with 32-bit loads and transposing them with byte permutes; each of
// its 4 output rows leaves as one 16-byte run.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) transpose_weight_128x128_kernel(const __grid_constant__ CUtensorMap tmQ,
                                                                       int64_t NB, int64_t KB,
                                                                       const float* __restrict__ sw,
                                                                       uint4* __restrict__ qt, int64_t ldqt_v,
                                                                       float* __restrict__ swt, unsigned* status,
                                                                       uint64_t timeout_ns) {
  pdl_wait();
  __shared__ __align__(128) uint8_t blk[128 * 128];
  __shared__ __align__(8) uint64_t bar_storage;
  const uint32_t bar = smem_u32(&bar_storage);
  const int cg = threadIdx.x & 31;  // input columns 4 cg .. 4 cg + 3 = output rows
  const int rg = threadIdx.x >> 5;  // input rows 16 rg .. 16 rg + 15 = output columns
  const int64_t nb = blockIdx.x;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    prefetch_tmap(&tmQ);
  }
  __syncthreads();
  uint32_t parity = 0;
  for (int64_t kb = blockIdx.y; kb < KB; kb += gridDim.y) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(bar, 128 * 128);
      tma_load_2d(smem_u32(blk), &tmQ, bar, static_cast<int32_t>(kb * 128), static_cast<int32_t>(nb * 128));
    }
    const bool landed = mbar_wait(bar, parity, nullptr, timeout_ns);
    if (!__syncthreads_and(landed)) {
      // let the copy in flight land before shared memory goes away
      if (threadIdx.x == 0) {
        record_status(status, kStatusTimeout);
        (void)mbar_wait(bar, parity, nullptr, timeout_ns);
      }
      return;
    }
    parity ^= 1u;
    uint32_t o[4][4];  // o[c][w]: output row 4 cg + c, bytes of input rows 16 rg + 4 w .. + 3
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const uint8_t* src = blk + (16 * rg + 4 * w) * 128 + 4 * cg;
      const uint32_t a0 = *reinterpret_cast<const uint32_t*>(src);
      const uint32_t a1 = *reinterpret_cast<const uint32_t*>(src + 128);
      const uint32_t a2 = *reinterpret_cast<const uint32_t*>(src + 256);
      const uint32_t a3 = *reinterpret_cast<const uint32_t*>(src + 384);
      const uint32_t t0 = __byte_perm(a0, a1, 0x5140), t1 = __byte_perm(a0, a1, 0x7362);
      const uint32_t t2 = __byte_perm(a2, a3, 0x5140), t3 = __byte_perm(a2, a3, 0x7362);
      o[0][w] = __byte_perm(t0, t2, 0x5410);
      o[1][w] = __byte_perm(t0, t2, 0x7632);
      o[2][w] = __byte_perm(t1, t3, 0x5410);
      o[3][w] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      qt[(kb * 128 + 4 * cg + c) * ldqt_v + nb * 8 + rg] = make_uint4(o[c][0], o[c][1], o[c][2], o[c][3]);
    }
    if (threadIdx.x == 0) swt[kb * NB + nb] = sw[nb * KB + kb];
    __syncthreads();  // blk is refilled for the next block of this CTA
  }
}

constexpr int64_t kMaxGridY = 65535;

}  // namespace

template <bool FROM_FP8>
cudaError_t launch_quant_t(const DeviceInfo& dev, const CUtensorMap& tmX, int64_t M, int64_t K, void* qt,
                           int64_t ldqt, float* st, int64_t ld_st, const float* sa, int64_t ld_sa,
                           cudaStream_t stream) {
  const int64_t MB = M / 128, KB = K / 128;
  constexpr int kSmem = TQuant<FROM_FP8>::kSmem;
  cudaError_t e =
      cudaFuncSetAttribute(quant_act_1x128_t_kernel<FROM_FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int64_t tiles = MB * KB;
  const int64_t resident = static_cast<int64_t>(dev.num_sms) * TQuant<FROM_FP8>::kCtasPerSm;
  const int grid = static_cast<int>(tiles < resident ? tiles : resident);
  (void)launch_pdl(quant_act_1x128_t_kernel<FROM_FP8>, grid, 256, kSmem, stream,
      tmX, MB, KB, static_cast<uint4*>(qt), ldqt / 16, st, ld_st, sa, ld_sa, dev.status, wait_timeout_ns());
  return cudaGetLastError();
}

cudaError_t launch_quant_act_1x128_t(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* qt, int64_t ldqt, float* st, int64_t ld_st, cudaStream_t stream) {
  CUtensorMap tmX;
  if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, K, M, ldx * 2, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_quant_t<false>(dev, tmX, M, K, qt, ldqt, st, ld_st, nullptr, 0, stream);
}

cudaError_t launch_requant_act_1x128_t(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                       int64_t ld_sa, int64_t M, int64_t K, void* qt, int64_t ldqt, float* st,
                                       int64_t ld_st, cudaStream_t stream) {
  CUtensorMap tmX;
  if (!make_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, ldqa, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  return launch_quant_t<true>(dev, tmX, M, K, qt, ldqt, st, ld_st, sa, ld_sa, stream);
}

cudaError_t launch_transpose_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                            const float* sw, void* qt, int64_t ldqt, float* swt,
                                            cudaStream_t stream) {
  const int64_t NB = N / 128, KB = K / 128;
  CUtensorMap tmQ;
  if (!make_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_UINT8, q, K, N, ldq, 128, 128, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(NB), static_cast<unsigned>(KB < kMaxGridY ? KB : kMaxGridY));
  (void)launch_pdl(transpose_weight_128x128_kernel, grid, 256, 0, stream, tmQ, NB, KB, sw, static_cast<uint4*>(qt),
                   ldqt / 16, swt, dev.status, wait_timeout_ns());
  return cudaGetLastError();
}

}  // namespace fp8bs
