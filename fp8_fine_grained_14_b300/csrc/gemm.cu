// gemm.cu — block-scaled FP8 GEMM with per-128-K-chunk FP32 promotion for
// sm_103a (tcgen05 + TMA), dense and grouped (MoE) variants.
//
// Method ("The Definitive Information To Deepseek"): FP8 GEMM inputs, BF16
// output (paragraph 4); activation scales per 1x128 tile and weight scales per
// 128x128 block ("Figure 7 (a)", paragraph 3); partial sums are promoted to a
// higher-precision accumulator while the next MMA runs (paragraph 1, where
// H800 alternates two warpgroups between WGMMA and promotion).  On sm_103a
// the same overlap comes from two TMEM accumulator buffers:
//
//   warp 0      TMA producer: A (128x128 codes) and B (BNx128 codes) per K
//               chunk into a STAGES-deep shared-memory ring (mbarrier full/empty)
//   warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma kind::f8f6f4
//               (K = 32 each) per chunk into TMEM buffer (chunk & 1), then
//               tcgen05.commit to free the smem stage and publish the chunk
//   warps 2..3  idle (their warpgroup gives registers to the promotion warps)
//   warps 4..11 promotion: tcgen05.ld the chunk (one row per thread, 64
//               columns per load), hand the TMEM buffer back as soon as the
//               chunk is in registers, then acc += chunk * (sa[kb][m] *
//               sw[nb][kb]) with packed FP32 FMAs (two columns per instruction);
//               after the last chunk, BF16 (RNE) -> swizzled smem -> TMA store
//               (dense) or row-masked coalesced stores (grouped)
//
// While the promotion warps drain buffer b, the MMA warp fills buffer b^1.
// The kernel is persistent: CTA i handles tiles i, i + grid, ...; tiles are
// ordered M-fastest so a wave of CTAs shares a few weight column blocks
// (L2-resident) and the whole activation matrix.
//
// Every mbarrier wait is bounded (see ptx.cuh).  A wait that gives up records
// a timeout in the status word and raises a CTA-wide abort flag; every role
// then leaves its loop, the producer drains its TMA loads, the MMA warp waits
// for its last commits, and TMEM is released before the CTA exits.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

constexpr int BM = 128;               // rows per tile (= MMA M, one TMEM lane per row)
constexpr int BK = 128;               // K chunk = one scale group = one 128-byte swizzle row
constexpr int MMA_K = 32;             // K per tcgen05.mma for 8-bit operands
constexpr int kThreads = 384;         // 12 warps = 3 warpgroups
constexpr int kEpiWarps = 8;          // warps 4..11
constexpr int kFirstEpiWarp = 4;
constexpr int kStagingBytes = 4096;   // per promotion warp: 32 rows x 64 BF16
constexpr int kEpiCols = 64;          // columns per TMA store box
// Register split for 256-wide tiles (setmaxnreg): warpgroup 0 (TMA, MMA,
// idle) drops to RegSplit::low, the two promotion warpgroups rise to
// RegSplit::high.  Every SM sub-partition hosts one warp of each warpgroup, so
// the split is balanced per sub-partition: low + 2 * high == 3 * launch.  The
// grouped tile walker needs a few more registers on the producer side.
constexpr int kRegsLaunch = 168;
static_assert(kRegsLaunch * kThreads <= 65536, "register file");
template <bool GROUPED>
struct RegSplit {
  static constexpr int low = GROUPED ? 72 : 56;
  static constexpr int high = GROUPED ? 216 : 224;
  static_assert(low + 2 * high == 3 * kRegsLaunch, "register split must match the launch allocation");
  static_assert(low % 8 == 0 && high % 8 == 0, "setmaxnreg takes multiples of 8");
};

struct Params {
  const float* sa;
  int64_t ld_sa;
  const float* sw;
  __nv_bfloat16* y;     // grouped: direct stores
  int64_t ldy;
  int32_t M;            // rows of A (M_total when grouped)
  int32_t N;
  int32_t KB;           // K / 128
  const int32_t* offsets;  // grouped only, [G+1]
  int32_t G;
  unsigned* status;
  uint64_t timeout_ns;
};

template <int BN, int STAGES>
struct Smem {
  static constexpr int kA = BM * BK;
  static constexpr int kB = BN * BK;
  static constexpr int kOffA = 0;
  static constexpr int kOffB = kOffA + STAGES * kA;
  static constexpr int kOffStaging = kOffB + STAGES * kB;
  static constexpr int kOffBar = kOffStaging + kEpiWarps * kStagingBytes;
  // full[STAGES], empty[STAGES], tmem_full[2], tmem_empty[2]
  static constexpr int kOffSlot = kOffBar + (2 * STAGES + 4) * 8;
  static constexpr int kOffAbort = kOffSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kDynamic = kBytes + 1024;  // + alignment slack
};

// Tile walker shared by all roles: yields (a_row, row_end, b_row, n0, group)
// for this CTA's tiles in order.  Dense: one group of M rows.  Grouped:
// group g has rows off[g] .. off[g+1]-1 and weight rows g*N .. g*N+N-1.
template <bool GROUPED, int BN>
struct TileWalker {
  const Params& p;
  int64_t next;        // next global tile index for this CTA
  int32_t n_tiles;     // N / BN
  // grouped state
  int32_t g;
  int64_t tiles_before;  // tiles of groups < g
  int32_t g_row0, g_row1, g_mtiles;

  __device__ TileWalker(const Params& p_) : p(p_), next(blockIdx.x), n_tiles(p_.N / BN), g(0), tiles_before(0) {
    if (GROUPED) load_group();
  }
  __device__ void load_group() {
    if (g >= p.G) return;
    int32_t r0 = __ldg(p.offsets + g), r1 = __ldg(p.offsets + g + 1);
    if (r0 < 0 || r1 < r0 || r1 > p.M) {
      record_status(p.status, kStatusBadOffsets);
      r1 = r0 = 0;
    }
    g_row0 = r0;
    g_row1 = r1;
    g_mtiles = (r1 - r0 + BM - 1) / BM;
  }
  // Returns false when this CTA has no more tiles.
  __device__ bool get(int32_t& a_row, int32_t& row_end, int32_t& b_row, int32_t& n0, int32_t& group) {
    const int64_t t = next;
    next += gridDim.x;
    if (!GROUPED) {
      const int32_t m_tiles = (p.M + BM - 1) / BM;
      if (t >= static_cast<int64_t>(m_tiles) * n_tiles) return false;
      const int32_t mt = static_cast<int32_t>(t % m_tiles);
      const int32_t nt = static_cast<int32_t>(t / m_tiles);
      a_row = mt * BM;
      row_end = p.M;
      n0 = nt * BN;
      b_row = n0;
      group = 0;
      return true;
    } else {
      while (g < p.G && t >= tiles_before + static_cast<int64_t>(g_mtiles) * n_tiles) {
        tiles_before += static_cast<int64_t>(g_mtiles) * n_tiles;
        ++g;
        load_group();
      }
      if (g >= p.G) return false;
      const int64_t local = t - tiles_before;
      const int32_t mt = static_cast<int32_t>(local % g_mtiles);
      const int32_t nt = static_cast<int32_t>(local / g_mtiles);
      a_row = g_row0 + mt * BM;
      row_end = g_row1;
      n0 = nt * BN;
      b_row = g * p.N + n0;
      group = g;
      return true;
    }
  }
};

__device__ __forceinline__ void abort_cta(volatile int* abort_flag, unsigned* status) {
  *abort_flag = 1;
  record_status(status, kStatusTimeout);
}

template <int BN, int STAGES, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1)
    blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmY, const Params p) {
  using L = Smem<BN, STAGES>;
  constexpr int kTmemCols = 2 * BN;   // two accumulator buffers
  constexpr int kHalfCols = BN / 2;   // columns per promotion warp
  constexpr uint32_t kStageTx = L::kA + L::kB;
  constexpr uint32_t kIdesc = idesc_e4m3_f32(BM, BN);
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
  static_assert(kHalfCols % kEpiCols == 0, "epilogue boxes");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;  // 1024-aligned for the 128B swizzle
  uint8_t* smem = smem_raw + (base - raw_addr);

  const uint32_t bar_full = base + L::kOffBar;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  const uint32_t bar_tfull = bar_empty + STAGES * 8;
  const uint32_t bar_tempty = bar_tfull + 2 * 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kOffSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kEpiWarps);
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (!GROUPED) prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    tmem_alloc(base + L::kOffSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;

  TileWalker<GROUPED, BN> tiles(p);
  int32_t a_row, row_end, b_row, n0, group;

  if (warp < kFirstEpiWarp) {
    // 128 FP32 accumulators per promotion thread (BN = 256) need more than the
    // launch allocation: this warpgroup hands registers to the other two.
    if (BN == 256) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<GROUPED>::low));
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer ----------------
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // per stage: ever issued / parity of last issue
      bool ok = true;
      while (ok && tiles.get(a_row, row_end, b_row, n0, group)) {
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns)) {
            abort_cta(abort_flag, p.status);
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * stage;
          mbar_arrive_expect_tx(full, kStageTx);
          tma_load_2d(base + L::kOffA + stage * L::kA, &tmA, full, kb * BK, a_row);
          tma_load_2d(base + L::kOffB + stage * L::kB, &tmB, full, kb * BK, b_row);
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every load already issued land before shared memory goes away.
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s))
            (void)mbar_wait(bar_full + 8 * s, (issued_parity >> s) & 1u, nullptr, p.timeout_ns);
      }
    } else if (warp == 1 && lane == 0) {
      // ---------------- MMA issuer ----------------
      uint32_t stage = 0, phase = 0, buf = 0, bphase = 0;
      uint32_t committed = 0, committed_parity = 0;  // per TMEM buffer: ever committed / parity of last commit
      bool ok = true;
      while (ok && tiles.get(a_row, row_end, b_row, n0, group)) {
        for (int kb = 0; kb < p.KB; ++kb) {
          if (!mbar_wait(bar_tempty + 8 * buf, bphase ^ 1u, abort_flag, p.timeout_ns) ||
              !mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.timeout_ns)) {
            abort_cta(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d = tmem_base + buf * BN;
          const uint64_t adesc = smem_desc_k128_sw128(base + L::kOffA + stage * L::kA);
          const uint64_t bdesc = smem_desc_k128_sw128(base + L::kOffB + stage * L::kB);
#pragma unroll
          for (int k = 0; k < BK / MMA_K; ++k) {
            // advance the start address by 32 bytes (2 units of 16 B) per K step
            mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
          }
          mma_commit(bar_empty + 8 * stage);  // smem stage reusable once these MMAs finish
          mma_commit(bar_tfull + 8 * buf);    // chunk kb ready in TMEM buffer `buf`
          committed |= 1u << buf;
          committed_parity = (committed_parity & ~(1u << buf)) | (bphase << buf);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          buf ^= 1u;
          if (buf == 0) bphase ^= 1u;
        }
      }
      if (!ok) {
        // No MMA may still be writing TMEM when it is released.
        for (int b = 0; b < 2; ++b)
          if (committed & (1u << b))
            (void)mbar_wait(bar_tfull + 8 * b, (committed_parity >> b) & 1u, nullptr, p.timeout_ns);
      }
    }
  } else {
    if (BN == 256) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RegSplit<GROUPED>::high));
    // ---------------- promotion + epilogue (warps 4..11) ----------------
    const int q = warp & 3;                        // TMEM lane quarter this warp may access
    const int half = (warp - kFirstEpiWarp) >> 2;  // which half of the tile's columns
    const int epi = warp - kFirstEpiWarp;
    const uint32_t staging = base + L::kOffStaging + epi * kStagingBytes;
    uint8_t* staging_ptr = smem + L::kOffStaging + epi * kStagingBytes;
    uint32_t buf = 0, bphase = 0;
    bool ok = true;
    while (ok && tiles.get(a_row, row_end, b_row, n0, group)) {
      const int32_t row = a_row + q * 32 + lane;  // this thread's output row
      const bool row_ok = row < row_end;
      // rows past the end read a valid row's scale (no divergent loads) and drop it
      const float* sa_col = p.sa + (row_ok ? row : a_row);
      const float row_mask = row_ok ? 1.0f : 0.0f;
      const int32_t col0 = n0 + half * kHalfCols;  // first column of this warp
      const float* sw_row = p.sw + (static_cast<int64_t>(group) * (p.N / 128) + col0 / 128) * p.KB;
      // Pairs of FP32 accumulators, updated with packed FP32 FMAs.
      float2 acc[kHalfCols / 2];
#pragma unroll
      for (int i = 0; i < kHalfCols / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

      float sa_next = __ldg(sa_col);
      float sw_next = __ldg(sw_row);
      for (int kb = 0; kb < p.KB; ++kb) {
        const float scale = sa_next * sw_next * row_mask;
        const float2 scale2 = make_float2(scale, scale);
        const int kn = kb + 1 < p.KB ? kb + 1 : kb;  // prefetch the next chunk's scales
        sa_next = __ldg(sa_col + static_cast<int64_t>(kn) * p.ld_sa);
        sw_next = __ldg(sw_row + kn);
        const bool waited = mbar_wait(bar_tfull + 8 * buf, bphase, abort_flag, p.timeout_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          abort_cta(abort_flag, p.status);
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + half * kHalfCols;
#pragma unroll
        for (int c = 0; c < kHalfCols / 64; ++c) {
          uint32_t r[64];
          tmem_ld_x64(taddr + c * 64, r);
          tmem_wait_ld(r);
          if (c == kHalfCols / 64 - 1) {
            // the whole chunk is in registers: hand the buffer back to the
            // MMA warp before the last FMAs
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_tempty + 8 * buf);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j)
            acc[c * 32 + j] =
                __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), scale2,
                           acc[c * 32 + j]);
        }
        buf ^= 1u;
        if (buf == 0) bphase ^= 1u;
      }
      if (!ok) break;

      // ---- epilogue: BF16 (RNE), swizzled staging, store ----
#pragma unroll
      for (int piece = 0; piece < kHalfCols / kEpiCols; ++piece) {
        if (!GROUPED) {
          if (lane == 0) tma_store_wait_read_all();  // staging free again
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int c0 = (piece * kEpiCols + j * 8) / 2;
          __nv_bfloat162 h0 = __float22bfloat162_rn(acc[c0 + 0]);
          __nv_bfloat162 h1 = __float22bfloat162_rn(acc[c0 + 1]);
          __nv_bfloat162 h2 = __float22bfloat162_rn(acc[c0 + 2]);
          __nv_bfloat162 h3 = __float22bfloat162_rn(acc[c0 + 3]);
          uint4 v;
          v.x = *reinterpret_cast<uint32_t*>(&h0);
          v.y = *reinterpret_cast<uint32_t*>(&h1);
          v.z = *reinterpret_cast<uint32_t*>(&h2);
          v.w = *reinterpret_cast<uint32_t*>(&h3);
          // 128-byte swizzle: 16-byte chunk j of row `lane` sits at chunk j ^ (lane % 8)
          *reinterpret_cast<uint4*>(staging_ptr + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
        }
        if (!GROUPED) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, staging, col0 + piece * kEpiCols, a_row + q * 32);
            tma_store_commit();
          }
        } else {
          __syncwarp();
          // 32 rows x 128 bytes: lane reads chunk (lane % 8) of rows lane/8 + 4i
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (lane >> 3) + 4 * i;
            const int ch = lane & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(staging_ptr + r * 128 + ((ch ^ (r & 7)) << 4));
            const int32_t grow = a_row + q * 32 + r;
            if (grow < row_end)
              *reinterpret_cast<uint4*>(p.y + static_cast<int64_t>(grow) * p.ldy + col0 + piece * kEpiCols + ch * 8) =
                  v;
          }
          __syncwarp();
        }
      }
    }
    if (!GROUPED && lane == 0) tma_store_wait_all();
  }

  // ---------------- teardown ----------------
  __syncwarp();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

template <int BN, int STAGES, bool GROUPED>
cudaError_t launch_kernel(const DeviceInfo& dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                          const CUtensorMap& tmY, const Params& p, int grid, cudaStream_t stream) {
  using L = Smem<BN, STAGES>;
  auto kernel = blockscaled_gemm_kernel<BN, STAGES, GROUPED>;
  if (BN == 256) {
    // setmaxnreg.inc only completes if the launch holds kRegsLaunch registers
    // per thread; refuse to launch a build that does not.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.numRegs != kRegsLaunch) return cudaErrorInvalidConfiguration;
  }
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamic);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, L::kDynamic, stream>>>(tmA, tmB, tmY, p);
  return cudaGetLastError();
}

constexpr int kStages256 = 4;
constexpr int kStages128 = 6;
static_assert(Smem<256, kStages256>::kDynamic <= 232448, "shared memory budget (BN=256)");
static_assert(Smem<128, kStages128>::kDynamic <= 232448, "shared memory budget (BN=128)");

Params make_params(const DeviceInfo& dev, const float* sa, int64_t ld_sa, const float* sw, void* y, int64_t ldy,
                   int64_t M, int64_t N, int64_t K, const int32_t* offsets, int32_t G) {
  Params p;
  p.sa = sa;
  p.ld_sa = ld_sa;
  p.sw = sw;
  p.y = static_cast<__nv_bfloat16*>(y);
  p.ldy = ldy;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.KB = static_cast<int32_t>(K / BK);
  p.offsets = offsets;
  p.G = G;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return p;
}

}  // namespace

cudaError_t launch_blockscaled_gemm(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                    int64_t ld_sa, const void* qw, int64_t ldqw, const float* sw, void* y,
                                    int64_t ldy, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
  // Wide tiles (BN = 256) halve the operand traffic per FLOP; narrow ones keep
  // every SM busy when there are few tiles (skinny, decode-shaped M).
  const int64_t m_tiles = (M + BM - 1) / BM;
  const bool wide = (N % 256 == 0) && m_tiles * (N / 256) >= dev.num_sms;
  const int BN = wide ? 256 : 128;
  CUtensorMap tmA, tmB, tmY;
  if (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, ldqa, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, K, N, ldqw, BK, BN, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M, ldy * 2, kEpiCols, 32,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const Params p = make_params(dev, sa, ld_sa, sw, y, ldy, M, N, K, nullptr, 1);
  const int64_t tiles = m_tiles * (N / BN);
  const int grid = static_cast<int>(tiles < dev.num_sms ? tiles : dev.num_sms);
  if (wide) return launch_kernel<256, kStages256, false>(dev, tmA, tmB, tmY, p, grid, stream);
  return launch_kernel<128, kStages128, false>(dev, tmA, tmB, tmY, p, grid, stream);
}

cudaError_t launch_blockscaled_grouped_gemm(const DeviceInfo& dev, int32_t G, const int32_t* offsets,
                                            int64_t M_total, const void* qa, int64_t ldqa, const float* sa,
                                            int64_t ld_sa, const void* qw, const float* sw, void* y, int64_t ldy,
                                            int64_t N, int64_t K, cudaStream_t stream) {
  const bool wide = (N % 256 == 0);
  const int BN = wide ? 256 : 128;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M_total, ldqa, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, K, static_cast<uint64_t>(G) * N, K, BK, BN,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const CUtensorMap& tmY = tmA;  // unused by the grouped epilogue
  const Params p = make_params(dev, sa, ld_sa, sw, y, ldy, M_total, N, K, offsets, G);
  // Upper bound on the tile count without reading the offsets: every group
  // can add at most one partial M tile.
  const int64_t max_tiles = ((M_total + BM - 1) / BM + G) * (N / BN);
  const int grid = static_cast<int>(max_tiles < dev.num_sms ? max_tiles : dev.num_sms);
  if (wide) return launch_kernel<256, kStages256, true>(dev, tmA, tmB, tmY, p, grid, stream);
  return launch_kernel<128, kStages128, true>(dev, tmA, tmB, tmY, p, grid, stream);
}

}  // namespace fp8bs
