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
//   warp 0      TMA producer: A (128x128 codes) and B (BN/CG x 128 codes) per
//               K chunk into a STAGES-deep shared-memory ring (mbarrier
//               full/empty)
//   warp 1      TMEM owner and MMA issuer: 4 x tcgen05.mma kind::f8f6f4
//               (K = 32 each) per chunk into the next TMEM buffer, then one
//               tcgen05.commit that publishes the chunk (the first promotion
//               warp then frees the chunk's shared-memory stage)
//   warps 2..3  idle (their warpgroup gives registers to the promotion warps)
//   warps 4..11 promotion: tcgen05.ld the chunk (one row per thread, 64
//               columns per load), acc += chunk * (sa[kb][m] * sw[nb][kb])
//               with packed FP32 FMAs (two columns per instruction), handing
//               the TMEM buffer back as soon as the whole chunk has been read
//               (for 128 columns per warp the FMAs of the first 64 run between
//               the two loads: accumulators and 128 loaded columns do not fit
//               in registers together); after the last chunk, BF16 (RNE) or
//               FP32 -> swizzled smem -> TMA store (dense) or row-masked
//               coalesced stores (grouped).  A template variant (RES) adds a
//               BF16 residual to the FP32 result before the rounding.
//
// B normally arrives by a tensor-map load of BN/CG rows x 128 bytes per stage.
// With packed weights (Params::b_packed, single-CTA tiles) each 128-row part
// of a stage is already stored as its 16 KB swizzled image and arrives by one
// contiguous bulk copy.
//
// Wide tiles run on CTA pairs (CG = 2, a cluster of two CTAs on two SMs):
// the pair computes a 256 x 256 tile with tcgen05 cta_group::2 MMAs issued by
// the even CTA.  Each CTA holds its 128 rows of A and half (128 columns) of B
// per stage, so a stage is 32 KB and six stages fit beside the epilogue
// staging: deep enough to cover the L2 latency of the operand loads at the
// tensor pipe's rate.  Each CTA's TMEM holds its 128 rows of the accumulator,
// and each CTA promotes and stores its own rows.  Narrow tiles (BN = 128, for
// skinny M) run on single CTAs (CG = 1).
//
// The kernel is persistent: cluster c handles work items c, c + clusters, ...;
// dense tiles are ordered M-fastest when A is the smaller operand (a wave then
// shares a few weight column blocks and the whole, L2-resident, activation
// matrix) and N-fastest otherwise.  When the last round of dense tiles, or
// the only one, would fill at most half of the clusters, those tiles are cut
// into K slices whose FP32 partials a second kernel sums (split-K tail).
//
// Every mbarrier wait is bounded (see ptx.cuh).  A wait that gives up records
// a timeout in the status word and raises a CTA-wide abort flag; every role
// then leaves its loop, the producer drains its TMA loads, the MMA warp waits
// for its last commits, and TMEM is released before the CTA exits.  The peer
// of an aborting CTA stops on its own bounded waits.
#include <cuda_bf16.h>

#include <atomic>

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
constexpr int kEpiRowBytes = 128;     // bytes of one staged output row (one 128B-swizzle row)
constexpr int kResPrefetchChunks = 4;  // residual epilogue: L2 prefetch this many chunks before the end
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
  const float* sw;        // 128x128 block scales of B (unless row-scaled)
  const float* sb;        // row-scaled B: 1x128 scales sb[kb * ld_sb + n]
  int64_t ld_sb;
  void* y;              // grouped: direct stores (BF16 or FP32)
  int64_t ldy;
  int32_t M;            // rows of A (M_total when grouped)
  int32_t N;
  int32_t n_fastest;    // dense: walk tiles N-fastest (see make_params)
  int32_t KB;           // K / 128
  const int32_t* offsets;  // grouped only, [G+1]
  int32_t G;
  unsigned* status;
  uint64_t timeout_ns;
  // Dense split-K tail: work items 0 .. t_full - 1 are whole tiles; the
  // remaining tiles are cut into `split` K slices each (items t_full .. n_items
  // - 1), whose FP32 partial accumulators go to ws and are summed by
  // split_tail_reduce_kernel.  split == 1: every item is a whole tile.
  int32_t n_items;
  int32_t t_full;
  int32_t split;
  float* ws;
  // Dense only: BF16 residual R [M, N] (row stride ldr) added to the FP32
  // result before the output rounding; null when there is none.
  const uint16_t* res;
  int64_t ldr;
  // Dense single-CTA tiles only: B as packed 128x128 tiles, each the 16 KB
  // shared-memory image of its stage (see fp8_pack_weight_128x128), loaded
  // by one bulk copy per tile instead of a tensor-map load; null otherwise.
  const uint8_t* b_packed;
};

constexpr uint32_t kPackedTileBytes = 128 * 128;

// Untiled bulk copy global -> shared of `bytes` (a multiple of 16; both
// addresses 16-byte aligned), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

// Bring the 128-byte line holding `ptr` into L2 (a hint; no fault on any
// address the caller may also load).
__device__ __forceinline__ void prefetch_l2(const void* ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(ptr)));
}

// Adds a pair of BF16 residual values (one 32-bit word) to a pair of FP32
// accumulators, each sum rounded to FP32.
__device__ __forceinline__ float2 add_bf16_pair(float2 a, uint32_t r) {
  return make_float2(__fadd_rn(a.x, bf16lo_to_f32(r)), __fadd_rn(a.y, bf16hi_to_f32(r)));
}

// Origin of dense cluster tile `tile` (see TileWalker for the order).
template <int BN, int CM>
__device__ __forceinline__ void dense_tile_origin(const Params& p, int64_t tile, int32_t rank, int32_t& a_row,
                                                  int32_t& n0) {
  const int32_t n_tiles = p.N / BN;
  const int32_t m_groups = ((p.M + BM - 1) / BM + CM - 1) / CM;
  // M-fastest keeps a wave on a few weight column tiles and streams A, which
  // stays L2-resident when it is the smaller operand; N-fastest re-reads B
  // instead (the choice: make_params)
  const int32_t mg = static_cast<int32_t>(p.n_fastest ? tile / n_tiles : tile % m_groups);
  const int32_t nt = static_cast<int32_t>(p.n_fastest ? tile % n_tiles : tile / m_groups);
  a_row = (mg * CM + rank) * BM;
  n0 = nt * BN;
}

// Accumulator buffers in tensor memory, each 128 lanes x BN FP32 columns
// holding one K chunk.  Two 256-wide buffers fill the 512 columns, so the
// MMAs of a 256-wide tile run at most one chunk ahead of promotion.  (Four
// 128-wide buffers with 256 x 128 pair tiles would let them run three
// chunks ahead, but such tiles double the operand bytes per FLOP through
// L2 and ran the up-projection GEMM 1.57x slower; narrow tiles measured
// the same with two or four buffers.)
template <int BN, int CG>
__host__ __device__ constexpr int num_tmem_bufs() {
  return 2;
}

// Shared-memory layout.  Stage s holds its A tile at a_off(s) and its share
// of the B tile at b_off(s).  HALF_A (M <= 64): only 64 rows of A are loaded
// and each stage is laid out [A 8 KB][B], so the M = 128 MMA's read of A rows
// 64 .. 127 falls on the same stage's B bytes, which have landed; those
// accumulator rows are never stored.
template <int BN, int STAGES, int CG, bool RS = false, bool HALF_A = false>
struct Smem {
  static constexpr int kARows = HALF_A ? BM / 2 : BM;
  static constexpr int kA = kARows * BK;
  static constexpr int kB = (BN / CG) * BK;  // this CTA's share of the B tile
  static constexpr int kStage = kA + kB;
  __host__ __device__ static constexpr uint32_t a_off(uint32_t s) { return HALF_A ? s * kStage : s * kA; }
  __host__ __device__ static constexpr uint32_t b_off(uint32_t s) { return HALF_A ? s * kStage + kA : STAGES * kA + s * kB; }
  static constexpr int kOffStaging = STAGES * kStage;
  // row-scaled B: per promotion warp, two chunks x (BN / 2) column scales
  static constexpr int kOffColScale = kOffStaging + kEpiWarps * kStagingBytes;
  static constexpr int kColScaleBytes = RS ? kEpiWarps * 2 * (BN / 2) * 4 : 0;
  static constexpr int kOffBar = kOffColScale + kColScaleBytes;
  // full[STAGES], empty[STAGES], tmem_full[NBUF], tmem_empty[NBUF]
  static constexpr int kOffSlot = kOffBar + (2 * STAGES + 2 * num_tmem_bufs<BN, CG>()) * 8;
  static constexpr int kOffAbort = kOffSlot + 4;
  static constexpr int kBytes = kOffAbort + 4;
  static constexpr int kDynamic = kBytes + 1024;  // + alignment slack
};

// Tile walker shared by all roles (dense tiles in M-fastest or N-fastest order,
// see Params::n_fastest).  Tiles are visited in "cluster tiles" of
// CM consecutive 128-row tiles x one BN-column tile; the CM CTAs of a
// cluster walk the same cluster tiles in the same order and CTA `rank` takes
// row tile CM * m + rank of each.  Yields (a_row, row_end, b_row, n0, group)
// per tile; b_row is the first weight row of the whole BN-column tile.  A row
// tile may lie wholly past row_end (an odd count of row tiles): its CTA still
// loads and takes part in the pair's MMAs, and its outputs are masked.  Dense: one group of M rows.  Grouped: group g has rows
// off[g] .. off[g+1]-1 and weight rows g*N .. g*N+N-1.
template <bool GROUPED, int BN, int CM>
struct TileWalker {
  const Params& p;
  int64_t next;          // next cluster tile of this cluster
  int64_t stride;        // clusters in the grid
  int32_t rank;          // this CTA's rank in its cluster
  int32_t n_tiles;       // N / BN
  // grouped state
  int32_t g;
  int64_t tiles_before;  // cluster tiles of groups < g
  int32_t g_row0, g_row1, g_mgroups;

  __device__ TileWalker(const Params& p_, int32_t rank_)
      : p(p_), next(blockIdx.x / CM), stride(gridDim.x / CM), rank(rank_), n_tiles(p_.N / BN), g(0),
        tiles_before(0) {
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
    g_mgroups = ((r1 - r0 + BM - 1) / BM + CM - 1) / CM;
  }
  // Returns false when this CTA has no more work items.  [kb0, kb1) is the
  // item's range of K chunks; unit >= 0 numbers a split-K unit of the tail.
  __device__ bool get(int32_t& a_row, int32_t& row_end, int32_t& b_row, int32_t& n0, int32_t& group, int32_t& kb0,
                      int32_t& kb1, int32_t& unit) {
    const int64_t t = next;
    next += stride;
    kb0 = 0;
    kb1 = p.KB;
    unit = -1;
    if (!GROUPED) {
      if (t >= p.n_items) return false;
      int64_t tile = t;
      if (t >= p.t_full) {
        const int32_t u = static_cast<int32_t>(t - p.t_full);
        const int32_t slice = u % p.split;
        tile = p.t_full + u / p.split;
        kb0 = slice * p.KB / p.split;
        kb1 = (slice + 1) * p.KB / p.split;
        unit = u;
      }
      dense_tile_origin<BN, CM>(p, tile, rank, a_row, n0);
      row_end = p.M;
      b_row = n0;
      group = 0;
      return true;
    } else {
      while (g < p.G && t >= tiles_before + static_cast<int64_t>(g_mgroups) * n_tiles) {
        tiles_before += static_cast<int64_t>(g_mgroups) * n_tiles;
        ++g;
        load_group();
      }
      if (g >= p.G) return false;
      const int64_t local = t - tiles_before;
      const int32_t mg = static_cast<int32_t>(local % g_mgroups);
      const int32_t nt = static_cast<int32_t>(local / g_mgroups);
      a_row = g_row0 + (mg * CM + rank) * BM;
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

template <int BN, int STAGES, bool GROUPED, int CG, bool F32, bool RS, bool HALF_A = false, bool RES = false>
__global__ void __launch_bounds__(kThreads, 1)
    blockscaled_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                            const __grid_constant__ CUtensorMap tmY, const Params p) {
  using L = Smem<BN, STAGES, CG, RS, HALF_A>;
  static_assert(!HALF_A || (CG == 1 && !GROUPED), "64-row A tiles are a dense single-CTA variant");
  static_assert(!(RS && GROUPED), "row-scaled B is a dense-only variant");
  static_assert(!RES || (!GROUPED && !RS && !F32), "the residual epilogue is a dense BF16-output variant");
  static_assert(CG == 1 || CG == 2, "single CTAs or CTA pairs");
  constexpr int NBUF = num_tmem_bufs<BN, CG>();
  constexpr int kTmemCols = NBUF * BN;  // NBUF accumulator buffers of this CTA's 128 rows x BN
  constexpr int kHalfCols = BN / 2;   // columns per promotion warp
  constexpr uint32_t kStageTx = CG * (L::kA + L::kB);  // bytes landing per stage (whole pair)
  constexpr uint32_t kIdesc = idesc_e4m3_f32(BM * CG, BN);
  constexpr uint16_t kPairMask = 0x3;
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation must be a power of two");
  constexpr int kOutBytes = F32 ? 4 : 2;
  constexpr int kPieceCols = kEpiRowBytes / kOutBytes;  // output columns per staged piece
  static_assert(kHalfCols % kPieceCols == 0, "epilogue boxes");

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t base = (raw_addr + 1023u) & ~1023u;  // 1024-aligned for the 128B swizzle
  uint8_t* smem = smem_raw + (base - raw_addr);

  const uint32_t bar_full = base + L::kOffBar;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  const uint32_t bar_tfull = bar_empty + STAGES * 8;
  const uint32_t bar_tempty = bar_tfull + NBUF * 8;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(smem + L::kOffSlot);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffAbort);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int32_t rank = CG > 1 ? static_cast<int32_t>(cluster_ctarank()) : 0;
  const bool leader = rank == 0;  // issues the pair's MMAs and owns its full / tempty barriers

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);   // the leader's producer arrives; all loads of the pair credit bytes
      mbar_init(bar_empty + 8 * s, 1);  // released by this CTA's first promotion warp (see below)
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(bar_tfull + 8 * b, 1);
      mbar_init(bar_tempty + 8 * b, kEpiWarps * CG);  // every promotion warp of the pair
    }
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    if (!GROUPED) prefetch_tmap(&tmY);
  }
  if (warp == 1) {
    if (CG == 1) {
      tmem_alloc(base + L::kOffSlot, kTmemCols);
      tmem_relinquish();
    } else {
      tmem_alloc_pair(base + L::kOffSlot, kTmemCols);
      tmem_relinquish_pair();
    }
  }
  // Barriers and TMEM must be ready in both CTAs of a pair before either
  // signals the other.
  tc_fence_before_sync();
  if (CG > 1)
    cluster_sync_all();
  else
    __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  if (!GROUPED && warp == 0 && lane == 0) {
    // While the previous kernel of the stream finishes, pull this CTA's
    // weight stages of its first item into L2 (dense tiles: their
    // coordinates need no global memory); the loads after the wait then
    // start from L2.  A prefetch changes no value read, so it is safe
    // whatever that kernel writes.
    TileWalker<false, BN, CG> first(p, rank);
    int32_t a0, r0, b0, c0, g0, k0, k1, u0;
    if (first.get(a0, r0, b0, c0, g0, k0, k1, u0)) {
      const int32_t kend = k1 - k0 < STAGES ? k1 : k0 + STAGES;
      for (int32_t kb = k0; kb < kend; ++kb) {
        if (p.b_packed != nullptr && CG == 1) {
          const uint8_t* src = p.b_packed + (static_cast<int64_t>(b0 / 128) * p.KB + kb) * kPackedTileBytes;
#pragma unroll
          for (int h = 0; h < BN / 128; ++h)
            bulk_prefetch_l2(src + static_cast<int64_t>(h) * p.KB * kPackedTileBytes, kPackedTileBytes);
        } else {
          tma_prefetch_l2_2d(&tmB, kb * BK, b0 + rank * (BN / CG));
        }
      }
    }
  }
  // Everything above touches only this CTA's (or pair's) shared and tensor
  // memory (and L2 through hints); from here on the kernel reads and writes
  // global memory.
  pdl_wait();
  // The pair's full and tempty barriers live in the leader.
  const uint32_t full_base = CG > 1 ? map_shared_rank(bar_full, 0) : bar_full;
  const uint32_t tempty_base = CG > 1 ? map_shared_rank(bar_tempty, 0) : bar_tempty;

  TileWalker<GROUPED, BN, CG> tiles(p, rank);
  int32_t a_row, row_end, b_row, n0, group, kb0, kb1, unit;

  if (warp < kFirstEpiWarp) {
    // 128 FP32 accumulators per promotion thread (BN = 256) need more than the
    // launch allocation: this warpgroup hands registers to the other two.
    if (BN == 256) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RegSplit<GROUPED>::low));
    if (warp == 0 && lane == 0) {
      // ---------------- TMA producer (both CTAs of a pair) ----------------
      uint32_t stage = 0, phase = 0;
      uint32_t issued_mask = 0, issued_parity = 0;  // per stage: ever issued / parity of last issue
      bool ok = true;
      while (ok && tiles.get(a_row, row_end, b_row, n0, group, kb0, kb1, unit)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(bar_empty + 8 * stage, phase ^ 1u, abort_flag, p.timeout_ns)) {
            abort_cta(abort_flag, p.status);
            ok = false;
            break;
          }
          const uint32_t a_dst = base + L::a_off(stage);
          const uint32_t b_dst = base + L::b_off(stage);
          if (CG == 1) {
            const uint32_t full = bar_full + 8 * stage;
            mbar_arrive_expect_tx(full, kStageTx);
            tma_load_2d(a_dst, &tmA, full, kb * BK, a_row);
            if (!GROUPED && p.b_packed != nullptr) {
              // BN / 128 packed tiles (rows b_row.., chunk kb), each one
              // contiguous 16 KB image of its part of the stage
              const uint8_t* src = p.b_packed + (static_cast<int64_t>(b_row / 128) * p.KB + kb) * kPackedTileBytes;
#pragma unroll
              for (int h = 0; h < BN / 128; ++h)
                bulk_load_1d(b_dst + h * kPackedTileBytes, src + static_cast<int64_t>(h) * p.KB * kPackedTileBytes,
                             kPackedTileBytes, full);
            } else {
              tma_load_2d(b_dst, &tmB, full, kb * BK, b_row);
            }
          } else {
            // the leader expects the whole pair's bytes; each CTA loads its
            // own A rows and its half of B and credits the leader's barrier
            if (leader) mbar_arrive_expect_tx(bar_full + 8 * stage, kStageTx);
            const uint32_t full = full_base + 8 * stage;
            tma_load_2d_pair(a_dst, &tmA, full, kb * BK, a_row);
            tma_load_2d_pair(b_dst, &tmB, full, kb * BK, b_row + rank * (BN / CG));
          }
          issued_mask |= 1u << stage;
          issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every load already issued land before shared memory goes away
        // (the pair's loads are counted on the leader's barriers).
        if (leader)
          for (int s = 0; s < STAGES; ++s)
            if (issued_mask & (1u << s))
              (void)mbar_wait(bar_full + 8 * s, (issued_parity >> s) & 1u, nullptr, p.timeout_ns);
      } else {
        // Wait for the last release of every stage, so that no MMA still
        // reads this CTA's shared memory and no commit still targets it.
        for (int s = 0; s < STAGES; ++s)
          if (issued_mask & (1u << s))
            (void)mbar_wait(bar_empty + 8 * s, (issued_parity >> s) & 1u, abort_flag, p.timeout_ns);
      }
    } else if (warp == 1 && lane == 0 && leader) {
      // ---------------- MMA issuer (the leader of a pair) ----------------
      uint32_t stage = 0, phase = 0, buf = 0, bphase = 0;
      uint32_t committed = 0, committed_parity = 0;  // per TMEM buffer: ever committed / parity of last commit
      bool ok = true;
      while (ok && tiles.get(a_row, row_end, b_row, n0, group, kb0, kb1, unit)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          // (with a pair, the peer's promotion warps also release the buffer)
          const bool drained = CG == 1 ? mbar_wait(bar_tempty + 8 * buf, bphase ^ 1u, abort_flag, p.timeout_ns)
                                       : mbar_wait_cluster(bar_tempty + 8 * buf, bphase ^ 1u, abort_flag,
                                                           p.timeout_ns);
          if (!drained || !mbar_wait(bar_full + 8 * stage, phase, abort_flag, p.timeout_ns)) {
            abort_cta(abort_flag, p.status);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint32_t d = tmem_base + buf * BN;
          const uint64_t adesc = smem_desc_k128_sw128(base + L::a_off(stage));
          const uint64_t bdesc = smem_desc_k128_sw128(base + L::b_off(stage));
#pragma unroll
          for (int k = 0; k < BK / MMA_K; ++k) {
            // advance the start address by 32 bytes (2 units of 16 B) per K step
            if (CG == 1)
              mma_f8f6f4(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
            else
              mma_f8f6f4_pair(d, adesc + 2u * k, bdesc + 2u * k, kIdesc, k > 0 ? 1u : 0u);
          }
          // One commit per chunk: chunk kb is in TMEM buffer `buf` (for a pair,
          // in both CTAs' accumulator rows).  The same completion frees the
          // operand stage, which the promotion side releases when it sees the
          // commit: a second commit per chunk would cost the tensor pipe more
          // than the later release costs the producer, which runs stages ahead.
          if (CG == 1)
            mma_commit(bar_tfull + 8 * buf);
          else
            mma_commit_pair(bar_tfull + 8 * buf, kPairMask);
          committed |= 1u << buf;
          committed_parity = (committed_parity & ~(1u << buf)) | (bphase << buf);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (++buf == NBUF) {
            buf = 0;
            bphase ^= 1u;
          }
        }
      }
      if (!ok) {
        // No MMA may still be writing TMEM when it is released.
        for (int b = 0; b < NBUF; ++b)
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
    uint32_t rel_stage = 0;  // operand stage of the next chunk (the producer's order)
    bool ok = true;
    const bool live = !HALF_A || q < 2;  // the warp's TMEM lanes can hold output rows
    while (ok && tiles.get(a_row, row_end, b_row, n0, group, kb0, kb1, unit)) {
      const int32_t row = a_row + q * 32 + lane;  // this thread's output row
      const bool row_ok = row < row_end;
      // rows past the end read a valid row's scale and drop the result
      const float* sa_col = p.sa + min(row, p.M - 1);
      const float row_mask = row_ok ? 1.0f : 0.0f;
      const int32_t col0 = n0 + half * kHalfCols;  // first column of this warp
      const float* sw_row = p.sw + (static_cast<int64_t>(group) * (p.N / 128) + col0 / 128) * p.KB;
      // Pairs of FP32 accumulators, updated with packed FP32 FMAs.
      float2 acc[kHalfCols / 2];
#pragma unroll
      for (int i = 0; i < kHalfCols / 2; ++i) acc[i] = make_float2(0.0f, 0.0f);

      // Row-scaled B: this warp's kHalfCols column scales per chunk, staged in
      // a two-chunk shared-memory ring one chunk ahead (lane l fetches
      // kColVec consecutive scales); every lane then reads all of them.
      constexpr int kColVec = kHalfCols / 32;
      float* colscale = reinterpret_cast<float*>(smem + L::kOffColScale) + epi * 2 * kHalfCols;
      const float* sb_col = RS ? p.sb + col0 + lane * kColVec : nullptr;
      float cs_next[kColVec];
      if (RS) {
#pragma unroll
        for (int v = 0; v < kColVec; ++v)
          colscale[lane * kColVec + v] = __ldg(sb_col + static_cast<int64_t>(kb0) * p.ld_sb + v);
        const int k1 = kb0 + 1 < kb1 ? kb0 + 1 : kb0;
#pragma unroll
        for (int v = 0; v < kColVec; ++v) cs_next[v] = __ldg(sb_col + static_cast<int64_t>(k1) * p.ld_sb + v);
        __syncwarp();
      }

      float sa_next = __ldg(sa_col + static_cast<int64_t>(kb0) * p.ld_sa);
      float sw_next = RS ? 1.0f : __ldg(sw_row + kb0);
      for (int kb = kb0; kb < kb1; ++kb) {
        const float scale = sa_next * sw_next * row_mask;
        const float2 scale2 = make_float2(scale, scale);
        const int kn = kb + 1 < kb1 ? kb + 1 : kb;  // prefetch the next chunk's scales
        sa_next = __ldg(sa_col + static_cast<int64_t>(kn) * p.ld_sa);
        if (!RS) sw_next = __ldg(sw_row + kn);
        const float* cs = colscale + ((kb - kb0) & 1) * kHalfCols;  // this chunk's column scales (RS)
        if (RES && row_ok && kb == (kb1 - kb0 > kResPrefetchChunks ? kb1 - kResPrefetchChunks : kb0)) {
          // a few chunks before the epilogue: pull this row's residual
          // segment into L2 so that the epilogue's loads do not wait on DRAM
          const uint16_t* rp = p.res + static_cast<int64_t>(row) * p.ldr + col0;
#pragma unroll
          for (int l = 0; l < kHalfCols / 64; ++l) prefetch_l2(rp + 64 * l);
        }
        const bool waited = mbar_wait(bar_tfull + 8 * buf, bphase, abort_flag, p.timeout_ns);
        if (!__all_sync(0xffffffffu, waited)) {
          abort_cta(abort_flag, p.status);
          ok = false;
          break;
        }
        // The chunk's MMAs have completed, so they no longer read this CTA's
        // operand stage: hand it back to the producer.
        if (epi == 0 && lane == 0) mbar_arrive(bar_empty + 8 * rel_stage);
        if (++rel_stage == STAGES) rel_stage = 0;
        tc_fence_after_sync();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN + half * kHalfCols;
        if (!live) {
          // lanes 64 .. 127 of a 64-row A tile hold no output: release at once
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_relaxed(bar_tempty + 8 * buf);
        }
#pragma unroll
        for (int c = 0; c < (live ? kHalfCols / 64 : 0); ++c) {
          uint32_t r[64];
          tmem_ld_x64(taddr + c * 64, r);
          tmem_wait_ld(r);
          if (c == kHalfCols / 64 - 1) {
            // the whole chunk is in registers: hand the buffer back to the
            // MMA warp (of the pair's leader) before the last FMAs
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) {
              if (CG == 1)
                mbar_arrive_relaxed(bar_tempty + 8 * buf);
              else
                mbar_arrive_cluster_relaxed(tempty_base + 8 * buf);
            }
          }
          if (!RS) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              acc[c * 32 + j] =
                  __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), scale2,
                             acc[c * 32 + j]);
          } else {
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              const float4 cs4 = *reinterpret_cast<const float4*>(cs + c * 64 + 2 * j);
              const float2 s01 = __fmul2_rn(scale2, make_float2(cs4.x, cs4.y));
              const float2 s23 = __fmul2_rn(scale2, make_float2(cs4.z, cs4.w));
              acc[c * 32 + j] =
                  __ffma2_rn(make_float2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1])), s01,
                             acc[c * 32 + j]);
              acc[c * 32 + j + 1] =
                  __ffma2_rn(make_float2(__uint_as_float(r[2 * j + 2]), __uint_as_float(r[2 * j + 3])), s23,
                             acc[c * 32 + j + 1]);
            }
          }
        }
        if (RS) {
          // stage the next chunk's column scales (the slot was last read in
          // chunk kb - 1) and fetch the one after
          __syncwarp();
#pragma unroll
          for (int v = 0; v < kColVec; ++v)
            colscale[((kb - kb0 + 1) & 1) * kHalfCols + lane * kColVec + v] = cs_next[v];
          const int k2 = kb + 2 < kb1 ? kb + 2 : kb1 - 1;
#pragma unroll
          for (int v = 0; v < kColVec; ++v) cs_next[v] = __ldg(sb_col + static_cast<int64_t>(k2) * p.ld_sb + v);
          __syncwarp();
        }
        if (++buf == NBUF) {
          buf = 0;
          bphase ^= 1u;
        }
      }
      if (!ok) break;

      if (!GROUPED && unit >= 0) {
        // split-K unit of a tail tile: this warp's FP32 partial (32 rows x
        // kHalfCols) to the workspace, float4 j of lane l at j * 32 + l so that
        // each store instruction covers 512 contiguous bytes
        float4* part = reinterpret_cast<float4*>(p.ws) +
                       ((static_cast<int64_t>(unit) * CG + rank) * kEpiWarps + epi) * (8 * kHalfCols) + lane;
#pragma unroll
        for (int j = 0; j < kHalfCols / 4; ++j)
          part[j * 32] = make_float4(acc[2 * j].x, acc[2 * j].y, acc[2 * j + 1].x, acc[2 * j + 1].y);
        continue;
      }

      // ---- epilogue: BF16 (RNE) or FP32, swizzled staging, store ----
#pragma unroll
      for (int piece = 0; piece < (live ? kHalfCols / kPieceCols : 0); ++piece) {
        if (!GROUPED) {
          if (lane == 0) tma_store_wait_read_all();  // staging free again
        }
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          // 16 bytes: 8 BF16 or 4 FP32 outputs of this thread's row
          const int c0 = (piece * kPieceCols + j * (16 / kOutBytes)) / 2;
          if (RES && row_ok) {
            // residual epilogue: R added to the FP32 result, one rounding after
            const uint16_t* rp =
                p.res + static_cast<int64_t>(row) * p.ldr + col0 + piece * kPieceCols + j * (16 / kOutBytes);
            if (F32) {
              const uint2 rr = *reinterpret_cast<const uint2*>(rp);
              acc[c0] = add_bf16_pair(acc[c0], rr.x);
              acc[c0 + 1] = add_bf16_pair(acc[c0 + 1], rr.y);
            } else {
              const uint4 rr = *reinterpret_cast<const uint4*>(rp);
              acc[c0] = add_bf16_pair(acc[c0], rr.x);
              acc[c0 + 1] = add_bf16_pair(acc[c0 + 1], rr.y);
              acc[c0 + 2] = add_bf16_pair(acc[c0 + 2], rr.z);
              acc[c0 + 3] = add_bf16_pair(acc[c0 + 3], rr.w);
            }
          }
          uint4 v;
          if (F32) {
            v = make_uint4(__float_as_uint(acc[c0].x), __float_as_uint(acc[c0].y), __float_as_uint(acc[c0 + 1].x),
                           __float_as_uint(acc[c0 + 1].y));
          } else {
            __nv_bfloat162 h0 = __float22bfloat162_rn(acc[c0 + 0]);
            __nv_bfloat162 h1 = __float22bfloat162_rn(acc[c0 + 1]);
            __nv_bfloat162 h2 = __float22bfloat162_rn(acc[c0 + 2]);
            __nv_bfloat162 h3 = __float22bfloat162_rn(acc[c0 + 3]);
            v.x = *reinterpret_cast<uint32_t*>(&h0);
            v.y = *reinterpret_cast<uint32_t*>(&h1);
            v.z = *reinterpret_cast<uint32_t*>(&h2);
            v.w = *reinterpret_cast<uint32_t*>(&h3);
          }
          // 128-byte swizzle: 16-byte chunk j of row `lane` sits at chunk j ^ (lane % 8)
          *reinterpret_cast<uint4*>(staging_ptr + lane * 128 + ((j ^ (lane & 7)) << 4)) = v;
        }
        if (!GROUPED) {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, staging, col0 + piece * kPieceCols, a_row + q * 32);
            tma_store_commit();
          }
        } else {
          __syncwarp();
          // 32 rows x 128 bytes: lane reads chunk (lane % 8) of rows lane/8 + 4i
          uint8_t* ybytes = static_cast<uint8_t*>(p.y);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int r = (lane >> 3) + 4 * i;
            const int ch = lane & 7;
            const uint4 v = *reinterpret_cast<const uint4*>(staging_ptr + r * 128 + ((ch ^ (r & 7)) << 4));
            const int32_t grow = a_row + q * 32 + r;
            if (grow < row_end)
              *reinterpret_cast<uint4*>(ybytes + (static_cast<int64_t>(grow) * p.ldy + col0 + piece * kPieceCols) *
                                                     kOutBytes +
                                        ch * 16) = v;
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
  if (CG > 1)
    cluster_sync_all();  // no CTA leaves while its peer may still signal it or use its TMEM
  else
    __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) {
    if (CG == 1)
      tmem_dealloc(tmem_base, kTmemCols);
    else
      tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Split-K tail: sums the FP32 partials of each tail tile in slice order (the
// result does not depend on which unit finished first) and writes Y.  One CTA
// per (tail tile, CTA rank of the tile, promotion-warp region of 32 rows x
// BN / 2 columns); thread t sums float4 columns t / 32, t / 32 + 8, .. of row
// t % 32.
template <int BN, int CG, bool F32>
__global__ void __launch_bounds__(256) split_tail_reduce_kernel(const Params p) {
  pdl_wait();
  constexpr int kHalfCols = BN / 2;
  constexpr int64_t kRegion = 8 * kHalfCols;  // float4 per warp region
  const int32_t region = static_cast<int32_t>(blockIdx.x % kEpiWarps);
  const int32_t rank = static_cast<int32_t>((blockIdx.x / kEpiWarps) % CG);
  const int32_t tail = static_cast<int32_t>(blockIdx.x / (kEpiWarps * CG));
  int32_t a_row, n0;
  dense_tile_origin<BN, CG>(p, static_cast<int64_t>(p.t_full) + tail, rank, a_row, n0);
  const int lane = threadIdx.x & 31;
  const int32_t row = a_row + (region & 3) * 32 + lane;
  const int32_t col0 = n0 + (region >> 2) * kHalfCols;
  const int64_t slice_stride = static_cast<int64_t>(CG) * kEpiWarps * kRegion;
  const float4* part = reinterpret_cast<const float4*>(p.ws) +
                       ((static_cast<int64_t>(tail) * p.split * CG + rank) * kEpiWarps + region) * kRegion + lane;
  for (int j = threadIdx.x >> 5; j < kHalfCols / 4; j += 8) {
    float4 sum = __ldcg(part + j * 32);
    for (int sl = 1; sl < p.split; ++sl) {
      const float4 v = __ldcg(part + sl * slice_stride + j * 32);
      sum.x = __fadd_rn(sum.x, v.x);
      sum.y = __fadd_rn(sum.y, v.y);
      sum.z = __fadd_rn(sum.z, v.z);
      sum.w = __fadd_rn(sum.w, v.w);
    }
    if (row < p.M) {
      if (p.res != nullptr) {
        const uint2 rr = *reinterpret_cast<const uint2*>(p.res + static_cast<int64_t>(row) * p.ldr + col0 + 4 * j);
        const float2 lo = add_bf16_pair(make_float2(sum.x, sum.y), rr.x);
        const float2 hi = add_bf16_pair(make_float2(sum.z, sum.w), rr.y);
        sum = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
      const int64_t off = static_cast<int64_t>(row) * p.ldy + col0 + 4 * j;
      if (F32) {
        *reinterpret_cast<float4*>(static_cast<float*>(p.y) + off) = sum;
      } else {
        const __nv_bfloat162 lo = __float22bfloat162_rn(make_float2(sum.x, sum.y));
        const __nv_bfloat162 hi = __float22bfloat162_rn(make_float2(sum.z, sum.w));
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.y) + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
      }
    }
  }
}

// Largest number of clusters of this kernel variant that can be resident at
// once on the current device (queried once per device and variant).
template <int BN, int STAGES, bool GROUPED, int CG, bool F32, bool RS, bool HALF_A, bool RES>
int max_resident_clusters(const DeviceInfo& dev, const cudaLaunchConfig_t& cfg) {
  static std::atomic<int> cache[64];
  const int idx = dev.ordinal & 63;
  int n = cache[idx].load(std::memory_order_relaxed);
  if (n > 0) return n;
  n = dev.num_sms / CG;
  if (CG > 1) {
    int q = 0;
    if (cudaOccupancyMaxActiveClusters(&q, blockscaled_gemm_kernel<BN, STAGES, GROUPED, CG, F32, RS, HALF_A, RES>, &cfg) == cudaSuccess &&
        q > 0)
      n = q;
    else
      (void)cudaGetLastError();
  }
  cache[idx].store(n, std::memory_order_relaxed);
  return n;
}

// Smallest K slice of a split tail tile, in 128-K chunks.
constexpr int kMinSplitChunks = 4;

// Persistent launch: one cluster of CG CTAs per CG SMs, at most one per work
// item.  When the dense tiles leave a last round (or a single round) that
// fills at most half of the resident clusters, those tiles are split along K
// over the idle clusters (FP32 partials in a workspace, see Workspace) and
// summed by split_tail_reduce_kernel.  A split tail has at most one unit per
// resident cluster, so the workspace never exceeds BM x BN FP32 values per SM.
template <int BN, int STAGES, bool GROUPED, int CG, bool F32, bool RS, bool HALF_A = false, bool RES = false>
cudaError_t launch_kernel(const DeviceInfo& dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                          const CUtensorMap& tmY, const Params& p0, int64_t cluster_tiles, cudaStream_t stream,
                          Workspace* ws) {
  using L = Smem<BN, STAGES, CG, RS, HALF_A>;
  auto kernel = blockscaled_gemm_kernel<BN, STAGES, GROUPED, CG, F32, RS, HALF_A, RES>;
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
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeClusterDimension;
  attrs[0].val.clusterDim.x = CG;
  attrs[0].val.clusterDim.y = 1;
  attrs[0].val.clusterDim.z = 1;
  attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attrs[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kDynamic;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = 2;
  cfg.gridDim = dim3(CG, 1, 1);
  const int resident = max_resident_clusters<BN, STAGES, GROUPED, CG, F32, RS, HALF_A, RES>(dev, cfg);
  Params p = p0;
  p.n_items = static_cast<int32_t>(cluster_tiles);
  p.t_full = static_cast<int32_t>(cluster_tiles);
  p.split = 1;
  p.ws = nullptr;
  int64_t tail = 0, split = 1;
  size_t bytes = 0;
  if constexpr (!GROUPED) {
    // the last round's tiles (all of them when the grid fills at most half of
    // the resident clusters, e.g. skinny products with few column tiles)
    tail = cluster_tiles % resident;
    if (tail > 0 && 2 * tail <= resident) {
      split = resident / tail;
      if (split > p.KB / kMinSplitChunks) split = p.KB / kMinSplitChunks;
      if (split < 2) split = 1;
      bytes = split > 1 ? static_cast<size_t>(tail * split) * CG * BM * BN * sizeof(float) : 0;
    }
  }
  if (ws != nullptr) {
    ws->needed = bytes;
    if (ws->plan_only) return cudaSuccess;
    if (ws->scratch != nullptr && bytes > ws->scratch_bytes) {
      ws->too_small = true;
      return cudaSuccess;
    }
  }
  bool owned = false;
  if (bytes > 0) {
    float* buf = nullptr;
    if (ws != nullptr && ws->scratch != nullptr) {
      buf = ws->scratch;
    } else {
      cudaMemPool_t pool = gemm_workspace_pool(dev);
      if (pool != nullptr &&
          cudaMallocFromPoolAsync(reinterpret_cast<void**>(&buf), bytes, pool, stream) == cudaSuccess) {
        owned = true;
      } else {
        (void)cudaGetLastError();  // no workspace: run the tail tiles whole
        buf = nullptr;
      }
    }
    if (buf != nullptr) {
      p.ws = buf;
      p.split = static_cast<int32_t>(split);
      p.t_full = static_cast<int32_t>(cluster_tiles - tail);
      p.n_items = static_cast<int32_t>(p.t_full + tail * split);
    }
  }
  const int64_t clusters = p.n_items < resident ? p.n_items : resident;
  cfg.gridDim = dim3(static_cast<unsigned>(clusters * CG), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmY, p);
  if (e == cudaSuccess && p.split > 1) {
    const unsigned blocks = static_cast<unsigned>((p.n_items - p.t_full) / p.split) * CG * kEpiWarps;
    (void)launch_pdl(split_tail_reduce_kernel<BN, CG, F32>, blocks, 256, 0, stream, p);
    e = cudaGetLastError();
  }
  if (owned) {
    const cudaError_t f = cudaFreeAsync(p.ws, stream);
    if (e == cudaSuccess) e = f;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// BN = 256 on a CTA pair: 32 KB stages.  Four measured faster than six or
// five (up projection 431 -> 420 us, down 448 -> 443 us) and than three (439
// us): the shared memory left over serves as L1.
constexpr int kStagesPair = 4;
// Whether wide tiles run on CTA pairs (cta_group::2) or single CTAs.
constexpr bool kUsePairs = true;
constexpr int kStages256 = 4;    // BN = 256 on one CTA: 48 KB stages
constexpr int kStages128 = 6;    // BN = 128 on one CTA: 32 KB stages
constexpr int kStages128HalfA = 6;  // BN = 128, 64-row A tiles (M <= 64): 24 KB stages (6 measured 1% faster than 8, 4 slower)
// Row-scaled B stages its column scales in shared memory: one stage fewer.
constexpr int kStagesPairRS = 5;
constexpr int kStages256RS = 3;
constexpr int kStages128RS = 5;
static_assert(Smem<256, kStagesPairRS, 2, true>::kDynamic <= 232448, "shared memory budget (BN=256, pair, RS)");
static_assert(Smem<256, kStages256RS, 1, true>::kDynamic <= 232448, "shared memory budget (BN=256, RS)");
static_assert(Smem<128, kStages128RS, 1, true>::kDynamic <= 232448, "shared memory budget (BN=128, RS)");
static_assert(Smem<256, kStagesPair, 2>::kDynamic <= 232448, "shared memory budget (BN=256, pair)");

static_assert(Smem<256, kStages256, 1>::kDynamic <= 232448, "shared memory budget (BN=256)");
static_assert(Smem<128, kStages128, 1>::kDynamic <= 232448, "shared memory budget (BN=128)");
static_assert(Smem<128, kStages128HalfA, 1, false, true>::kDynamic <= 232448, "shared memory budget (64-row A)");

Params make_params(const DeviceInfo& dev, const float* sa, int64_t ld_sa, const float* sw, void* y, int64_t ldy,
                   int64_t M, int64_t N, int64_t K, const int32_t* offsets, int32_t G) {
  Params p;
  p.sa = sa;
  p.ld_sa = ld_sa;
  p.sw = sw;
  p.sb = nullptr;
  p.ld_sb = 0;
  p.res = nullptr;
  p.ldr = 0;
  p.b_packed = nullptr;
  p.y = y;
  p.ldy = ldy;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  // N-fastest when A is the larger operand, and for long-K products whose
  // weights are the narrower side (the 4096 x 7168 x 18432 down projection and
  // its dgrad ran 3% faster so; the 4096 x 18432 x 7168 up projection 18%
  // slower): a measured rule, not a model.
  p.n_fastest = (M > N || K > 2 * N) ? 1 : 0;
  p.KB = static_cast<int32_t>(K / BK);
  p.offsets = offsets;
  p.G = G;
  p.status = dev.status;
  p.timeout_ns = wait_timeout_ns();
  return p;
}


// Tile shapes: narrow (BN = 128, one CTA), wide (BN = 256, one CTA) and
// pair (BN = 256 on a CTA pair, 256 x 256 per pair).
enum class Shape { kNarrow, kNarrowHalfA, kWide, kPair };

template <bool GROUPED, bool F32, bool RS = false, bool RES = false>
cudaError_t launch_shape(Shape shape, const DeviceInfo& dev, const CUtensorMap& tmA, const CUtensorMap& tmB,
                         const CUtensorMap& tmY, const Params& p, int64_t cluster_tiles, cudaStream_t stream,
                         Workspace* ws = nullptr) {
  switch (shape) {
    case Shape::kNarrow:
      return launch_kernel<128, RS ? kStages128RS : kStages128, GROUPED, 1, F32, RS, false, RES>(
          dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws);
    case Shape::kNarrowHalfA:
      if constexpr (!GROUPED && !RS)
        return launch_kernel<128, kStages128HalfA, false, 1, F32, false, true, RES>(dev, tmA, tmB, tmY, p,
                                                                                   cluster_tiles, stream, ws);
      return cudaErrorInvalidValue;
    case Shape::kWide:
      return launch_kernel<256, RS ? kStages256RS : kStages256, GROUPED, 1, F32, RS, false, RES>(
          dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws);
    case Shape::kPair:
      return launch_kernel<256, RS ? kStagesPairRS : kStagesPair, GROUPED, 2, F32, RS, false, RES>(
          dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_blockscaled_gemm(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                    int64_t ld_sa, const void* qw, int64_t ldqw, const float* sw, void* y,
                                    int64_t ldy, bool y_f32, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                                    Workspace* ws, const void* res, int64_t ldr) {
  // Wide tiles (BN = 256) halve the operand traffic per FLOP; narrow ones keep
  // every SM busy when there are few tiles (skinny, decode-shaped M).
  const int64_t m_tiles = (M + BM - 1) / BM;
  const bool wide = (N % 256 == 0) && m_tiles * (N / 256) >= dev.num_sms;
  const Shape shape = !wide ? (M <= BM / 2 ? Shape::kNarrowHalfA : Shape::kNarrow)
                             : (kUsePairs && m_tiles >= 2 ? Shape::kPair : Shape::kWide);
  const int CG = shape == Shape::kPair ? 2 : 1;
  const int BN = wide ? 256 : 128;
  const int out_bytes = y_f32 ? 4 : 2;
  const uint32_t a_rows = shape == Shape::kNarrowHalfA ? BM / 2 : BM;
  CUtensorMap tmA = {}, tmB = {}, tmY = {};
  const bool plan_only = ws != nullptr && ws->plan_only;  // the maps are not needed to plan
  if (!plan_only &&
      (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, ldqa, BK, a_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
       !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, K, N, ldqw, BK, BN / CG, CU_TENSOR_MAP_SWIZZLE_128B) ||
       !make_tmap_2d(&tmY, y_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M,
                     ldy * out_bytes, kEpiRowBytes / out_bytes, 32, CU_TENSOR_MAP_SWIZZLE_128B)))
    return cudaErrorInvalidValue;
  Params p = make_params(dev, sa, ld_sa, sw, y, ldy, M, N, K, nullptr, 1);
  p.res = static_cast<const uint16_t*>(res);
  p.ldr = ldr;
  const int64_t cluster_tiles = (m_tiles + CG - 1) / CG * (N / BN);
  if (res != nullptr) {
    // the residual epilogue is its own kernel variant (BF16 output only), so
    // the plain GEMM keeps its register budget
    if (y_f32) return cudaErrorInvalidValue;
    return launch_shape<false, false, false, true>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws);
  }
  return y_f32 ? launch_shape<false, true>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws)
               : launch_shape<false, false>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream, ws);
}

cudaError_t launch_blockscaled_gemm_packed(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                           int64_t ld_sa, const void* wp, const float* sw, void* y, int64_t ldy,
                                           bool y_f32, int64_t M, int64_t N, int64_t K, cudaStream_t stream) {
  // Single-CTA tiles only (a pair's B half would credit the peer's barrier).
  const int64_t m_tiles = (M + BM - 1) / BM;
  const bool wide = (N % 256 == 0) && m_tiles * (N / 256) >= dev.num_sms;
  const Shape shape = wide ? Shape::kWide : (M <= BM / 2 ? Shape::kNarrowHalfA : Shape::kNarrow);
  const int BN = wide ? 256 : 128;
  const int out_bytes = y_f32 ? 4 : 2;
  const uint32_t a_rows = shape == Shape::kNarrowHalfA ? BM / 2 : BM;
  CUtensorMap tmA, tmY;
  if (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, ldqa, BK, a_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmY, y_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M,
                    ldy * out_bytes, kEpiRowBytes / out_bytes, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const CUtensorMap& tmB = tmA;  // unused: B arrives by bulk copies
  Params p = make_params(dev, sa, ld_sa, sw, y, ldy, M, N, K, nullptr, 1);
  p.b_packed = static_cast<const uint8_t*>(wp);
  const int64_t cluster_tiles = m_tiles * (N / BN);
  return y_f32 ? launch_shape<false, true>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream)
               : launch_shape<false, false>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream);
}

cudaError_t launch_blockscaled_grouped_gemm(const DeviceInfo& dev, int32_t G, const int32_t* offsets,
                                            int64_t M_total, const void* qa, int64_t ldqa, const float* sa,
                                            int64_t ld_sa, const void* qw, const float* sw, void* y, int64_t ldy,
                                            bool y_f32, int64_t N, int64_t K, cudaStream_t stream) {
  const bool wide = (N % 256 == 0);
  const Shape shape = !wide ? Shape::kNarrow : (kUsePairs ? Shape::kPair : Shape::kWide);
  const int CG = shape == Shape::kPair ? 2 : 1;
  const int BN = wide ? 256 : 128;
  CUtensorMap tmA, tmB;
  if (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M_total, ldqa, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qw, K, static_cast<uint64_t>(G) * N, K, BK, BN / CG,
                    CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  const CUtensorMap& tmY = tmA;  // unused by the grouped epilogue
  const Params p = make_params(dev, sa, ld_sa, sw, y, ldy, M_total, N, K, offsets, G);
  // Upper bound on the cluster-tile count without reading the offsets: each
  // group adds at most one partial row tile and one partial cluster tile.
  const int64_t max_ctiles = (((M_total + BM - 1) / BM + G) / CG + G) * (N / BN);
  return y_f32 ? launch_shape<true, true>(shape, dev, tmA, tmB, tmY, p, max_ctiles, stream)
               : launch_shape<true, false>(shape, dev, tmA, tmB, tmY, p, max_ctiles, stream);
}

cudaError_t launch_blockscaled_gemm_rowscaled(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                              int64_t ld_sa, const void* qb, int64_t ldqb, const float* sb,
                                              int64_t ld_sb, void* y, int64_t ldy, bool y_f32, int64_t M, int64_t N,
                                              int64_t K, cudaStream_t stream) {
  const int64_t m_tiles = (M + BM - 1) / BM;
  const bool wide = (N % 256 == 0) && m_tiles * (N / 256) >= dev.num_sms;
  const Shape shape = !wide ? Shape::kNarrow : (kUsePairs && m_tiles >= 2 ? Shape::kPair : Shape::kWide);
  const int CG = shape == Shape::kPair ? 2 : 1;
  const int BN = wide ? 256 : 128;
  const int out_bytes = y_f32 ? 4 : 2;
  CUtensorMap tmA, tmB, tmY;
  if (!make_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, qa, K, M, ldqa, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, qb, K, N, ldqb, BK, BN / CG, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_tmap_2d(&tmY, y_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M,
                    ldy * out_bytes, kEpiRowBytes / out_bytes, 32, CU_TENSOR_MAP_SWIZZLE_128B))
    return cudaErrorInvalidValue;
  Params p = make_params(dev, sa, ld_sa, nullptr, y, ldy, M, N, K, nullptr, 1);
  p.sb = sb;
  p.ld_sb = ld_sb;
  const int64_t cluster_tiles = (m_tiles + CG - 1) / CG * (N / BN);
  return y_f32 ? launch_shape<false, true, true>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream)
               : launch_shape<false, false, true>(shape, dev, tmA, tmB, tmY, p, cluster_tiles, stream);
}

}  // namespace fp8bs
