// ptx.cuh — thin inline-PTX wrappers for sm_103a: mbarriers with bounded
// waits, TMA (cp.async.bulk.tensor) loads/stores, and the tcgen05 tensor-core
// instructions (TMEM alloc, MMA kind::f8f6f4, commit, TMEM loads).
#pragma once

#include <cstdint>
#include <cuda.h>

namespace fp8bs {

// Values a kernel may record in the per-device status word.
constexpr unsigned kStatusTimeout = 5;      // a bounded wait gave up
constexpr unsigned kStatusBadOffsets = 1;   // grouped GEMM: malformed offset table

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Record a device-side failure: first writer wins.
__device__ __forceinline__ void record_status(unsigned* status, unsigned code) {
  atomicCAS(status, 0u, code);
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// True once the phase with parity `parity` has completed (a fresh barrier is
// in phase 0, so waiting for parity 1 succeeds at once).
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Slow path of a bounded wait: spin until the phase completes, the CTA-wide
// abort flag is raised by another role, or `timeout_ns` of wall time passes.
// Inlined on purpose: a real call inside a setmaxnreg region defeats the
// register allocation of that region.
__device__ __forceinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                               uint64_t timeout_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 16; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                          uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  return mbar_wait_slow(bar, parity, abort_flag, timeout_ns);
}

// ---------------------------------------------------------------------------
// TMA (tensor-map bulk copies)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 2-D tile load global -> shared; completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// 2-D tile store shared -> global (out-of-range rows/columns are dropped).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}
__device__ __forceinline__ void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void tma_store_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Make generic-proxy shared-memory writes visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and 5th-generation MMA
// ---------------------------------------------------------------------------
// Whole-warp TMEM allocation; the base address is written to shared memory.
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, FP8 operands, FP32 accumulator.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every MMA this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile stored as rows of
// 128 bytes with the 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B): 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc_k128_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
  d |= static_cast<uint64_t>(1u) << 16;                 // leading-dim offset (unused when swizzled K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;         // stride between 8-row groups
  d |= static_cast<uint64_t>(1u) << 46;                 // descriptor version for tcgen05
  d |= static_cast<uint64_t>(2u) << 61;                 // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f8f6f4, A = B = E4M3, D = F32, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n) {
  return (1u << 4)                                  // D format F32
         | (0u << 7) | (0u << 10)                   // A, B format E4M3
         | (static_cast<uint32_t>(n >> 3) << 17)    // N / 8
         | (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

// TMEM -> registers, 32 lanes x 32 consecutive 32-bit columns; thread i of the
// warp receives lane (base lane + i).  The registers are valid only after
// tcgen05.wait::ld (see tmem_wait_fma32).
__device__ __forceinline__ void tmem_ld_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

// Promotion step: wait for this warp's outstanding TMEM loads, then
// acc[i] += chunk[i] * scale for 32 columns.  Wait and FMAs form one asm
// statement: the loaded registers are read only after the wait, and each
// chunk's FMAs stay between its load and the next one, which bounds the
// number of live registers.
__device__ __forceinline__ void tmem_wait_fma32(float* acc, const uint32_t (&r)[32], float scale) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;\n\t"
      "fma.rn.f32 %0, %32, %64, %0;\n\t fma.rn.f32 %1, %33, %64, %1;\n\t"
      "fma.rn.f32 %2, %34, %64, %2;\n\t fma.rn.f32 %3, %35, %64, %3;\n\t"
      "fma.rn.f32 %4, %36, %64, %4;\n\t fma.rn.f32 %5, %37, %64, %5;\n\t"
      "fma.rn.f32 %6, %38, %64, %6;\n\t fma.rn.f32 %7, %39, %64, %7;\n\t"
      "fma.rn.f32 %8, %40, %64, %8;\n\t fma.rn.f32 %9, %41, %64, %9;\n\t"
      "fma.rn.f32 %10, %42, %64, %10;\n\t fma.rn.f32 %11, %43, %64, %11;\n\t"
      "fma.rn.f32 %12, %44, %64, %12;\n\t fma.rn.f32 %13, %45, %64, %13;\n\t"
      "fma.rn.f32 %14, %46, %64, %14;\n\t fma.rn.f32 %15, %47, %64, %15;\n\t"
      "fma.rn.f32 %16, %48, %64, %16;\n\t fma.rn.f32 %17, %49, %64, %17;\n\t"
      "fma.rn.f32 %18, %50, %64, %18;\n\t fma.rn.f32 %19, %51, %64, %19;\n\t"
      "fma.rn.f32 %20, %52, %64, %20;\n\t fma.rn.f32 %21, %53, %64, %21;\n\t"
      "fma.rn.f32 %22, %54, %64, %22;\n\t fma.rn.f32 %23, %55, %64, %23;\n\t"
      "fma.rn.f32 %24, %56, %64, %24;\n\t fma.rn.f32 %25, %57, %64, %25;\n\t"
      "fma.rn.f32 %26, %58, %64, %26;\n\t fma.rn.f32 %27, %59, %64, %27;\n\t"
      "fma.rn.f32 %28, %60, %64, %28;\n\t fma.rn.f32 %29, %61, %64, %29;\n\t"
      "fma.rn.f32 %30, %62, %64, %30;\n\t fma.rn.f32 %31, %63, %64, %31;"
      : "+f"(acc[0]), "+f"(acc[1]), "+f"(acc[2]), "+f"(acc[3]), "+f"(acc[4]), "+f"(acc[5]), "+f"(acc[6]),
        "+f"(acc[7]), "+f"(acc[8]), "+f"(acc[9]), "+f"(acc[10]), "+f"(acc[11]), "+f"(acc[12]), "+f"(acc[13]),
        "+f"(acc[14]), "+f"(acc[15]), "+f"(acc[16]), "+f"(acc[17]), "+f"(acc[18]), "+f"(acc[19]), "+f"(acc[20]),
        "+f"(acc[21]), "+f"(acc[22]), "+f"(acc[23]), "+f"(acc[24]), "+f"(acc[25]), "+f"(acc[26]), "+f"(acc[27]),
        "+f"(acc[28]), "+f"(acc[29]), "+f"(acc[30]), "+f"(acc[31])
      : "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]),
        "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "f"(scale)
      : "memory");
}

// ---------------------------------------------------------------------------
// Conversions and memory helpers
// ---------------------------------------------------------------------------
// Two FP32 values -> two E4M3 codes (round to nearest even, saturating to
// +-448); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint32_t out;
  asm("{\n\t.reg .b16 t;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u16 %0, t;\n\t}"
      : "=r"(out)
      : "f"(hi), "f"(lo));
  return out;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

}  // namespace fp8bs
