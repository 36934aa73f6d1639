// api.cu — the C ABI declared in include/fp8bs.h: argument validation,
// per-device state (SM count, status word), tensor-map encoding and the
// bounded-wait self test.  Validation happens before any CUDA call, so a bad
// argument is reported synchronously and nothing is launched.
#include <atomic>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "../../include/fp8bs.h"
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {

// One status word per device (each device holds its own copy of a __device__
// variable).  Kernels record failures here; fp8bs_last_device_error reads it.
__device__ unsigned g_status_word;

// Fixed split-K workspace of fp8_blockscaled_gemm_noalloc, one per device
// (every device that loads the library holds it until the process exits).
// 20 MiB covers the largest split tail of a device with up to 160 SMs: a
// split tail has at most one work unit per resident cluster, each unit 128
// rows x 256 columns of FP32 per CTA, i.e. 128 KiB per SM.  Nothing in it
// needs to start at zero: each unit writes its whole partial before the
// reduction kernel reads it.
constexpr size_t kGemmScratchBytes = size_t(20) << 20;
static __device__ __align__(256) unsigned char g_gemm_scratch[kGemmScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;  // 1 s

std::atomic<uint64_t> g_timeout_ns{kDefaultTimeoutNs};

struct DeviceSlot {
  std::once_flag once;
  DeviceInfo info;
  cudaError_t err = cudaSuccess;
  // the GEMM workspace pool, created at the first split tail that needs it
  std::once_flag pool_once;
  cudaMemPool_t pool = nullptr;
  // this device's address of g_gemm_scratch, looked up at the first
  // fp8_blockscaled_gemm_noalloc call on the device
  std::once_flag scratch_once;
  float* scratch = nullptr;
  cudaError_t scratch_err = cudaSuccess;
};
DeviceSlot g_devices[kMaxDevices];

// Text of the last CUDA failure seen by a call on this host thread.
thread_local char t_detail[256] = "";

std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

void resolve_encode() {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Largest sizes the kernels index with 32-bit coordinates.
constexpr int64_t kMaxDim = (int64_t{1} << 31) - 1;

fp8bs_status cuda_failure(const char* where, cudaError_t e) {
  std::snprintf(t_detail, sizeof(t_detail), "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
  return FP8BS_ERR_CUDA;
}

}  // namespace

const DeviceInfo* current_device_info(cudaError_t* err) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = (e != cudaSuccess) ? e : cudaErrorInvalidDevice;
    return nullptr;
  }
  DeviceSlot& slot = g_devices[dev];
  std::call_once(slot.once, [&slot, dev]() {
    slot.info.ordinal = dev;
    slot.err = cudaDeviceGetAttribute(&slot.info.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (slot.err == cudaSuccess)
      slot.err = cudaDeviceGetAttribute(&slot.info.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    void* addr = nullptr;
    if (slot.err == cudaSuccess) slot.err = cudaGetSymbolAddress(&addr, g_status_word);
    slot.info.status = static_cast<unsigned*>(addr);
    const unsigned zero = 0;
    if (slot.err == cudaSuccess) slot.err = cudaMemcpy(addr, &zero, sizeof(zero), cudaMemcpyHostToDevice);
  });
  if (slot.err != cudaSuccess) {
    *err = slot.err;
    return nullptr;
  }
  *err = cudaSuccess;
  return &slot.info;
}

cudaMemPool_t gemm_workspace_pool(const DeviceInfo& dev) {
  DeviceSlot& slot = g_devices[dev.ordinal];
  std::call_once(slot.pool_once, [&slot, &dev]() {
    cudaMemPoolProps props = {};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev.ordinal;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
      cuuint64_t keep = ~static_cast<cuuint64_t>(0);
      (void)cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      slot.pool = pool;
    } else {
      (void)cudaGetLastError();  // no pool: GEMM tails run unsplit
    }
  });
  return slot.pool;
}

// Device address of this device's g_gemm_scratch (the host-side name is only
// a stand-in), looked up once per device with that device current.
float* gemm_scratch_address(const DeviceInfo& dev, cudaError_t* err) {
  DeviceSlot& slot = g_devices[dev.ordinal];
  std::call_once(slot.scratch_once, [&slot]() {
    void* addr = nullptr;
    slot.scratch_err = cudaGetSymbolAddress(&addr, g_gemm_scratch);
    slot.scratch = slot.scratch_err == cudaSuccess ? static_cast<float*>(addr) : nullptr;
  });
  *err = slot.scratch_err;
  return slot.scratch;
}

uint64_t wait_timeout_ns() { return g_timeout_ns.load(std::memory_order_relaxed); }

bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle) {
  std::call_once(g_encode_once, resolve_encode);
  if (g_encode == nullptr) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = g_encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

__global__ void selftest_wait_kernel(unsigned* status, uint64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) {
    // Nothing ever arrives on `bar`: the bounded wait must give up.
    if (!mbar_wait(smem_u32(&bar), 0, &abort_flag, timeout_ns)) record_status(status, kStatusTimeout);
  }
}

// One thread: waits, as every kernel of this library does, until the grid
// before it on the stream has completed and its writes are visible, then
// records the device's global nanosecond timer.  Launched between two kernels
// of a sequence, it marks where the first ended without the serialising
// launch gap that an event record brings back.  With `release` set it lets
// the next kernel launch before its own wait, as the kernel before it did.
__global__ void stream_timestamp_kernel(uint64_t* dst, int release) {
  if (release) pdl_launch_dependents();
  pdl_wait();
  *dst = globaltimer_ns();
}

}  // namespace

cudaError_t launch_stream_timestamp(uint64_t* dst, int release, cudaStream_t stream) {
  return launch_pdl(stream_timestamp_kernel, dim3(1), dim3(1), 0, stream, dst, release);
}

cudaError_t launch_selftest_wait(const DeviceInfo& dev, uint64_t timeout_ns, cudaStream_t stream) {
  selftest_wait_kernel<<<1, 32, 0, stream>>>(dev.status, timeout_ns);
  return cudaGetLastError();
}

}  // namespace fp8bs

using fp8bs::aligned16;
using fp8bs::cuda_failure;
using fp8bs::kMaxDim;

extern "C" {

const char* fp8bs_status_string(fp8bs_status s) {
  switch (s) {
    case FP8BS_OK: return "ok";
    case FP8BS_ERR_INVALID_ARG: return "invalid argument";
    case FP8BS_ERR_MISALIGNED: return "misaligned pointer or stride";
    case FP8BS_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case FP8BS_ERR_CUDA: return "CUDA error";
    case FP8BS_ERR_TIMEOUT: return "in-kernel wait timed out";
  }
  return "unknown status";
}

const char* fp8bs_last_error_detail(void) { return fp8bs::t_detail; }

void fp8bs_set_wait_timeout_ns(uint64_t timeout_ns) {
  fp8bs::g_timeout_ns.store(timeout_ns ? timeout_ns : fp8bs::kDefaultTimeoutNs, std::memory_order_relaxed);
}

fp8bs_status fp8_quant_act_1x128(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* qa, int64_t ldq,
                                 float* sa, int64_t ld_sa, cudaStream_t stream) {
  if (M < 0 || K < 0 || ldx < 0 || ldq < 0 || ld_sa < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || K > kMaxDim || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || ldq < K || ld_sa < M) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (x_bf16 == nullptr || qa == nullptr || sa == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(qa) || !aligned16(sa) || ldx % 8 != 0 || ldq % 16 != 0 || ld_sa % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_quant_act_1x128(*dev, x_bf16, M, K, ldx, qa, ldq, sa, ld_sa, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_quant_act_1x128 launch", e);
}

fp8bs_status fp8_quant_weight_128x128(const void* w_bf16, int64_t N, int64_t K, int64_t ldw, void* qw, int64_t ldq,
                                      float* sw, cudaStream_t stream) {
  if (N < 0 || K < 0 || ldw < 0 || ldq < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldw < K || ldq < K) return FP8BS_ERR_INVALID_ARG;
  if (w_bf16 == nullptr || qw == nullptr || sw == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(w_bf16) || !aligned16(qw) || !aligned16(sw) || ldw % 8 != 0 || ldq % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_quant_weight_128x128(*dev, w_bf16, N, K, ldw, qw, ldq, sw, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_quant_weight_128x128 launch", e);
}

}  // extern "C"

namespace {

// Shared validation and launch of the dense GEMM; out_bytes is 2 (BF16 y) or
// 4 (FP32 y) and sets the row-stride rule for y.
fp8bs_status dense_gemm(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, const void* qw, int64_t ldqw,
                        const float* sw, void* y, int64_t ldy, int out_bytes, int64_t M, int64_t N, int64_t K,
                        cudaStream_t stream, const char* name, bool use_static_scratch = false,
                        const void* res = nullptr, int64_t ldr = 0) {
  if (M < 0 || N < 0 || K < 0 || ldqa < 0 || ld_sa < 0 || ldqw < 0 || ldy < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim || M > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldqa < K || ldqw < K || ldy < N || ld_sa < M) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (qa == nullptr || sa == nullptr || qw == nullptr || sw == nullptr || y == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qw) || !aligned16(sw) || !aligned16(y) || ldqa % 16 != 0 ||
      ldqw % 16 != 0 || (ldy * out_bytes) % 16 != 0 || ld_sa % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  fp8bs::Workspace ws;
  if (use_static_scratch) {
    ws.scratch = fp8bs::gemm_scratch_address(*dev, &e);
    if (ws.scratch == nullptr) return cuda_failure("scratch address", e);
    ws.scratch_bytes = fp8bs::kGemmScratchBytes;
  }
  e = fp8bs::launch_blockscaled_gemm(*dev, qa, ldqa, sa, ld_sa, qw, ldqw, sw, y, ldy, out_bytes == 4, M, N, K,
                                     stream, &ws, res, ldr);
  if (e != cudaSuccess) return cuda_failure(name, e);
  if (ws.too_small) {
    std::snprintf(fp8bs::t_detail, sizeof(fp8bs::t_detail),
                  "%s: the split-K tail needs %zu bytes of workspace, more than the %zu-byte static scratch", name,
                  ws.needed, ws.scratch_bytes);
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  }
  return FP8BS_OK;
}

fp8bs_status grouped_gemm(int32_t G, const int32_t* group_offsets_dev, int64_t M_total, const void* qa, int64_t ldqa,
                          const float* sa, int64_t ld_sa, const void* qw, const float* sw, void* y, int64_t ldy,
                          int out_bytes, int64_t N, int64_t K, cudaStream_t stream, const char* name) {
  if (G <= 0 || G > 65536 || M_total < 0 || N < 0 || K < 0 || ldqa < 0 || ld_sa < 0 || ldy < 0)
    return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || M_total > kMaxDim ||
      static_cast<int64_t>(G) * N > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldqa < K || ldy < N || ld_sa < M_total) return FP8BS_ERR_INVALID_ARG;
  if (group_offsets_dev == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (M_total == 0) return FP8BS_OK;
  if (qa == nullptr || sa == nullptr || qw == nullptr || sw == nullptr || y == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qw) || !aligned16(sw) || !aligned16(y) ||
      (reinterpret_cast<uintptr_t>(group_offsets_dev) & 3u) != 0 || ldqa % 16 != 0 || (ldy * out_bytes) % 16 != 0 ||
      ld_sa % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_blockscaled_grouped_gemm(*dev, G, group_offsets_dev, M_total, qa, ldqa, sa, ld_sa, qw, sw, y,
                                             ldy, out_bytes == 4, N, K, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure(name, e);
}

fp8bs_status rowscaled_gemm(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, const void* qb,
                           int64_t ldqb, const float* sb, int64_t ld_sb, void* y, int64_t ldy, int out_bytes,
                           int64_t M, int64_t N, int64_t K, cudaStream_t stream, const char* name) {
  if (M < 0 || N < 0 || K < 0 || ldqa < 0 || ld_sa < 0 || ldqb < 0 || ld_sb < 0 || ldy < 0)
    return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim || M > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldqa < K || ldqb < K || ldy < N || ld_sa < M || ld_sb < N) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (qa == nullptr || sa == nullptr || qb == nullptr || sb == nullptr || y == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb) || !aligned16(y) || ldqa % 16 != 0 ||
      ldqb % 16 != 0 || (ldy * out_bytes) % 16 != 0 || ld_sa % 4 != 0 || ld_sb % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_blockscaled_gemm_rowscaled(*dev, qa, ldqa, sa, ld_sa, qb, ldqb, sb, ld_sb, y, ldy, out_bytes == 4,
                                               M, N, K, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure(name, e);
}

}  // namespace

extern "C" {

fp8bs_status fp8_blockscaled_gemm_rowscaled(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                            const void* qb, int64_t ldqb, const float* sb, int64_t ld_sb,
                                            void* y_bf16, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                            cudaStream_t stream) {
  return rowscaled_gemm(qa, ldqa, sa, ld_sa, qb, ldqb, sb, ld_sb, y_bf16, ldy, 2, M, N, K, stream,
                        "fp8_blockscaled_gemm_rowscaled launch");
}

fp8bs_status fp8_blockscaled_gemm_rowscaled_f32(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                                const void* qb, int64_t ldqb, const float* sb, int64_t ld_sb,
                                                float* y_f32, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                                cudaStream_t stream) {
  return rowscaled_gemm(qa, ldqa, sa, ld_sa, qb, ldqb, sb, ld_sb, y_f32, ldy, 4, M, N, K, stream,
                        "fp8_blockscaled_gemm_rowscaled_f32 launch");
}

fp8bs_status fp8_quant_act_1x128_t(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* qt, int64_t ldqt,
                                   float* st, int64_t ld_st, cudaStream_t stream) {
  if (M < 0 || K < 0 || ldx < 0 || ldqt < 0 || ld_st < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || M % 128 != 0 || K > kMaxDim || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || ldqt < M || ld_st < K) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (x_bf16 == nullptr || qt == nullptr || st == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(qt) || !aligned16(st) || ldx % 8 != 0 || ldqt % 16 != 0 || ld_st % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_quant_act_1x128_t(*dev, x_bf16, M, K, ldx, qt, ldqt, st, ld_st, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_quant_act_1x128_t launch", e);
}

fp8bs_status fp8_pack_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, void* wp,
                                      cudaStream_t stream) {
  if (N < 0 || K < 0 || ldq < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldq < K) return FP8BS_ERR_INVALID_ARG;
  if (qw == nullptr || wp == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qw) || !aligned16(wp) || ldq % 16 != 0) return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_pack_weight_128x128(*dev, qw, N, K, ldq, wp, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_pack_weight_128x128 launch", e);
}

fp8bs_status fp8_blockscaled_gemm_packed(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                         const void* wp, const float* sw, void* y_bf16, int64_t ldy, int64_t M,
                                         int64_t N, int64_t K, cudaStream_t stream) {
  if (M < 0 || N < 0 || K < 0 || ldqa < 0 || ld_sa < 0 || ldy < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim || M > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldqa < K || ldy < N || ld_sa < M) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (qa == nullptr || sa == nullptr || wp == nullptr || sw == nullptr || y_bf16 == nullptr)
    return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(wp) || !aligned16(sw) || !aligned16(y_bf16) || ldqa % 16 != 0 ||
      ld_sa % 4 != 0 || ldy % 8 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_blockscaled_gemm_packed(*dev, qa, ldqa, sa, ld_sa, wp, sw, y_bf16, ldy, false, M, N, K, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_blockscaled_gemm_packed launch", e);
}

fp8bs_status fp8_requant_act_1x128_t(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, int64_t M,
                                     int64_t K, void* qt, int64_t ldqt, float* st, int64_t ld_st,
                                     cudaStream_t stream) {
  if (M < 0 || K < 0 || ldqa < 0 || ld_sa < 0 || ldqt < 0 || ld_st < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || M % 128 != 0 || K > kMaxDim || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldqa < K || ld_sa < M || ldqt < M || ld_st < K) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (qa == nullptr || sa == nullptr || qt == nullptr || st == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qa) || !aligned16(sa) || !aligned16(qt) || !aligned16(st) || ldqa % 16 != 0 || ld_sa % 4 != 0 ||
      ldqt % 16 != 0 || ld_st % 4 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_requant_act_1x128_t(*dev, qa, ldqa, sa, ld_sa, M, K, qt, ldqt, st, ld_st, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_requant_act_1x128_t launch", e);
}

fp8bs_status fp8_transpose_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, const float* sw,
                                          void* qwt, int64_t ldqt, float* swt, cudaStream_t stream) {
  if (N < 0 || K < 0 || ldq < 0 || ldqt < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldq < K || ldqt < N) return FP8BS_ERR_INVALID_ARG;
  if (qw == nullptr || sw == nullptr || qwt == nullptr || swt == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qw) || !aligned16(qwt) || (reinterpret_cast<uintptr_t>(sw) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(swt) & 3u) != 0 || ldq % 16 != 0 || ldqt % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_transpose_weight_128x128(*dev, qw, N, K, ldq, sw, qwt, ldqt, swt, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_transpose_weight_128x128 launch", e);
}

fp8bs_status fp8_quant_per_token(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                                 float* s, cudaStream_t stream) {
  if (M < 0 || K < 0 || ldx < 0 || ldq < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 8 != 0 || K > 32768 || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || ldq < K) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (x_bf16 == nullptr || q == nullptr || s == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s) & 3u) != 0 || ldx % 8 != 0 ||
      ldq % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_quant_per_token(*dev, x_bf16, M, K, ldx, q, ldq, s, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_quant_per_token launch", e);
}

fp8bs_status fp8_quant_per_channel(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                                   float* s, cudaStream_t stream) {
  if (M < 0 || K < 0 || ldx < 0 || ldq < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 8 != 0 || K > kMaxDim || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldx < K || ldq < K) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (x_bf16 == nullptr || q == nullptr || s == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(q) || !aligned16(s) || ldx % 8 != 0 || ldq % 16 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_quant_per_channel(*dev, x_bf16, M, K, ldx, q, ldq, s, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_quant_per_channel launch", e);
}

fp8bs_status fp8bs_e5m6_encode_bf16(const void* x_bf16, int64_t n, void* codes, cudaStream_t stream) {
  if (n < 0) return FP8BS_ERR_INVALID_ARG;
  if (n % 8 != 0 || n > (int64_t{1} << 40)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return FP8BS_OK;
  if (x_bf16 == nullptr || codes == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(x_bf16) || !aligned16(codes)) return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_cast_e5m6(*dev, x_bf16, n, codes, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8bs_e5m6_encode_bf16 launch", e);
}

fp8bs_status fp8bs_e5m6_decode_bf16(const void* codes, int64_t n, void* y_bf16, cudaStream_t stream) {
  if (n < 0) return FP8BS_ERR_INVALID_ARG;
  if (n % 8 != 0 || n > (int64_t{1} << 40)) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (n == 0) return FP8BS_OK;
  if (codes == nullptr || y_bf16 == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(y_bf16)) return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_e5m6_to_bf16(*dev, codes, n, y_bf16, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8bs_e5m6_decode_bf16 launch", e);
}

fp8bs_status fp8_swiglu_quant_act_1x128(const void* gate_up_bf16, int64_t M, int64_t F, int64_t ld, void* qa,
                                        int64_t ldq, float* sa, int64_t ld_sa, void* h_bf16, int64_t ldh,
                                        cudaStream_t stream) {
  if (M < 0 || F < 0 || ld < 0 || ldq < 0 || ld_sa < 0 || ldh < 0) return FP8BS_ERR_INVALID_ARG;
  if (F == 0 || F % 128 != 0 || F > kMaxDim / 2 || M > kMaxDim) return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ld < 2 * F || ldq < F || ld_sa < M || (h_bf16 != nullptr && ldh < F)) return FP8BS_ERR_INVALID_ARG;
  if (M == 0) return FP8BS_OK;
  if (gate_up_bf16 == nullptr || qa == nullptr || sa == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(gate_up_bf16) || !aligned16(qa) || !aligned16(sa) || ld % 8 != 0 || ldq % 16 != 0 ||
      ld_sa % 4 != 0 || (h_bf16 != nullptr && (!aligned16(h_bf16) || ldh % 8 != 0)))
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_swiglu_quant_act_1x128(*dev, gate_up_bf16, M, F, ld, qa, ldq, sa, ld_sa, h_bf16, ldh, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_swiglu_quant_act_1x128 launch", e);
}

fp8bs_status fp8_blockscaled_gemm(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, const void* qw,
                                  int64_t ldqw, const float* sw, void* y_bf16, int64_t ldy, int64_t M, int64_t N,
                                  int64_t K, cudaStream_t stream) {
  return dense_gemm(qa, ldqa, sa, ld_sa, qw, ldqw, sw, y_bf16, ldy, 2, M, N, K, stream, "fp8_blockscaled_gemm launch");
}

fp8bs_status fp8_blockscaled_gemm_residual(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                           const void* qw, int64_t ldqw, const float* sw, const void* r_bf16,
                                           int64_t ldr, void* y_bf16, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                           cudaStream_t stream) {
  if (ldr < 0) return FP8BS_ERR_INVALID_ARG;
  if (M > 0) {
    if (r_bf16 == nullptr || ldr < N) return FP8BS_ERR_INVALID_ARG;
    if (r_bf16 == y_bf16 && ldr != ldy) return FP8BS_ERR_INVALID_ARG;  // in place: same layout
    if (!aligned16(r_bf16) || ldr % 8 != 0) return FP8BS_ERR_MISALIGNED;
  }
  return dense_gemm(qa, ldqa, sa, ld_sa, qw, ldqw, sw, y_bf16, ldy, 2, M, N, K, stream,
                    "fp8_blockscaled_gemm_residual launch", false, r_bf16, ldr);
}

fp8bs_status fp8_blockscaled_gemm_noalloc(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, const void* qw,
                                          int64_t ldqw, const float* sw, void* y_bf16, int64_t ldy, int64_t M, int64_t N,
                                          int64_t K, cudaStream_t stream) {
  return dense_gemm(qa, ldqa, sa, ld_sa, qw, ldqw, sw, y_bf16, ldy, 2, M, N, K, stream,
                    "fp8_blockscaled_gemm_noalloc launch", true);
}

fp8bs_status fp8_blockscaled_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t* bytes) {
  if (bytes == nullptr || M < 0 || N < 0 || K < 0) return FP8BS_ERR_INVALID_ARG;
  *bytes = 0;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim || M > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return FP8BS_OK;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  fp8bs::Workspace ws;
  ws.plan_only = true;
  e = fp8bs::launch_blockscaled_gemm(*dev, nullptr, K, nullptr, M, nullptr, K, nullptr, nullptr, N, false, M, N, K,
                                     nullptr, &ws);
  if (e != cudaSuccess) return cuda_failure("fp8_blockscaled_gemm_workspace_bytes", e);
  *bytes = ws.needed;
  return FP8BS_OK;
}

fp8bs_status fp8_blockscaled_gemm_f32(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa, const void* qw,
                                      int64_t ldqw, const float* sw, float* y_f32, int64_t ldy, int64_t M, int64_t N,
                                      int64_t K, cudaStream_t stream) {
  return dense_gemm(qa, ldqa, sa, ld_sa, qw, ldqw, sw, y_f32, ldy, 4, M, N, K, stream,
                    "fp8_blockscaled_gemm_f32 launch");
}

fp8bs_status fp8_blockscaled_grouped_gemm(int32_t G, const int32_t* group_offsets_dev, int64_t M_total,
                                          const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                          const void* qw, const float* sw, void* y_bf16, int64_t ldy, int64_t N,
                                          int64_t K, cudaStream_t stream) {
  return grouped_gemm(G, group_offsets_dev, M_total, qa, ldqa, sa, ld_sa, qw, sw, y_bf16, ldy, 2, N, K, stream,
                      "fp8_blockscaled_grouped_gemm launch");
}

fp8bs_status fp8_blockscaled_grouped_gemm_f32(int32_t G, const int32_t* group_offsets_dev, int64_t M_total,
                                              const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                              const void* qw, const float* sw, float* y_f32, int64_t ldy, int64_t N,
                                              int64_t K, cudaStream_t stream) {
  return grouped_gemm(G, group_offsets_dev, M_total, qa, ldqa, sa, ld_sa, qw, sw, y_f32, ldy, 4, N, K, stream,
                      "fp8_blockscaled_grouped_gemm_f32 launch");
}

fp8bs_status fp8_dequant_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, const float* sw,
                                        void* y_bf16, int64_t ldy, cudaStream_t stream) {
  if (N < 0 || K < 0 || ldq < 0 || ldy < 0) return FP8BS_ERR_INVALID_ARG;
  if (K == 0 || K % 128 != 0 || N == 0 || N % 128 != 0 || K > kMaxDim || N > kMaxDim)
    return FP8BS_ERR_UNSUPPORTED_SHAPE;
  if (ldq < K || ldy < K) return FP8BS_ERR_INVALID_ARG;
  if (qw == nullptr || sw == nullptr || y_bf16 == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (!aligned16(qw) || !aligned16(y_bf16) || (reinterpret_cast<uintptr_t>(sw) & 3u) != 0 || ldq % 16 != 0 ||
      ldy % 8 != 0)
    return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_dequant_weight_128x128(*dev, qw, N, K, ldq, sw, y_bf16, ldy, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("fp8_dequant_weight_128x128 launch", e);
}

fp8bs_status fp8bs_last_device_error(cudaStream_t stream) {
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) return cuda_failure("stream synchronize", e);
  unsigned word = 0;
  const unsigned zero = 0;
  if ((e = cudaMemcpy(&word, dev->status, sizeof(word), cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_failure("status read", e);
  if (word != 0 && (e = cudaMemcpy(dev->status, &zero, sizeof(zero), cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_failure("status clear", e);
  switch (word) {
    case 0: return FP8BS_OK;
    case fp8bs::kStatusTimeout: return FP8BS_ERR_TIMEOUT;
    case fp8bs::kStatusBadOffsets: return FP8BS_ERR_INVALID_ARG;
  }
  return FP8BS_ERR_CUDA;
}

fp8bs_status fp8bs_stream_timestamp(uint64_t* dst, int release_next, cudaStream_t stream) {
  if (dst == nullptr) return FP8BS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(dst) % 8 != 0) return FP8BS_ERR_MISALIGNED;
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_stream_timestamp(dst, release_next != 0, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("timestamp launch", e);
}

fp8bs_status fp8bs_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream) {
  cudaError_t e;
  const fp8bs::DeviceInfo* dev = fp8bs::current_device_info(&e);
  if (dev == nullptr) return cuda_failure("device query", e);
  e = fp8bs::launch_selftest_wait(*dev, timeout_ns, stream);
  return e == cudaSuccess ? FP8BS_OK : cuda_failure("self-test launch", e);
}

}  // extern "C"
