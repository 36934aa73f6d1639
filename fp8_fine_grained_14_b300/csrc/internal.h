// internal.h — launchers shared between the C-ABI layer (api.cu) and the
// kernel translation units.  Arguments arrive here already validated.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8bs {

// Launches `kernel` with programmatic stream serialisation: the launch may
// be processed while the previous kernel on `stream` is still running, which
// shortens the gap between dependent kernels (about 1 us instead of 3-6 us
// on B300).  Every kernel of the library starts with pdl_wait() (ptx.cuh), so
// it still sees all the writes of the work before it.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

struct DeviceInfo {
  int ordinal;
  int num_sms;
  int max_smem_optin;
  unsigned* status;  // device address of this device's status word
};

// Per-device facts, looked up once per device (thread-safe).  Returns nullptr
// and sets *err when the device cannot be queried.
const DeviceInfo* current_device_info(cudaError_t* err);

// Library-owned stream-ordered memory pool of a device for GEMM split-K
// workspaces, created on first use (thread-safe).  It keeps freed memory for
// reuse instead of returning it at every synchronisation.  Null when the
// device offers no memory pools (split tails then run unsplit).
cudaMemPool_t gemm_workspace_pool(const DeviceInfo& dev);

// Where the FP32 partials of a split-K tail go (see launch_blockscaled_gemm).
struct Workspace {
  float* scratch = nullptr;   // a fixed device region; null: the device's workspace pool
  size_t scratch_bytes = 0;   // its size
  bool plan_only = false;     // decide the tile plan and report `needed`; launch nothing
  size_t needed = 0;          // out: workspace bytes the split tail needs (0: no split)
  bool too_small = false;     // out: scratch given and smaller than `needed` (nothing launched)
};

uint64_t wait_timeout_ns();

// Encodes a 2-D row-major tensor map; returns false on failure.
bool make_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                  uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle);

cudaError_t launch_quant_act_1x128(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                   void* q, int64_t ldq, float* sa, int64_t ld_sa, cudaStream_t stream);

cudaError_t launch_quant_weight_128x128(const DeviceInfo& dev, const void* w, int64_t N, int64_t K, int64_t ldw,
                                        void* q, int64_t ldq, float* sw, cudaStream_t stream);

// Returns cudaErrorInvalidValue when a tensor map cannot be encoded.
// y is BF16 (y_f32 false) or FP32 (y_f32 true); ldy in elements of that type.
// When the last round of tiles would leave most SMs idle, the tail tiles are
// split along K; their FP32 partials go to ws->scratch, or, when that is null,
// to stream-ordered memory from gemm_workspace_pool (allocated and freed on
// `stream` around the two kernels).  ws->needed reports the bytes; with a
// scratch region smaller than that, nothing is launched and ws->too_small is
// set.  With ws->plan_only only ws->needed is computed.  ws may be null (the
// pool).  res (BF16, row stride ldr elements), when not null, is added to the
// FP32 result before the output rounding; it may be y itself (same stride)
// for an in-place update.
cudaError_t launch_blockscaled_gemm(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                    int64_t ld_sa, const void* qw, int64_t ldqw, const float* sw, void* y,
                                    int64_t ldy, bool y_f32, int64_t M, int64_t N, int64_t K, cudaStream_t stream,
                                    Workspace* ws = nullptr, const void* res = nullptr, int64_t ldr = 0);

// As launch_blockscaled_gemm with B as packed 128x128 tiles wp[N/128][K/128]
// (fp8_pack_weight_128x128's layout); single-CTA tile shapes only.
cudaError_t launch_blockscaled_gemm_packed(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                           int64_t ld_sa, const void* wp, const float* sw, void* y, int64_t ldy,
                                           bool y_f32, int64_t M, int64_t N, int64_t K, cudaStream_t stream);

// Codes W [N, K] -> packed tiles wp[N/128][K/128][128 x 128 bytes], each the
// 128B-swizzled K-major image that a GEMM stage holds.
cudaError_t launch_pack_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                       void* wp, cudaStream_t stream);

cudaError_t launch_blockscaled_grouped_gemm(const DeviceInfo& dev, int32_t G, const int32_t* offsets,
                                            int64_t M_total, const void* qa, int64_t ldqa, const float* sa,
                                            int64_t ld_sa, const void* qw, const float* sw, void* y, int64_t ldy,
                                            bool y_f32, int64_t N, int64_t K, cudaStream_t stream);

cudaError_t launch_dequant_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                          const float* sw, void* y, int64_t ldy, cudaStream_t stream);

// Y = sum_kb sa[kb][m] * sb[kb][n] * chunk product (1x128 scales on both operands).
cudaError_t launch_blockscaled_gemm_rowscaled(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                              int64_t ld_sa, const void* qb, int64_t ldqb, const float* sb,
                                              int64_t ld_sb, void* y, int64_t ldy, bool y_f32, int64_t M, int64_t N,
                                              int64_t K, cudaStream_t stream);

// 1x128 quantisation of X^T: codes [K, M] (row stride ldqt bytes), scales
// st[m / 128][k] (row stride ld_st).  M % 128 == 0.
cudaError_t launch_quant_act_1x128_t(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* qt, int64_t ldqt, float* st, int64_t ld_st, cudaStream_t stream);

// The same from X's FP8 cache (1x128 codes [M, K], stride ldqa; scales
// sa[kb * ld_sa + m]): each value is dequantised to BF16 first.
cudaError_t launch_requant_act_1x128_t(const DeviceInfo& dev, const void* qa, int64_t ldqa, const float* sa,
                                       int64_t ld_sa, int64_t M, int64_t K, void* qt, int64_t ldqt, float* st,
                                       int64_t ld_st, cudaStream_t stream);

cudaError_t launch_transpose_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                            const float* sw, void* qt, int64_t ldqt, float* swt,
                                            cudaStream_t stream);

// Quantisation variants (variants.cu).
cudaError_t launch_quant_per_token(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx, void* q,
                                   int64_t ldq, float* s, cudaStream_t stream);
cudaError_t launch_quant_per_channel(const DeviceInfo& dev, const void* x, int64_t M, int64_t K, int64_t ldx,
                                     void* q, int64_t ldq, float* s, cudaStream_t stream);
cudaError_t launch_cast_e5m6(const DeviceInfo& dev, const void* x, int64_t n, void* codes, cudaStream_t stream);
cudaError_t launch_e5m6_to_bf16(const DeviceInfo& dev, const void* codes, int64_t n, void* y, cudaStream_t stream);
cudaError_t launch_swiglu_quant_act_1x128(const DeviceInfo& dev, const void* gate_up, int64_t M, int64_t F,
                                          int64_t ld, void* q, int64_t ldq, float* sa, int64_t ld_sa, void* h,
                                          int64_t ldh, cudaStream_t stream);

cudaError_t launch_selftest_wait(const DeviceInfo& dev, uint64_t timeout_ns, cudaStream_t stream);
cudaError_t launch_stream_timestamp(uint64_t* dst, int release, cudaStream_t stream);

}  // namespace fp8bs
