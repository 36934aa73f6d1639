// pack.cu — weight codes in the GEMM's stage layout, for weight-streaming
// (decode-shaped) GEMMs on sm_103a.
//
// A block-scaled GEMM stage holds B's 128 rows x 128 K-bytes of one 128x128
// block in the 128B-swizzled K-major layout that the tensor-core descriptors
// read: row r at byte 128 r, its 16-byte chunk c at chunk position c ^ (r % 8).
// Read from row-major codes, every stage is 128 runs of 128 bytes, one per
// weight row, 7 KB or more apart.  Packed, the same stage is one contiguous
// 16 KB run that a single bulk copy moves, which keeps DRAM pages open when
// the weights stream through once per call (decode).  The codes and the block
// scales are those of fp8_quant_weight_128x128 ("The Definitive Information To
// Deepseek", "Figure 7 (a)" item (2): one scale per 128x128 block); only the
// byte order changes.
#include "internal.h"
#include "ptx.cuh"

namespace fp8bs {
namespace {

// One 128x128 block per iteration: thread t copies half of row t / 2
// (chunks 4 (t % 2) .. + 3) to their swizzled positions in the block's image.
__global__ void __launch_bounds__(256) pack_weight_128x128_kernel(const uint4* __restrict__ q, int64_t NB,
                                                                  int64_t KB, int64_t ldq_v, uint4* __restrict__ wp) {
  pdl_wait();
  const int r = threadIdx.x >> 1;
  const int h = threadIdx.x & 1;
  for (int64_t tile = blockIdx.x; tile < NB * KB; tile += gridDim.x) {
    const int64_t nb = tile / KB, kb = tile % KB;
    const uint4* src = q + (nb * 128 + r) * ldq_v + kb * 8 + 4 * h;
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldcs(src + i);
    uint4* dst = wp + tile * (128 * 8) + r * 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[(4 * h + i) ^ (r & 7)] = v[i];
  }
}

}  // namespace

cudaError_t launch_pack_weight_128x128(const DeviceInfo& dev, const void* q, int64_t N, int64_t K, int64_t ldq,
                                       void* wp, cudaStream_t stream) {
  const int64_t NB = N / 128, KB = K / 128;
  const int64_t cap = static_cast<int64_t>(dev.num_sms) * 8;
  const int64_t tiles = NB * KB;
  (void)launch_pdl(pack_weight_128x128_kernel, static_cast<unsigned>(tiles < cap ? tiles : cap), 256, 0, stream,
      static_cast<const uint4*>(q), NB, KB, ldq / 16, static_cast<uint4*>(wp));
  return cudaGetLastError();
}

}  // namespace fp8bs
