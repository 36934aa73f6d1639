/*
 * fp8bs.h — C ABI of the fine-grained FP8 block-scaled linear layer for
 * B300 (sm_103a).
 *
 * Method: the DeepSeek-V3 FP8 mixed-precision framework as excerpted in
 * "The Definitive Information To Deepseek":
 *   - paragraph 3, "Figure 7 (a)": activations are grouped and scaled on 1x128
 *     tiles (per token per 128 channels), weights on 128x128 blocks (per 128
 *     input channels per 128 output channels);
 *   - paragraph 2, last sentence: each group's scaling factor is derived
 *     online and the tensor is quantised into FP8;
 *   - paragraph 4, first sentence: the GEMM takes FP8 tensors and writes BF16;
 *   - paragraph 1, last sentence: partial sums are promoted to a higher
 *     precision accumulator while the next MMA proceeds.
 * Readings of what the excerpt leaves open: FP8 is OCP E4M3FN; a group's
 * scale is s = fl32(amax / 448) (IEEE float32 division, no flush to zero);
 * codes are E4M3(fl32(x / s)) rounded to nearest even and saturated to +-448;
 * an all-zero group has s = 0 and codes 0x00; promotion happens once per
 * 128-wide K chunk with the factor sa * sw.
 *
 * Conventions shared by every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates, frees or retains them.  Base pointers must be 16-byte
 *     aligned (FP8BS_ERR_MISALIGNED otherwise).
 *   - Memory the library owns: per device, one status word (a __device__
 *     variable) and the fixed 20 MiB static scratch array of
 *     fp8_blockscaled_gemm_noalloc (both part of the loaded module), and one
 *     stream-ordered memory pool for the split-K workspace of
 *     fp8_blockscaled_gemm, _f32 and _residual.  The pool is created by the
 *     first of those calls whose last round of tiles is split; each such call
 *     takes at most 128 KiB per SM of the device (18.5 MiB on 148 SMs) from it
 *     on its stream and returns it on the same stream after the two kernels.
 *     The pool keeps freed memory for reuse (it is never trimmed while the
 *     process runs), so repeated calls do not allocate from the device again.
 *     fp8_blockscaled_gemm_workspace_bytes tells how much a shape takes.
 *     Nothing else is allocated.
 *   - Matrices are row-major; "ld" arguments are row strides in ELEMENTS.
 *     BF16 and FP8 row strides must make 16-byte multiples (ld % 8 == 0 for
 *     BF16, ld % 16 == 0 for FP8 codes).
 *   - FP8 codes are OCP E4M3FN bytes (bit-compatible with torch.float8_e4m3fn).
 *   - Activation scales are stored TRANSPOSED: sa[kb * ld_sa + m] is the scale
 *     of row m, channels 128*kb .. 128*kb+127; ld_sa >= M and ld_sa % 4 == 0.
 *     Weight scales are sw[nb * (K/128) + kb] for rows 128*nb.., columns 128*kb...
 *   - Shape rules: K % 128 == 0 and K > 0; N % 128 == 0 and N > 0;
 *     M >= 0 is arbitrary (M == 0 is a no-op).  Violations return
 *     FP8BS_ERR_UNSUPPORTED_SHAPE (or FP8BS_ERR_INVALID_ARG for negative sizes,
 *     short strides and null pointers) before anything is launched.
 *   - Every call is asynchronous on `stream` (0 = legacy default stream) and
 *     returns after validation and launch.  A launch failure returns
 *     FP8BS_ERR_CUDA (fp8bs_last_error_detail() names the CUDA error).
 *     Kernel waits are bounded; a wait that gives up records
 *     FP8BS_ERR_TIMEOUT in a per-device status word, which
 *     fp8bs_last_device_error() reports.
 *   - No CPU fallback exists: without a usable CUDA device the calls fail.
 *   - Thread safety: calls may be made concurrently from several host threads.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FP8BS_OK = 0,
  FP8BS_ERR_INVALID_ARG = 1,       /* null pointer, negative size, short stride or bad group offsets */
  FP8BS_ERR_MISALIGNED = 2,        /* pointer or row stride breaks the 16-byte rules above */
  FP8BS_ERR_UNSUPPORTED_SHAPE = 3, /* K or N not a positive multiple of 128, or sizes too large */
  FP8BS_ERR_CUDA = 4,              /* a CUDA runtime/driver call or a launch failed */
  FP8BS_ERR_TIMEOUT = 5            /* a bounded in-kernel wait gave up (reported asynchronously) */
} fp8bs_status;

/*
 * 1x128 activation quantisation ("Figure 7 (a)" item (1); online scaling of
 * paragraph 2).
 *   x_bf16 : [M, K] BF16, row stride ldx (elements).
 *   qa     : [M, K] E4M3 codes out, row stride ldq (bytes).
 *   sa     : [K/128, ld_sa] FP32 scales out, sa[kb*ld_sa + m].
 * Columns m >= M of sa are left untouched.
 */
fp8bs_status fp8_quant_act_1x128(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                 void* qa, int64_t ldq, float* sa, int64_t ld_sa,
                                 cudaStream_t stream);

/*
 * 128x128 weight quantisation ("Figure 7 (a)" item (2)).
 *   w_bf16 : [N, K] BF16 (row = output channel), row stride ldw.
 *   qw     : [N, K] E4M3 codes out, row stride ldq.
 *   sw     : [N/128, K/128] FP32 scales out, row-major, contiguous.
 * A stack of G expert weights [G, N, K] can be passed as one [G*N, K] matrix:
 * blocks never straddle experts because N % 128 == 0.
 */
fp8bs_status fp8_quant_weight_128x128(const void* w_bf16, int64_t N, int64_t K, int64_t ldw,
                                      void* qw, int64_t ldq, float* sw, cudaStream_t stream);

/*
 * Block-scaled FP8 GEMM with per-128-K-chunk promotion (paragraphs 1 and 4):
 *   Y[m, n] = bf16( sum_kb sa[kb*ld_sa + m] * sw[(n/128)*(K/128) + kb]
 *                   * sum_{k in chunk kb} dec(qa[m, k]) * dec(qw[n, k]) ).
 *   qa : [M, K] codes, row stride ldqa (bytes);  qw : [N, K] codes, stride ldqw.
 *   y  : [M, N] BF16 out, row stride ldy (elements).
 * Chunk products accumulate in FP32 tensor memory; each chunk is scaled and
 * added to an FP32 register accumulator; the result is rounded to BF16
 * (round to nearest even).
 * Workspace: when the last round of output tiles would leave at least half
 * of the SMs idle, those tiles are split along K over the idle SMs, and their
 * FP32 partial sums go to a workspace drawn from the library's per-device
 * pool on `stream` (at most 128 KiB per SM; see the conventions above and
 * fp8_blockscaled_gemm_workspace_bytes).  A second kernel sums the slices in
 * a fixed order, so results do not depend on timing.  Without a pool on the
 * device the tail runs unsplit (same results).
 */
fp8bs_status fp8_blockscaled_gemm(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                  const void* qw, int64_t ldqw, const float* sw,
                                  void* y_bf16, int64_t ldy,
                                  int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * As fp8_blockscaled_gemm, with FP32 output (paragraph 4: the FP8 GEMMs
 * "produce outputs in BF16 or FP32"): y[m, n] is the FP32 accumulator itself,
 * not rounded further.  y : [M, N] FP32, row stride ldy (elements, ldy % 4 == 0).
 * Split-K workspace from the library's pool as for fp8_blockscaled_gemm.
 */
fp8bs_status fp8_blockscaled_gemm_f32(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                      const void* qw, int64_t ldqw, const float* sw,
                                      float* y_f32, int64_t ldy,
                                      int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * Grouped (per-expert) block-scaled GEMM for MoE row groups.  Rows
 * off[g] .. off[g+1]-1 of qa, sa and y belong to expert g and are multiplied
 * by expert g's weights:
 *   group_offsets_dev : DEVICE int32 [G+1], off[0] == 0, non-decreasing,
 *                       off[G] == M_total (checked on the device: a bad table
 *                       records FP8BS_ERR_INVALID_ARG in the status word and
 *                       the offending groups are skipped).
 *   M_total           : host copy of off[G] (sizes the launch; 0 is a no-op).
 *   qa [M_total, K] (stride ldqa), sa [K/128, ld_sa] with ld_sa >= M_total,
 *   qw [G, N, K] contiguous codes, sw [G, N/128, K/128] contiguous scales,
 *   y [M_total, N] BF16 (stride ldy).  Empty groups are allowed.
 *   1 <= G <= 65536.
 */
fp8bs_status fp8_blockscaled_grouped_gemm(int32_t G, const int32_t* group_offsets_dev, int64_t M_total,
                                          const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                          const void* qw, const float* sw,
                                          void* y_bf16, int64_t ldy,
                                          int64_t N, int64_t K, cudaStream_t stream);

/*
 * As fp8_blockscaled_grouped_gemm, with FP32 output (ldy % 4 == 0).
 */
fp8bs_status fp8_blockscaled_grouped_gemm_f32(int32_t G, const int32_t* group_offsets_dev, int64_t M_total,
                                              const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                              const void* qw, const float* sw,
                                              float* y_f32, int64_t ldy,
                                              int64_t N, int64_t K, cudaStream_t stream);

/*
 * 128x128 block dequantisation, the inverse of fp8_quant_weight_128x128: the
 * BF16 conversion of FP8 weights that the DeepSeek-V3 model card (section 6,
 * "How to Run Locally") provides for its FP8-only checkpoints.
 *   qw : [N, K] E4M3 codes, row stride ldq (bytes).
 *   sw : [N/128, K/128] FP32 block scales, row-major, contiguous (4-byte aligned).
 *   y  : [N, K] BF16 out, row stride ldy (elements):
 *        y[n, k] = bf16_rn(fl32(dec(qw[n, k]) * sw[n/128][k/128])).
 * N % 128 == 0, K % 128 == 0.  A stack of experts passes as [G*N, K].
 */
fp8bs_status fp8_dequant_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, const float* sw,
                                        void* y_bf16, int64_t ldy, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Backward GEMMs of the linear layer.  The excerpt keeps the activation in
 * FP8 for the backward pass (paragraph 2) and splits the backward into its
 * input-gradient and weight-gradient parts (paragraph 3):
 *   dX = dY . W    : fp8_quant_act_1x128(dY) and fp8_transpose_weight_128x128
 *                    of W's codes, then fp8_blockscaled_gemm;
 *   dW = dY^T . X  : fp8_quant_act_1x128_t of dY and of X (1x128 tiles of the
 *                    transposes: per channel per 128 tokens), then
 *                    fp8_blockscaled_gemm_rowscaled(_f32).
 * ------------------------------------------------------------------------ */

/*
 * Weight codes in the GEMM's stage layout, for weight-streaming
 * (decode-shaped) GEMMs.  The codes and block scales stay those of
 * fp8_quant_weight_128x128 ("Figure 7 (a)" item (2)); only the byte order
 * changes: packed tile (nb, kb) is 16384 contiguous bytes at
 * wp + (nb * K/128 + kb) * 16384, holding rows 128 nb + r (r < 128) and
 * columns 128 kb + c (c < 128) of qw with byte (r, c) at
 *     128 r + 16 ((c / 16) XOR (r % 8)) + (c % 16),
 * the 128-byte-swizzled K-major image that a GEMM stage holds.
 *   qw : [N, K] codes, row stride ldq (bytes, % 16 == 0).
 *   wp : N * K bytes out, 16-byte aligned.
 * N % 128 == 0 and K % 128 == 0.
 */
fp8bs_status fp8_pack_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, void* wp,
                                     cudaStream_t stream);

/*
 * fp8_blockscaled_gemm with B given as packed tiles (fp8_pack_weight_128x128):
 * the same Y, bit for bit, but every B stage arrives as one contiguous bulk
 * copy.  Meant for skinny M, where streaming the weights is the whole cost;
 * large grids run on single-CTA tiles (no CTA pairs).  sw as for
 * fp8_blockscaled_gemm; other arguments and errors likewise.
 */
fp8bs_status fp8_blockscaled_gemm_packed(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                         const void* wp, const float* sw, void* y_bf16, int64_t ldy,
                                         int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * 1x128 quantisation of X^T for X [M, K] BF16 (row stride ldx): each run of
 * 128 rows of one column is a group.
 *   qt : [K, M] E4M3 codes of X^T out, row stride ldqt (bytes, % 16 == 0).
 *   st : [M/128, ld_st] FP32 scales out, st[mb * ld_st + k] (ld_st >= K,
 *        ld_st % 4 == 0) -- the activation-scale layout of X^T.
 * M % 128 == 0 and K % 128 == 0 (FP8BS_ERR_UNSUPPORTED_SHAPE otherwise).
 * Codes and scales equal fp8_quant_act_1x128 applied to X^T.
 */
fp8bs_status fp8_quant_act_1x128_t(const void* x_bf16, int64_t M, int64_t K, int64_t ldx,
                                   void* qt, int64_t ldqt, float* st, int64_t ld_st, cudaStream_t stream);

/*
 * fp8_quant_act_1x128_t with X taken from its FP8 cache: the forward's 1x128
 * codes and scales of X, kept for the backward pass instead of BF16 X
 * ("The Definitive Information To Deepseek", paragraph 2).  Each cached value
 * is dequantised to BF16, x = bf16_rn(fl32(dec(qa[m, k]) * sa[kb][m])) (the
 * conversion of fp8_dequant_weight_128x128 with the 1x128 grouping), and the
 * result is quantised on 1x128 tiles of X^T exactly as fp8_quant_act_1x128_t
 * does; the BF16 values never reach HBM.
 *   qa : [M, K] E4M3 codes, row stride ldqa (bytes, % 16 == 0).
 *   sa : [K/128, ld_sa] FP32 scales, sa[kb * ld_sa + m] (ld_sa >= M,
 *        ld_sa % 4 == 0, 16-byte aligned) -- fp8_quant_act_1x128's layout.
 *   qt, st : as fp8_quant_act_1x128_t.
 * M % 128 == 0 and K % 128 == 0 (FP8BS_ERR_UNSUPPORTED_SHAPE otherwise).
 */
fp8bs_status fp8_requant_act_1x128_t(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                     int64_t M, int64_t K, void* qt, int64_t ldqt, float* st, int64_t ld_st,
                                     cudaStream_t stream);

/*
 * Codes and block scales of W^T from those of W [N, K]: a 128x128 block is
 * a block either way round ("Figure 7 (a)" item (2)), so nothing is
 * requantised.
 *   qw  : [N, K] codes (row stride ldq);   sw  : [N/128, K/128] scales.
 *   qwt : [K, N] codes out (row stride ldqt, % 16 == 0);
 *   swt : [K/128, N/128] scales out, contiguous.
 */
fp8bs_status fp8_transpose_weight_128x128(const void* qw, int64_t N, int64_t K, int64_t ldq, const float* sw,
                                          void* qwt, int64_t ldqt, float* swt, cudaStream_t stream);

/*
 * Block-scaled FP8 GEMM with 1x128 scales on BOTH operands (the weight-gradient
 * GEMM, whose operands are quantised along the token dimension):
 *   Y[m, n] = sum_kb sa[kb*ld_sa + m] * sb[kb*ld_sb + n]
 *             * sum_{k in chunk kb} dec(qa[m, k]) * dec(qb[n, k]),
 * promoted per 128-wide K chunk in FP32.  qa [M, K] (stride ldqa), qb [N, K]
 * (stride ldqb), ld_sa >= M, ld_sb >= N, both % 4 == 0.  Y BF16 [M, N]
 * (stride ldy), or FP32 for the _f32 variant (ldy % 4 == 0).
 */
fp8bs_status fp8_blockscaled_gemm_rowscaled(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                            const void* qb, int64_t ldqb, const float* sb, int64_t ld_sb,
                                            void* y_bf16, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                            cudaStream_t stream);
fp8bs_status fp8_blockscaled_gemm_rowscaled_f32(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                                const void* qb, int64_t ldqb, const float* sb, int64_t ld_sb,
                                                float* y_f32, int64_t ldy, int64_t M, int64_t N, int64_t K,
                                                cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Quantisation variants.  The TileKernels release ("DeepSeek starts updating
 * frequently", the tile kernels' features, item "Quantification") converts to
 * FP8 / E5M6 per token, per block and per channel and fuses SwiGLU with the
 * quantisation; the V3 excerpt (paragraph 3) keeps certain activations in a
 * custom E5M6 format.  The FP8 variants use the 1x128 quantiser's rule
 * s = fl32(amax / 448), codes E4M3_RNE_satfinite(fl32(x / s)).
 * ------------------------------------------------------------------------ */

/*
 * Per token: one scale per row of X [M, K] BF16 over all K channels.
 *   q : [M, K] codes (row stride ldq bytes);  s : [M] FP32 scales, contiguous.
 * K % 8 == 0 and K <= 32768.
 */
fp8bs_status fp8_quant_per_token(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                                 float* s, cudaStream_t stream);

/*
 * Per channel: one scale per column of X [M, K] BF16 over all M rows.
 *   q : [M, K] codes (row stride ldq);  s : [K] FP32 scales, contiguous,
 *   16-byte aligned.  K % 8 == 0.  X is read twice (maxima, then codes), in
 *   one kernel; while X fits in L2 the second read is served from there.
 */
fp8bs_status fp8_quant_per_channel(const void* x_bf16, int64_t M, int64_t K, int64_t ldx, void* q, int64_t ldq,
                                   float* s, cudaStream_t stream);

/*
 * E5M6 activation format: sign, 5 exponent bits (bias 15), 6 mantissa bits
 * in the low 12 bits of a 16-bit word; subnormals 2^-14 * m / 64; exponent
 * field 31 reserved (decoded as inf / NaN).  Encoding rounds to nearest even
 * and saturates magnitudes above 65024 (no scale factor).  n BF16 values in,
 * n 16-bit codes out (n % 8 == 0, 16-byte aligned buffers); decoding back to
 * BF16 is exact.
 */
fp8bs_status fp8bs_e5m6_encode_bf16(const void* x_bf16, int64_t n, void* codes_u16, cudaStream_t stream);
fp8bs_status fp8bs_e5m6_decode_bf16(const void* codes_u16, int64_t n, void* y_bf16, cudaStream_t stream);

/*
 * SwiGLU fused with 1x128 quantisation.  gate_up : [M, 2F] BF16 (row stride
 * ld): gate in columns [0, F), up projection in [F, 2F).
 *   h = bf16_rn(silu(g) * u), silu(g) = g / (1 + exp(-g)) evaluated in FP32
 *   as g * sigmoid(g) from exp(-|g|) and a reciprocal of 1 + exp(-|g|)
 *   (within a few FP32 ulps of the exact value wherever that is a normal
 *   FP32 number, before the BF16 rounding), and h is
 *   quantised exactly as fp8_quant_act_1x128 would: qa [M, F] codes (stride
 *   ldq), sa [F/128, ld_sa] scales.  h itself is written to h_bf16 (stride
 *   ldh) when h_bf16 is not null.  F % 128 == 0.
 */
fp8bs_status fp8_swiglu_quant_act_1x128(const void* gate_up_bf16, int64_t M, int64_t F, int64_t ld,
                                        void* qa, int64_t ldq, float* sa, int64_t ld_sa,
                                        void* h_bf16, int64_t ldh, cudaStream_t stream);

/*
 * fp8_blockscaled_gemm with a residual: Y = bf16_rn(fl32(sum) + R), where the
 * FP32 result of the block-scaled GEMM and the BF16 residual R [M, N] (row
 * stride ldr elements) are added before the single rounding to BF16
 * ("The Definitive Information To Deepseek", paragraph 4: BF16 or FP32
 * outputs; the addition fuses the block's residual stream into the
 * epilogue).  R and Y are either the same buffer with the same stride (an
 * in-place update of the residual stream) or disjoint.  R must be 16-byte
 * aligned with ldr % 8 == 0 and ldr >= N; otherwise as fp8_blockscaled_gemm,
 * split-K workspace from the library's pool included.
 */
fp8bs_status fp8_blockscaled_gemm_residual(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                           const void* qw, int64_t ldqw, const float* sw,
                                           const void* r_bf16, int64_t ldr, void* y_bf16, int64_t ldy,
                                           int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * fp8_blockscaled_gemm for callers that cannot allocate device memory.  The
 * pages have no counterpart of this call; it serves code that runs where a
 * cudaMalloc or a memory-pool allocation is not allowed or not safe: a host
 * whose device memory is all handed out by another allocator (a framework,
 * or a fixed arena planned ahead of time), code that must not add the
 * implicit synchronisation or the latency of an allocation to its step, or
 * code that must not fail for lack of memory half-way through a step.
 *
 * Arguments, layouts, results (bit for bit) and errors are those of
 * fp8_blockscaled_gemm, except for the workspace of a split-K tail: its FP32
 * partials go to a fixed static device array of 20 MiB in the library (one
 * per device, part of the loaded module, held until the process exits)
 * instead of the pool.  The call makes no cudaMalloc, cudaFree or pool
 * allocation and creates no pool.  Nothing in the array needs clearing
 * between calls (every partial is written before it is read).
 *   - A shape whose split tail would need more than 20 MiB returns
 *     FP8BS_ERR_UNSUPPORTED_SHAPE and launches nothing
 *     (fp8_blockscaled_gemm_workspace_bytes tells the need; devices with up
 *     to 160 SMs never need more).
 *   - Every call on a device shares the array: calls whose work overlaps on
 *     the GPU (different streams without ordering between them) race on it
 *     and may return wrong results.  Order them on one stream, or with events.
 *   - The first call on a device, like the first call of any entry point,
 *     sets up per-device state with synchronous runtime calls (device
 *     attributes, the addresses of the library's device variables, clearing
 *     the status word).  Make that first call before any stream capture.
 */
fp8bs_status fp8_blockscaled_gemm_noalloc(const void* qa, int64_t ldqa, const float* sa, int64_t ld_sa,
                                          const void* qw, int64_t ldqw, const float* sw,
                                          void* y_bf16, int64_t ldy,
                                          int64_t M, int64_t N, int64_t K, cudaStream_t stream);

/*
 * Split-K workspace, in bytes, that fp8_blockscaled_gemm takes from the
 * library's pool for an M x N x K product on the current device (and that
 * fp8_blockscaled_gemm_noalloc needs in its static array): 0 when the shape's
 * tiles are not split.  No counterpart in the pages.  Nothing is launched or
 * allocated.  Shape errors as for fp8_blockscaled_gemm; null `bytes`
 * returns FP8BS_ERR_INVALID_ARG.
 */
fp8bs_status fp8_blockscaled_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, size_t* bytes);

/*
 * Text naming the CUDA error (and the step) behind the last FP8BS_ERR_CUDA
 * returned to the calling host thread; "" if none.  Valid until the thread's
 * next call into the library.
 */
const char* fp8bs_last_error_detail(void);

/* Static, human-readable name of a status code. */
const char* fp8bs_status_string(fp8bs_status s);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns FP8BS_OK, FP8BS_ERR_TIMEOUT, FP8BS_ERR_INVALID_ARG (a bad
 * group-offset table) or FP8BS_ERR_CUDA (the synchronisation failed).
 */
fp8bs_status fp8bs_last_device_error(cudaStream_t stream);

/*
 * Limit, in nanoseconds, of every bounded in-kernel wait launched after the
 * call (default 1e9 = 1 s; 0 restores the default).  Process-wide.
 */
void fp8bs_set_wait_timeout_ns(uint64_t timeout_ns);

/*
 * Self-test of the bounded-wait path: launches one warp that waits on a
 * barrier nothing will ever signal, with a limit of `timeout_ns`.  The wait
 * gives up, records FP8BS_ERR_TIMEOUT in the status word and the kernel
 * returns; the context stays usable.  No counterpart in the method; it exists
 * so failure detection can be exercised without faulting or hanging a GPU.
 */
fp8bs_status fp8bs_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

/*
 * Measurement aid, no counterpart in the method.  Enqueues on `stream` a
 * one-thread kernel that waits until the work before it on the stream has
 * completed, then writes the device's global timer (nanoseconds) to *dst
 * (device memory, 8-byte aligned, owned by the caller).  The library's
 * kernels launch as programmatic dependents of the work before them, and
 * fp8_quant_act_1x128 lets the next kernel launch before it finishes, so
 * that a GEMM after it sets up early; release_next != 0 makes the timestamp
 * do the same (pass it for a timestamp placed right after that call).
 * Placed between kernels this way, consecutive timestamps split a sequence
 * into per-kernel intervals (each including the short dependent-launch gap
 * before its kernel) without the full launch gap that a recorded event adds.
 * Returns FP8BS_ERR_INVALID_ARG for a null dst, FP8BS_ERR_MISALIGNED for an
 * unaligned one.
 */
fp8bs_status fp8bs_stream_timestamp(uint64_t* dst, int release_next, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
