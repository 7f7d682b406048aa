/*
 * nvfp4moe_testing.h -- test and inspection entry points of libnvfp4moe.so.
 *
 * These run the same device functions as the forward (the NVFP4 group
 * quantizer, the SiTU + requant epilogue, the hardware FP4/FP8 conversions,
 * the block-scaled tcgen05 MMA with the forward's operand staging) on
 * caller-given inputs, so that each step can be checked in isolation against
 * an independent implementation.  Same conventions as nvfp4moe.h: device
 * pointers unless marked "host", caller-owned memory, asynchronous on
 * `stream`, host validation errors returned synchronously.
 */
#ifndef NVFP4MOE_TESTING_H_
#define NVFP4MOE_TESTING_H_

#include "nvfp4moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Hardware conversions over n consecutive fp32 bit patterns start..start+n-1:
 *   e2m1_lo[i] = cvt.rn.satfinite.e2m1x2 with the value in the low nibble (4-bit code),
 *   e2m1_hi[i] = the same conversion with the value in the high nibble (4-bit code),
 *   e4m3[i]    = cvt.rn.satfinite.e4m3x2 of the value (byte).
 * Any output may be NULL.  start + n <= 2^32. */
moe_status_t moe_test_codec_sweep(uint32_t start, int64_t n, uint8_t* e2m1_lo, uint8_t* e2m1_hi, uint8_t* e4m3,
                                  cudaStream_t stream);

/* Group-16 NVFP4 quantization of fp32 rows ("Cake SiTU backend": group-16
 * NVFP4 with an encode scale) with the device quantizer of the forward:
 *   x [rows, cols] fp32 (cols % 16 == 0), q_per_row [rows] fp32 encode scales;
 *   packed [rows, cols/2] (even element in the low nibble), sf [rows, cols/16]. */
moe_status_t moe_test_quantize_rows(const float* x, int64_t rows, int32_t cols, const float* q_per_row,
                                    uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* The FC1 epilogue's SiTU + requant on given pre-activations ("Cake SiTU
 * backend": SiTU, intermediate NVFP4 requantization):
 *   z [rows, 2I] fp32 rows of [g | u] (already multiplied by dX*dW13);
 *   a_out [rows, I] fp32 SiTU outputs; packed [rows, I/2]; sf [rows, I/16].
 * I % 32 == 0. */
moe_status_t moe_test_situ_requant(const float* z, int64_t rows, int32_t inter, float qA, float beta, float lam,
                                   float* a_out, uint8_t* packed, uint8_t* sf, cudaStream_t stream);

/* The FC1 epilogue's requant alone (one value per lane, 16-lane groups) on
 * given activations act [rows, I] fp32 with encode scale qA:
 * packed [rows, I/2], sf [rows, I/16].  I % 32 == 0. */
moe_status_t moe_test_requant_lanes(const float* act, int64_t rows, int32_t inter, float qA, uint8_t* packed,
                                    uint8_t* sf, cudaStream_t stream);

/* Throughput of the block-scaled FP4 tensor-core MMA as the GEMMs issue it
 * (tcgen05.mma kind::mxf4nvf4, scale_vec::4X, M = 128, N = n, K = 64, the
 * "Cake SiTU backend" page's NVFP4 x NVFP4 product with 16-element E4M3
 * scales): `grid` CTAs (one per SM; up to the SM count), each with resident
 * operands in shared memory, issue `mmas` MMAs back to back from one thread
 * into `accs` accumulators in turn (1: every MMA depends on the previous
 * one, as the K-steps of one output tile do), plus `copies` scale-atom copies to TMEM (tcgen05.cp 32x128b.warpx4) after
 * every four MMAs, as FC1 issues them per k-block (0 for the bare MMA rate).
 * cycles [grid] (device, int64): SM clock cycles from the first issue to the
 * completion of the last MMA in each CTA, -1 if its bounded wait gave up
 * (status [1], device, then holds MOE_DEVSTAT_TIMEOUT).  FLOPs per CTA are
 * 2 * 128 * n * 64 * mmas; time the call with events on `stream`.
 * 16 <= n <= 256, n % 16 == 0; mmas % 4 == 0, 4 <= mmas <= 1 << 24;
 * 0 <= copies <= 16; accs in {1, 2, 4}, accs * n <= 384. */
moe_status_t moe_test_mma_peak(int32_t grid, int32_t n, int32_t mmas, int32_t copies, int32_t accs, int64_t* cycles,
                               int32_t* status, cudaStream_t stream);

/* One block-scaled FP4 tile product on tcgen05 with the operand staging of
 * FC1 (kind::mxf4nvf4, 16-element E4M3 scales, 128B-swizzled K-major tiles):
 *   a [128, k/2] packed E2M1 (even element in the low nibble), b [n, k/2];
 *   sfa_atoms / sfb_atoms: their block scales in the 128x4 atom layout of
 *   the "Nvfp4 Tensor" page (k/64 atoms of 512 B, rows padded to 128);
 *   d [128, n] fp32 = sum_k a*sfa * b*sfb;  status [1] device status word.
 * 1 <= n <= 128, k % 256 == 0; a, b 256-byte aligned. */
moe_status_t moe_test_mma_fp4(const uint8_t* a, const uint8_t* sfa_atoms, const uint8_t* b, const uint8_t* sfb_atoms,
                              int32_t n, int32_t k, float* d, int32_t* status, cudaStream_t stream);

/* Byte offsets of the internal workspace regions of a workspace of ws_bytes
 * (its carve-up depends only on the shape and its size), for inspection of
 * intermediates in tests (host out struct).  Routing arrays are int32;
 * xq holds the packed X codes once per token ([tokens, H/2]; FC1 gathers them
 * per tile row), aq the packed A codes of the padded expanded rows
 * ([rows, I/2]); sfx/sfa are the block scales of the padded expanded rows
 * (X and A) in the 128x4 atom layout; sft holds X's block scales once per
 * token ([tokens, H/16]) where a forward writes them token-major (above 4096
 * routed pairs, before the atom pass; and at the batch sizes where FC1 runs
 * on the CUDA cores, which read them there and leave sfx unwritten); row_pos maps a
 * flat pair t*k+j to its padded row; acc [tokens, H] fp32 is the FC2
 * combine accumulator (route-weighted sums before the BF16 rounding). */
typedef struct {
  int64_t max_tokens, pairs_max, padded_rows_max, tiles_max;
  int64_t header, count, cumsum, offs, poffs, sorted_row, gather, row_pos, prow_pair, tt_list;
  int64_t xq, sfx, sft, aq, sfa, acc, total;
} moe_ws_layout_t;

moe_status_t moe_workspace_layout(const moe_shape_t* shape, size_t ws_bytes, moe_ws_layout_t* layout);

/* Number of kernel launches one moe_forward enqueues for this shape and T
 * (host out). */
moe_status_t moe_forward_launch_count(const moe_shape_t* shape, int64_t num_tokens, int32_t* launches);

/* Which kernels one moe_forward runs for FC1 and FC2 at this shape and T
 * (host outs): 1 = the decode kernel (weights streamed through a bulk-copy
 * ring, products on warp-level mma.sync; by default FC1 up to 32 tokens,
 * FC2 up to 16), 0 = the tcgen05 block-scaled GEMM.  Follows the same
 * environment overrides as the forward (NVFP4MOE_FC1_GEMV, NVFP4MOE_FC2_GEMV). */
moe_status_t moe_forward_kernels(const moe_shape_t* shape, int64_t num_tokens, int32_t* fc1_decode,
                                 int32_t* fc2_decode);

/* Stage timing (tracing): after moe_profile_start(max_calls), each of the
 * next max_calls moe_forward calls records a CUDA timing event before each of
 * its five stages (routing, X quantization, FC1, FC2 with the combine, BF16
 * finalize) and one after the last, on the call's stream.  moe_profile_stop
 * synchronizes on those events, writes the summed milliseconds per stage to
 * stage_ms[0..4] and the
 * number of recorded calls to *calls (HOST pointers), and frees the events.
 * Events recorded between stages make the stages run back to back (no launch
 * overlap across stage boundaries).  Not thread-safe against concurrent
 * moe_forward calls; not for use inside stream capture. */
moe_status_t moe_profile_start(int32_t max_calls);
moe_status_t moe_profile_stop(float* stage_ms, int32_t* calls);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_TESTING_H_ */
