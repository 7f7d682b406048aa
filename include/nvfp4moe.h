/*
 * nvfp4moe.h -- C ABI of the GB300 (sm_103a) routed NVFP4 SiTU MoE forward.
 *
 * The operation ("Cake SiTU backend", FlashInfer tutorial, intro): BF16 x is
 * routed to top-k experts, quantized to group-16 NVFP4, run through FC1 (gate
 * and up), SiTU = (beta*tanh(g/beta)*sigmoid(g)) * (lambda*tanh(u/lambda))
 * (defaults 4 and 25), requantized to NVFP4, run through FC2 and combined with
 * the BF16 route weights into a BF16 output.  Init-routing follows the
 * torch_npu page "npu_moe_init_routing_v2", section 计算公式 (formulas 1-5).
 *
 * Conventions for every entry point:
 *  - Pointers are DEVICE pointers owned by the caller unless marked "host".
 *  - The library allocates no memory, never synchronizes the stream (except
 *    moe_read_status, a test helper), and never reads routing values on the
 *    host ("Cake SiTU backend", section "Caller-owned execution": routing
 *    values never participate in host dispatch; submission makes no CUDA
 *    allocation).  All work is enqueued on `stream` in order, so a complete
 *    call can be captured in a CUDA graph and replayed.
 *  - Host-side validation failures return a status synchronously and launch
 *    nothing.  Device-side anomalies (an expert id outside [0, E), a bounded
 *    wait that gave up) never trap: they are OR-ed into a status word in the
 *    workspace, read by moe_read_status.
 *  - Concurrent calls need separate workspace and output buffers.
 *
 * Tuning overrides, read from the environment (none is needed; the defaults
 * are the measured best):
 *  - NVFP4MOE_PDL=0: launch without programmatic dependent launch (each
 *    kernel then starts only after its predecessor has finished); read once.
 *  Read at every forward unless noted:
 *  - NVFP4MOE_FC1_GEMV=0/1, NVFP4MOE_FC2_GEMV=0/1: FC1 / FC2 on the decode
 *    kernel (warp-level MMAs over the streamed weights) or on the tcgen05
 *    GEMM (default: the decode kernel up to 32 tokens for FC1, 16 for FC2).
 *  - NVFP4MOE_FC1_PAIR=1 or 2: W13 tiles per work unit of FC1's tcgen05
 *    GEMM (default 1 up to 16 tokens, else 2).
 *  - NVFP4MOE_FC1_DYNAMIC=0, NVFP4MOE_FC2_DYNAMIC=0: the GEMMs' CTAs take
 *    their units by a static stride instead of the routing-seeded counters.
 *  - NVFP4MOE_FC2_GROUP=n: output tiles per FC2 work unit (tcgen05: a
 *    divisor of the pass width, else ignored; decode kernel: any n >= 1).
 *  - NVFP4MOE_FC2_TAIL=n: FC2's last units split into parts about 1/n as
 *    wide (default 4; 1 = no split).
 *  - NVFP4MOE_FC2_TILE_STAGES=0: FC2 ring stages of one k-block instead of a
 *    whole output tile.
 *  - NVFP4MOE_ACC_PASS_MB=n: L2 budget in MiB of one FC2 pass over H (the
 *    accumulator slice T x H/passes fp32; default 64).
 */
#ifndef NVFP4MOE_H_
#define NVFP4MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, bad size, bad option, misaligned pointer */
  MOE_ERR_UNSUPPORTED = 2,          /* shape or option outside what the kernels implement */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below moe_workspace_size for this call */
  MOE_ERR_NOT_PREPARED = 4,         /* token count not passed to moe_prepare_workspace on this ws */
  MOE_ERR_CUDA = 5,                 /* a CUDA runtime/driver call failed (launch, tensor map) */
  MOE_ERR_DEVICE_STATUS = 6         /* moe_read_status found a non-zero device status */
} moe_status_t;

/* H (hidden), I (intermediate), E (local experts), k (top-k).
 * Supported: H % 256 == 0, I % 128 == 0, I <= 512, 1 <= E <= 1024, 1 <= k <= min(32, E).
 * The pages' shape is H=3584, I=384, E=896, k=16 ("Cake SiTU backend", intro). */
typedef struct {
  int32_t hidden, inter, num_experts, top_k;
} moe_shape_t;

/* Device status word bits (moe_read_status). */
#define MOE_DEVSTAT_INVALID_EXPERT 1  /* an expert id outside [0, E) was skipped */
#define MOE_DEVSTAT_TIMEOUT 2         /* a bounded wait inside a kernel gave up */
#define MOE_DEVSTAT_BAD_TILE 4        /* a tile descriptor failed a bounds check */
#define MOE_DEVSTAT_NOT_PREPARED 32   /* the workspace held no preparation stamp: the call did nothing
                                         (its output is left zero or untouched) */

/* Workspace bytes for any token count 1..max_tokens ("Cake SiTU backend",
 * "The size query uses host metadata only").  *bytes is a HOST pointer.
 * The workspace holds a header (status word, counts, preparation stamp), the
 * routing arrays, the quantized activations, the quantized intermediate, the
 * fp32 combine accumulator [max_tokens, H] (the route-weighted sum of a
 * token's FC2 outputs before the BF16 rounding) and the default SiTU
 * constants.  Its carve-up depends only on the shape and its byte size, so
 * a maximum-size workspace serves every smaller token count. */
moe_status_t moe_workspace_size(const moe_shape_t* shape, int64_t max_tokens, size_t* bytes);

/* Bytes of each prepared weight buffer.  They equal the canonical sizes
 * ("Cake SiTU backend", "Prepared weights and scales": uint8 [E,2I,H/2] and
 * [E,H,I/2], block scales [E,2I,H/16] and [E,H,I/16]).  Host out pointers. */
moe_status_t moe_prepared_weight_bytes(const moe_shape_t* shape, size_t* w13_bytes, size_t* sf13_bytes,
                                       size_t* w2_bytes, size_t* sf2_bytes);

/* Weight preparation, run once per model ("Cake SiTU backend", "Prepared
 * weights and scales": prepare once, scales carried with the packed bytes).
 * Input is the canonical layout: w13 [E, 2I, H/2] packed E2M1 with the even
 * element in the low nibble, rows 0..I-1 the gate (w1) and I..2I-1 the up
 * projection (w3); sf13 [E, 2I, H/16] E4M3 row-major; w2 [E, H, I/2];
 * sf2 [E, H, I/16].  Output is this library's private layout (same byte
 * counts): codes tiled per MMA tile, gate and up tiles side by side, block
 * scales in the 128x4 atom layout of the "Nvfp4 Tensor" page (block_scale).
 * In and out must not overlap; outputs 256-byte aligned.  Asynchronous. */
moe_status_t moe_prepare_weights(const moe_shape_t* shape, const uint8_t* w13, const uint8_t* sf13,
                                 const uint8_t* w2, const uint8_t* sf2, uint8_t* w13_out, uint8_t* sf13_out,
                                 uint8_t* w2_out, uint8_t* sf2_out, cudaStream_t stream);

/* Per-token-count preparation ("Cake SiTU backend": "Prepare every token
 * count before its first submission"; it initializes the default SiTU
 * constants and allocates nothing).  Writes the default beta = 4 and
 * lambda = 25 arrays, clears the status word and writes a preparation stamp
 * (shape and token capacity) into the header of `ws` (256-byte aligned), and
 * records (ws, ws_bytes, num_tokens) as prepared in a host-side table (one
 * entry per workspace address; a preparation with another size or shape
 * replaces it).  Must be stream-ordered before the first moe_forward /
 * moe_init_routing with this num_tokens.  The first kernel of every call
 * checks the stamp: memory that is no longer the prepared workspace (freed,
 * then handed out again at the same address) makes the call skip its work
 * and set MOE_DEVSTAT_NOT_PREPARED instead of computing from stale state. */
moe_status_t moe_prepare_workspace(const moe_shape_t* shape, void* ws, size_t ws_bytes, int64_t num_tokens,
                                   cudaStream_t stream);

/* The forward ("Cake SiTU backend", whole page):
 *   x [T, H] bf16; expert_ids [T, k] int32 in [0, E); route_weights [T, k] bf16;
 *   w13, sf13, w2, sf2 prepared by moe_prepare_weights (w13, w2 256-byte aligned);
 *   qX [1], dX_dW13 [E], qA [E], dA_dW2 [E] fp32 (the six quant_scales minus
 *   the two block-scale tensors; qX = 1/dX, qA = 1/dA);
 *   situ_beta, situ_linear_beta [E] fp32 or NULL (then 4 and 25);
 *   out [T, H] bf16, written completely.
 * T = num_tokens must be prepared on ws.  Ids outside [0, E) are skipped and
 * flagged in the status word. */
moe_status_t moe_forward(const moe_shape_t* shape, int64_t num_tokens, const void* x, const int32_t* expert_ids,
                         const void* route_weights, const uint8_t* w13, const uint8_t* sf13, const uint8_t* w2,
                         const uint8_t* sf2, const float* qX, const float* dX_dW13, const float* qA,
                         const float* dA_dW2, const float* situ_beta, const float* situ_linear_beta, void* ws,
                         size_t ws_bytes, void* out, cudaStream_t stream);

/* The forward over a contiguous slice of the experts, as one expert-parallel
 * rank runs it ("npu_moe_init_routing_v2": active_expert_range, the
 * EP-local routing of a rank's experts).  shape.num_experts is the slice
 * size; w13/sf13/w2/sf2 and dX_dW13/qA/dA_dW2/situ_* hold the slice's
 * experts, expert_begin .. expert_begin + num_experts - 1 (prepared with that
 * shape).  expert_ids are global: pairs routed outside the slice contribute
 * nothing here and are not errors (negative ids are still skipped and
 * flagged).  out [T, H] bf16 = the rank's partial output, the route-weighted
 * sum over its own experts only (zero for tokens with no pair on the rank);
 * summing the ranks' partial outputs is the caller's collective.  Everything
 * else is as in moe_forward; the workspace is prepared for shape. */
moe_status_t moe_forward_local_experts(const moe_shape_t* shape, int32_t expert_begin, int64_t num_tokens,
                                       const void* x, const int32_t* expert_ids, const void* route_weights,
                                       const uint8_t* w13, const uint8_t* sf13, const uint8_t* w2, const uint8_t* sf2,
                                       const float* qX, const float* dX_dW13, const float* qA, const float* dA_dW2,
                                       const float* situ_beta, const float* situ_linear_beta, void* ws,
                                       size_t ws_bytes, void* out, cudaStream_t stream);

/* Options of moe_init_routing (torch_npu "npu_moe_init_routing_v2",
 * parameter list: drop_pad_mode, expert_capacity, row_idx_type,
 * expert_tokens_num_type, quant_mode, active_expert_range, active_num,
 * scale, offset).  With the fields after quant_mode zero, the op routes every
 * expert, dropless, with no input scale. */
typedef struct {
  int32_t drop_pad;         /* 0 dropless, 1 pad/drop every expert to expert_capacity rows */
  int32_t expert_capacity;  /* C, used when drop_pad == 1 */
  int32_t row_idx_type;     /* 0 gather form (default), 1 scatter form */
  int32_t tokens_num_type;  /* 0 inclusive cumsum (default), 1 count, 2 key_value */
  int32_t quant_mode;       /* -1 no quant (bf16 rows), 0 static int8, 1 dynamic int8 */
  int32_t expert_start;     /* active expert range [expert_start, expert_end); */
  int32_t expert_end;       /*   both 0 = every expert; drop/pad needs every expert */
  int64_t active_num;       /* > 0 (dropless only): move only the first active_num sorted rows */
  const float* scale;       /* device; quant -1: [num_rows] carried to expanded_scale, or NULL;
                               quant 0: [1] (required); quant 1: smooth scale [scale_rows, hidden] or NULL */
  int32_t scale_rows;       /* quant 1 with a smooth scale: 1 (shared) or expert_end - expert_start */
  const float* offset;      /* device; quant 0: [1] (required) */
  int32_t* available_out;   /* device [1] or NULL: availableIdxNum, the pairs whose id is in the range */
} moe_routing_opts_t;

/* Init-routing alone ("npu_moe_init_routing_v2", formulas 1-6):
 *   x [num_rows, hidden] bf16; expert_ids [num_rows, k] int32;
 *   Only pairs whose id lies in the active range are routed (ids outside
 *   [0, E) are also skipped, and flagged in the status word).
 *   expanded_x: dropless [num_rows*k, hidden] (Active: its first
 *     min(active_num, available) rows), drop/pad [E*C, hidden] (int8 when
 *     quant_mode is 0 or 1, else bf16); rows in expert-sorted order; drop/pad
 *     slots beyond an expert's count are zero;
 *     quant 0: rint(x*scale + offset), half to even, saturated to [-128, 127];
 *     quant 1: xs = x (times the smooth row of the pair's expert, or the shared
 *     row), s = row_max|xs|/127, rint(xs / s) clamped to +-127;
 *   expanded_row_idx [num_rows*k] int32: gather form out[sortedRowIdx[i]] = i
 *     for moved rows (drop/pad: e*C + rank), -1 for pairs not moved; or
 *     scatter form out[i] = sortedRowIdx[i] for the available pairs, then -1;
 *   tokens_cumsum_or_count: cumsum or count [expert_end - expert_start] int32
 *     (not clipped by the capacity), or key_value [E, 2]: (expert id, count) of
 *     the in-range experts with a non-zero count in expert order, then zeros;
 *   expanded_scale [rows of expanded_x] fp32: quant 1 the row scale s; quant
 *     -1 with a scale: the token's scale; 0 on unfilled slots; else may be NULL.
 * The sort is stable (ties by flat row index t*k+j).  ws: a workspace of
 * moe_workspace_size(shape) for at least num_rows tokens (shape.inter is
 * used only for that size), prepared for num_rows.  Options out of range
 * return MOE_ERR_INVALID_ARG. */
moe_status_t moe_init_routing(const moe_shape_t* shape, int64_t num_rows, const void* x, const int32_t* expert_ids,
                              const moe_routing_opts_t* opts, void* expanded_x, int32_t* expanded_row_idx,
                              int32_t* tokens_cumsum_or_count, float* expanded_scale, void* ws, size_t ws_bytes,
                              cudaStream_t stream);

/* Init-routing without a workspace, for callers that cannot allocate device
 * memory (code running inside an allocator or memory-pool callback, plug-ins
 * under a framework that owns every device allocation, processes that must
 * not grow their device footprint after start-up).  The pages have no
 * counterpart of this entry point.  Same arguments, outputs and kernels as
 * moe_init_routing, minus ws/ws_bytes: the routing scratch lives in one
 * 2 MiB static device array of the library, held by every GPU that loads it
 * until the process exits.
 *  - Limits: num_rows * top_k <= 65536 routed pairs and num_experts <= 1024;
 *    larger calls return MOE_ERR_WORKSPACE_TOO_SMALL and launch nothing.
 *  - The first call on each device looks up the array's device address and
 *    sets kernel attributes (no allocation); make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array and clears its header on
 *    entry; calls whose work overlaps on the GPU (different streams, other
 *    threads) race on it.  Serialize them.
 *  - The device status word (skipped ids) is kept in the shared array and is
 *    not reported by this entry point. */
moe_status_t moe_init_routing_static(const moe_shape_t* shape, int64_t num_rows, const void* x,
                                     const int32_t* expert_ids, const moe_routing_opts_t* opts, void* expanded_x,
                                     int32_t* expanded_row_idx, int32_t* tokens_cumsum_or_count,
                                     float* expanded_scale, cudaStream_t stream);

/* Test helper: synchronizes `stream`, copies the device status word and the
 * count of skipped expert ids to host_status[0..1] (HOST pointer) and clears
 * them.  Returns MOE_ERR_DEVICE_STATUS if the status word was non-zero. */
moe_status_t moe_read_status(const void* ws, int32_t* host_status, cudaStream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MOE_H_ */
