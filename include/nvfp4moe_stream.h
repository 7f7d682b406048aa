/* nvfp4moe_stream.h -- chunk-ready streaming front end of the routed NVFP4
 * MoE forward, for one GPU (one rank).
 *
 * The protocol follows the "[RFC] Chunk-ready symmetric-buffer protocol for
 * streaming MegaMoE inputs" page (DeepGEMM issue), sections "Fixed-capacity
 * ring", "Independent readiness generations", "Memory ordering", "Chunk-aware
 * dispatch scheduling" and "Progress and deadlock requirements":
 *
 *   - A caller-owned ring of num_slots slots, each holding up to
 *     tokens_per_slot tokens of one chunk (a token micro-batch of one MoE
 *     invocation): activations x [C, H] bf16, expert ids [C, k] int32 and
 *     route weights [C, k] bf16, plus the chunk's logical token base and
 *     valid-token count (C = tokens_per_slot).
 *   - Per slot three monotonic 64-bit generations: route_ready (ids and
 *     weights published), layout_ready (x published) and consumed (the slot
 *     may be reused).  The generation of chunk c is (epoch << 32) | (c + 1);
 *     chunk c lives in slot c % num_slots.  The epoch is a device word that
 *     moe_stream_begin increments, so a captured CUDA graph that starts with
 *     moe_stream_begin never confuses one replay's chunks with another's.
 *   - Publishing writes the payload, then stores the generation with release
 *     semantics (GPU scope); the forward of a chunk reads both generations
 *     with acquire semantics before it reads the slot, and stores consumed
 *     with release semantics once the chunk's combine is complete (the
 *     conservative reuse rule of the page).  A publish first waits until the
 *     slot's previous chunk (c - num_slots) has been consumed.
 *   - Scheduling is chunk-local: each chunk is routed and padded into expert
 *     tiles on its own; outputs go to rows token_base .. token_base + n - 1 of
 *     the caller's [out_rows, H] output.
 *   - Progress: no kernel of this library ever waits for work that is not
 *     already ahead of it in stream order.  Producers and consumers on one
 *     stream are ordered by the stream; on two streams the caller orders each
 *     chunk's forward after its publish with an event (cudaEventRecord /
 *     cudaStreamWaitEvent).  The generation checks are bounded waits
 *     (wait_us, default 1 s when 0): one that gives up records a status and
 *     the call degrades to no work (a publish copies nothing and publishes
 *     nothing; a forward writes no output rows and does not mark the slot
 *     consumed).  Serialized execution is always valid.
 *
 * Every pointer is a device pointer owned by the caller unless marked host.
 * Nothing here allocates, synchronizes (except moe_stream_read_status) or
 * reads device values on the host; every call is capturable.  Errors: host
 * validation returns a status synchronously and launches nothing.
 */
#pragma once
#include <stddef.h>
#include <stdint.h>

#include "nvfp4moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Ring geometry: 1 <= num_slots <= 64, 1 <= tokens_per_slot.  max_sms >= 0
 * caps the SMs that a chunk forward's kernels occupy (its persistent GEMM
 * grids and its grid-stride kernels are sized to it), leaving the rest of
 * the GPU to a producer publishing on another stream; 0 (or at least the
 * device's count): all SMs.  It does not change the ring's size. */
typedef struct {
  int32_t num_slots;
  int32_t tokens_per_slot;
  int32_t max_sms;
} moe_stream_ring_t;

/* Parts of a chunk that moe_stream_publish copies and publishes. */
#define MOE_STREAM_ROUTE 1  /* expert ids, route weights, token base and count -> route_ready */
#define MOE_STREAM_LAYOUT 2 /* activations x -> layout_ready */

/* Ring status bits (moe_stream_read_status). */
#define MOE_STREAM_PRODUCER_TIMEOUT 1 /* a publish gave up waiting for its slot to be consumed */

/* Device status bits of a chunk forward, in the workspace status word
 * (moe_read_status), beside the MOE_DEVSTAT_* bits of nvfp4moe.h. */
#define MOE_DEVSTAT_STREAM_WAIT 8     /* the chunk's generations were not published in time */
#define MOE_DEVSTAT_STREAM_BOUNDS 16  /* token_base + n exceeds out_rows: no rows written */

/* Bytes of a ring for this shape and geometry (host out). */
moe_status_t moe_stream_ring_size(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, size_t* bytes);

/* Clears a ring of ring_bytes (>= moe_stream_ring_size; 256-byte aligned):
 * epoch 0, every generation 0, status 0, payload zero.  Once, before first
 * use. */
moe_status_t moe_stream_ring_init(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                  size_t ring_bytes, cudaStream_t stream);

/* Starts one streamed invocation: epoch += 1 on the device and every slot
 * marked consumed for chunk sequence 0 of the new epoch, so chunks 0 ..
 * num_slots - 1 may be published at once.  Chunk indices restart at 0. */
moe_status_t moe_stream_begin(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                              size_t ring_bytes, cudaStream_t stream);

/* Producer: chunk `chunk` (>= 0) of the current invocation, n tokens
 * (0 <= n <= tokens_per_slot) whose first logical token is token_base (>= 0).
 * parts = MOE_STREAM_ROUTE, MOE_STREAM_LAYOUT or both: ROUTE copies
 * expert_ids [n, k] and route_weights [n, k] (rows n .. C-1 of the slot get
 * the id num_experts, which the forward skips, and weight 0) and the base and
 * count; LAYOUT copies x [n, H].  A part's pointers may be NULL when the part
 * is not published.  Waits (bounded) for the slot's previous chunk to be
 * consumed, copies, then publishes the part's generation. */
moe_status_t moe_stream_publish(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                size_t ring_bytes, int64_t chunk, int64_t token_base, int32_t n, int32_t parts,
                                const void* x /* bf16 [n, H] */, const int32_t* expert_ids /* [n, k] */,
                                const void* route_weights /* bf16 [n, k] */, uint32_t wait_us, cudaStream_t stream);

/* Consumer: the forward of chunk `chunk` (moe_forward's weights, scales and
 * SiTU parameters, see nvfp4moe.h) into out [out_rows, H] bf16, rows
 * token_base .. token_base + n - 1 only.  ws must have been prepared with
 * moe_prepare_workspace for tokens_per_slot tokens.  Waits (bounded) for the
 * chunk's route_ready and layout_ready generations, runs the path on the
 * slot's tokens, then marks the slot consumed. */
moe_status_t moe_stream_forward(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                size_t ring_bytes, int64_t chunk, const uint8_t* w13, const uint8_t* sf13,
                                const uint8_t* w2, const uint8_t* sf2, const float* qX, const float* dX_dW13,
                                const float* qA, const float* dA_dW2, const float* situ_beta,
                                const float* situ_linear_beta, void* ws, size_t ws_bytes, void* out,
                                int64_t out_rows, uint32_t wait_us, cudaStream_t stream);

/* Reads and clears the ring status word (MOE_STREAM_* bits) into *host_status
 * (host out).  Synchronizes the stream; test and diagnostics use. */
moe_status_t moe_stream_read_status(const void* ring, int32_t* host_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
