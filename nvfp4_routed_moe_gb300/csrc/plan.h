// plan.h -- internal: shape constants, workspace carve-up and the kernel
// parameter blocks shared by the host launcher and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>

#include "nvfp4moe.h"

namespace moe {

// Tile geometry (fixed by the kernels).
constexpr int kTileRows = 128;      // weight rows per MMA (M) and token rows per tile
constexpr int kFc1KBlock = 256;     // FP4 elements per FC1 k-block (128 B per row, 128B swizzle)
constexpr int kFc2KBlock = 128;     // FP4 elements per FC2 k-sub-block (64 B per row, 64B swizzle)
constexpr int kTokChunk = 16;       // rows per activation TMA box (and MMA N granule)
constexpr int kRouteSmallMax = 4096;  // pairs handled by the one-CTA routing kernel
constexpr int kRouteChunk = 4096;     // largest number of pairs per CTA of the multi-CTA routing kernels
constexpr int kRouteChunkMin = 512;   // smallest (more CTAs for mid-size batches)
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr size_t kSmemOptin = 232448;  // dynamic shared memory a CTA may opt into on sm_103 (227 KB)
constexpr size_t kAccPassBytes = 64u << 20;  // default L2 budget of one combine pass over H

// Workspace header words (int32).
enum : int {
  HDR_STATUS = 0,      // OR of DEVSTAT_* codes
  HDR_INVALID = 1,     // count of skipped (out-of-range) expert ids
  HDR_NUM_TT = 2,      // number of token tiles this call
  HDR_PPAD = 3,        // padded rows this call
  HDR_DONE = 4,        // last-arriver ticket of the multi-CTA routing
  HDR_NVALID = 5,      // routed pairs this call
  HDR_MAXROWS = 6,     // largest number of pairs routed to one expert this call
  HDR_STREAM_OK = 7,   // streamed chunk: 1 once its generations were seen published
  HDR_STREAM_N = 8,    // streamed chunk: valid tokens
  HDR_SKIP = 9,        // 1: routing found no valid preparation stamp and did nothing; later kernels skip too
  HDR_STREAM_BASE = 10,  // streamed chunk: first logical token (int64, words 10-11)
  HDR_FC2_NEXT = 12,   // FC2's work counter: next unit to take (seeded to 0 by routing on every call)
  HDR_FC1_NEXT = 13,   // FC1's work counter, likewise
  HDR_STAMP = 16,      // preparation stamp, kStampWords words: magic, H, I, E, k, token capacity
  HDR_WORDS = 64,
};

// Written into the header by moe_prepare_workspace and checked by the first
// kernel of every call, so that memory handed back by an allocator at the
// address of a workspace prepared earlier is not mistaken for a prepared one.
constexpr int kStampWords = 6;
constexpr int32_t kStampMagic = 0x4E564634;   // "NVF4"


// One tensor map per activation-row box height (16, 32, 64, 128 rows).
struct RowMaps {
  CUtensorMap m16, m32, m64, m128;
};

struct Shape {
  int32_t H, I, E, k;
};

// Byte offsets of every region of the workspace (all 1024-B aligned).
struct WsLayout {
  int64_t max_tokens, Pmax, PpadMax, TTmax, nblkMax;
  size_t header, count, cumsum, offs, poffs, ttoffs;
  size_t sorted_row, gather, row_pos, prow_pair, tt_list, blockhist;
  size_t xq, sfx, sft, aq, sfa, acc, wrow, beta_def, lam_def;
  size_t total;
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline int64_t tt_bound(int64_t P, int64_t E) {  // max token tiles for P pairs
  return P / kTileRows + (P < E ? P : E);
}

inline WsLayout make_layout(const Shape& s, int64_t max_tokens) {
  WsLayout L{};
  L.max_tokens = max_tokens;
  L.Pmax = max_tokens * s.k;
  const int64_t padded = L.Pmax + (int64_t)(kTileRows - 1) * (L.Pmax < s.E ? L.Pmax : s.E);
  L.PpadMax = (int64_t)align_up((size_t)padded, kTileRows);
  L.TTmax = tt_bound(L.Pmax, s.E);
  L.nblkMax = (L.Pmax + kRouteChunkMin - 1) / kRouteChunkMin;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + (bytes ? bytes : 1), 1024);
    return at;
  };
  L.header = take(HDR_WORDS * 4);
  L.count = take((size_t)s.E * 4);
  L.cumsum = take((size_t)s.E * 4);
  L.offs = take((size_t)(s.E + 1) * 4);
  L.poffs = take((size_t)(s.E + 1) * 4);
  L.ttoffs = take((size_t)(s.E + 1) * 4);
  L.sorted_row = take((size_t)L.Pmax * 4);
  L.gather = take((size_t)L.Pmax * 4);
  L.row_pos = take((size_t)L.Pmax * 4);
  L.prow_pair = take((size_t)L.PpadMax * 4);
  L.tt_list = take((size_t)L.TTmax * 16);
  L.blockhist = take((size_t)L.nblkMax * s.E * 4);
  L.xq = take((size_t)max_tokens * (s.H / 2));
  L.sfx = take((size_t)(L.PpadMax / kTileRows) * (s.H / 64) * 512);
  L.sft = take((size_t)max_tokens * (s.H / 16));
  L.aq = take((size_t)L.PpadMax * (s.I / 2));
  L.sfa = take((size_t)(L.PpadMax / kTileRows) * (s.I / 64) * 512);
  L.acc = take((size_t)max_tokens * s.H * 4);
  L.wrow = take((size_t)L.PpadMax * 4);
  L.beta_def = take((size_t)s.E * 4);
  L.lam_def = take((size_t)s.E * 4);
  L.total = o;
  return L;
}

// Routing outputs (device pointers into the workspace).
struct RouteArgs {
  const int32_t* ids;
  int64_t P;
  int32_t k, E;       // E: experts routed, ids id_base .. id_base + E - 1
  int32_t id_base;    // first routed expert id
  int32_t E_all;      // ids outside [0, E_all) are flagged as invalid; in-range ids outside the routed range are skipped silently
  int32_t* hdr;
  int32_t* count;
  int32_t* cumsum;
  int32_t* offs;
  int32_t* poffs;
  int32_t* ttoffs;
  int32_t* sorted_row;
  int32_t* gather;
  int32_t* row_pos;
  int32_t* prow_pair;
  int32_t* tt_list;   // int4 {expert, row0, rows, 0}
  int32_t* blockhist;
  int32_t nblk;
  int32_t chunk;      // pairs per CTA of the multi-CTA kernels (a multiple of 256)
  int32_t check_stamp;            // 1: compare hdr[HDR_STAMP..] with `stamp` before any work
  int32_t stamp[kStampWords];
};

struct Fc1Args {
  const uint8_t* w13p;      // prepared W13 codes (the decode kernel; the tcgen05 kernel uses a tensor map)
  const uint8_t* sf13p;
  const uint8_t* xq;        // [T, H/2] token-major X codes, gathered per tile row
  const uint8_t* sft;       // [T, H/16] token-major X block scales (decode kernel)
  const int32_t* prow_pair; // [Ppad] flat pair of each padded row (-1: padding)
  const uint8_t* sfx;
  const int32_t* tt_list;
  const int32_t* hdr;
  const float* dXdW13;
  const float* qA;
  const float* beta;
  const float* lam;
  uint8_t* aq;
  uint8_t* sfa;
  int32_t* status;
  int32_t H, I, E, k;
  int32_t max_tiles;      // capacity of the tile list
  int64_t max_rows;       // padded rows of the workspace
  int64_t num_pairs;      // T * k of this call
  int32_t* next;          // work counter (hdr + HDR_FC1_NEXT): CTAs take units from it when `dynamic`
  int32_t dynamic;        // 1: units by the work counter; 0: the static stride blockIdx.x + i * gridDim.x
};

struct Fc2Args {
  const uint8_t* w2p;       // prepared W2 codes (the decode kernel; the tcgen05 kernel uses a tensor map)
  const uint8_t* sf2p;
  const uint8_t* aq;        // [Ppad, I/2] A codes (the decode kernel; the tcgen05 kernel uses tensor maps)
  const uint8_t* sfa;
  const int32_t* tt_list;
  const int32_t* hdr;
  const int32_t* prow_pair;
  const float* wrow;        // [Ppad] route weight of the pair in each padded row
  const float* dAdW2;
  float* acc;               // [T, H] fp32: sum over a token's pairs of route weight x FC2 output
  int32_t* status;
  int32_t H, I, E, k;
  int32_t nq;               // passes over H (H/128 divisible by nq)
  int32_t kbs_per_stage;    // k-blocks per W2 ring stage: I/128 (a whole output tile) or 1 (selects the kernel)
  int32_t group;            // output tiles per work unit (decode kernel; tcgen05 kernel: 0 = its own choice)
  int32_t tail_div;         // tcgen05 kernel: the last units split into parts about 1/tail_div as wide (<= 1: none)
  int32_t* next;            // work counter (hdr + HDR_FC2_NEXT): CTAs take units from it when `dynamic`
  int32_t dynamic;          // 1: units by the work counter; 0: the static stride blockIdx.x + i * gridDim.x
  int32_t max_tiles;
  int64_t max_rows;
  int64_t num_pairs;      // T * k of this call
};

struct InitMoveArgs {
  const int32_t* hdr;         // workspace header (HDR_SKIP)
  const uint16_t* x;          // [T, H] bf16
  const int32_t* ids;         // [T, k]
  const int32_t* gather;      // dropless sorted position per flat pair (ws)
  const int32_t* offs;        // [E] (ws)
  int64_t T;
  int32_t k, E, H, drop_pad, C, quant_mode, row_idx_type;
  const float* scale;         // quant 0: [1]
  const float* offset;        // quant 0: [1]
  void* expanded_x;
  float* expanded_scale;
  int32_t* expanded_row_idx;
};

struct InitFinishArgs {
  const int32_t* count;
  const int32_t* cumsum;
  const int32_t* sorted_row;
  const int32_t* gather;    // sorted position of each pair, -1 if not routed
  const int32_t* ids;
  const int32_t* hdr;
  int64_t P, active_num;
  int32_t E, H, C, drop_pad, row_idx_type, tokens_num_type, esize;
  int32_t E_all, id_base;
  int32_t gather_idx;       // write the gather form of expanded_row_idx here (row-driven move)
  void* expanded_x;
  float* expanded_scale;
  int32_t* expanded_row_idx;
  int32_t* tokens_out;
  int32_t* available_out;   // [1] or null
};

// Row-driven init-routing move: one warp per moved row, every option.
struct InitRowsArgs {
  const uint16_t* x;
  const int32_t* ids;
  const int32_t* sorted_row;
  const int32_t* count;
  const int32_t* cumsum;
  const int32_t* hdr;
  int64_t T, active_num;
  int32_t k, E, id_base, H, drop_pad, C, quant_mode;
  const float* scale;       // quant -1: [T] or null; quant 0: [1]; quant 1: smooth [scale_rows, H] or null
  int32_t scale_rows;
  const float* offset;      // quant 0: [1]
  void* expanded_x;
  float* expanded_scale;
};

struct QuantXArgs {
  const uint16_t* x;        // [T, H] bf16
  const int32_t* row_pos;   // [T*k] padded expanded row of each pair, -1 if not routed
  const uint16_t* route_w;  // [T*k] bf16 route weights
  float* wrow;              // [Ppad] out: route weight of each padded row (fp32), unless the atom pass runs
  float* acc;               // [T, H] out: zeroed
  const float* qX;          // [1]
  uint8_t* xq;              // [T, H/2] token-major codes
  uint8_t* sfx;             // atom layout, H/16 chunks per row: written here when sft is null, by the atom
                            // pass when both are set; null: no atoms (FC1's decode kernel reads sft)
  uint8_t* sft;             // [T, H/16] token-major block scales, or null
  int64_t T;
  int32_t H, k;
  int64_t max_rows;         // padded rows of the workspace
};

// Block scales of X from token-major rows into the atom layout of the padded rows.
struct SfAtomArgs {
  const uint8_t* sft;       // [T, H/16]
  const int32_t* prow_pair; // [Ppad] flat pair of each padded row
  const int32_t* tt_list;   // int4 {expert, row0, rows, 0} per 128-row tile, in row order
  const int32_t* hdr;
  const uint16_t* route_w;  // [T*k] bf16 route weights
  float* wrow;              // [Ppad] out: route weight of each routed padded row (fp32)
  uint32_t* sfx;            // atom layout
  int64_t num_pairs;
  int32_t H, k, max_tiles;
};

struct PrepArgs {
  const uint8_t *w13, *sf13, *w2, *sf2;
  uint8_t *w13o, *sf13o, *w2o, *sf2o;
  int32_t H, I, E;
};

// ---------------------------------------------------------------- streaming
// Ring of a chunk-ready stream: header | slot metadata | x | ids | weights.
struct RingHeader {
  uint64_t epoch;        // incremented by every moe_stream_begin
  int32_t status;        // MOE_STREAM_* bits
  int32_t pad[61];
};
static_assert(sizeof(RingHeader) == 256, "ring header");

struct SlotMeta {
  uint64_t route_gen, layout_gen, consumed_gen;
  int64_t token_base;
  int32_t n;
  int32_t done[2];       // CTAs of the publish in flight that have finished copying (ROUTE[+LAYOUT], LAYOUT)
  int32_t fail[2];       // ... and whether one of them gave up waiting for the slot
  int32_t pad[3];
};
static_assert(sizeof(SlotMeta) == 64, "slot metadata");

struct RingLayout {
  int32_t S;
  int64_t C;
  size_t header, meta, x, ids, w, total;
};

inline RingLayout make_ring_layout(const Shape& s, int32_t S, int64_t C) {
  RingLayout R{};
  R.S = S;
  R.C = C;
  size_t o = 0;
  R.header = o;
  o += sizeof(RingHeader);
  R.meta = o;
  o = align_up(o + (size_t)S * sizeof(SlotMeta), 256);
  R.x = o;
  o = align_up(o + (size_t)S * C * s.H * 2, 256);
  R.ids = o;
  o = align_up(o + (size_t)S * C * s.k * 4, 256);
  R.w = o;
  o = align_up(o + (size_t)S * C * s.k * 2, 256);
  R.total = o;
  return R;
}

struct StreamArgs {
  RingHeader* hdr;
  SlotMeta* meta;
  int32_t S;
  int64_t chunk;         // chunk index of this invocation; slot chunk % S
  uint64_t wait_ns;
};

struct PublishArgs {
  StreamArgs r;
  int64_t token_base, C;
  int32_t n, H, k, E, parts;
  const uint16_t* x;     // [n, H]
  const int32_t* ids;    // [n, k]
  const uint16_t* w;     // [n, k]
  uint16_t* slot_x;      // [C, H]
  int32_t* slot_ids;     // [C, k]
  uint16_t* slot_w;      // [C, k]
};

cudaError_t launch_stream_begin(const StreamArgs& r, cudaStream_t st);
cudaError_t launch_stream_publish(const PublishArgs& a, int num_sms, cudaStream_t st);
cudaError_t launch_stream_gate(const StreamArgs& r, int64_t C, int32_t* ws_hdr, cudaStream_t st);
cudaError_t launch_stream_release(const StreamArgs& r, const int32_t* ws_hdr, cudaStream_t st);
cudaError_t launch_finalize_rows(const float* acc, uint16_t* out, int64_t out_rows, int H, int32_t* ws_hdr,
                                 int64_t C, int num_sms, cudaStream_t st);

// Shape check of the routing kernels alone (H, E, k; I is not used by them),
// shared by moe_init_routing and moe_init_routing_static.
moe_status_t routing_shape_supported(const moe_shape_t* s);

// Init-routing shared by moe_init_routing and moe_init_routing_static: the
// host check of the options (fills the routed expert range) and the
// launches that follow the routing arrays' placement in `ra`.
moe_status_t init_routing_check(const moe_shape_t* shape, const moe_routing_opts_t* o, int32_t* base,
                                int32_t* range);
cudaError_t init_routing_enqueue(RouteArgs ra, int32_t base, int32_t range, const moe_shape_t* shape, int64_t T,
                                 const void* x, const int32_t* ids, const moe_routing_opts_t* o, void* expanded_x,
                                 int32_t* expanded_row_idx, int32_t* tokens_out, float* expanded_scale, int sms,
                                 cudaStream_t st);

}  // namespace moe
