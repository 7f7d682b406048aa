// static_scratch.cu -- init-routing for callers that cannot allocate device
// memory.
//
// Some callers can't hand this library a workspace: code that runs where
// cudaMalloc is not allowed (inside an allocator or memory-pool callback,
// under a framework that owns every device allocation and exposes none to
// plug-ins, or in a process that must not grow its device footprint after
// start-up).  moe_init_routing_static runs the same routing and token-move
// kernels as moe_init_routing, but keeps its routing scratch in one
// file-scope device array instead of a caller workspace.  The array is
// kStaticScratchBytes (2 MiB) and is held by every GPU that loads the
// library until the process exits.  It covers at most kStaticMaxPairs routed
// pairs (num_rows * k) and kMaxExperts experts; larger calls are refused.
#include <mutex>

#include "nvfp4moe.h"
#include "plan.h"
#include "ptx.cuh"

namespace moe {

cudaError_t launch_routing(const RouteArgs& a, cudaStream_t st, int* launches);
cudaError_t routing_set_attributes(int E);
cudaError_t launch_init_move(const InitMoveArgs& a, cudaStream_t st);
cudaError_t launch_init_finish(const InitFinishArgs& a, cudaStream_t st, int num_sms);

constexpr int64_t kStaticMaxPairs = 65536;
constexpr size_t kStaticScratchBytes = 2u << 20;

// The routing scratch shared by every moe_init_routing_static call on a GPU.
static __device__ __align__(256) uint8_t g_route_scratch[kStaticScratchBytes];

// Carve-up of the static array: the routing regions of a workspace, sized
// for kStaticMaxPairs pairs and kMaxExperts experts.
struct StaticLayout {
  size_t header, count, cumsum, offs, poffs, ttoffs, sorted_row, gather, row_pos, prow_pair, tt_list, blockhist,
      total;
};

static StaticLayout static_layout() {
  StaticLayout L{};
  const size_t P = kStaticMaxPairs, E = kMaxExperts;
  // the same bound as the workspace carve-up: every expert padded to whole tiles
  const size_t ppad = align_up(P + (size_t)(kTileRows - 1) * E, kTileRows);
  const size_t tiles = P / kTileRows + E;
  const size_t nblk = (P + kRouteChunk - 1) / kRouteChunk;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = (o + bytes + 255) / 256 * 256;
    return at;
  };
  L.header = take(HDR_WORDS * 4);
  L.count = take(E * 4);
  L.cumsum = take(E * 4);
  L.offs = take((E + 1) * 4);
  L.poffs = take((E + 1) * 4);
  L.ttoffs = take((E + 1) * 4);
  L.sorted_row = take(P * 4);
  L.gather = take(P * 4);
  L.row_pos = take(P * 4);
  L.prow_pair = take(ppad * 4);
  L.tt_list = take(tiles * 16);
  L.blockhist = take(nblk * E * 4);
  L.total = o;
  return L;
}

// Per-device set-up, done by the first call on each device: the device
// address of the static array (the host-side name is only a stand-in for it)
// and the kernels' shared-memory limits.
struct StaticDevice {
  bool ready = false;
  uint8_t* scratch = nullptr;
  int sms = 0;
};
static std::mutex g_static_mu;
static StaticDevice g_static_dev[64];

static cudaError_t static_setup(uint8_t** scratch, int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticDevice& d = g_static_dev[dev];
  if (!d.ready) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_route_scratch);
    if (err != cudaSuccess) return err;
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = routing_set_attributes(kMaxExperts);
    if (err != cudaSuccess) return err;
    d.scratch = static_cast<uint8_t*>(p);
    d.ready = true;
  }
  *scratch = d.scratch;
  *sms = d.sms;
  return cudaSuccess;
}

static_assert(kStaticMaxPairs % kRouteChunk == 0, "routing blocks tile the static pair capacity");

}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_init_routing_static(const moe_shape_t* shape, int64_t num_rows, const void* x,
                                                const int32_t* expert_ids, const moe_routing_opts_t* opts,
                                                void* expanded_x, int32_t* expanded_row_idx,
                                                int32_t* tokens_cumsum_or_count, float* expanded_scale,
                                                cudaStream_t stream) {
  // the routing kernels' own limits, as moe_init_routing applies them (the
  // intermediate size is not used here)
  const moe_status_t sst = routing_shape_supported(shape);
  if (sst != MOE_OK) return sst;
  if (!x || !expert_ids || !opts || !expanded_x || !expanded_row_idx || !tokens_cumsum_or_count || num_rows < 1)
    return MOE_ERR_INVALID_ARG;
  if (num_rows > kStaticMaxPairs / shape->top_k) return MOE_ERR_WORKSPACE_TOO_SMALL;  // beyond the static scratch
  int32_t base = 0, range = 0;
  const moe_status_t ost = init_routing_check(shape, opts, &base, &range);
  if (ost != MOE_OK) return ost;
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(expanded_x)) % 16 != 0)
    return MOE_ERR_INVALID_ARG;

  const StaticLayout L = static_layout();
  if (L.total > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED;
  uint8_t* w = nullptr;
  int sms = 0;
  if (static_setup(&w, &sms) != cudaSuccess) return MOE_ERR_CUDA;

  // Header words (status, skipped-id count, tile count, ticket of the
  // multi-CTA routing) must start at zero on every call.
  if (cudaMemsetAsync(w + L.header, 0, HDR_WORDS * 4, stream) != cudaSuccess) return MOE_ERR_CUDA;

  const int32_t k = shape->top_k, E = shape->num_experts;
  RouteArgs ra{};
  ra.ids = expert_ids;
  ra.P = num_rows * k;
  ra.k = k;
  ra.E = E;
  ra.hdr = reinterpret_cast<int32_t*>(w + L.header);
  ra.count = reinterpret_cast<int32_t*>(w + L.count);
  ra.cumsum = reinterpret_cast<int32_t*>(w + L.cumsum);
  ra.offs = reinterpret_cast<int32_t*>(w + L.offs);
  ra.poffs = reinterpret_cast<int32_t*>(w + L.poffs);
  ra.ttoffs = reinterpret_cast<int32_t*>(w + L.ttoffs);
  ra.sorted_row = reinterpret_cast<int32_t*>(w + L.sorted_row);
  ra.gather = reinterpret_cast<int32_t*>(w + L.gather);
  ra.row_pos = reinterpret_cast<int32_t*>(w + L.row_pos);
  ra.prow_pair = reinterpret_cast<int32_t*>(w + L.prow_pair);
  ra.tt_list = reinterpret_cast<int32_t*>(w + L.tt_list);
  ra.blockhist = reinterpret_cast<int32_t*>(w + L.blockhist);
  ra.chunk = kRouteChunk;
  ra.check_stamp = 0;   // the header was cleared just above; there is no caller workspace to stamp
  ra.nblk = (int32_t)((ra.P + kRouteChunk - 1) / kRouteChunk);
  if (init_routing_enqueue(ra, base, range, shape, num_rows, x, expert_ids, opts, expanded_x, expanded_row_idx,
                           tokens_cumsum_or_count, expanded_scale, sms, stream) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
