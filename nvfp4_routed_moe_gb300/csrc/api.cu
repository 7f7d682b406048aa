// api.cu -- the C ABI: host validation, workspace planning, tensor maps and
// the launch sequence of the forward and of the standalone init-routing.
#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <unordered_map>
#include <vector>

#include "nvfp4moe.h"
#include "nvfp4moe_stream.h"
#include "nvfp4moe_testing.h"
#include "plan.h"
#include "ptx.cuh"

namespace moe {

// launchers defined next to their kernels
cudaError_t launch_routing(const RouteArgs& a, cudaStream_t st, int* launches);
cudaError_t routing_set_attributes(int E);
cudaError_t launch_init_move(const InitMoveArgs& a, cudaStream_t st);
cudaError_t launch_init_finish(const InitFinishArgs& a, cudaStream_t st, int num_sms);
cudaError_t launch_init_rows(const InitRowsArgs& a, int64_t P, cudaStream_t st, int num_sms);
cudaError_t launch_quant_x(const QuantXArgs& a, cudaStream_t st);
cudaError_t launch_sf_atoms(const SfAtomArgs& a, int64_t max_tiles, int num_sms, cudaStream_t st);
cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t T, int H, int num_sms, cudaStream_t st);
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st, int num_sms);
cudaError_t launch_codec_sweep(uint32_t start, int64_t n, uint8_t* lo, uint8_t* hi, uint8_t* e4, cudaStream_t st,
                               int num_sms);
cudaError_t launch_quant_rows(const float* x, int64_t rows, int cols, const float* qpr, uint8_t* packed, uint8_t* sf,
                              cudaStream_t st, int num_sms);
cudaError_t launch_situ_requant(const float* z, int64_t rows, int I, float qA, float beta, float lam, float* a_out,
                                uint8_t* packed, uint8_t* sf, cudaStream_t st);
cudaError_t launch_requant_lanes(const float* act, int64_t rows, int I, float qA, uint8_t* packed, uint8_t* sf,
                                 cudaStream_t st);
cudaError_t gemm_set_attributes();
cudaError_t launch_fc1(const CUtensorMap& w13, const Fc1Args& a, int pair, int grid,
                       cudaStream_t st);
cudaError_t launch_fc2(const CUtensorMap& w2, const RowMaps& aq, const Fc2Args& a, int grid, cudaStream_t st);
cudaError_t gemv_set_attributes();
size_t fc1_gemv_smem(int H);
cudaError_t launch_fc1_gemv(const CUtensorMap& w13, const Fc1Args& a, int grid, cudaStream_t st);
size_t fc2_gemv_smem(int I);
cudaError_t launch_fc2_gemv(const Fc2Args& a, int grid, cudaStream_t st);
cudaError_t launch_mma_check(const CUtensorMap& a, const CUtensorMap& b, const uint8_t* sfa, const uint8_t* sfb,
                             int N, int K, float* d, int32_t* status, cudaStream_t st);
cudaError_t launch_mma_peak(int grid, int n, int mmas, int copies, int accs, long long* cycles, int32_t* status,
                            cudaStream_t st);

__global__ void fill_f32_kernel(float* p, int n, float v) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) p[i] = v;
}

struct Stamp {
  int32_t w[kStampWords];
};

__global__ void stamp_kernel(int32_t* hdr, const Stamp st) {
  if (threadIdx.x < kStampWords) hdr[HDR_STAMP + threadIdx.x] = st.w[threadIdx.x];
}

// The preparation stamp of a workspace: the shape and the token capacity of
// its carve-up, behind a magic word.
static Stamp make_stamp(const moe_shape_t* s, int64_t cap) {
  return Stamp{{kStampMagic, s->hidden, s->inter, s->num_experts, s->top_k, (int32_t)cap}};
}

// Programmatic dependent launch: a kernel may be scheduled while its
// predecessor drains; every kernel of this library waits (griddepcontrol.wait)
// before it reads memory an earlier kernel of the call writes, or writes
// memory an earlier kernel may still read.  The one exception is by design:
// the X quantization writes its token-major codes and zeroes the accumulator
// before its wait, which is safe because the routing kernel before it starts
// only after the previous forward has completed and touches neither buffer.
// NVFP4MOE_PDL=0 turns the attribute off.
static bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("NVFP4MOE_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

// ------------------------------------------------------------ device state
struct DeviceInfo {
  int sms = 0;
  bool attrs = false;
};
static std::mutex g_mu;
static DeviceInfo g_dev[64];

static cudaError_t device_ready(int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.attrs) {
    err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
    err = routing_set_attributes(kMaxExperts);
    if (err != cudaSuccess) return err;
    err = gemm_set_attributes();
    if (err != cudaSuccess) return err;
    err = gemv_set_attributes();
    if (err != cudaSuccess) return err;
    d.attrs = true;
  }
  *sms = d.sms;
  return cudaSuccess;
}

// ------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static bool make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                     const uint32_t* box, CUtensorMapSwizzle sw) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], s[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) s[i] = strides[i];
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Row-major [rows, row_bytes] byte matrix seen through boxes of inner_bytes x
// {16, 32, 64, 128} rows.
static bool make_row_maps(RowMaps* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t inner_bytes,
                          CUtensorMapSwizzle sw) {
  const uint64_t d[2] = {row_bytes, rows};
  const uint64_t str[1] = {row_bytes};
  CUtensorMap* out[4] = {&m->m16, &m->m32, &m->m64, &m->m128};
  for (int i = 0; i < 4; ++i) {
    const uint32_t box[2] = {inner_bytes, (uint32_t)(kTokChunk << i)};
    if (!make_map(out[i], base, 2, d, str, box, sw)) return false;
  }
  return true;
}

// ------------------------------------------------------------ validation
moe_status_t routing_shape_supported(const moe_shape_t* s) {
  if (!s || s->hidden <= 0 || s->num_experts <= 0 || s->top_k <= 0) return MOE_ERR_INVALID_ARG;
  if (s->hidden % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (s->num_experts > kMaxExperts || s->top_k > kMaxTopK || s->top_k > s->num_experts) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)s->hidden * s->top_k > (int64_t)1 << 30) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

// The routing limits plus the intermediate size the GEMMs (and the workspace
// carve-up) support.
static moe_status_t shape_supported(const moe_shape_t* s) {
  const moe_status_t st = routing_shape_supported(s);
  if (st != MOE_OK) return st;
  if (s->inter <= 0) return MOE_ERR_INVALID_ARG;
  if (s->inter % 128 != 0 || s->inter > 512) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}
static Shape to_shape(const moe_shape_t* s) { return Shape{s->hidden, s->inter, s->num_experts, s->top_k}; }

// Largest token count whose layout fits in `bytes` (the carve-up of a
// workspace is a function of its size, so every call on it agrees).
static int64_t capacity_tokens(const Shape& s, size_t bytes) {
  int64_t lo = 0, hi = 1;
  while (hi < ((int64_t)1 << 31) / s.k && make_layout(s, hi).total <= bytes) {
    lo = hi;
    hi *= 2;
  }
  while (hi - lo > 1) {
    const int64_t mid = (lo + hi) / 2;
    if (make_layout(s, mid).total <= bytes) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Host record of prepared workspaces: one entry per workspace address, with
// the byte size and shape it was prepared for and the token counts prepared
// on it.  A preparation with another size or shape at the same address
// replaces the entry.  The device-side stamp is the second check: it catches
// an address whose memory was freed and handed out again since.
struct PreparedEntry {
  size_t bytes;
  Shape shape;
  std::set<int64_t> T;
};
static std::unordered_map<const void*, PreparedEntry> g_prepared;

static bool same_shape(const Shape& a, const Shape& b) { return a.H == b.H && a.I == b.I && a.E == b.E && a.k == b.k; }

static bool is_prepared(const void* ws, size_t bytes, int64_t T, const Shape& s) {
  std::lock_guard<std::mutex> lock(g_mu);
  const auto it = g_prepared.find(ws);
  return it != g_prepared.end() && it->second.bytes == bytes && same_shape(it->second.shape, s) &&
         it->second.T.count(T) != 0;
}

static void record_prepared(const void* ws, size_t bytes, int64_t T, const Shape& s) {
  std::lock_guard<std::mutex> lock(g_mu);
  PreparedEntry& p = g_prepared[ws];
  if (p.bytes != bytes || !same_shape(p.shape, s)) {
    p.bytes = bytes;
    p.shape = s;
    p.T.clear();
  }
  p.T.insert(T);
}

static bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define MOE_CUDA(x)                              \
  do {                                           \
    if ((x) != cudaSuccess) return MOE_ERR_CUDA; \
  } while (0)

static RouteArgs route_args(const moe_shape_t* shape, const WsLayout& L, uint8_t* ws, const int32_t* ids,
                            int64_t T) {
  const Shape s = to_shape(shape);
  RouteArgs a{};
  const Stamp st = make_stamp(shape, L.max_tokens);
  a.check_stamp = 1;
  for (int i = 0; i < kStampWords; ++i) a.stamp[i] = st.w[i];
  a.ids = ids;
  a.P = T * s.k;
  a.k = s.k;
  a.E = s.E;
  a.id_base = 0;
  a.E_all = s.E;
  a.hdr = reinterpret_cast<int32_t*>(ws + L.header);
  a.count = reinterpret_cast<int32_t*>(ws + L.count);
  a.cumsum = reinterpret_cast<int32_t*>(ws + L.cumsum);
  a.offs = reinterpret_cast<int32_t*>(ws + L.offs);
  a.poffs = reinterpret_cast<int32_t*>(ws + L.poffs);
  a.ttoffs = reinterpret_cast<int32_t*>(ws + L.ttoffs);
  a.sorted_row = reinterpret_cast<int32_t*>(ws + L.sorted_row);
  a.gather = reinterpret_cast<int32_t*>(ws + L.gather);
  a.row_pos = reinterpret_cast<int32_t*>(ws + L.row_pos);
  a.prow_pair = reinterpret_cast<int32_t*>(ws + L.prow_pair);
  a.tt_list = reinterpret_cast<int32_t*>(ws + L.tt_list);
  a.blockhist = reinterpret_cast<int32_t*>(ws + L.blockhist);
  // about 32 routing CTAs (the last one's prefix over the per-CTA histograms
  // grows with their number): chunk = ceil(P / 32) rounded up to 256, within [512, 4096]
  int64_t chunk = ((a.P + 31) / 32 + 255) / 256 * 256;
  a.chunk = (int32_t)(chunk < kRouteChunkMin ? kRouteChunkMin : chunk > kRouteChunk ? kRouteChunk : chunk);
  a.nblk = (int32_t)((a.P + a.chunk - 1) / a.chunk);
  return a;
}

// Above this many routed pairs the X block scales are written token-major
// and laid out in atoms by a second kernel (scattered 4-byte atom writes from
// the quantizer cost more from here on; the same bound as routing's one-CTA
// path).
constexpr int64_t kSfTwoPassMin = 4096;
// Largest batch for which FC1 works on one W13 tile per unit.
constexpr int64_t kFc1SingleMaxTokens = 16;

// W13 tiles per FC1 work unit: two (shared X loads and scale copies) unless
// the batch is so small that single tiles are needed to keep the SMs busy
// (NVFP4MOE_FC1_PAIR=1/2 overrides).
static int fc1_pair(const Shape&, int64_t T) {
  if (const char* v = std::getenv("NVFP4MOE_FC1_PAIR")) {
    if (v[0] == '1') return 1;
    if (v[0] == '2') return 2;
  }
  return T <= kFc1SingleMaxTokens ? 1 : 2;
}

// Largest batch for which FC1 runs on the decode kernel (weights streamed at
// HBM rate, a few tokens per expert tile): the whole forward is faster with it
// up to about 36 tokens (T = 24: 0.159 against 0.171 ms, T = 32: 0.192
// against 0.198), the tcgen05 GEMM from 40; NVFP4MOE_FC1_GEMV=0/1 overrides.
constexpr int64_t kFc1GemvMaxTokens = 32;

static bool fc1_gemv(const Shape& s, int64_t T) {
  if (fc1_gemv_smem(s.H) > kSmemOptin) return false;   // the X slots for this H do not fit
  if (const char* v = std::getenv("NVFP4MOE_FC1_GEMV")) {
    if (v[0] == '0') return false;
    if (v[0] == '1') return true;
  }
  return T <= kFc1GemvMaxTokens;
}

// Largest batch for which FC2 runs the same way; NVFP4MOE_FC2_GEMV=0/1 overrides.
constexpr int64_t kFc2GemvMaxTokens = 16;

static bool fc2_gemv(const Shape& s, int64_t T) {
  if (fc2_gemv_smem(s.I) > kSmemOptin) return false;
  if (const char* v = std::getenv("NVFP4MOE_FC2_GEMV")) {
    if (v[0] == '0') return false;
    if (v[0] == '1') return true;
  }
  return T <= kFc2GemvMaxTokens;
}

// Output tiles per unit of the decode FC2: long units stream best (each
// job's A rows take a few microseconds to arrive, and units are claimed one
// at a time), so about 0.8 units per SM for the batch's tile bound, at most
// half of H/128 (measured at T = 1, 2, 4, 8, 16: 4, 7, 14, 14-28, 14 tiles).
// NVFP4MOE_FC2_GROUP overrides.
static int fc2_gemv_group(const Shape& s, int64_t tiles, int sms) {
  if (const char* v = std::getenv("NVFP4MOE_FC2_GROUP")) {
    const int g = std::atoi(v);
    if (g >= 1) return g;
  }
  const int64_t nmt = s.H / 128, g = (tiles * nmt * 5 + 4 * (int64_t)sms - 1) / (4 * (int64_t)sms);
  return (int)std::max<int64_t>(1, std::min<int64_t>(std::max<int64_t>(1, nmt / 2), g));
}

// The tcgen05 FC2's output tiles per unit: its own choice from the tile
// count (0) unless NVFP4MOE_FC2_GROUP names a divisor of its pass width.
static int fc2_tc_group() {
  const char* v = std::getenv("NVFP4MOE_FC2_GROUP");
  return v ? std::max(0, std::atoi(v)) : 0;
}

// The tcgen05 FC2's last units (one tile per CTA) are split into parts about
// 1/kFc2TailDiv as wide, so that its CTAs finish together
// (NVFP4MOE_FC2_TAIL overrides; 1 = no split).
constexpr int kFc2TailDiv = 4;
static int fc2_tail_div() {
  const char* v = std::getenv("NVFP4MOE_FC2_TAIL");
  return v ? std::max(1, std::atoi(v)) : kFc2TailDiv;
}

// Above kSfTwoPassMin pairs the X scales take the token-major + atom pass
// route, unless FC1 runs on the decode kernel (which reads them token-major).
static bool sf_atom_pass(const Shape& s, int64_t T) { return T * s.k > kSfTwoPassMin && !fc1_gemv(s, T); }

static int forward_launches(const Shape& s, int64_t T) {
  return (T * s.k <= kRouteSmallMax ? 1 : 2) + 4 + (sf_atom_pass(s, T) ? 1 : 0);
}

// The GEMMs' CTAs take their units from work counters that routing seeds on
// every call (NVFP4MOE_FC1_DYNAMIC=0 / NVFP4MOE_FC2_DYNAMIC=0: the static
// stride instead).
static int gemm_dynamic(const char* env) {
  const char* v = std::getenv(env);
  return (v && v[0] == '0') ? 0 : 1;
}

// FC2's ring stages hold a whole output tile (all I/128 k-blocks): one wait,
// fence and commit of the issuing thread per output tile instead of one per
// k-block, faster at every batch size measured (T = 1 .. 16384).  Stages of
// one k-block remain selectable (NVFP4MOE_FC2_TILE_STAGES=0).
static bool fc2_tile_stages(int64_t) {
  const char* v = std::getenv("NVFP4MOE_FC2_TILE_STAGES");
  return !(v && v[0] == '0');
}

// Passes of the FC2 combine over H: the fewest (a divisor of H/128) whose
// accumulator slice, T x H/nq fp32, fits the L2 budget (NVFP4MOE_ACC_PASS_MB
// overrides the default budget).
static int combine_passes(const Shape& s, int64_t T) {
  size_t budget = kAccPassBytes;
  if (const char* v = std::getenv("NVFP4MOE_ACC_PASS_MB")) {
    const long mb = std::strtol(v, nullptr, 10);
    if (mb > 0) budget = (size_t)mb << 20;
  }
  const int NMT = s.H / 128;
  for (int d = 1; d < NMT; ++d)
    if (NMT % d == 0 && (size_t)T * (size_t)s.H * 4u / (size_t)d <= budget) return d;
  return NMT;
}

// ------------------------------------------------------------ stage timing
// While a profile is open, every moe_forward records a timing event before
// each stage and one after the last, from a pool created by moe_profile_start.
constexpr int kStages = 5;  // routing, quant X, FC1, FC2 with the combine, BF16 finalize
struct Profile {
  bool on = false;
  int max_calls = 0, calls = 0;
  std::vector<cudaEvent_t> ev;  // (kStages + 1) per call
};
static Profile g_prof;

static void prof_mark(int stage, cudaStream_t st) {
  if (!g_prof.on || g_prof.calls >= g_prof.max_calls) return;
  cudaEventRecord(g_prof.ev[(size_t)g_prof.calls * (kStages + 1) + stage], st);
}
static void prof_end_call(cudaStream_t st) {
  if (!g_prof.on || g_prof.calls >= g_prof.max_calls) return;
  prof_mark(kStages, st);
  ++g_prof.calls;
}

moe_status_t init_routing_check(const moe_shape_t* shape, const moe_routing_opts_t* o, int32_t* base,
                                int32_t* range) {
  if (o->drop_pad != 0 && o->drop_pad != 1) return MOE_ERR_INVALID_ARG;
  if (o->drop_pad && o->expert_capacity < 1) return MOE_ERR_INVALID_ARG;
  if (o->row_idx_type != 0 && o->row_idx_type != 1) return MOE_ERR_INVALID_ARG;
  if (o->tokens_num_type < 0 || o->tokens_num_type > 2) return MOE_ERR_INVALID_ARG;
  if (o->quant_mode < -1 || o->quant_mode > 1) return MOE_ERR_INVALID_ARG;
  int32_t lo = o->expert_start, hi = o->expert_end;
  if (lo == 0 && hi == 0) hi = shape->num_experts;
  if (lo < 0 || hi <= lo || hi > shape->num_experts) return MOE_ERR_INVALID_ARG;
  if (o->drop_pad && (lo != 0 || hi != shape->num_experts || o->active_num > 0)) return MOE_ERR_INVALID_ARG;
  if (o->quant_mode == 0 && (!o->scale || !o->offset)) return MOE_ERR_INVALID_ARG;
  if (o->quant_mode == 1 && o->scale && o->scale_rows != 1 && o->scale_rows != hi - lo) return MOE_ERR_INVALID_ARG;
  *base = lo;
  *range = hi - lo;
  return MOE_OK;
}

cudaError_t init_routing_enqueue(RouteArgs ra, int32_t base, int32_t range, const moe_shape_t* shape, int64_t T,
                                 const void* x, const int32_t* ids, const moe_routing_opts_t* o, void* expanded_x,
                                 int32_t* expanded_row_idx, int32_t* tokens_out, float* expanded_scale, int sms,
                                 cudaStream_t st) {
  ra.id_base = base;
  ra.E = range;
  ra.E_all = shape->num_experts;
  int nl = 0;
  cudaError_t err = launch_routing(ra, st, &nl);
  if (err != cudaSuccess) return err;
  // Token-driven move (each token quantized once, written to its routed
  // pairs' rows; pairs outside the expert range have no row) when there is
  // no Active limit and the row does not depend on the expert (static int8's
  // scalar scale and offset, or no input scale); row-driven (scatter form)
  // for the others.  Drop/pad always spans every expert.
  const bool plain = o->active_num <= 0 && (o->quant_mode == 0 || !o->scale);
  float* sc_out = (o->quant_mode == 1 || (o->quant_mode == -1 && o->scale)) ? expanded_scale : nullptr;
  if (plain) {
    InitMoveArgs ma{};
    ma.hdr = ra.hdr;
    ma.x = static_cast<const uint16_t*>(x);
    ma.ids = ids;
    ma.gather = ra.gather;
    ma.offs = ra.offs;
    ma.T = T;
    ma.k = shape->top_k;
    ma.E = range;
    ma.H = shape->hidden;
    ma.drop_pad = o->drop_pad;
    ma.C = o->expert_capacity;
    ma.quant_mode = o->quant_mode;
    ma.row_idx_type = o->row_idx_type;
    ma.scale = o->scale;
    ma.offset = o->offset;
    ma.expanded_x = expanded_x;
    ma.expanded_scale = sc_out;
    ma.expanded_row_idx = expanded_row_idx;
    err = launch_init_move(ma, st);
  } else {
    InitRowsArgs wa{};
    wa.x = static_cast<const uint16_t*>(x);
    wa.ids = ids;
    wa.sorted_row = ra.sorted_row;
    wa.count = ra.count;
    wa.cumsum = ra.cumsum;
    wa.hdr = ra.hdr;
    wa.T = T;
    wa.active_num = o->active_num;
    wa.k = shape->top_k;
    wa.E = range;
    wa.id_base = base;
    wa.H = shape->hidden;
    wa.drop_pad = o->drop_pad;
    wa.C = o->expert_capacity;
    wa.quant_mode = o->quant_mode;
    wa.scale = o->scale;
    wa.scale_rows = o->scale_rows;
    wa.offset = o->offset;
    wa.expanded_x = expanded_x;
    wa.expanded_scale = sc_out;
    err = launch_init_rows(wa, ra.P, st, sms);
  }
  if (err != cudaSuccess) return err;
  InitFinishArgs fa{};
  fa.count = ra.count;
  fa.cumsum = ra.cumsum;
  fa.sorted_row = ra.sorted_row;
  fa.gather = ra.gather;
  fa.ids = ids;
  fa.hdr = ra.hdr;
  fa.P = ra.P;
  fa.active_num = o->active_num;
  fa.E = range;
  fa.H = shape->hidden;
  fa.C = o->expert_capacity;
  fa.drop_pad = o->drop_pad;
  fa.row_idx_type = o->row_idx_type;
  fa.tokens_num_type = o->tokens_num_type;
  fa.esize = o->quant_mode == -1 ? 2 : 1;
  fa.E_all = shape->num_experts;
  fa.id_base = base;
  fa.gather_idx = plain ? 0 : 1;
  fa.expanded_x = expanded_x;
  fa.expanded_scale = sc_out;
  fa.expanded_row_idx = expanded_row_idx;
  fa.tokens_out = tokens_out;
  fa.available_out = o->available_out;
  return launch_init_finish(fa, st, sms);
}

static moe_status_t forward_impl(const moe_shape_t* shape, int32_t expert_begin, int32_t id_limit,
                                 int64_t num_tokens, const void* x, const int32_t* expert_ids,
                                 const void* route_weights, const uint8_t* w13, const uint8_t* sf13,
                                 const uint8_t* w2, const uint8_t* sf2, const float* qX, const float* dX_dW13,
                                 const float* qA, const float* dA_dW2, const float* situ_beta,
                                 const float* situ_linear_beta, void* ws, size_t ws_bytes, void* out,
                                 cudaStream_t stream, int64_t stream_out_rows = -1, int max_sms = 0) {
  // stream_out_rows >= 0: a streamed chunk; the finalize writes the chunk's
  // rows (count and base from the workspace header) into out [stream_out_rows, H].
  // max_sms > 0: the kernels' grids are sized to at most that many SMs.
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!x || !expert_ids || !route_weights || !w13 || !sf13 || !w2 || !sf2 || !qX || !dX_dW13 || !qA || !dA_dW2 ||
      !ws || !out || num_tokens < 1)
    return MOE_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(out, 16) || !aligned(ws, 256) || !aligned(w13, 256) || !aligned(w2, 256) ||
      !aligned(sf13, 16) || !aligned(sf2, 16))
    return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  const int64_t cap = capacity_tokens(s, ws_bytes);
  if (cap < num_tokens) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!is_prepared(ws, ws_bytes, num_tokens, s)) return MOE_ERR_NOT_PREPARED;
  const WsLayout L = make_layout(s, cap);
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  if (max_sms > 0 && max_sms < sms) sms = max_sms;
  uint8_t* w = static_cast<uint8_t*>(ws);
  const int64_t T = num_tokens, P = T * s.k;
  const int NIT = s.I / 64, NKB = s.H / kFc1KBlock, NMT = s.H / 128, NKB2 = s.I / kFc2KBlock;

  CUtensorMap tm_w13, tm_w2;
  RowMaps tm_aq;
  {
    const uint64_t d[3] = {128, 128, (uint64_t)s.E * NIT * NKB};
    const uint64_t str[2] = {128, 16384};
    const uint32_t box[3] = {128, 128, 1};
    if (!make_map(&tm_w13, w13, 3, d, str, box, CU_TENSOR_MAP_SWIZZLE_128B)) return MOE_ERR_CUDA;
  }
  {
    const uint64_t d[3] = {64, 128, (uint64_t)s.E * NMT * NKB2};
    const uint64_t str[2] = {64, 8192};
    const uint32_t box[3] = {64, 128, 1};
    if (!make_map(&tm_w2, w2, 3, d, str, box, CU_TENSOR_MAP_SWIZZLE_64B)) return MOE_ERR_CUDA;
  }
  if (!make_row_maps(&tm_aq, w + L.aq, (uint64_t)s.I / 2, (uint64_t)L.PpadMax, 64, CU_TENSOR_MAP_SWIZZLE_64B))
    return MOE_ERR_CUDA;

  // 1. routing
  prof_mark(0, stream);
  RouteArgs ra = route_args(shape, L, w, expert_ids, T);
  ra.id_base = expert_begin;
  ra.E_all = id_limit;
  int nl = 0;
  MOE_CUDA(launch_routing(ra, stream, &nl));

  // 2. quantize X (token-major codes; block scales into the padded rows' atoms)
  QuantXArgs qa{};
  qa.x = static_cast<const uint16_t*>(x);
  qa.row_pos = ra.row_pos;
  qa.route_w = static_cast<const uint16_t*>(route_weights);
  qa.wrow = reinterpret_cast<float*>(w + L.wrow);
  const int nq = combine_passes(s, T);
  qa.acc = reinterpret_cast<float*>(w + L.acc);
  qa.qX = qX;
  qa.xq = w + L.xq;
  const bool gemv = fc1_gemv(s, T);
  qa.sfx = gemv ? nullptr : w + L.sfx;
  qa.sft = (gemv || sf_atom_pass(s, T)) ? w + L.sft : nullptr;
  qa.T = T;
  qa.H = s.H;
  qa.k = s.k;
  qa.max_rows = L.PpadMax;
  prof_mark(1, stream);
  MOE_CUDA(launch_quant_x(qa, stream));
  if (qa.sft && qa.sfx) {
    SfAtomArgs sa{};
    sa.sft = qa.sft;
    sa.prow_pair = ra.prow_pair;
    sa.tt_list = ra.tt_list;
    sa.hdr = ra.hdr;
    sa.route_w = qa.route_w;
    sa.wrow = qa.wrow;
    sa.sfx = reinterpret_cast<uint32_t*>(w + L.sfx);
    sa.num_pairs = P;
    sa.H = s.H;
    sa.k = s.k;
    sa.max_tiles = (int32_t)std::min<int64_t>(L.TTmax, L.PpadMax / kTileRows);   // atoms exist for the padded rows
    MOE_CUDA(launch_sf_atoms(sa, tt_bound(P, s.E), sms, stream));
  }

  // 3. FC1 + SiTU + requant
  const int64_t tt = tt_bound(P, s.E);
  Fc1Args f1{};
  f1.w13p = static_cast<const uint8_t*>(w13);
  f1.sf13p = sf13;
  f1.xq = w + L.xq;
  f1.sft = w + L.sft;
  f1.prow_pair = ra.prow_pair;
  f1.k = s.k;
  f1.num_pairs = P;
  f1.sfx = w + L.sfx;
  f1.tt_list = ra.tt_list;
  f1.hdr = ra.hdr;
  f1.dXdW13 = dX_dW13;
  f1.qA = qA;
  f1.beta = situ_beta ? situ_beta : reinterpret_cast<const float*>(w + L.beta_def);
  f1.lam = situ_linear_beta ? situ_linear_beta : reinterpret_cast<const float*>(w + L.lam_def);
  f1.aq = w + L.aq;
  f1.sfa = w + L.sfa;
  f1.status = ra.hdr + HDR_STATUS;
  f1.H = s.H;
  f1.I = s.I;
  f1.E = s.E;
  f1.max_tiles = (int32_t)L.TTmax;
  f1.max_rows = L.PpadMax;
  f1.next = ra.hdr + HDR_FC1_NEXT;
  f1.dynamic = gemm_dynamic("NVFP4MOE_FC1_DYNAMIC");
  prof_mark(2, stream);
  if (gemv) {
    MOE_CUDA(launch_fc1_gemv(tm_w13, f1, (int)std::min<int64_t>(sms, tt * (s.I / 64)), stream));
  } else {
    const int pair = fc1_pair(s, T);
    const int grid1 = (int)std::min<int64_t>(sms, tt * (s.I / 64 / pair));
    MOE_CUDA(launch_fc1(tm_w13, f1, pair, grid1, stream));
  }

  // 4. FC2 with the route-weighted combine into the fp32 accumulator
  Fc2Args f2{};
  f2.w2p = w2;
  f2.sf2p = sf2;
  f2.aq = w + L.aq;
  f2.sfa = w + L.sfa;
  f2.tt_list = ra.tt_list;
  f2.hdr = ra.hdr;
  f2.prow_pair = ra.prow_pair;
  f2.wrow = reinterpret_cast<const float*>(w + L.wrow);
  f2.dAdW2 = dA_dW2;
  f2.acc = reinterpret_cast<float*>(w + L.acc);
  f2.nq = nq;
  f2.kbs_per_stage = fc2_tile_stages(T) ? NKB2 : 1;
  f2.next = ra.hdr + HDR_FC2_NEXT;
  f2.dynamic = gemm_dynamic("NVFP4MOE_FC2_DYNAMIC");
  f2.status = ra.hdr + HDR_STATUS;
  f2.H = s.H;
  f2.I = s.I;
  f2.E = s.E;
  f2.k = s.k;
  f2.max_tiles = (int32_t)L.TTmax;
  f2.max_rows = L.PpadMax;
  f2.num_pairs = P;
  prof_mark(3, stream);
  if (fc2_gemv(s, T)) {
    f2.group = fc2_gemv_group(s, tt, sms);
    const int64_t units = tt * ((NMT + f2.group - 1) / f2.group);
    MOE_CUDA(launch_fc2_gemv(f2, (int)std::min<int64_t>(sms, units), stream));
  } else {
    f2.group = fc2_tc_group();
    f2.tail_div = fc2_tail_div();
    MOE_CUDA(launch_fc2(tm_w2, tm_aq, f2, (int)std::min<int64_t>(sms, tt * NMT), stream));
  }

  // 5. BF16 finalize
  prof_mark(4, stream);
  if (stream_out_rows >= 0)
    MOE_CUDA(launch_finalize_rows(reinterpret_cast<const float*>(w + L.acc), static_cast<uint16_t*>(out),
                                  stream_out_rows, s.H, ra.hdr, T, sms, stream));
  else
    MOE_CUDA(launch_finalize(reinterpret_cast<const float*>(w + L.acc), static_cast<uint16_t*>(out), T, s.H, sms,
                             stream));

  prof_end_call(stream);
  return MOE_OK;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char* moe_status_string(moe_status_t st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "MOE_ERR_WORKSPACE_TOO_SMALL";
    case MOE_ERR_NOT_PREPARED: return "MOE_ERR_NOT_PREPARED";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE_STATUS: return "MOE_ERR_DEVICE_STATUS";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status_t moe_workspace_size(const moe_shape_t* shape, int64_t max_tokens, size_t* bytes) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!bytes || max_tokens < 1) return MOE_ERR_INVALID_ARG;
  if (max_tokens * shape->top_k >= ((int64_t)1 << 31) - (int64_t)kTileRows * kMaxExperts)
    return MOE_ERR_UNSUPPORTED;
  *bytes = make_layout(to_shape(shape), max_tokens).total;
  return MOE_OK;
}

moe_status_t moe_prepared_weight_bytes(const moe_shape_t* shape, size_t* w13_bytes, size_t* sf13_bytes,
                                       size_t* w2_bytes, size_t* sf2_bytes) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!w13_bytes || !sf13_bytes || !w2_bytes || !sf2_bytes) return MOE_ERR_INVALID_ARG;
  const size_t E = shape->num_experts, H = shape->hidden, I = shape->inter;
  *w13_bytes = E * 2 * I * (H / 2);
  *sf13_bytes = E * 2 * I * (H / 16);
  *w2_bytes = E * H * (I / 2);
  *sf2_bytes = E * H * (I / 16);
  return MOE_OK;
}

moe_status_t moe_prepare_weights(const moe_shape_t* shape, const uint8_t* w13, const uint8_t* sf13,
                                 const uint8_t* w2, const uint8_t* sf2, uint8_t* w13_out, uint8_t* sf13_out,
                                 uint8_t* w2_out, uint8_t* sf2_out, cudaStream_t stream) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!w13 || !sf13 || !w2 || !sf2 || !w13_out || !sf13_out || !w2_out || !sf2_out) return MOE_ERR_INVALID_ARG;
  if (!aligned(w13, 16) || !aligned(w2, 16) || !aligned(w13_out, 256) || !aligned(w2_out, 256) ||
      !aligned(sf13_out, 16) || !aligned(sf2_out, 16))
    return MOE_ERR_INVALID_ARG;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  PrepArgs a{w13, sf13, w2, sf2, w13_out, sf13_out, w2_out, sf2_out, shape->hidden, shape->inter,
             shape->num_experts};
  MOE_CUDA(launch_prep(a, stream, sms));
  return MOE_OK;
}

moe_status_t moe_prepare_workspace(const moe_shape_t* shape, void* ws, size_t ws_bytes, int64_t num_tokens,
                                   cudaStream_t stream) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!ws || num_tokens < 1 || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  const int64_t cap = capacity_tokens(s, ws_bytes);
  if (cap < num_tokens) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout L = make_layout(s, cap);
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  uint8_t* w = static_cast<uint8_t*>(ws);
  MOE_CUDA(cudaMemsetAsync(w + L.header, 0, HDR_WORDS * 4, stream));
  fill_f32_kernel<<<4, 256, 0, stream>>>(reinterpret_cast<float*>(w + L.beta_def), s.E, 4.0f);
  fill_f32_kernel<<<4, 256, 0, stream>>>(reinterpret_cast<float*>(w + L.lam_def), s.E, 25.0f);
  stamp_kernel<<<1, 32, 0, stream>>>(reinterpret_cast<int32_t*>(w + L.header), make_stamp(shape, cap));
  MOE_CUDA(cudaGetLastError());
  record_prepared(ws, ws_bytes, num_tokens, s);
  return MOE_OK;
}

moe_status_t moe_forward(const moe_shape_t* shape, int64_t num_tokens, const void* x, const int32_t* expert_ids,
                         const void* route_weights, const uint8_t* w13, const uint8_t* sf13, const uint8_t* w2,
                         const uint8_t* sf2, const float* qX, const float* dX_dW13, const float* qA,
                         const float* dA_dW2, const float* situ_beta, const float* situ_linear_beta, void* ws,
                         size_t ws_bytes, void* out, cudaStream_t stream) {
  if (!shape) return MOE_ERR_INVALID_ARG;
  return forward_impl(shape, 0, shape->num_experts, num_tokens, x, expert_ids, route_weights, w13, sf13, w2, sf2, qX,
                      dX_dW13, qA, dA_dW2, situ_beta, situ_linear_beta, ws, ws_bytes, out, stream);
}

moe_status_t moe_forward_local_experts(const moe_shape_t* shape, int32_t expert_begin, int64_t num_tokens,
                                       const void* x, const int32_t* expert_ids, const void* route_weights,
                                       const uint8_t* w13, const uint8_t* sf13, const uint8_t* w2, const uint8_t* sf2,
                                       const float* qX, const float* dX_dW13, const float* qA, const float* dA_dW2,
                                       const float* situ_beta, const float* situ_linear_beta, void* ws,
                                       size_t ws_bytes, void* out, cudaStream_t stream) {
  if (!shape || expert_begin < 0 || (int64_t)expert_begin + shape->num_experts > (int64_t)INT32_MAX)
    return MOE_ERR_INVALID_ARG;
  // negative ids are flagged; ids past the slice belong to other ranks
  return forward_impl(shape, expert_begin, INT32_MAX, num_tokens, x, expert_ids, route_weights, w13, sf13, w2, sf2,
                      qX, dX_dW13, qA, dA_dW2, situ_beta, situ_linear_beta, ws, ws_bytes, out, stream);
}

moe_status_t moe_init_routing(const moe_shape_t* shape, int64_t num_rows, const void* x, const int32_t* expert_ids,
                              const moe_routing_opts_t* opts, void* expanded_x, int32_t* expanded_row_idx,
                              int32_t* tokens_cumsum_or_count, float* expanded_scale, void* ws, size_t ws_bytes,
                              cudaStream_t stream) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!x || !expert_ids || !opts || !expanded_x || !expanded_row_idx || !tokens_cumsum_or_count || !ws ||
      num_rows < 1)
    return MOE_ERR_INVALID_ARG;
  int32_t base = 0, range = 0;
  st = init_routing_check(shape, opts, &base, &range);
  if (st != MOE_OK) return st;
  if (!aligned(x, 16) || !aligned(expanded_x, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  const int64_t cap = capacity_tokens(s, ws_bytes);
  if (cap < num_rows) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!is_prepared(ws, ws_bytes, num_rows, s)) return MOE_ERR_NOT_PREPARED;
  const WsLayout L = make_layout(s, cap);
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  RouteArgs ra = route_args(shape, L, static_cast<uint8_t*>(ws), expert_ids, num_rows);
  MOE_CUDA(init_routing_enqueue(ra, base, range, shape, num_rows, x, expert_ids, opts, expanded_x, expanded_row_idx,
                                tokens_cumsum_or_count, expanded_scale, sms, stream));
  return MOE_OK;
}

// ------------------------------------------------------------ streaming
static moe_status_t ring_check(const moe_shape_t* shape, const moe_stream_ring_t* cfg, const void* ring,
                               size_t ring_bytes, RingLayout* R) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!cfg || cfg->num_slots < 1 || cfg->num_slots > 64 || cfg->tokens_per_slot < 1 || cfg->max_sms < 0)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)cfg->tokens_per_slot * shape->top_k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  *R = make_ring_layout(to_shape(shape), cfg->num_slots, cfg->tokens_per_slot);
  if (ring) {
    if (!aligned(ring, 256)) return MOE_ERR_INVALID_ARG;
    if (ring_bytes < R->total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  }
  return MOE_OK;
}

static StreamArgs stream_args(const RingLayout& R, void* ring, int64_t chunk, uint32_t wait_us) {
  uint8_t* b = static_cast<uint8_t*>(ring);
  StreamArgs r{};
  r.hdr = reinterpret_cast<RingHeader*>(b + R.header);
  r.meta = reinterpret_cast<SlotMeta*>(b + R.meta);
  r.S = R.S;
  r.chunk = chunk;
  r.wait_ns = (uint64_t)(wait_us ? wait_us : 1000000u) * 1000u;
  return r;
}

static bool chunk_ok(int64_t chunk) { return chunk >= 0 && chunk < ((int64_t)1 << 32) - 1; }

moe_status_t moe_stream_ring_size(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, size_t* bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  RingLayout R;
  moe_status_t st = ring_check(shape, ring_cfg, nullptr, 0, &R);
  if (st != MOE_OK) return st;
  *bytes = R.total;
  return MOE_OK;
}

moe_status_t moe_stream_ring_init(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                  size_t ring_bytes, cudaStream_t stream) {
  if (!ring) return MOE_ERR_INVALID_ARG;
  RingLayout R;
  moe_status_t st = ring_check(shape, ring_cfg, ring, ring_bytes, &R);
  if (st != MOE_OK) return st;
  MOE_CUDA(cudaMemsetAsync(ring, 0, R.total, stream));
  return MOE_OK;
}

moe_status_t moe_stream_begin(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                              size_t ring_bytes, cudaStream_t stream) {
  if (!ring) return MOE_ERR_INVALID_ARG;
  RingLayout R;
  moe_status_t st = ring_check(shape, ring_cfg, ring, ring_bytes, &R);
  if (st != MOE_OK) return st;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  MOE_CUDA(launch_stream_begin(stream_args(R, ring, 0, 0), stream));
  return MOE_OK;
}

moe_status_t moe_stream_publish(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                size_t ring_bytes, int64_t chunk, int64_t token_base, int32_t n, int32_t parts,
                                const void* x, const int32_t* expert_ids, const void* route_weights, uint32_t wait_us,
                                cudaStream_t stream) {
  if (!ring || !chunk_ok(chunk) || token_base < 0 || n < 0 || parts < 1 || parts > 3) return MOE_ERR_INVALID_ARG;
  RingLayout R;
  moe_status_t st = ring_check(shape, ring_cfg, ring, ring_bytes, &R);
  if (st != MOE_OK) return st;
  if (n > R.C) return MOE_ERR_INVALID_ARG;
  if ((parts & MOE_STREAM_LAYOUT) && n > 0 && (!x || !aligned(x, 16))) return MOE_ERR_INVALID_ARG;
  if ((parts & MOE_STREAM_ROUTE) && n > 0 && (!expert_ids || !route_weights)) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  uint8_t* b = static_cast<uint8_t*>(ring);
  const int64_t slot = chunk % R.S;
  PublishArgs a{};
  a.r = stream_args(R, ring, chunk, wait_us);
  a.token_base = token_base;
  a.C = R.C;
  a.n = n;
  a.H = shape->hidden;
  a.k = shape->top_k;
  a.E = shape->num_experts;
  a.parts = parts;
  a.x = static_cast<const uint16_t*>(x);
  a.ids = expert_ids;
  a.w = static_cast<const uint16_t*>(route_weights);
  a.slot_x = reinterpret_cast<uint16_t*>(b + R.x) + slot * R.C * a.H;
  a.slot_ids = reinterpret_cast<int32_t*>(b + R.ids) + slot * R.C * a.k;
  a.slot_w = reinterpret_cast<uint16_t*>(b + R.w) + slot * R.C * a.k;
  MOE_CUDA(launch_stream_publish(a, sms, stream));
  return MOE_OK;
}

moe_status_t moe_stream_forward(const moe_shape_t* shape, const moe_stream_ring_t* ring_cfg, void* ring,
                                size_t ring_bytes, int64_t chunk, const uint8_t* w13, const uint8_t* sf13,
                                const uint8_t* w2, const uint8_t* sf2, const float* qX, const float* dX_dW13,
                                const float* qA, const float* dA_dW2, const float* situ_beta,
                                const float* situ_linear_beta, void* ws, size_t ws_bytes, void* out,
                                int64_t out_rows, uint32_t wait_us, cudaStream_t stream) {
  if (!ring || !chunk_ok(chunk) || !out || out_rows < 1 || !ws) return MOE_ERR_INVALID_ARG;
  RingLayout R;
  moe_status_t st = ring_check(shape, ring_cfg, ring, ring_bytes, &R);
  if (st != MOE_OK) return st;
  if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  const int64_t cap = capacity_tokens(s, ws_bytes);
  if (cap < R.C) return MOE_ERR_WORKSPACE_TOO_SMALL;
  if (!is_prepared(ws, ws_bytes, R.C, s)) return MOE_ERR_NOT_PREPARED;
  if (!w13 || !sf13 || !w2 || !sf2 || !qX || !dX_dW13 || !qA || !dA_dW2) return MOE_ERR_INVALID_ARG;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  uint8_t* b = static_cast<uint8_t*>(ring);
  const int64_t slot = chunk % R.S;
  const StreamArgs r = stream_args(R, ring, chunk, wait_us);
  int32_t* ws_hdr = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + make_layout(s, cap).header);
  MOE_CUDA(launch_stream_gate(r, R.C, ws_hdr, stream));
  // the slot's C tokens; rows past the chunk's count carry the id E, which the
  // routing skips without flagging it (ids above E are still flagged)
  st = forward_impl(shape, 0, shape->num_experts + 1, R.C, reinterpret_cast<uint16_t*>(b + R.x) + slot * R.C * s.H,
                    reinterpret_cast<int32_t*>(b + R.ids) + slot * R.C * s.k,
                    reinterpret_cast<uint16_t*>(b + R.w) + slot * R.C * s.k, w13, sf13, w2, sf2, qX, dX_dW13, qA,
                    dA_dW2, situ_beta, situ_linear_beta, ws, ws_bytes, out, stream, out_rows, ring_cfg->max_sms);
  if (st != MOE_OK) return st;
  MOE_CUDA(launch_stream_release(r, ws_hdr, stream));
  return MOE_OK;
}

moe_status_t moe_stream_read_status(const void* ring, int32_t* host_status, cudaStream_t stream) {
  if (!ring || !host_status) return MOE_ERR_INVALID_ARG;
  int32_t* d = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(const_cast<void*>(ring)) + offsetof(RingHeader, status));
  int32_t h = 0;
  MOE_CUDA(cudaMemcpyAsync(&h, d, sizeof(h), cudaMemcpyDeviceToHost, stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  MOE_CUDA(cudaMemsetAsync(d, 0, sizeof(h), stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  *host_status = h;
  return MOE_OK;
}

moe_status_t moe_read_status(const void* ws, int32_t* host_status, cudaStream_t stream) {
  if (!ws || !host_status) return MOE_ERR_INVALID_ARG;
  int32_t h[2] = {0, 0};
  MOE_CUDA(cudaMemcpyAsync(h, ws, sizeof(h), cudaMemcpyDeviceToHost, stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  MOE_CUDA(cudaMemsetAsync(const_cast<void*>(ws), 0, sizeof(h), stream));
  MOE_CUDA(cudaStreamSynchronize(stream));
  host_status[0] = h[0];
  host_status[1] = h[1];
  return h[0] ? MOE_ERR_DEVICE_STATUS : MOE_OK;
}

moe_status_t moe_test_codec_sweep(uint32_t start, int64_t n, uint8_t* e2m1_lo, uint8_t* e2m1_hi, uint8_t* e4m3,
                                  cudaStream_t stream) {
  if (n < 0 || (uint64_t)start + (uint64_t)n > ((uint64_t)1 << 32)) return MOE_ERR_INVALID_ARG;
  if (n == 0) return MOE_OK;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  MOE_CUDA(launch_codec_sweep(start, n, e2m1_lo, e2m1_hi, e4m3, stream, sms));
  return MOE_OK;
}

moe_status_t moe_test_quantize_rows(const float* x, int64_t rows, int32_t cols, const float* q_per_row,
                                    uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!x || !q_per_row || !packed || !sf || rows < 0 || cols <= 0 || cols % 16 != 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(packed, 8)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  MOE_CUDA(launch_quant_rows(x, rows, cols, q_per_row, packed, sf, stream, sms));
  return MOE_OK;
}

moe_status_t moe_test_situ_requant(const float* z, int64_t rows, int32_t inter, float qA, float beta, float lam,
                                   float* a_out, uint8_t* packed, uint8_t* sf, cudaStream_t stream) {
  if (!z || !a_out || !packed || !sf || rows < 0 || inter <= 0 || inter % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(packed, 4)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  MOE_CUDA(launch_situ_requant(z, rows, inter, qA, beta, lam, a_out, packed, sf, stream));
  return MOE_OK;
}

moe_status_t moe_test_requant_lanes(const float* act, int64_t rows, int32_t inter, float qA, uint8_t* packed,
                                    uint8_t* sf, cudaStream_t stream) {
  if (!act || !packed || !sf || rows < 0 || inter <= 0 || inter % 32 != 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(packed, 4)) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  MOE_CUDA(launch_requant_lanes(act, rows, inter, qA, packed, sf, stream));
  return MOE_OK;
}

moe_status_t moe_test_mma_fp4(const uint8_t* a, const uint8_t* sfa_atoms, const uint8_t* b, const uint8_t* sfb_atoms,
                              int32_t n, int32_t k, float* d, int32_t* status, cudaStream_t stream) {
  if (!a || !sfa_atoms || !b || !sfb_atoms || !d || !status) return MOE_ERR_INVALID_ARG;
  if (n < 1 || n > 128 || k < 256 || k % 256 != 0) return MOE_ERR_INVALID_ARG;
  if (!aligned(a, 256) || !aligned(b, 256) || !aligned(sfa_atoms, 16) || !aligned(sfb_atoms, 16))
    return MOE_ERR_INVALID_ARG;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  CUtensorMap ta, tb;
  const uint64_t da[2] = {(uint64_t)k / 2, 128}, db[2] = {(uint64_t)k / 2, (uint64_t)n};
  const uint64_t str[1] = {(uint64_t)k / 2};
  const uint32_t ba[2] = {128, 128}, bb[2] = {128, 16};
  if (!make_map(&ta, a, 2, da, str, ba, CU_TENSOR_MAP_SWIZZLE_128B)) return MOE_ERR_CUDA;
  if (!make_map(&tb, b, 2, db, str, bb, CU_TENSOR_MAP_SWIZZLE_128B)) return MOE_ERR_CUDA;
  MOE_CUDA(launch_mma_check(ta, tb, sfa_atoms, sfb_atoms, n, k, d, status, stream));
  return MOE_OK;
}

moe_status_t moe_test_mma_peak(int32_t grid, int32_t n, int32_t mmas, int32_t copies, int32_t accs, int64_t* cycles,
                               int32_t* status, cudaStream_t stream) {
  if (!cycles || !status || n < 16 || n > 256 || n % 16 != 0 || mmas < 4 || mmas % 4 != 0 || mmas > (1 << 24) ||
      copies < 0 || copies > 16 || (accs != 1 && accs != 2 && accs != 4) || accs * n > 384)
    return MOE_ERR_INVALID_ARG;
  int sms = 0;
  MOE_CUDA(device_ready(&sms));
  if (grid < 1 || grid > sms) return MOE_ERR_INVALID_ARG;
  MOE_CUDA(launch_mma_peak(grid, n, mmas, copies, accs, reinterpret_cast<long long*>(cycles), status, stream));
  return MOE_OK;
}

moe_status_t moe_workspace_layout(const moe_shape_t* shape, size_t ws_bytes, moe_ws_layout_t* out) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!out) return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  const int64_t cap = capacity_tokens(s, ws_bytes);
  if (cap < 1) return MOE_ERR_WORKSPACE_TOO_SMALL;
  const WsLayout L = make_layout(s, cap);
  out->max_tokens = L.max_tokens;
  out->pairs_max = L.Pmax;
  out->padded_rows_max = L.PpadMax;
  out->tiles_max = L.TTmax;
  out->header = (int64_t)L.header;
  out->count = (int64_t)L.count;
  out->cumsum = (int64_t)L.cumsum;
  out->offs = (int64_t)L.offs;
  out->poffs = (int64_t)L.poffs;
  out->sorted_row = (int64_t)L.sorted_row;
  out->gather = (int64_t)L.gather;
  out->row_pos = (int64_t)L.row_pos;
  out->prow_pair = (int64_t)L.prow_pair;
  out->tt_list = (int64_t)L.tt_list;
  out->xq = (int64_t)L.xq;
  out->sfx = (int64_t)L.sfx;
  out->sft = (int64_t)L.sft;
  out->aq = (int64_t)L.aq;
  out->sfa = (int64_t)L.sfa;
  out->acc = (int64_t)L.acc;
  out->total = (int64_t)L.total;
  return MOE_OK;
}

moe_status_t moe_profile_start(int32_t max_calls) {
  if (max_calls < 1 || max_calls > 100000) return MOE_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_prof.on) return MOE_ERR_INVALID_ARG;
  g_prof.ev.assign((size_t)max_calls * (kStages + 1), nullptr);
  for (auto& e : g_prof.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return MOE_ERR_CUDA;
  g_prof.max_calls = max_calls;
  g_prof.calls = 0;
  g_prof.on = true;
  return MOE_OK;
}

moe_status_t moe_profile_stop(float* stage_ms, int32_t* calls) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_prof.on) return MOE_ERR_INVALID_ARG;
  moe_status_t st = MOE_OK;
  float acc[kStages] = {0, 0, 0, 0, 0};
  for (int c = 0; c < g_prof.calls && st == MOE_OK; ++c) {
    cudaEvent_t* e = &g_prof.ev[(size_t)c * (kStages + 1)];
    if (cudaEventSynchronize(e[kStages]) != cudaSuccess) st = MOE_ERR_CUDA;
    for (int i = 0; i < kStages && st == MOE_OK; ++i) {
      float ms = 0.f;
      if (cudaEventElapsedTime(&ms, e[i], e[i + 1]) != cudaSuccess) st = MOE_ERR_CUDA;
      acc[i] += ms;
    }
  }
  if (stage_ms)
    for (int i = 0; i < kStages; ++i) stage_ms[i] = acc[i];
  if (calls) *calls = g_prof.calls;
  for (auto& e : g_prof.ev) cudaEventDestroy(e);
  g_prof.ev.clear();
  g_prof.on = false;
  g_prof.calls = g_prof.max_calls = 0;
  return st;
}

moe_status_t moe_forward_kernels(const moe_shape_t* shape, int64_t num_tokens, int32_t* fc1_decode,
                                 int32_t* fc2_decode) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!fc1_decode || !fc2_decode || num_tokens < 1) return MOE_ERR_INVALID_ARG;
  const Shape s = to_shape(shape);
  *fc1_decode = fc1_gemv(s, num_tokens) ? 1 : 0;
  *fc2_decode = fc2_gemv(s, num_tokens) ? 1 : 0;
  return MOE_OK;
}

moe_status_t moe_forward_launch_count(const moe_shape_t* shape, int64_t num_tokens, int32_t* launches) {
  moe_status_t st = shape_supported(shape);
  if (st != MOE_OK) return st;
  if (!launches || num_tokens < 1) return MOE_ERR_INVALID_ARG;
  *launches = forward_launches(to_shape(shape), num_tokens);
  return MOE_OK;
}

}  // extern "C"
