// gemm.cu -- the two block-scaled NVFP4 grouped GEMMs on tcgen05.
//
// FC1 ("Cake SiTU backend": FC1 over gate and up, SiTU, intermediate NVFP4
// requantization): the MMA takes the routed tokens of one expert tile on its
// M side (128 rows, gathered per row from the token-major quantized X; a
// decode-sized group fills only the first rows, which costs the tensor pipe
// no more than a narrow N would) and prepared W13 tiles on its N side: 128
// rows holding 64 intermediate features with gate and up rows interleaved
// (row 2i = gate of feature i, row 2i+1 = up).  A work unit is one token tile
// and two such W13 tiles (128 features), which form one 256-row operand: per
// k-block of 256 FP4 elements one N = 256 MMA per K-step, and the X tile and
// its scale atoms serve both tiles (12 scale-atom copies to TMEM instead of
// 16, 54 KB of loads for a [128 x 256] product instead of 72).  The
// accumulators (256 TMEM columns) are single-buffered; the epilogue releases
// them as soon as it has read them.  In the epilogue a thread owns one token
// row: it reads 16 features' gate/up pairs, forms z = acc * dX*dW13[e] and
// a = SiTU(z_g, z_u), and quantizes the 16 values with qA[e] in registers
// into the token's padded row of A (codes and atom-layout scale) -- no
// cross-lane traffic.  Below 17 tokens a unit is one W13 tile (N = 128), for
// more units to spread over the SMs.
//
// FC2 ("Cake SiTU backend": FC2, BF16 weighted finalization): weights on the
// MMA's M side (128 output features), tokens on N (16..128).  A work unit is
// one token tile and a group of G consecutive 128-feature output tiles.  The
// tile's quantized activations (K = I, all k-blocks) are loaded into a shared
// memory slot once and stay there while the group's W2 tiles stream through
// the ring; each output tile accumulates [128 x N] over K = I in k-blocks of
// 128.  The epilogue scales by dA*dW2[e] and the route weight and adds each
// routed pair's 128 outputs into its token's fp32 accumulator row with L2
// reductions (one coalesced 128-byte reduction per warp and token).  Groups
// run outermost (in nq passes over H), so the accumulator columns of one
// group are the reductions' working set; the per-pair FC2 rows never reach
// memory.  The finalize kernel rounds the sums to BF16.  When the tiles are
// heavy, the last unit of one tile per CTA is split into narrower parts that
// are taken last, so that the CTAs finish together.
//
// Warp roles (FC2; FC1's are listed with its constants): warp 0 issues TMA,
// warp 1 owns TMEM and issues MMAs, the next warps drain TMEM (each 32-lane
// quarter by several warps taking alternate 16-column chunks), and the last
// one copies each stage's W2 scale atoms to TMEM (outside the MMA thread,
// whose commits then cover its MMAs alone).  In FC1 warps 0 and 1 gather the
// X rows.  Persistent CTAs take their work units from a counter that routing
// seeds; the stage ring and the barrier phases carry across units.  Every
// wait is bounded.
#include "nvfp4.cuh"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

constexpr uint32_t kTmemCols = 512;

// FC1 stage: X [128 tokens x 128 B, gathered] | W [PAIR tiles of 128 interleaved
// gate/up rows x 128 B] | X scale atoms | W scale atoms (4 of 512 B per tile).
// PAIR = 2 shares the X tile and its atoms between two W13 tiles (single-
// buffered accumulators); PAIR = 1 keeps double-buffered accumulators and a
// deeper ring, better when few units would leave SMs idle.
template <int PAIR>
struct Fc1Cfg {
  static constexpr int kStage = 16384 * (1 + PAIR) + 2048 * (1 + PAIR);
  static constexpr int kStages = 221184 / kStage;            // 6 or 4
  static constexpr int kX = 0, kW = 16384, kSX = 16384 * (1 + PAIR), kSW = kSX + 2048;
  static constexpr int kBufs = PAIR == 1 ? 2 : 1;            // accumulator buffers of PAIR x 128 columns
  static constexpr int kSfCols = 16 * (1 + PAIR);            // TMEM scale columns per stage
  static constexpr size_t kSmem = (size_t)kStages * kStage + 1024 + 1024;
};
static_assert(Fc1Cfg<1>::kBufs * 128 + Fc1Cfg<1>::kStages * Fc1Cfg<1>::kSfCols <= 512 &&
                  Fc1Cfg<2>::kBufs * 256 + Fc1Cfg<2>::kStages * Fc1Cfg<2>::kSfCols <= 512,
              "FC1 TMEM plan");
constexpr int kFc1EpiWarps = 16;
// FC1 warps: 0 and 1 gather X rows, 2 TMA producer, 3 MMA issuer and TMEM
// owner, 4.. epilogue.  TMEM lane quarter q is read by warps w with
// w % 4 == q, which share a scheduler; tiles fill the low quarters first, so
// the two issuing warps sit on the schedulers of quarters 2 and 3.
constexpr int kFc1Producer = 2, kFc1Mma = 3, kFc1Epi0 = 4;
constexpr int kFc1Gather = 32 * kFc1Producer;   // gather threads (warps 0 and 1)
constexpr int kFc1Threads = 32 * (kFc1Epi0 + kFc1EpiWarps);
// FC2 shared memory: barriers (1 KB) | two activation slots (a token tile's
// A codes [I/128 k-blocks][128 rows x 64 B] + its I/64 scale atoms) | ring of
// W2 stages of KS k-blocks of one 128-feature output tile: their codes
// [KS][128 rows x 64 B] then their 2*KS scale atoms (9 KB per k-block).  KS
// is 1 or I/128 (a whole output tile, so that the issuing thread waits,
// fences and commits once per tile, which pays at small and medium batches);
// the stage count follows from I and KS.
constexpr int kMaxStages = 20;
constexpr int kFc2KbBytes = 9216;   // codes (8 KB) + scale atoms (1 KB) of one k-block
constexpr int kFc2EpiWarps = 16;
// FC2 warps: 0 TMA producer, 1 MMA issuer and TMEM owner, 2 .. 2 + kFc2EpiWarps - 1
// epilogue, then the thread that copies each W2 stage's scale atoms to TMEM.
constexpr int kFc2CopyWarp = 2 + kFc2EpiWarps;
constexpr int kFc2Threads = 32 * (kFc2CopyWarp + 1);
constexpr int kFc2MaxI = 512;
constexpr uint32_t kFc2SfbCol = 448;   // TMEM column of the activation slots' scale factors

constexpr int kMaxAccSlots = 8;
constexpr int kUnitQueue = 8;   // entries of a CTA's work-unit queue

struct Barriers {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t sready[kMaxStages];    // FC2: the stage's W2 scale atoms are in TMEM (the copy thread's commit)
  uint64_t tmem_full[kMaxAccSlots];
  uint64_t tmem_empty[kMaxAccSlots];
  uint64_t act_full[2];
  uint64_t act_empty[2];
  uint64_t drain;
  uint64_t drain_cp;              // FC2: the copy thread's last copies complete
  uint64_t uq_full[kUnitQueue];   // work-unit queue: entry published by the producer thread
  uint64_t uq_empty[kUnitQueue];  // ... read by every consuming role
  int4 uq_tile[kUnitQueue];
  int32_t uq_unit[kUnitQueue];
  uint32_t tmem_base;
  volatile int32_t abort_flag;
  int32_t fc2_g;         // FC2: output tiles per work unit, chosen by thread 0 during setup
  int32_t fc2_gs;        // FC2: output tiles per part of a split tail unit (= fc2_g: no split)
};
static_assert(sizeof(Barriers) <= 1024, "barrier block");

constexpr size_t kFc2Smem = 232448;    // the opt-in maximum; carved up at run time

__host__ __device__ constexpr int fc2_act_bytes(int I) { return (128 * (I / 2) + (I / 64) * 512 + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int fc2_stages(int I, int KS) {
  return ((int)kFc2Smem - 1024 - 1024 - 2 * fc2_act_bytes(I)) / (KS * kFc2KbBytes) < kMaxStages
             ? ((int)kFc2Smem - 1024 - 1024 - 2 * fc2_act_bytes(I)) / (KS * kFc2KbBytes)
             : kMaxStages;
}
// per stage 2*KS scale atoms of 4 TMEM columns from column 256, below the
// activation slots' scale columns
constexpr bool fc2_plan_ok(int I) {
  return fc2_stages(I, I / 128) >= 4 && 256 + fc2_stages(I, I / 128) * (I / 64) * 4 <= (int)kFc2SfbCol &&
         256 + fc2_stages(I, 1) * 8 <= (int)kFc2SfbCol;
}
static_assert(fc2_plan_ok(128) && fc2_plan_ok(256) && fc2_plan_ok(384) && fc2_plan_ok(512) &&
                  kFc2SfbCol + 2 * (kFc2MaxI / 64) * 4 <= kTmemCols,
              "FC2 shared memory / TMEM plan");

// Activation rows of a tile arrive in boxes of 128, 64, 32 or 16 rows,
// largest first: at most four copies per k-block.

__device__ __forceinline__ void load_rows(uint8_t* dst, const RowMaps& maps, int32_t x, int32_t row0, int nch,
                                          uint32_t chunk_bytes, uint64_t* bar) {
  int r = 0;
  while (r < nch) {
    const int left = nch - r;
    const CUtensorMap* m;
    int n;
    if (left >= 8) { m = &maps.m128; n = 8; }
    else if (left >= 4) { m = &maps.m64; n = 4; }
    else if (left >= 2) { m = &maps.m32; n = 2; }
    else { m = &maps.m16; n = 1; }
    tma_load_2d(dst + r * chunk_bytes, m, x, row0 + r * kTokChunk, bar);
    r += n;
  }
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ uint64_t sf_desc(const uint8_t* p) { return smem_desc(smem_u32(p), 0, 128, kLayoutNone); }

template <int STAGES, int EPI_WARPS>
__device__ void gemm_setup(Barriers* bars, int warp, int tmem_warp, uint32_t full_arrivals = 1,
                           uint32_t uq_consumers = 1) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], full_arrivals);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->sready[s], 1);
    }
    for (int b = 0; b < kMaxAccSlots; ++b) {
      mbar_init(&bars->tmem_full[b], 1);
      mbar_init(&bars->tmem_empty[b], EPI_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->act_full[b], 1);
      mbar_init(&bars->act_empty[b], 1);
    }
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->drain_cp, 1);
    for (int q = 0; q < kUnitQueue; ++q) {
      mbar_init(&bars->uq_full[q], 1);
      mbar_init(&bars->uq_empty[q], uq_consumers);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == tmem_warp) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Waits that fail raise the CTA-wide abort flag; every role then leaves its
// loop, drains what it issued, and the CTA frees TMEM and exits.
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, Barriers* bars, int32_t* status) {
  if (bars->abort_flag) return false;
  if (mbar_wait(bar, parity, status)) return true;
  bars->abort_flag = 1;
  return false;
}

// Work-unit queue of a persistent GEMM CTA.  The producer thread takes the
// CTA's next unit (from the call's work counter, or the static stride) and
// publishes (unit, tile descriptor) entries in order, one entry ahead of the
// unit it streams; the other roles read them in the same order, each entry
// and the one after it, and release an entry once past it.  Unit -1 ends the
// sequence.  Waits are bounded like every other.
__device__ __forceinline__ bool uq_publish(Barriers* bars, int j, int unit, int4 tile, int32_t* status) {
  const int q = j % kUnitQueue;
  if (!wait_or_abort(&bars->uq_empty[q], ((uint32_t)(j / kUnitQueue) & 1u) ^ 1u, bars, status)) return false;
  volatile int* t = reinterpret_cast<volatile int*>(bars->uq_tile + q);
  t[0] = tile.x;
  t[1] = tile.y;
  t[2] = tile.z;
  t[3] = tile.w;
  reinterpret_cast<volatile int32_t*>(bars->uq_unit)[q] = unit;
  mbar_arrive(&bars->uq_full[q]);
  return true;
}

// Unit of entry j (-1: the end; -2: the wait gave up) and its tile descriptor.
__device__ __forceinline__ int uq_read(Barriers* bars, int j, int4& tile, int32_t* status) {
  const int q = j % kUnitQueue;
  if (!wait_or_abort(&bars->uq_full[q], (uint32_t)(j / kUnitQueue) & 1u, bars, status)) return -2;
  const volatile int* t = reinterpret_cast<const volatile int*>(bars->uq_tile + q);
  tile = make_int4(t[0], t[1], t[2], t[3]);
  return reinterpret_cast<const volatile int32_t*>(bars->uq_unit)[q];
}

__device__ __forceinline__ void uq_release(Barriers* bars, int j) { mbar_arrive(&bars->uq_empty[j % kUnitQueue]); }

// A tile descriptor from the routing kernel is trusted only after a bounds
// check; a bad one is skipped by every role alike and flagged.
__device__ __forceinline__ bool tile_ok(const int4& t, int E, int64_t max_rows) {
  return t.x >= 0 && t.x < E && t.y >= 0 && (t.y & (kTileRows - 1)) == 0 && t.z >= 1 && t.z <= kTileRows &&
         (int64_t)t.y + t.z <= max_rows;
}

__device__ __forceinline__ int clamp_tiles(int n, int max_tiles) { return n < 0 ? 0 : (n > max_tiles ? max_tiles : n); }

// Tile descriptor of work unit `unit` (units_per_tile units share a token
// tile), or an invalid descriptor past the end.  Issued one or two units
// ahead so the load latency hides under the current unit.
__device__ __forceinline__ int4 next_tile(const int4* tiles, int unit, int num_units, int units_per_tile) {
  return unit < num_units ? tiles[unit / units_per_tile] : make_int4(-1, 0, 0, 0);
}

// dX*dW13, qA, beta, lambda of the expert of a tile (zeros for an invalid tile).
__device__ __forceinline__ float4 unit_scalars(const Fc1Args& p, const int4& t) {
  if (t.x < 0 || t.x >= p.E) return make_float4(0.f, 0.f, 0.f, 0.f);
  return make_float4(__ldg(p.dXdW13 + t.x), __ldg(p.qA + t.x), __ldg(p.beta + t.x), __ldg(p.lam + t.x));
}

// FC2 work unit -> (token tile, group of G consecutive 128-feature tiles);
// groups outermost, so the groups of one pass over H run together.
// FC2's work units.  Unit u < U0 is (tile u % ntiles, output tiles
// [(u / ntiles) * G, + G)), groups outermost; with Gs < G the last `ntail`
// tiles of the last group are split into S = G / Gs parts of Gs output tiles
// each and come last, so that the units taken at the end are short and the
// CTAs finish together (the parts reload their tile's activations, so the
// split is kept to one tile per CTA).
struct Fc2Units {
  int ntiles, G, NG, S, Gs, ntail, U0, num;
  __device__ __forceinline__ void init(int nt, int NMT, int G_, int Gs_, int grid) {
    ntiles = nt;
    G = G_;
    NG = NMT / G;
    Gs = Gs_;
    S = G / Gs;
    ntail = (S > 1 && nt > 0) ? min(nt, grid) : 0;
    U0 = nt * NG - ntail;
    num = U0 + ntail * S;
  }
  __device__ __forceinline__ int tile_index(int u) const {
    return u < U0 ? u % ntiles : ntiles - ntail + (u - U0) / S;
  }
  __device__ __forceinline__ int first_mt(int u) const {
    return u < U0 ? (u / ntiles) * G : (NG - 1) * G + ((u - U0) % S) * Gs;
  }
  __device__ __forceinline__ int width(int u) const { return u < U0 ? G : Gs; }
  // the unit as the MMA and epilogue warps see it: first output tile << 8 | count (a negative u passes through)
  __device__ __forceinline__ int code(int u) const { return u < 0 ? u : (first_mt(u) << 8) | width(u); }
};

// Width of the split tail units: the widest divisor of G that is at most
// G / tail_div, or G itself (no split) when tail_div <= 1 or the tiles hold
// fewer than kFc2TailMinRows routed pairs on average (there the weight
// stream, not the tiles' reductions, sets the units' cost and the extra
// activation loads of the parts do not pay).
constexpr int kFc2TailMinRows = 48;
__device__ __forceinline__ int fc2_tail_width(int G, int tail_div, int ntiles, int64_t pairs) {
  if (tail_div <= 1 || ntiles <= 0 || pairs < (int64_t)kFc2TailMinRows * ntiles) return G;
  int gs = 1;
  for (int d = 2; d <= G; ++d)
    if (G % d == 0 && d * tail_div <= G) gs = d;
  return gs;
}

__device__ __forceinline__ int4 fc2_next_tile(const int4* tiles, int unit, const Fc2Units& us) {
  return (unit >= 0 && unit < us.num) ? tiles[us.tile_index(unit)] : make_int4(-1, 0, 0, 0);
}

// Feature tiles per FC2 unit: the divisor G of the pass width npu that
// minimizes the busiest CTA's work, ceil(units / grid) * (G + 2), where each
// unit streams G W2 tiles and costs about two more in activation loads and
// hand-over.  Small batches get long units (few tiles, overhead dominates);
// large batches short ones.  G is at most half of H/128: units over all of H
// are never faster, and under skewed routing the shorter units of G = H/256
// balance better (Zipf T = 4096: FC2 0.293 -> 0.279 ms).
constexpr int kFc2MaxGroup = 255;   // a unit's output-tile count travels in 8 bits
__device__ __forceinline__ int fc2_group(int ntiles, int NMT, int npu, int grid) {
  int best = 1, best_cost = -1;
  for (int G = 1; G <= min(min(npu, kFc2MaxGroup), max(1, NMT / 2)); ++G) {
    if (npu % G) continue;
    const int units = ntiles * (NMT / G);
    const int cost = (units + grid - 1) / grid * (G + 2);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = G;
    }
  }
  return best;
}

// nvfp4_quant16 over 16 activations held in the even slots of two
// 16-register arrays (activation i in lo[2i] for i < 8, hi[2i-16] after).
__device__ __forceinline__ uint32_t quant16_even(const uint32_t (&lo)[16], const uint32_t (&hi)[16], float q,
                                                 uint2& packed) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(lo[2 * i])), fabsf(__uint_as_float(hi[2 * i]))));
  float r;
  const uint32_t sf = nvfp4_scale(amax, q, r);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const float a0 = __uint_as_float(m < 4 ? lo[4 * m] : hi[4 * m - 16]);
    const float a1 = __uint_as_float(m < 4 ? lo[4 * m + 2] : hi[4 * m - 14]);
    w[m >> 2] |= cvt_e2m1x2(__fmul_rn(a1, r), __fmul_rn(a0, r)) << (8 * (m & 3));
  }
  packed = make_uint2(w[0], w[1]);
  return sf;
}

// ================================================================== FC1
template <int PAIR>
__global__ void __launch_bounds__(kFc1Threads, 1)
    fc1_kernel(const __grid_constant__ CUtensorMap tm_w13, const Fc1Args p) {
  using C = Fc1Cfg<PAIR>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + C::kStages * C::kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NIT = p.I / 64, NP = NIT / PAIR, NKB = p.H / kFc1KBlock;
  if (warp == kFc1Producer && lane == 0) tma_prefetch_desc(&tm_w13);
  // a stage is full once the producer's copies and every gather thread's rows have landed
  gemm_setup<C::kStages, kFc1EpiWarps>(bars, warp, kFc1Mma, 1u + kFc1Gather, kFc1Producer + 1 + kFc1EpiWarps);
  const uint32_t tmem = bars->tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  const int num_units = clamp_tiles(p.hdr[HDR_NUM_TT], p.max_tiles) * NP;   // (token tile, PAIR W13 tiles)
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp < kFc1Producer) {
    // -------------------------------------------------------------- gather
    // The tile's X rows come from the token-major codes: row r of the tile is
    // routed pair prow_pair[row0 + r], i.e. token pair / k.  Eight lanes copy
    // one row's 128-byte k-block slice as 16-byte chunks (chunk c to position
    // c ^ (r % 8) of the 128B-swizzled row), so one warp instruction moves four
    // whole lines; thread (warp w, lane l) takes rows 8i + 4w + l/8, i < 16.
    // Rows past the tile's fill are not copied (their outputs are discarded).
    const int c = lane & 7, rsub = (warp << 2) + (lane >> 3);
    const uint32_t dst0 = (uint32_t)(rsub * 128 + ((c ^ rsub) << 4));
    const size_t H2 = (size_t)p.H / 2;
    // The next unit's pair indices are loaded a unit ahead and only turned
    // into token rows when that unit starts, so their latency stays hidden.
    auto pairs = [&](const int4& t, int (&f)[16]) {
      const bool ok = tile_ok(t, p.E, p.max_rows);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int r = 8 * i + rsub;
        f[i] = (ok && r < t.z) ? __ldg(p.prow_pair + t.y + r) : -1;
      }
    };
    uint32_t stage = 0, phase = 0;
    bool ok = true;
    int qj = 0;
    int4 nxt;
    int unit_nxt = uq_read(bars, 0, nxt, p.status);
    int f_nxt[16];
    pairs(nxt, f_nxt);
    while (unit_nxt >= 0 && ok) {
      const int4 tl = nxt;
      int tok[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) tok[i] = (f_nxt[i] >= 0 && f_nxt[i] < p.num_pairs) ? f_nxt[i] / p.k : -1;
      unit_nxt = uq_read(bars, qj + 1, nxt, p.status);
      __syncwarp();
      if (lane == 0) uq_release(bars, qj);
      ++qj;
      if (unit_nxt == -2) break;
      pairs(nxt, f_nxt);                                      // in flight while this unit streams
      if (!tile_ok(tl, p.E, p.max_rows)) continue;
      for (int kb = 0; kb < NKB; ++kb) {
        if (!wait_or_abort(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
          ok = false;
          break;
        }
        uint8_t* xs = smem + stage * C::kStage + C::kX + dst0;
        const uint8_t* src = p.xq + (size_t)kb * 128 + c * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (tok[i] >= 0) cp_async16(xs + i * 1024, src + (size_t)tok[i] * H2);
        cp_async_mbar_arrive(&bars->full[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait_all();   // every issued copy has landed before the CTA may exit
  } else if (warp == kFc1Producer) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, last_phase = 0;  // bit s: stage s armed; its last armed phase
      bool ok = true;
      // The CTA's units: taken from the work counter (seeded by routing on
      // every call) or by the static stride, and published two units ahead
      // of the one whose loads this thread issues (the gather warps look one
      // unit ahead as they start a unit, about when this thread does).
      int taken = 0;
      auto take = [&]() -> int {
        const int u = p.dynamic ? atomicAdd(p.next, 1) : (int)blockIdx.x + taken * (int)gridDim.x;
        ++taken;
        return (u >= 0 && u < num_units) ? u : -1;
      };
      int qj = 0;
      int unit = take();
      int4 tl0 = next_tile(tiles, unit < 0 ? num_units : unit, num_units, NP);
      ok = uq_publish(bars, qj++, unit, tl0, p.status);
      int unit1 = -1;
      int4 tl1 = make_int4(-1, 0, 0, 0);
      if (ok && unit >= 0) {
        unit1 = take();
        tl1 = next_tile(tiles, unit1 < 0 ? num_units : unit1, num_units, NP);
        ok = uq_publish(bars, qj++, unit1, tl1, p.status);
      }
      while (ok && unit >= 0) {
        int unit2 = -1;
        int4 tl2 = make_int4(-1, 0, 0, 0);
        if (unit1 >= 0) {
          unit2 = take();
          tl2 = next_tile(tiles, unit2 < 0 ? num_units : unit2, num_units, NP);
          if (!uq_publish(bars, qj++, unit2, tl2, p.status)) break;
        }
        const int4 tl = tl0;
        const int cur = unit;
        unit = unit1;
        tl0 = tl1;
        unit1 = unit2;
        tl1 = tl2;
        if (!tile_ok(tl, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
          continue;
        }
        const int e = tl.x, row0 = tl.y;
        const int w0 = (e * NIT + PAIR * (cur % NP)) * NKB;   // first W13 tile; the next is NKB later
        const uint32_t tx = (uint32_t)PAIR * 16384u + (1u + PAIR) * 2048u;
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * C::kStage;
          mbar_arrive_expect_tx(&bars->full[stage], tx);
          armed |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          bulk_g2s(st + C::kSX, p.sfx + ((size_t)(row0 >> 7) * (p.H / 64) + (size_t)kb * 4) * 512u, 2048u,
                   &bars->full[stage]);
#pragma unroll
          for (int j = 0; j < PAIR; ++j) {
            tma_load_3d(st + C::kW + j * 16384, &tm_w13, 0, 0, w0 + j * NKB + kb, &bars->full[stage]);
            bulk_g2s(st + C::kSW + j * 2048, p.sf13p + (size_t)(w0 + j * NKB + kb) * 2048u, 2048u, &bars->full[stage]);
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every issued copy has landed before the CTA may exit
      for (int s = 0; s < C::kStages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
    }
  } else if (warp == kFc1Mma) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      // TMEM: accumulator buffer b holds the unit's PAIR blocks at columns
      // (b*PAIR + j)*128; the scale atoms of stage s at 256 + kSfCols*s: X's
      // four (K-steps 0..3), then per K-step the PAIR W tiles' atoms.
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      const uint32_t idesc = idesc_mxf4nvf4(128, 128 * PAIR);
      // Descriptors of stage 0 are computed once; a stage, K-step or scale
      // atom only moves their start-address field (address >> 4), so the
      // issuing thread spends its time on the tcgen05 instructions rather
      // than on dependent address arithmetic.
      const uint64_t xd0 = smem_desc(smem_u32(smem + C::kX), 16, 1024, kLayoutSW128);
      const uint64_t wd0 = smem_desc(smem_u32(smem + C::kW), 16, 1024, kLayoutSW128);
      const uint64_t sd0 = sf_desc(smem + C::kSX);   // X atom 0 of stage 0; W atoms follow at kSW
      uint32_t soff = 0;                              // (stage * kStage) >> 4
      uint32_t sfc = tmem + 256;                      // the stage's scale columns
      int qj = 0;
      int4 nxt;
      int unit_nxt = uq_read(bars, 0, nxt, p.status);
      while (unit_nxt >= 0 && ok) {
        const int4 tl = nxt;
        unit_nxt = uq_read(bars, qj + 1, nxt, p.status);
        uq_release(bars, qj++);
        if (unit_nxt == -2) break;
        if (!tile_ok(tl, p.E, p.max_rows)) continue;
        const uint32_t buf = (uint32_t)local % C::kBufs, par = (((uint32_t)local / C::kBufs) & 1u) ^ 1u;
        const uint32_t dcol = tmem + buf * PAIR * 128;
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->full[stage], phase, bars, p.status)) {
            ok = false;
            break;
          }
          if (kb == 0) {   // the buffer's blocks drained by the epilogue of its previous unit
#pragma unroll
            for (int j = 0; j < PAIR; ++j)
              if (!wait_or_abort(&bars->tmem_empty[buf * PAIR + j], par, bars, p.status)) ok = false;
            if (!ok) break;
          }
          fence_proxy_async_shared();   // the gathered X rows (cp.async) before the MMA reads them
          tc_fence_after();
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            tmem_cp_32x128b_x4(sfc + a * 4, sd0 + soff + a * 32);
#pragma unroll
            for (int j = 0; j < PAIR; ++j)
              tmem_cp_32x128b_x4(sfc + 16 + (a * PAIR + j) * 4,
                                 sd0 + soff + (C::kSW - C::kSX + j * 2048 + a * 512) / 16);
          }
          // M = tokens (X tile), N = the PAIR W13 tiles as one operand of
          // PAIR*128 rows (contiguous in shared memory, their accumulators
          // contiguous in TMEM, their scale atoms side by side per K-step):
          // one long MMA per K-step, during which the tensor pipe also works
          // off the scale copies.
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_mxf4nvf4(dcol, xd0 + soff + 2 * ks, wd0 + soff + 2 * ks, idesc, sfc + ks * 4,
                         sfc + 16 + ks * 4 * PAIR, (kb | ks) ? 1u : 0u);
          tc_commit(&bars->empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
            soff = 0;
            sfc = tmem + 256;
          } else {
            soff += C::kStage / 16;
            sfc += C::kSfCols;
          }
        }
        if (ok) tc_commit(&bars->tmem_full[buf]);
        ++local;
      }
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w drains TMEM lanes 32*(w%4).. (its tokens); in each of the pair's
    // two accumulators, the 32 columns of 16 features: group (w-4)/4 of 4.
    const int q = warp & 3, grp = (warp - kFc1Epi0) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int I2 = p.I / 2, KC = p.I / 16;
    const int r = q * 32 + lane;                      // token row within the tile
    int local = 0;
    int qj = 0;
    int4 nxt;
    int unit_nxt = uq_read(bars, 0, nxt, p.status);
    float4 sc_nxt = unit_scalars(p, nxt);
    while (unit_nxt >= 0) {
      const int unit = unit_nxt;
      const int4 tl = nxt;
      const float4 sc = sc_nxt;
      unit_nxt = uq_read(bars, qj + 1, nxt, p.status);
      __syncwarp();
      if (lane == 0) uq_release(bars, qj);
      ++qj;
      if (unit_nxt == -2) break;
      sc_nxt = unit_scalars(p, nxt);                                  // one unit ahead
      if (!tile_ok(tl, p.E, p.max_rows)) continue;
      const int row0 = tl.y, rows = tl.z;
      const uint32_t buf = (uint32_t)local % C::kBufs;
      if (!wait_or_abort(&bars->tmem_full[buf], ((uint32_t)local / C::kBufs) & 1u, bars, p.status)) break;
      tc_fence_after();
      const float s13 = sc.x, qa = sc.y, be = sc.z, la = sc.w;
      const float inv_be = 1.0f / be, inv_la = 1.0f / la;
      const bool any = q * 32 < rows;                 // warp-uniform: this quarter holds tokens
      const int64_t prow = row0 + r;
      // read the unit's accumulators, release them, then compute: the MMA of a
      // later unit can start.  Columns 2i / 2i+1 = gate / up of feature
      // (PAIR*u + b)*64 + 16*grp + i.
      uint32_t v[PAIR][2][16];
      if (any) {
#pragma unroll
        for (int b = 0; b < PAIR; ++b) {
          tmem_ld16(tmem + lane_base + (buf * PAIR + b) * 128 + grp * 32, v[b][0]);
          tmem_ld16(tmem + lane_base + (buf * PAIR + b) * 128 + grp * 32 + 16, v[b][1]);
        }
        tmem_ld_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int b = 0; b < PAIR; ++b) mbar_arrive(&bars->tmem_empty[buf * PAIR + b]);
      }
      if (any && r < rows) {
#pragma unroll
        for (int b = 0; b < PAIR; ++b) {
          // SiTU in place: activation i overwrites the gate value it was computed from
#pragma unroll
          for (int i = 0; i < 16; ++i)
            v[b][i >> 3][(2 * i) & 15] = __float_as_uint(
                situ_f32(__fmul_rn(__uint_as_float(v[b][i >> 3][(2 * i) & 15]), s13),
                         __fmul_rn(__uint_as_float(v[b][i >> 3][(2 * i + 1) & 15]), s13), be, inv_be, la, inv_la));
          uint2 packed;
          const uint32_t sf = quant16_even(v[b][0], v[b][1], qa, packed);
          const int it = PAIR * (unit % NP) + b;
          *reinterpret_cast<uint2*>(p.aq + (size_t)prow * I2 + it * 32 + grp * 8) = packed;
          p.sfa[atom_offset(prow, it * 4 + grp, KC)] = (uint8_t)sf;
        }
      }
      ++local;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kFc1Mma) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================== FC2
// WHOLE: ring stages of a whole output tile (KS = I/128 k-blocks); else one
// k-block per stage.
template <bool WHOLE>
__global__ void __launch_bounds__(kFc2Threads, 1)
    fc2_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ RowMaps tm_aq,
               const Fc2Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NMT = p.H / 128, NKB = p.I / kFc2KBlock, NA = p.I / 64, npu = NMT / p.nq;
  const int KS = WHOLE ? NKB : 1;   // k-blocks per ring stage
  const int act_bytes = fc2_act_bytes(p.I), nstages = fc2_stages(p.I, KS), stage_bytes = KS * kFc2KbBytes;
  uint8_t* act = smem + 1024;                       // slot s at act + s * act_bytes
  uint8_t* ring = act + 2 * act_bytes;              // stage s at ring + s * stage_bytes
  const uint32_t act_sf = (uint32_t)(NKB * 8192);   // scale atoms after the codes of a slot
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w2);
    tma_prefetch_desc(&tm_aq.m16);
    tma_prefetch_desc(&tm_aq.m128);
  }
  if (threadIdx.x == 0) {
    // The tile count comes from the routing kernel, which completed before
    // FC1 started, so it is read before waiting for FC1; one thread picks the
    // group size and the setup barrier shares it.
    const int nt = clamp_tiles(__ldcg(p.hdr + HDR_NUM_TT), p.max_tiles);
    const int g = (p.group > 0 && p.group <= kFc2MaxGroup && npu % p.group == 0) ? p.group
                                                                                 : fc2_group(nt, NMT, npu, gridDim.x);
    bars->fc2_g = g;
    bars->fc2_gs = fc2_tail_width(g, p.tail_div, nt, p.num_pairs);
  }
  gemm_setup<kMaxStages, kFc2EpiWarps>(bars, warp, 1, 1, 2 + kFc2EpiWarps);
  const uint32_t tmem = bars->tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  const int ntiles = clamp_tiles(p.hdr[HDR_NUM_TT], p.max_tiles);
  const int G = bars->fc2_g;
  // Accumulator slots: the 256 accumulator columns split into slots as wide as
  // the widest token tile of this call, at least 32 columns (8 slots when
  // decoding), so that many narrow sub-units can be in flight between MMA and
  // epilogue.
  const int maxrows = min(max(p.hdr[HDR_MAXROWS], 1), kTileRows);
  const uint32_t slot_cols = maxrows <= 32 ? 32u : maxrows <= 64 ? 64u : 128u;
  const uint32_t nslots = 256u / slot_cols;
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, last_phase = 0;   // ring stages
      uint32_t act_armed = 0, act_last = 0;  // activation slots
      int local = 0;
      bool ok = true;
      // The CTA's units: taken from the work counter (seeded by routing on
      // every call) or by the static stride, each published one unit ahead
      // of the W2 stream that serves it.
      Fc2Units us;
      us.init(ntiles, NMT, G, bars->fc2_gs, (int)gridDim.x);
      const int num_units = us.num;
      int taken = 0;
      auto take = [&]() -> int {
        const int u = p.dynamic ? atomicAdd(p.next, 1) : (int)blockIdx.x + taken * (int)gridDim.x;
        ++taken;
        return (u >= 0 && u < num_units) ? u : -1;
      };
      int qj = 0;
      int unit = take();
      int4 tl = fc2_next_tile(tiles, unit, us);
      ok = uq_publish(bars, qj++, us.code(unit), tl, p.status);
      while (ok && unit >= 0) {
        const int un = take();
        const int4 tn = fc2_next_tile(tiles, un, us);
        if (!uq_publish(bars, qj++, us.code(un), tn, p.status)) break;
        const int cur = unit;
        const int4 ct = tl;
        unit = un;
        tl = tn;
        if (!tile_ok(ct, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
          continue;
        }
        const int4 tlc = ct;
        const int mt0 = us.first_mt(cur), cnt = us.width(cur);
        const int e = tlc.x, row0 = tlc.y, rows = tlc.z;
        const int nch = (rows + kTokChunk - 1) / kTokChunk;
        // the token tile's activations, once per unit
        const uint32_t slot = (uint32_t)local & 1u, sph = ((uint32_t)local >> 1) & 1u;
        if (!wait_or_abort(&bars->act_empty[slot], sph ^ 1u, bars, p.status)) break;
        uint8_t* as = act + slot * act_bytes;
        mbar_arrive_expect_tx(&bars->act_full[slot], (uint32_t)(NKB * nch * 1024 + NA * 512));
        act_armed |= 1u << slot;
        act_last = (act_last & ~(1u << slot)) | (sph << slot);
        for (int kb = 0; kb < NKB; ++kb) load_rows(as + kb * 8192, tm_aq, kb * 64, row0, nch, 1024u, &bars->act_full[slot]);
        bulk_g2s(as + act_sf, p.sfa + (size_t)(row0 >> 7) * NA * 512u, (uint32_t)(NA * 512), &bars->act_full[slot]);
        ++local;
        // the unit's W2 tiles through the ring
        for (int g = 0; g < cnt && ok; ++g) {
          const int mt = mt0 + g;
          for (int kb0 = 0; kb0 < NKB; kb0 += KS) {
            if (!wait_or_abort(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
              ok = false;
              break;
            }
            uint8_t* st = ring + stage * stage_bytes;
            mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)stage_bytes);
            armed |= 1u << stage;
            last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
            for (int j = 0; j < KS; ++j)
              tma_load_3d(st + j * 8192, &tm_w2, 0, 0, (e * NMT + mt) * NKB + kb0 + j, &bars->full[stage]);
            bulk_g2s(st + KS * 8192, p.sf2p + ((size_t)(e * NMT + mt) * NA + (size_t)kb0 * 2) * 512u,
                     (uint32_t)(KS * 1024), &bars->full[stage]);
            if (++stage == (uint32_t)nstages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // every issued copy has landed before the CTA may exit
      for (int s = 0; s < nstages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
      for (int s = 0; s < 2; ++s)
        if (act_armed & (1u << s)) mbar_wait(&bars->act_full[s], (act_last >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0;
      int local = 0, sub = 0;
      bool ok = true;
      // Ring descriptors of stage 0, moved by their start-address field only
      // (see FC1's issuing thread).
      const uint64_t rd0 = smem_desc(smem_u32(ring), 16, 512, kLayoutSW64);   // + 512 per k-block, + 2 per K-step
      uint32_t soff = 0;                     // (stage * stage_bytes) >> 4
      uint32_t sfc = tmem + 256;             // the stage's scale columns
      int qj = 0;
      int4 tn;
      int unit = uq_read(bars, 0, tn, p.status);
      while (unit >= 0 && ok) {
        const int4 tl = tn;
        const int cnt = unit & 0xFF;
        unit = uq_read(bars, qj + 1, tn, p.status);   // the next entry (published already or soon)
        uq_release(bars, qj++);
        if (unit == -2) break;
        if (!tile_ok(tl, p.E, p.max_rows)) continue;
        const uint32_t ncols = (uint32_t)((tl.z + kTokChunk - 1) / kTokChunk * kTokChunk);
        const uint32_t idesc = idesc_mxf4nvf4(128, ncols);
        const uint32_t slot = (uint32_t)local & 1u, sph = ((uint32_t)local >> 1) & 1u;
        ++local;
        if (!wait_or_abort(&bars->act_full[slot], sph, bars, p.status)) break;
        tc_fence_after();
        const uint8_t* as = act + slot * act_bytes;
        const uint32_t sfb = tmem + kFc2SfbCol + slot * (uint32_t)(NA * 4);
        for (int a = 0; a < NA; ++a) tmem_cp_32x128b_x4(sfb + a * 4, sf_desc(as + act_sf + a * 512));
        const uint64_t bd0 = smem_desc(smem_u32(as), 16, 512, kLayoutSW64);   // + 512 per k-block, + 2 per K-step
        for (int g = 0; g < cnt && ok; ++g, ++sub) {
          const uint32_t buf = (uint32_t)sub % nslots, use = (uint32_t)sub / nslots;
          if (!wait_or_abort(&bars->tmem_empty[buf], (use & 1u) ^ 1u, bars, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dcol = tmem + buf * slot_cols;
          for (int kb0 = 0; kb0 < NKB && ok; kb0 += KS) {
            // the stage has landed and the copy thread has put its scale atoms in TMEM
            if (!wait_or_abort(&bars->sready[stage], phase, bars, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 1
            for (int j = 0; j < KS; ++j) {
              const int kb = kb0 + j;
#pragma unroll
              for (int ks = 0; ks < 2; ++ks)
                mma_mxf4nvf4(dcol, rd0 + soff + (uint32_t)(j * 512 + 2 * ks), bd0 + (uint32_t)(kb * 512 + 2 * ks),
                             idesc, sfc + (j * 2 + ks) * 4, sfb + (kb * 2 + ks) * 4, (kb | ks) ? 1u : 0u);
            }
            tc_commit(&bars->empty[stage]);
            if (++stage == (uint32_t)nstages) {
              stage = 0;
              phase ^= 1u;
              soff = 0;
              sfc = tmem + 256;
            } else {
              soff += (uint32_t)(stage_bytes / 16);
              sfc += (uint32_t)(KS * 8);
            }
          }
          if (ok) tc_commit(&bars->tmem_full[buf]);
        }
        tc_commit(&bars->act_empty[slot]);   // the slot is free once these MMAs are done
      }
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.status);
    }
  } else if (warp == kFc2CopyWarp) {
    if (lane == 0) {
      // ---------------------------------------------------------- scale copies
      // Each ring stage's W2 scale atoms go to its TMEM scale columns as soon
      // as the stage lands, and a commit tells the MMA thread they are there.
      // Issued from their own thread, the copies are not part of the MMA
      // thread's commits, so a stage is released once its MMAs are done
      // rather than once the copies issued for later stages are too.
      uint32_t stage = 0, phase = 0, soff = 0, sfc = tmem + 256;
      const uint64_t rs0 = sf_desc(ring + KS * 8192);   // + 32 per scale atom
      bool ok = true;
      int qj = 0;
      int4 tn;
      int unit = uq_read(bars, 0, tn, p.status);
      while (unit >= 0 && ok) {
        const int4 tl = tn;
        const int cnt = unit & 0xFF;
        unit = uq_read(bars, qj + 1, tn, p.status);
        uq_release(bars, qj++);
        if (unit == -2) break;
        if (!tile_ok(tl, p.E, p.max_rows)) continue;
        for (int g = 0; g < cnt && ok; ++g) {
          for (int kb0 = 0; kb0 < NKB; kb0 += KS) {
            if (!wait_or_abort(&bars->full[stage], phase, bars, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll 2
            for (int a = 0; a < 2 * KS; ++a) tmem_cp_32x128b_x4(sfc + a * 4, rs0 + soff + a * 32);
            tc_commit(&bars->sready[stage]);
            if (++stage == (uint32_t)nstages) {
              stage = 0;
              phase ^= 1u;
              soff = 0;
              sfc = tmem + 256;
            } else {
              soff += (uint32_t)(stage_bytes / 16);
              sfc += (uint32_t)(KS * 8);
            }
          }
        }
      }
      tc_commit(&bars->drain_cp);
      mbar_wait(&bars->drain_cp, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr int NGRP = kFc2EpiWarps / 4;
    constexpr int NI = (kTileRows / kTokChunk + NGRP - 1) / NGRP;   // column chunks per warp
    const int q = warp & 3, grp = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int sub = 0;
    // Route weight and token (-1 if none) of this warp's columns of a tile,
    // fetched one unit ahead so their latency hides under the current unit.
    auto columns = [&](const int4& t, float (&w)[NI], int (&tk)[NI]) {
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int col = (grp + i * NGRP) * 16 + (lane & 15);
        w[i] = 0.0f;
        tk[i] = -1;
        if (t.x >= 0 && col < t.z) {
          const int f = __ldg(p.prow_pair + t.y + col);
          if (f >= 0 && f < p.num_pairs) {
            w[i] = __ldg(p.wrow + t.y + col);
            tk[i] = f / p.k;
          }
        }
      }
    };
    // The unit after the current one comes from the queue one entry ahead,
    // so its scale and columns load while the current unit drains.
    int qj = 0;
    int4 nxt;
    int unit_nxt = uq_read(bars, 0, nxt, p.status);
    float s2_nxt = (nxt.x >= 0 && nxt.x < p.E) ? __ldg(p.dAdW2 + nxt.x) : 0.0f;
    float wgt_nxt[NI];
    int tok_nxt[NI];
    if (tile_ok(nxt, p.E, p.max_rows)) columns(nxt, wgt_nxt, tok_nxt);
    else columns(make_int4(-1, 0, 0, 0), wgt_nxt, tok_nxt);
    bool ok = true;
    while (unit_nxt >= 0 && ok) {
      const int unit = unit_nxt;
      const int4 tl = nxt;
      const float s2 = s2_nxt;
      float wgt[NI];
      int tok[NI];
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        wgt[i] = wgt_nxt[i];
        tok[i] = tok_nxt[i];
      }
      unit_nxt = uq_read(bars, qj + 1, nxt, p.status);
      __syncwarp();
      if (lane == 0) uq_release(bars, qj);
      ++qj;
      if (unit_nxt == -2) break;
      s2_nxt = (nxt.x >= 0 && nxt.x < p.E) ? __ldg(p.dAdW2 + nxt.x) : 0.0f;
      if (tile_ok(nxt, p.E, p.max_rows)) columns(nxt, wgt_nxt, tok_nxt);
      else columns(make_int4(-1, 0, 0, 0), wgt_nxt, tok_nxt);
      if (!tile_ok(tl, p.E, p.max_rows)) continue;
      const int mt0 = unit >> 8, cnt = unit & 0xFF;
      const int rows = tl.z;
      const int nch = (rows + kTokChunk - 1) / kTokChunk;
      for (int g = 0; g < cnt; ++g, ++sub) {
        const uint32_t buf = (uint32_t)sub % nslots, use = (uint32_t)sub / nslots;
        if (!wait_or_abort(&bars->tmem_full[buf], use & 1u, bars, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // drain this warp's columns from TMEM first, so the MMA can refill the slot under the reductions
        uint32_t r[NI][16];
#pragma unroll
        for (int i = 0; i < NI; ++i)
          if (grp + i * NGRP < nch) tmem_ld16(tmem + lane_base + buf * slot_cols + (grp + i * NGRP) * 16, r[i]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->tmem_empty[buf]);
        float* accf = p.acc + (size_t)(mt0 + g) * 128 + q * 32 + lane;
#pragma unroll
        for (int i = 0; i < NI; ++i) {
          if (grp + i * NGRP >= nch) break;
          // per 8 columns: broadcast their weights and tokens first, then issue 8 reductions back to back
#pragma unroll
          for (int h = 0; h < 16; h += 8) {
            float wv[8];
            int tc[8];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
              wv[cc] = __shfl_sync(0xffffffffu, wgt[i], h + cc);
              tc[cc] = __shfl_sync(0xffffffffu, tok[i], h + cc);
            }
#pragma unroll
            for (int cc = 0; cc < 8; ++cc)
              if (tc[cc] >= 0)
                atomicAdd(accf + (size_t)tc[cc] * p.H,
                          __fmul_rn(__fmul_rn(__uint_as_float(r[i][h + cc]), s2), wv[cc]));
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================ MMA check
// One CTA, one tile: D[128, N] = sum_k (A[m,k]*sfa[m,k/16]) * (B[n,k]*sfb[n,k/16])
// with exactly the operand staging of FC1 (128B-swizzled K-major k-blocks of
// 256 FP4, scale atoms copied to TMEM, M = 128, K = 64 per MMA).  Used to
// check the MMA semantics in isolation.
__global__ void __launch_bounds__(128, 1)
    mma_check_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                     const uint8_t* sfa, const uint8_t* sfb, int N, int K, float* d, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;            // 16 KB
  uint8_t* sB = smem + 16384;    // 16 KB
  uint8_t* sSA = smem + 32768;   // 2 KB
  uint8_t* sSB = smem + 34816;   // 2 KB
  Barriers* bars = reinterpret_cast<Barriers*>(smem + 36864);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(&bars->full[0], 1);
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t ncols = (uint32_t)((N + 15) / 16 * 16);
  if (threadIdx.x == 0) {
    bool ok = true;
    const uint32_t idesc = idesc_mxf4nvf4(128, ncols);
    const int nch = (int)ncols / 16;
    for (int kb = 0; kb < K / 256 && ok; ++kb) {
      mbar_arrive_expect_tx(&bars->full[0], 16384u + (uint32_t)nch * 2048u + 4096u);
      tma_load_2d(sA, &tm_a, kb * 128, 0, &bars->full[0]);
      for (int c = 0; c < nch; ++c) tma_load_2d(sB + c * 2048, &tm_b, kb * 128, c * 16, &bars->full[0]);
      bulk_g2s(sSA, sfa + (size_t)kb * 2048, 2048u, &bars->full[0]);
      bulk_g2s(sSB, sfb + (size_t)kb * 2048, 2048u, &bars->full[0]);
      ok = mbar_wait(&bars->full[0], (uint32_t)kb & 1u, status);
      if (!ok) break;
      tc_fence_after();
      for (int a = 0; a < 4; ++a) {
        tmem_cp_32x128b_x4(tmem + 128 + a * 4, sf_desc(sSA + a * 512));
        tmem_cp_32x128b_x4(tmem + 144 + a * 4, sf_desc(sSB + a * 512));
      }
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ad = smem_desc(smem_u32(sA) + ks * 32, 16, 1024, kLayoutSW128);
        const uint64_t bd = smem_desc(smem_u32(sB) + ks * 32, 16, 1024, kLayoutSW128);
        mma_mxf4nvf4(tmem, ad, bd, idesc, tmem + 128 + ks * 4, tmem + 144 + ks * 4, (kb | ks) ? 1u : 0u);
      }
      tc_commit(&bars->drain);
      ok = mbar_wait(&bars->drain, (uint32_t)kb & 1u, status);
    }
    bars->abort_flag = ok ? 0 : 1;
  }
  __syncthreads();
  tc_fence_after();
  if (!bars->abort_flag) {
    for (int c = 0; c < (int)ncols / 16; ++c) {
      uint32_t r[16];
      tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + c * 16, r);
      tmem_ld_wait();
      for (int j = 0; j < 16; ++j)
        if (c * 16 + j < N) d[(size_t)(warp * 32 + lane) * N + c * 16 + j] = __uint_as_float(r[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

// ================================================================ MMA peak
// Tensor-pipe throughput of the block-scaled FP4 MMA as the GEMMs issue it:
// every CTA (one per SM) keeps one A tile [128 x 256 FP4], one B tile
// [n x 256 FP4] and their scale atoms resident in shared memory, copies the
// atoms to TMEM once, and one thread issues `mmas` MMAs (M = 128, N = n,
// K = 64, cycling over the four K-steps of the tile) into `accs` accumulators
// in turn (consecutive MMAs into one accumulator depend on each other; into
// different ones they do not), plus `copies` scale-atom copies (tcgen05.cp 32x128b.warpx4, into TMEM
// columns no MMA reads) after every fourth MMA, as FC1 issues them per
// k-block.  The operand values do not matter for throughput; they are
// fixed bytes.  cycles[blockIdx.x] = SM clock cycles from the first issue to
// the completion of the last MMA.
template <int ACCS>
__global__ void __launch_bounds__(128, 1)
    mma_peak_kernel(int n, int mmas, int copies, long long* cycles, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;              // 16 KB: 128 rows x 128 B, 128B-swizzled
  uint8_t* sB = smem + 16384;      // 32 KB: up to 256 rows x 128 B
  uint8_t* sSF = smem + 49152;     // 16 atoms of 512 B: 4 for A, 8 for B, 4 spare copy sources
  Barriers* bars = reinterpret_cast<Barriers*>(smem + 57344);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 57344 / 16; i += blockDim.x) {
    const uint32_t v = i < 49152 / 16 ? 0x3A2B1C0Du ^ (uint32_t)(i * 0x9E37u) : 0x38383838u;   // codes; scales 1.0
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(v, v ^ 0x11111111u, v ^ 0x22222222u, v ^ 0x44444444u);
  }
  if (threadIdx.x == 0) {
    mbar_init(&bars->drain, 1);
    fence_barrier_init();
  }
  fence_proxy_async_shared();
  if (warp == 0) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  if (threadIdx.x == 0) {
    // TMEM: accumulator a at columns [a n, (a + 1) n) (ACCS n <= 384); A atoms
    // at 384 + 4 ks; B atoms at 400 + 8 ks + 4 j; copy targets at 448 .. 511
    // (read by no MMA).  Descriptors and addresses are computed once, so the
    // loop issues little besides the tcgen05 instructions themselves.
    for (int a = 0; a < 4; ++a) tmem_cp_32x128b_x4(tmem + 384 + a * 4, sf_desc(sSF + a * 512));
    for (int a = 0; a < 8; ++a) tmem_cp_32x128b_x4(tmem + 400 + a * 4, sf_desc(sSF + 2048 + a * 512));
    const uint32_t idesc = idesc_mxf4nvf4(128, (uint32_t)n);
    uint64_t ad[4], bd[4];
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      ad[ks] = smem_desc(smem_u32(sA) + ks * 32, 16, 1024, kLayoutSW128);
      bd[ks] = smem_desc(smem_u32(sB) + ks * 32, 16, 1024, kLayoutSW128);
    }
    const uint64_t cpd0 = sf_desc(sSF);           // + 32 per 512-byte atom (address >> 4)
    const long long t0 = clock64();
    for (int i = 0; i < mmas; i += 4) {
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_mxf4nvf4(tmem + (uint32_t)((ks % ACCS) * n), ad[ks], bd[ks], idesc, tmem + 384 + ks * 4,
                     tmem + 400 + ks * 8, (i > 0 || ks >= ACCS) ? 1u : 0u);
      for (int c = 0; c < copies; ++c) tmem_cp_32x128b_x4(tmem + 448 + c * 4, cpd0 + (uint64_t)(c * 32));
    }
    tc_commit(&bars->drain);
    const bool ok = mbar_wait(&bars->drain, 0, status);
    cycles[blockIdx.x] = ok ? clock64() - t0 : -1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------ launchers
constexpr size_t kMmaCheckSmem = 36864 + sizeof(Barriers) + 1024;
constexpr size_t kMmaPeakSmem = 57344 + sizeof(Barriers) + 1024;

cudaError_t gemm_set_attributes() {
  cudaError_t err =
      cudaFuncSetAttribute((const void*)fc1_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)Fc1Cfg<1>::kSmem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute((const void*)fc1_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Fc1Cfg<2>::kSmem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute((const void*)fc2_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFc2Smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute((const void*)fc2_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)kFc2Smem);
  if (err != cudaSuccess) return err;
  for (const void* fn : {(const void*)mma_peak_kernel<1>, (const void*)mma_peak_kernel<2>,
                         (const void*)mma_peak_kernel<4>}) {
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kMmaPeakSmem);
    if (err != cudaSuccess) return err;
  }
  return cudaFuncSetAttribute((const void*)mma_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kMmaCheckSmem);
}

cudaError_t launch_fc1(const CUtensorMap& w13, const Fc1Args& a, int pair, int grid, cudaStream_t st) {
  CUtensorMap m0 = w13;
  Fc1Args args = a;
  void* kargs[] = {&m0, &args};
  if (pair == 2)
    return launch_with_pdl((const void*)fc1_kernel<2>, dim3(grid), dim3(kFc1Threads), Fc1Cfg<2>::kSmem, st, kargs);
  return launch_with_pdl((const void*)fc1_kernel<1>, dim3(grid), dim3(kFc1Threads), Fc1Cfg<1>::kSmem, st, kargs);
}

cudaError_t launch_fc2(const CUtensorMap& w2, const RowMaps& aq, const Fc2Args& a, int grid, cudaStream_t st) {
  CUtensorMap m0 = w2;
  RowMaps m1 = aq;
  Fc2Args args = a;
  void* kargs[] = {&m0, &m1, &args};
  const void* fn = a.kbs_per_stage > 1 ? (const void*)fc2_kernel<true> : (const void*)fc2_kernel<false>;
  return launch_with_pdl(fn, dim3(grid), dim3(kFc2Threads), kFc2Smem, st, kargs);
}

cudaError_t launch_mma_check(const CUtensorMap& a, const CUtensorMap& b, const uint8_t* sfa, const uint8_t* sfb,
                             int N, int K, float* d, int32_t* status, cudaStream_t st) {
  mma_check_kernel<<<1, 128, kMmaCheckSmem, st>>>(a, b, sfa, sfb, N, K, d, status);
  return cudaGetLastError();
}

cudaError_t launch_mma_peak(int grid, int n, int mmas, int copies, int accs, long long* cycles, int32_t* status,
                            cudaStream_t st) {
  if (accs == 4) mma_peak_kernel<4><<<grid, 128, kMmaPeakSmem, st>>>(n, mmas, copies, cycles, status);
  else if (accs == 2) mma_peak_kernel<2><<<grid, 128, kMmaPeakSmem, st>>>(n, mmas, copies, cycles, status);
  else mma_peak_kernel<1><<<grid, 128, kMmaPeakSmem, st>>>(n, mmas, copies, cycles, status);
  return cudaGetLastError();
}

}  // namespace moe
