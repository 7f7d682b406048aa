// gemm.cu -- the two block-scaled NVFP4 grouped GEMMs on tcgen05.
//
// Both kernels put the weights on the MMA's M side (128 weight rows per MMA)
// and the tokens routed to one expert on the N side (16..128 padded rows of
// the expert's segment), so one weight tile serves every token of the tile
// and decode-sized groups still fill the 128-row MMA.
//
// FC1 ("Cake SiTU backend": FC1 over gate and up, SiTU, intermediate NVFP4
// requantization): per work unit (token tile, intermediate tile of 128
// features) two accumulators D_g, D_u [128 features x N tokens] in TMEM
// collect K = H over k-blocks of 256 FP4 elements; the epilogue computes
// z = acc * dX*dW13[e], a = SiTU(z_g, z_u), and quantizes a per 16 features
// with qA[e] into the padded expanded rows of A (codes + atom-layout scales).
//
// FC2 ("Cake SiTU backend": FC2, BF16 weighted finalization): per work unit
// (token tile, 128 output features) one accumulator [128 x N] over K = I in
// k-blocks of 128; the epilogue scales by dA*dW2[e] and the route weight and
// adds the result into the fp32 [T, H] accumulator (one red per element).
//
// Warp roles (320 threads): warp 0 issues TMA, warp 1 owns TMEM and issues
// MMAs, warps 2..9 drain TMEM (two warps per 32-lane quarter, alternating
// 16-column chunks).  Persistent CTAs stride over the work units; the stage
// ring and the barrier phases carry across units.  Every wait is bounded.
#include "nvfp4.cuh"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

constexpr int kThreads = 320;
constexpr int kEpiWarps = 8;
constexpr uint32_t kTmemCols = 512;

// FC1 stage: A gate [128 x 128 B] | A up [128 x 128 B] | B [128 x 128 B] |
// SF gate 4 atoms | SF up 4 atoms | SF tokens 4 atoms.
constexpr int kFc1Stages = 4;
constexpr int F1_AG = 0, F1_AU = 16384, F1_B = 32768, F1_SG = 49152, F1_SU = 51200, F1_SB = 53248;
constexpr int kFc1StageBytes = 55296;
// FC2 stage: A [128 x 64 B] | B [128 x 64 B] | SF A 2 atoms | SF B 2 atoms.
constexpr int kFc2Stages = 12;
constexpr int F2_A = 0, F2_B = 8192, F2_SA = 16384, F2_SB = 17408;
constexpr int kFc2StageBytes = 18432;

struct Barriers {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t tmem_full[2];
  uint64_t tmem_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  volatile int32_t abort_flag;
};

constexpr size_t kFc1Smem = (size_t)kFc1Stages * kFc1StageBytes + sizeof(Barriers) + 1024;
constexpr size_t kFc2Smem = (size_t)kFc2Stages * kFc2StageBytes + sizeof(Barriers) + 1024;

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ uint64_t sf_desc(const uint8_t* p) { return smem_desc(smem_u32(p), 0, 128, kLayoutNone); }

template <int STAGES>
__device__ void gemm_setup(Barriers* bars, int warp) {
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->tmem_full[b], 1);
      mbar_init(&bars->tmem_empty[b], kEpiWarps);
    }
    mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
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

// A tile descriptor from the routing kernel is trusted only after a bounds
// check; a bad one is skipped by every role alike and flagged.
__device__ __forceinline__ bool tile_ok(const int4& t, int E, int64_t max_rows) {
  return t.x >= 0 && t.x < E && t.y >= 0 && (t.y & (kTileRows - 1)) == 0 && t.z >= 1 && t.z <= kTileRows &&
         (int64_t)t.y + t.z <= max_rows;
}

__device__ __forceinline__ int clamp_tiles(int n, int max_tiles) { return n < 0 ? 0 : (n > max_tiles ? max_tiles : n); }

// ================================================================== FC1
__global__ void __launch_bounds__(kThreads, 1)
    fc1_kernel(const __grid_constant__ CUtensorMap tm_w13, const __grid_constant__ CUtensorMap tm_xq,
               const Fc1Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kFc1Stages * kFc1StageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NIT = p.I / 128, NKB = p.H / kFc1KBlock;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w13);
    tma_prefetch_desc(&tm_xq);
  }
  gemm_setup<kFc1Stages>(bars, warp);
  const uint32_t tmem = bars->tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  const int num_units = clamp_tiles(p.hdr[HDR_NUM_TT], p.max_tiles) * NIT;
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, last_phase = 0;  // bit s: stage s armed; its last armed phase
      bool ok = true;
      for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
        const int4 tl = tiles[unit / NIT];
        const int it = unit % NIT;
        if (!tile_ok(tl, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
          continue;
        }
        const int e = tl.x, row0 = tl.y, rows = tl.z;
        const int nch = (rows + kTokChunk - 1) / kTokChunk;
        const uint32_t tx = 32768u + (uint32_t)nch * 2048u + 4096u + 2048u;
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * kFc1StageBytes;
          mbar_arrive_expect_tx(&bars->full[stage], tx);
          armed |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          tma_load_3d(st + F1_AG, &tm_w13, 0, 0, (e * NIT + it) * NKB + kb, &bars->full[stage]);
          for (int c = 0; c < nch; ++c)
            tma_load_2d(st + F1_B + c * 2048, &tm_xq, kb * 128, row0 + c * kTokChunk, &bars->full[stage]);
          bulk_g2s(st + F1_SG, p.sf13p + (size_t)((e * NIT + it) * NKB + kb) * 4096u, 4096u, &bars->full[stage]);
          bulk_g2s(st + F1_SB, p.sfx + ((size_t)(row0 >> 7) * (p.H / 64) + (size_t)kb * 4) * 512u, 2048u,
                   &bars->full[stage]);
          if (++stage == kFc1Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every issued copy has landed before the CTA may exit
      for (int s = 0; s < kFc1Stages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // --------------------------------------------------------------- MMA
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
        const int4 tl = tiles[unit / NIT];
        if (!tile_ok(tl, p.E, p.max_rows)) continue;
        const uint32_t ncols = (uint32_t)((tl.z + kTokChunk - 1) / kTokChunk * kTokChunk);
        const uint32_t idesc = idesc_mxf4nvf4(128, ncols);
        if (!wait_or_abort(&bars->tmem_empty[0], ((uint32_t)local & 1u) ^ 1u, bars, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->full[stage], phase, bars, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + stage * kFc1StageBytes;
          const uint32_t sfc = tmem + 256 + stage * 48;
#pragma unroll
          for (int a = 0; a < 4; ++a) {
            tmem_cp_32x128b_x4(sfc + a * 4, sf_desc(st + F1_SG + a * 512));
            tmem_cp_32x128b_x4(sfc + 16 + a * 4, sf_desc(st + F1_SU + a * 512));
            tmem_cp_32x128b_x4(sfc + 32 + a * 4, sf_desc(st + F1_SB + a * 512));
          }
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ag = smem_desc(smem_u32(st + F1_AG) + ks * 32, 16, 1024, kLayoutSW128);
            const uint64_t au = smem_desc(smem_u32(st + F1_AU) + ks * 32, 16, 1024, kLayoutSW128);
            const uint64_t bd = smem_desc(smem_u32(st + F1_B) + ks * 32, 16, 1024, kLayoutSW128);
            const uint32_t acc = (kb | ks) ? 1u : 0u;
            mma_mxf4nvf4(tmem + 0, ag, bd, idesc, sfc + ks * 4, sfc + 32 + ks * 4, acc);
            mma_mxf4nvf4(tmem + 128, au, bd, idesc, sfc + 16 + ks * 4, sfc + 32 + ks * 4, acc);
          }
          tc_commit(&bars->empty[stage]);
          if (++stage == kFc1Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&bars->tmem_full[0]);
        ++local;
      }
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.status);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    const int I2 = p.I / 2, KC = p.I / 16;
    int local = 0;
    for (int unit = blockIdx.x; unit < num_units; unit += gridDim.x) {
      const int4 tl = tiles[unit / NIT];
      if (!tile_ok(tl, p.E, p.max_rows)) continue;
      const int it = unit % NIT;
      const int e = tl.x, row0 = tl.y, rows = tl.z;
      if (!wait_or_abort(&bars->tmem_full[0], (uint32_t)local & 1u, bars, p.status)) break;
      tc_fence_after();
      const float s13 = __ldg(p.dXdW13 + e), qa = __ldg(p.qA + e);
      const float be = __ldg(p.beta + e), la = __ldg(p.lam + e);
      const int nch = (rows + kTokChunk - 1) / kTokChunk;
      const int feat = it * 128 + q * 32 + lane;  // intermediate feature of this lane
      for (int c = half; c < nch; c += 2) {
        uint32_t rg[16], ru[16];
        tmem_ld16(tmem + lane_base + c * 16, rg);
        tmem_ld16(tmem + lane_base + 128 + c * 16, ru);
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int n = c * 16 + cc;
          if (n < rows) {
            const float g = __fmul_rn(__uint_as_float(rg[cc]), s13);
            const float u = __fmul_rn(__uint_as_float(ru[cc]), s13);
            const float act = situ_f32(g, u, be, la);
            uint32_t word;
            const uint32_t sf = nvfp4_quant_lanes16(act, qa, word);
            const int64_t prow = row0 + n;
            if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(p.aq + (size_t)prow * I2 + feat / 2) = word;
            if ((lane & 15) == 0) p.sfa[atom_offset(prow, feat / 16, KC)] = (uint8_t)sf;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tmem_empty[0]);
      ++local;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ================================================================== FC2
__global__ void __launch_bounds__(kThreads, 1)
    fc2_kernel(const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_aq,
               const Fc2Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  Barriers* bars = reinterpret_cast<Barriers*>(smem + kFc2Stages * kFc2StageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NMT = p.H / 128, NKB = p.I / kFc2KBlock, NA = p.I / 64;
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w2);
    tma_prefetch_desc(&tm_aq);
  }
  gemm_setup<kFc2Stages>(bars, warp);
  const uint32_t tmem = bars->tmem_base;
  pdl_wait();
  pdl_launch_dependents();
  const int num_units = clamp_tiles(p.hdr[HDR_NUM_TT], p.max_tiles) * NMT;
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      uint32_t armed = 0, last_phase = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
        const int4 tl = tiles[unit / NMT];
        if (!tile_ok(tl, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
          continue;
        }
        const int mt = unit % NMT;
        const int e = tl.x, row0 = tl.y, rows = tl.z;
        const int nch = (rows + kTokChunk - 1) / kTokChunk;
        const uint32_t tx = 8192u + (uint32_t)nch * 1024u + 1024u + 1024u;
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
            ok = false;
            break;
          }
          uint8_t* st = smem + stage * kFc2StageBytes;
          mbar_arrive_expect_tx(&bars->full[stage], tx);
          armed |= 1u << stage;
          last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
          tma_load_3d(st + F2_A, &tm_w2, 0, 0, (e * NMT + mt) * NKB + kb, &bars->full[stage]);
          for (int c = 0; c < nch; ++c)
            tma_load_2d(st + F2_B + c * 1024, &tm_aq, kb * 64, row0 + c * kTokChunk, &bars->full[stage]);
          bulk_g2s(st + F2_SA, p.sf2p + ((size_t)(e * NMT + mt) * NA + (size_t)kb * 2) * 512u, 1024u,
                   &bars->full[stage]);
          bulk_g2s(st + F2_SB, p.sfa + ((size_t)(row0 >> 7) * NA + (size_t)kb * 2) * 512u, 1024u,
                   &bars->full[stage]);
          if (++stage == kFc2Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < kFc2Stages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int unit = blockIdx.x; unit < num_units && ok; unit += gridDim.x) {
        const int4 tl = tiles[unit / NMT];
        if (!tile_ok(tl, p.E, p.max_rows)) continue;
        const uint32_t ncols = (uint32_t)((tl.z + kTokChunk - 1) / kTokChunk * kTokChunk);
        const uint32_t idesc = idesc_mxf4nvf4(128, ncols);
        const uint32_t buf = (uint32_t)local & 1u;
        if (!wait_or_abort(&bars->tmem_empty[buf], (((uint32_t)local >> 1) & 1u) ^ 1u, bars, p.status)) break;
        tc_fence_after();
        const uint32_t dcol = tmem + buf * 128;
        for (int kb = 0; kb < NKB; ++kb) {
          if (!wait_or_abort(&bars->full[stage], phase, bars, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + stage * kFc2StageBytes;
          const uint32_t sfc = tmem + 256 + stage * 16;
#pragma unroll
          for (int a = 0; a < 2; ++a) {
            tmem_cp_32x128b_x4(sfc + a * 4, sf_desc(st + F2_SA + a * 512));
            tmem_cp_32x128b_x4(sfc + 8 + a * 4, sf_desc(st + F2_SB + a * 512));
          }
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) {
            const uint64_t ad = smem_desc(smem_u32(st + F2_A) + ks * 32, 16, 512, kLayoutSW64);
            const uint64_t bd = smem_desc(smem_u32(st + F2_B) + ks * 32, 16, 512, kLayoutSW64);
            mma_mxf4nvf4(dcol, ad, bd, idesc, sfc + ks * 4, sfc + 8 + ks * 4, (kb | ks) ? 1u : 0u);
          }
          tc_commit(&bars->empty[stage]);
          if (++stage == kFc2Stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&bars->tmem_full[buf]);
        ++local;
      }
      tc_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, p.status);
    }
  } else {
    const int q = warp & 3, half = (warp - 2) >> 2;
    const uint32_t lane_base = (uint32_t)(q * 32) << 16;
    int local = 0;
    for (int unit = blockIdx.x; unit < num_units; unit += gridDim.x) {
      const int4 tl = tiles[unit / NMT];
      if (!tile_ok(tl, p.E, p.max_rows)) continue;
      const int mt = unit % NMT;
      const int e = tl.x, row0 = tl.y, rows = tl.z;
      const uint32_t buf = (uint32_t)local & 1u;
      if (!wait_or_abort(&bars->tmem_full[buf], ((uint32_t)local >> 1) & 1u, bars, p.status)) break;
      tc_fence_after();
      const float s2 = __ldg(p.dAdW2 + e);
      const int nch = (rows + kTokChunk - 1) / kTokChunk;
      const int h = mt * 128 + q * 32 + lane;
      for (int c = half; c < nch; c += 2) {
        uint32_t r[16];
        tmem_ld16(tmem + lane_base + buf * 128 + c * 16, r);
        int pair = -1;
        float wgt = 0.0f;
        if (lane < 16 && c * 16 + lane < rows) {
          pair = p.prow_pair[row0 + c * 16 + lane];
          if (pair >= 0 && pair < p.num_pairs) wgt = bf16_bits_to_f32(p.route_w[pair]);
        }
        tmem_ld_wait();
#pragma unroll
        for (int cc = 0; cc < 16; ++cc) {
          const int pr = __shfl_sync(0xffffffffu, pair, cc);
          const float wv = __shfl_sync(0xffffffffu, wgt, cc);
          if (c * 16 + cc < rows && pr >= 0 && pr < p.num_pairs) {
            const float y = __fmul_rn(__uint_as_float(r[cc]), s2);
            atomicAdd(p.out_f32 + (size_t)(pr / p.k) * p.H + h, __fmul_rn(y, wv));
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->tmem_empty[buf]);
      ++local;
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

// ------------------------------------------------------------------ launchers
constexpr size_t kMmaCheckSmem = 36864 + sizeof(Barriers) + 1024;

cudaError_t gemm_set_attributes() {
  cudaError_t err =
      cudaFuncSetAttribute((const void*)fc1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFc1Smem);
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute((const void*)fc2_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFc2Smem);
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute((const void*)mma_check_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kMmaCheckSmem);
}

cudaError_t launch_fc1(const CUtensorMap& w13, const CUtensorMap& xq, const Fc1Args& a, int grid, cudaStream_t st) {
  CUtensorMap m0 = w13, m1 = xq;
  Fc1Args args = a;
  void* kargs[] = {&m0, &m1, &args};
  return launch_with_pdl((const void*)fc1_kernel, dim3(grid), dim3(kThreads), kFc1Smem, st, kargs);
}

cudaError_t launch_fc2(const CUtensorMap& w2, const CUtensorMap& aq, const Fc2Args& a, int grid, cudaStream_t st) {
  CUtensorMap m0 = w2, m1 = aq;
  Fc2Args args = a;
  void* kargs[] = {&m0, &m1, &args};
  return launch_with_pdl((const void*)fc2_kernel, dim3(grid), dim3(kThreads), kFc2Smem, st, kargs);
}

cudaError_t launch_mma_check(const CUtensorMap& a, const CUtensorMap& b, const uint8_t* sfa, const uint8_t* sfb,
                             int N, int K, float* d, int32_t* status, cudaStream_t st) {
  mma_check_kernel<<<1, 128, kMmaCheckSmem, st>>>(a, b, sfa, sfb, N, K, d, status);
  return cudaGetLastError();
}

}  // namespace moe
