// routing.cu -- init-routing kernels: stable counting sort of expert ids,
// expanded row index in gather and scatter form, per-expert histogram and
// inclusive cumsum, padded per-expert row offsets and the token-tile list the
// grouped GEMMs run over; plus the token move of the standalone init-routing
// (dynamic int8 quant, drop/pad).
//
// Definitions ("npu_moe_init_routing_v2", section 计算公式):
//   formula 1  sortedExpertIdx, sortedRowIdx = keyValueSort(expertIdx, rowIdx)
//              with rowIdx = t*k + j; the sort is stable (ties by rowIdx).
//   formula 2  scatter form expandedRowIdx[i] = sortedRowIdx[i];
//              gather form expandedRowIdx[sortedRowIdx[i]] = i.
//   formula 3  per-expert histogram of sortedExpertIdx.
//   formula 4  dynamic quant: scale = row_max(|x|)/127, q = round(x/scale).
//   formula 5  expandedX[i] = x[sortedRowIdx[i] // k] (drop/pad: pad every
//              expert to expertCapacity rows, drop the excess, zero-fill).
//
// Sorting method: each warp owns a contiguous run of pairs and walks it 32 at
// a time in order.  Pass 1 counts its pairs per expert in a private shared-
// memory histogram (warp match groups lanes with equal ids, the group leader
// adds the group size).  The per-(block, warp, expert) exclusive prefixes plus
// the per-expert offsets give every warp the first sorted slot of each
// expert; pass 2 walks the same run again and hands out slots in order
// (base + number of equal-id lanes below).  Walking runs in order makes the
// result stable without any comparison sort.
#include "nvfp4.cuh"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// The ids of a warp's run are loaded kIdBatch steps of 32 at a time, all in
// flight together, and then processed step by step in order.
constexpr int kIdBatch = 8;

// Pass 1: per-warp histogram of ids[begin, end) into hist_w[E] (shared).
// Counts do not depend on order, so each lane adds its own pair with a
// shared-memory atomic.
__device__ __forceinline__ void warp_histogram(const int32_t* ids, int64_t begin, int64_t end, int E,
                                               int* hist_w, int id_base) {
  const int lane = threadIdx.x & 31;
  for (int64_t base0 = begin; base0 < end; base0 += 32 * kIdBatch) {
    int raw[kIdBatch];
#pragma unroll
    for (int j = 0; j < kIdBatch; ++j) {
      const int64_t f = base0 + j * 32 + lane;
      raw[j] = f < end ? ids[f] : id_base - 1;   // generic load: ids may be in shared memory
    }
#pragma unroll
    for (int j = 0; j < kIdBatch; ++j) {
      const int id = raw[j] - id_base;
      if (id >= 0 && id < E) atomicAdd(hist_w + id, 1);
    }
  }
}

// Pass 2: hand out sorted slots.  base_w[e] holds the next slot of expert e
// for this warp, counted from the expert's first row when kRelative (else
// absolute); offs/poffs are the expert's first dropless / padded row.
template <bool kRelative>
__device__ __forceinline__ int warp_rank(const RouteArgs& a, const int32_t* ids, int64_t begin, int64_t end,
                                         int* base_w, const int* s_offs, const int* s_poffs) {
  const int lane = threadIdx.x & 31;
  int invalid = 0;
  for (int64_t base0 = begin; base0 < end; base0 += 32 * kIdBatch) {
   int rawb[kIdBatch];
#pragma unroll
   for (int j = 0; j < kIdBatch; ++j) {
     const int64_t f = base0 + j * 32 + lane;
     rawb[j] = f < end ? ids[f] : -1;   // generic load: ids may be in shared memory
   }
#pragma unroll
   for (int j = 0; j < kIdBatch; ++j) {
    if (base0 + j * 32 >= end) break;   // warp-uniform: the run is done
    const int64_t f = base0 + j * 32 + lane;
    const bool in = f < end;
    const int raw = in ? rawb[j] : -1;
    const int id = raw - a.id_base;
    const bool ok = in && id >= 0 && id < a.E;
    const uint32_t okmask = __ballot_sync(0xffffffffu, ok);
    if (ok) {
      const uint32_t peers = __match_any_sync(okmask, id);
      const int leader = __ffs(peers) - 1;
      const int rank = base_w[id] + __popc(peers & lanemask_lt());   // within the expert (kRelative) or absolute
      __syncwarp(okmask);
      if (lane == leader) base_w[id] += __popc(peers);
      const int slot = kRelative ? s_offs[id] + rank : rank;
      a.sorted_row[slot] = (int32_t)f;
      a.gather[f] = slot;
      const int prow = s_poffs[id] + (slot - s_offs[id]);
      a.row_pos[f] = prow;
      a.prow_pair[prow] = (int32_t)f;
    } else if (in) {
      a.gather[f] = -1;
      a.row_pos[f] = -1;
      if (raw < 0 || raw >= a.E_all) ++invalid;   // outside every expert; in-range ids outside E are skipped silently
    }
    __syncwarp();
   }
  }
  return invalid;
}

// Block-wide exclusive scan of (count, padded count, tile count) over experts
// and the tile list.  cnt_s[E] holds the counts on entry; on exit s_offs and
// s_poffs hold the dropless / padded first rows.  NT threads, E <= NT * 4.
template <int NT>
__device__ void scan_experts(const RouteArgs& a, const int* cnt_s, int* s_offs, int* s_poffs, int* s_tmp) {
  constexpr int NWARP = NT / 32;
  constexpr int PER = (kMaxExperts + NT - 1) / NT;   // experts per thread, at most
  static_assert(PER <= 4, "E <= NT * 4");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int E = a.E;
  const int per = (E + NT - 1) / NT;  // experts per thread (consecutive)
  const int e0 = tid * per;
  int c[PER];
  int v0 = 0, v1 = 0, v2 = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = e0 + i;
    const int n = (i < per && e < E) ? cnt_s[e] : 0;
    c[i] = n;
    v0 += n;
    v1 += (n + kTileRows - 1) / kTileRows * kTileRows;
    v2 += (n + kTileRows - 1) / kTileRows;
  }
  int i0 = v0, i1 = v1, i2 = v2;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t0 = __shfl_up_sync(0xffffffffu, i0, off);
    const int t1 = __shfl_up_sync(0xffffffffu, i1, off);
    const int t2 = __shfl_up_sync(0xffffffffu, i2, off);
    if (lane >= off) {
      i0 += t0;
      i1 += t1;
      i2 += t2;
    }
  }
  if (lane == 31) {
    s_tmp[warp * 3 + 0] = i0;
    s_tmp[warp * 3 + 1] = i1;
    s_tmp[warp * 3 + 2] = i2;
  }
  int mx = 0;   // largest expert group, for the GEMMs' accumulator sizing
#pragma unroll
  for (int i = 0; i < PER; ++i) mx = max(mx, c[i]);
  mx = __reduce_max_sync(0xffffffffu, mx);
  if (lane == 0) s_tmp[208 + warp] = mx;
  __syncthreads();
  if (warp == 0) {
    int w0 = lane < NWARP ? s_tmp[lane * 3 + 0] : 0;
    int w1 = lane < NWARP ? s_tmp[lane * 3 + 1] : 0;
    int w2 = lane < NWARP ? s_tmp[lane * 3 + 2] : 0;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t0 = __shfl_up_sync(0xffffffffu, w0, off);
      const int t1 = __shfl_up_sync(0xffffffffu, w1, off);
      const int t2 = __shfl_up_sync(0xffffffffu, w2, off);
      if (lane >= off) {
        w0 += t0;
        w1 += t1;
        w2 += t2;
      }
    }
    if (lane < NWARP) {
      s_tmp[96 + lane * 3 + 0] = w0;
      s_tmp[96 + lane * 3 + 1] = w1;
      s_tmp[96 + lane * 3 + 2] = w2;
    }
  }
  __syncthreads();
  const int wb0 = warp ? s_tmp[96 + (warp - 1) * 3 + 0] : 0;
  const int wb1 = warp ? s_tmp[96 + (warp - 1) * 3 + 1] : 0;
  const int wb2 = warp ? s_tmp[96 + (warp - 1) * 3 + 2] : 0;
  int o0 = wb0 + i0 - v0, o1 = wb1 + i1 - v1, o2 = wb2 + i2 - v2;  // exclusive
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int e = e0 + i;
    if (i < per && e < E) {
      const int n = c[i];
      const int nt = (n + kTileRows - 1) / kTileRows;
      s_offs[e] = o0;
      s_poffs[e] = o1;
      a.count[e] = n;
      a.cumsum[e] = o0 + n;
      a.offs[e] = o0;
      a.poffs[e] = o1;
      a.ttoffs[e] = o2;
      int4* tl = reinterpret_cast<int4*>(a.tt_list);
      for (int j = 0; j < nt; ++j) {
        const int rows = min(kTileRows, n - j * kTileRows);
        tl[o2 + j] = make_int4(e, o1 + j * kTileRows, rows, 0);
      }
      o0 += n;
      o1 += nt * kTileRows;
      o2 += nt;
    }
  }
  if (tid == NT - 1) {
    // the last thread's running sums are the grand totals
    a.offs[E] = o0;
    a.poffs[E] = o1;
    a.ttoffs[E] = o2;
    a.hdr[HDR_NVALID] = o0;
    a.hdr[HDR_PPAD] = o1;
    a.hdr[HDR_NUM_TT] = o2;
    a.hdr[HDR_FC2_NEXT] = 0;   // the GEMMs' work counters start over on every call
    a.hdr[HDR_FC1_NEXT] = 0;
    int m = 0;
    for (int w = 0; w < NWARP; ++w) m = max(m, s_tmp[208 + w]);
    a.hdr[HDR_MAXROWS] = m;
    s_tmp[200] = o0;
  }
  __syncthreads();
}

// The preparation stamp written by moe_prepare_workspace.  A workspace whose
// header does not hold it (memory an allocator handed back at the address of
// a workspace prepared earlier, or never prepared) is left alone: the call
// records DEVSTAT_NOT_PREPARED and zeroes the tile and row counts, so every
// later kernel of the call finds nothing to do.
__device__ __forceinline__ bool stamp_bad(const RouteArgs& a) {
  if (!a.check_stamp) return false;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kStampWords; ++i) bad |= __ldcg(a.hdr + HDR_STAMP + i) != a.stamp[i];
  return bad;
}

__device__ __forceinline__ void mark_not_prepared(const RouteArgs& a) {
  a.hdr[HDR_NUM_TT] = 0;
  a.hdr[HDR_PPAD] = 0;
  a.hdr[HDR_NVALID] = 0;
  a.hdr[HDR_MAXROWS] = 0;
  a.hdr[HDR_FC2_NEXT] = 0;
  a.hdr[HDR_FC1_NEXT] = 0;
  a.hdr[HDR_SKIP] = 1;
  atomicOr(a.hdr + HDR_STATUS, DEVSTAT_NOT_PREPARED);
}

// ---------------------------------------------------------------- small path
// One CTA of 1024 threads sorts up to kRouteSmallMax pairs in one launch.
// The ids are staged in shared memory once; as many warps as there are
// 32-pair chunks (at most 32) keep per-warp histograms.
__global__ void __launch_bounds__(1024, 1) route_small_kernel(const RouteArgs a) {
  extern __shared__ int sm[];
  const int E = a.E;
  const int NHW = a.P >= 1024 ? 32 : (int)((a.P + 31) / 32 > 0 ? (a.P + 31) / 32 : 1);   // histogram warps
  int* hist = sm;                  // [NHW][E]
  int* s_cnt = hist + NHW * E;     // [E]
  int* s_offs = s_cnt + E;         // [E]
  int* s_poffs = s_offs + E;       // [E]
  int* s_tmp = s_poffs + E;        // [256]
  int* s_ids = s_tmp + 256;        // [P]
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  __shared__ int s_bad;
  if (tid == 0) {
    s_bad = stamp_bad(a);
    if (s_bad) mark_not_prepared(a);
    else a.hdr[HDR_SKIP] = 0;
  }
  __syncthreads();
  if (s_bad) return;
  for (int i = tid; i < NHW * E; i += 1024) hist[i] = 0;
  for (int64_t i = tid; i < a.P; i += 1024) s_ids[i] = __ldg(a.ids + i);
  __syncthreads();
  const int64_t per = (a.P + NHW - 1) / NHW;
  const int64_t b = min(a.P, (int64_t)warp * per), en = min(a.P, b + per);
  if (warp < NHW) warp_histogram(s_ids, b, en, E, hist + warp * E, a.id_base);
  __syncthreads();
  for (int e = tid; e < E; e += 1024) {
    int run = 0;
    for (int w = 0; w < NHW; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    s_cnt[e] = run;
  }
  __syncthreads();
  scan_experts<1024>(a, s_cnt, s_offs, s_poffs, s_tmp);   // ends with a block barrier
  const int invalid = warp < NHW ? warp_rank<true>(a, s_ids, b, en, hist + warp * E, s_offs, s_poffs) : 0;
  const int nvalid = s_tmp[200];
  for (int64_t i = nvalid + tid; i < a.P; i += 1024) a.sorted_row[i] = -1;
  if (invalid) {
    atomicAdd(&a.hdr[HDR_INVALID], invalid);
    atomicOr(&a.hdr[HDR_STATUS], DEVSTAT_INVALID_EXPERT);
  }
}

// ---------------------------------------------------------------- large path
// Kernel 1: per-block histograms; the last block to finish (ticket counter,
// no waiting) scans them into per-(block, expert) bases and per-expert
// offsets, and writes the tile list.  256 threads, a.chunk pairs per block.
__global__ void __launch_bounds__(256) route_hist_kernel(const RouteArgs a) {
  extern __shared__ int sm[];
  const int E = a.E;
  int* hist = sm;                 // [8][E]
  int* s_cnt = hist + 8 * E;      // [E]
  int* s_offs = s_cnt + E;        // [E]
  int* s_poffs = s_offs + E;      // [E]
  int* s_tmp = s_poffs + E;       // [256]
  __shared__ int s_last, s_bad;
  const int tid = threadIdx.x, warp = tid >> 5;
  pdl_wait();
  pdl_launch_dependents();
  if (tid == 0) {
    s_bad = stamp_bad(a);
    if (blockIdx.x == 0) {
      if (s_bad) mark_not_prepared(a);
      else a.hdr[HDR_SKIP] = 0;
    }
  }
  __syncthreads();
  if (s_bad) return;   // before the ticket, which a foreign header does not hold at zero
  for (int i = tid; i < 8 * E; i += 256) hist[i] = 0;
  __syncthreads();
  const int64_t cb = (int64_t)blockIdx.x * a.chunk;
  const int64_t wb = cb + (int64_t)warp * (a.chunk / 8);
  warp_histogram(a.ids, min(wb, a.P), min(wb + a.chunk / 8, a.P), E, hist + warp * E, a.id_base);
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int s = 0;
    for (int w = 0; w < 8; ++w) s += hist[w * E + e];
    a.blockhist[(size_t)blockIdx.x * E + e] = s;
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = (atomicAdd(&a.hdr[HDR_DONE], 1) == a.nblk - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // Each thread scans the block counts of experts tid + 256 j (j < 4; E <=
  // 1024 here), 32 blocks at a time: 128 independent loads in flight per step.
  {
    int run[4] = {0, 0, 0, 0};
    for (int blk0 = 0; blk0 < a.nblk; blk0 += 32) {
      int c[4][32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const bool inb = blk0 + j < a.nblk;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = tid + 256 * q;
          c[q][j] = inb && e < E ? __ldcg(&a.blockhist[(size_t)(blk0 + j) * E + e]) : 0;
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int e = tid + 256 * q;
          if (blk0 + j < a.nblk && e < E) a.blockhist[(size_t)(blk0 + j) * E + e] = run[q];
          run[q] += c[q][j];
        }
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (tid + 256 * q < E) s_cnt[tid + 256 * q] = run[q];
  }
  __syncthreads();
  scan_experts<256>(a, s_cnt, s_offs, s_poffs, s_tmp);
}

// Kernel 2: every block recounts its pairs per warp and hands out slots.
__global__ void __launch_bounds__(256) route_rank_kernel(const RouteArgs a) {
  extern __shared__ int sm[];
  const int E = a.E;
  int* hist = sm;                 // [8][E]
  int* s_offs = hist + 8 * E;     // [E]
  int* s_poffs = s_offs + E;      // [E]
  const int tid = threadIdx.x, warp = tid >> 5;
  // The X quantization may start at once: this kernel itself starts only
  // after the histogram kernel has waited for the previous forward, and
  // the quantization reads nothing that routing writes before its own wait.
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_bad;
  if (tid == 0) s_bad = stamp_bad(a);
  __syncthreads();
  if (s_bad) return;
  if (blockIdx.x == 0 && tid == 0) a.hdr[HDR_DONE] = 0;  // re-arm the ticket for the next call
  for (int i = tid; i < 8 * E; i += 256) hist[i] = 0;
  for (int e = tid; e < E; e += 256) {
    s_offs[e] = a.offs[e];
    s_poffs[e] = a.poffs[e];
  }
  __syncthreads();
  const int64_t cb = (int64_t)blockIdx.x * a.chunk;
  const int64_t wb = cb + (int64_t)warp * (a.chunk / 8);
  const int64_t b = min(wb, a.P), en = min(wb + a.chunk / 8, a.P);
  warp_histogram(a.ids, b, en, E, hist + warp * E, a.id_base);
  __syncthreads();
  for (int e = tid; e < E; e += 256) {
    int run = s_offs[e] + a.blockhist[(size_t)blockIdx.x * E + e];
    for (int w = 0; w < 8; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  const int invalid = warp_rank<false>(a, a.ids, b, en, hist + warp * E, s_offs, s_poffs);
  const int nvalid = a.offs[E];
  const int64_t t0 = max((int64_t)nvalid, cb), t1 = min(a.P, cb + a.chunk);
  for (int64_t i = t0 + tid; i < t1; i += 256) a.sorted_row[i] = -1;
  if (invalid) {
    atomicAdd(&a.hdr[HDR_INVALID], invalid);
    atomicOr(&a.hdr[HDR_STATUS], DEVSTAT_INVALID_EXPERT);
  }
}

// -------------------------------------------------------- init-routing move
// One warp per token: dynamic int8 quant of the row (formula 4), static int8
// with the scalar scale and offset (formula 3), or a bf16
// copy, written to each destination row of the token's pairs (formula 5).
__global__ void __launch_bounds__(256) init_move_kernel(const InitMoveArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  pdl_wait();
  pdl_launch_dependents();
  if (t >= a.T || a.hdr[HDR_SKIP]) return;
  const uint16_t* xr = a.x + t * a.H;
  int dest = -1;
  if (lane < a.k) {
    const int64_t f = t * a.k + lane;
    const int i = a.gather[f];
    if (i >= 0) {
      if (!a.drop_pad) {
        dest = i;
      } else {
        const int e = a.ids[f];
        const int r = i - a.offs[e];
        dest = (r < a.C) ? e * a.C + r : -1;
      }
    }
    if (a.row_idx_type == 0) a.expanded_row_idx[f] = dest;
  }
  const int nvec = a.H / 8;  // 8 bf16 per 16-byte vector
  const uint4* xv = reinterpret_cast<const uint4*>(xr);
  if (a.quant_mode == 1) {
    float amax = 0.0f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[i] & 0xFFFFu)));
        amax = fmaxf(amax, fabsf(bf16_bits_to_f32(w[i] >> 16)));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t q[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
        int qi = 0;
        if (s != 0.0f) {
          float y = rintf(__fdiv_rn(bf16_bits_to_f32(bits), s));
          y = fminf(fmaxf(y, -127.0f), 127.0f);
          qi = (int)y;
        }
        q[i >> 2] |= ((uint32_t)qi & 0xFFu) << (8 * (i & 3));
      }
      for (int j = 0; j < a.k; ++j) {
        const int d = __shfl_sync(0xffffffffu, dest, j);
        if (d >= 0)
          *reinterpret_cast<uint2*>(static_cast<int8_t*>(a.expanded_x) + (int64_t)d * a.H + v * 8) =
              make_uint2(q[0], q[1]);
      }
    }
    for (int j = 0; j < a.k; ++j) {
      const int d = __shfl_sync(0xffffffffu, dest, j);
      if (d >= 0 && lane == 0 && a.expanded_scale) a.expanded_scale[d] = s;
    }
  } else if (a.quant_mode == 0) {
    // static int8: q = rint(x*scale + offset) in fp32, saturated to [-128, 127]
    const float sc = __ldg(a.scale), of = __ldg(a.offset);
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      uint32_t q[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t bits = (i & 1) ? (w[i >> 1] >> 16) : (w[i >> 1] & 0xFFFFu);
        float y = rintf(__fadd_rn(__fmul_rn(bf16_bits_to_f32(bits), sc), of));
        y = fminf(fmaxf(y, -128.0f), 127.0f);
        q[i >> 2] |= ((uint32_t)(int)y & 0xFFu) << (8 * (i & 3));
      }
      for (int j = 0; j < a.k; ++j) {
        const int d = __shfl_sync(0xffffffffu, dest, j);
        if (d >= 0)
          *reinterpret_cast<uint2*>(static_cast<int8_t*>(a.expanded_x) + (int64_t)d * a.H + v * 8) =
              make_uint2(q[0], q[1]);
      }
    }
  } else {
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      for (int j = 0; j < a.k; ++j) {
        const int d = __shfl_sync(0xffffffffu, dest, j);
        if (d >= 0) reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.expanded_x) + (int64_t)d * a.H)[v] = u;
      }
    }
  }
}

// Row-driven move ("npu_moe_init_routing_v2", formula 5 in scatter form:
// expandedX[i] = quantResult[scatterRowIdx[i] // K]), for every option: one
// warp per sorted position i of a routed pair; the row goes to position i
// (dropless, i < the Active limit) or to slot e*C + rank (drop/pad).
//   quant -1: bf16 copy; with a [T] scale the row's scale is its token's
//   quant  0: q = rint(x*scale + offset) in fp32, saturated to [-128, 127]
//   quant  1: xs = x * smooth row (of the pair's expert, or the one shared
//             row, or 1); s = row_max|xs| / 127; q = rint(xs / s), +-127
__global__ void __launch_bounds__(256) init_rows_kernel(const InitRowsArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  if (a.hdr[HDR_SKIP]) return;
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * 256 + threadIdx.x) >> 5, nw = ((int64_t)gridDim.x * 256) >> 5;
  const int64_t avail = a.hdr[HDR_NVALID];
  const int64_t nmove = (!a.drop_pad && a.active_num > 0 && a.active_num < avail) ? a.active_num : avail;
  const int nvec = a.H / 8;   // 8 bf16 per 16-byte vector
  for (int64_t i = w0; i < nmove; i += nw) {
    const int f = a.sorted_row[i];
    const int e = a.ids[f] - a.id_base;
    int64_t dest = i;
    if (a.drop_pad) {
      const int r = (int)(i - (a.cumsum[e] - a.count[e]));
      if (r >= a.C) continue;
      dest = (int64_t)e * a.C + r;
    }
    const int64_t t = f / a.k;
    const uint4* xv = reinterpret_cast<const uint4*>(a.x + t * a.H);
    if (a.quant_mode == -1) {
      uint4* dv = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.expanded_x) + dest * a.H);
      for (int v = lane; v < nvec; v += 32) dv[v] = __ldg(xv + v);
      if (lane == 0 && a.scale && a.expanded_scale) a.expanded_scale[dest] = __ldg(a.scale + t);
      continue;
    }
    int8_t* drow = static_cast<int8_t*>(a.expanded_x) + dest * a.H;
    if (a.quant_mode == 0) {
      const float sc = __ldg(a.scale), of = __ldg(a.offset);
      for (int v = lane; v < nvec; v += 32) {
        const uint4 u = __ldg(xv + v);
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
        uint32_t q[2] = {0u, 0u};
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t bits = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu);
          float y = rintf(__fadd_rn(__fmul_rn(bf16_bits_to_f32(bits), sc), of));
          y = fminf(fmaxf(y, -128.0f), 127.0f);
          q[j >> 2] |= ((uint32_t)(int)y & 0xFFu) << (8 * (j & 3));
        }
        *reinterpret_cast<uint2*>(drow + v * 8) = make_uint2(q[0], q[1]);
      }
      continue;
    }
    const float* sm = (a.scale && a.scale_rows > 0) ? a.scale + (a.scale_rows == 1 ? 0 : (int64_t)e) * a.H : nullptr;
    float amax = 0.0f;
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t bits = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu);
        float x = bf16_bits_to_f32(bits);
        if (sm) x = __fmul_rn(x, __ldg(sm + v * 8 + j));
        amax = fmaxf(amax, fabsf(x));
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.0f);
    for (int v = lane; v < nvec; v += 32) {
      const uint4 u = __ldg(xv + v);
      const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
      uint32_t q[2] = {0u, 0u};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t bits = (j & 1) ? (wd[j >> 1] >> 16) : (wd[j >> 1] & 0xFFFFu);
        float x = bf16_bits_to_f32(bits);
        if (sm) x = __fmul_rn(x, __ldg(sm + v * 8 + j));
        int qi = 0;
        if (s != 0.0f) qi = (int)fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
        q[j >> 2] |= ((uint32_t)qi & 0xFFu) << (8 * (j & 3));
      }
      *reinterpret_cast<uint2*>(drow + v * 8) = make_uint2(q[0], q[1]);
    }
    if (lane == 0 && a.expanded_scale) a.expanded_scale[dest] = s;
  }
}

// Histogram output (formula 3: inclusive cumsum or count over the routed
// experts, or key_value rows), expanded_row_idx in scatter form (formula 2)
// or -- after a row-driven move -- in gather form, availableIdxNum (formula
// 6), and the zero fill of unfilled drop/pad slots.
static_assert(4 * 256 >= kMaxExperts, "init_finish: four experts per thread of one 256-thread block");
__global__ void __launch_bounds__(256) init_finish_kernel(const InitFinishArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  if (a.hdr[HDR_SKIP]) return;
  const int64_t gtid = (int64_t)blockIdx.x * 256 + threadIdx.x;
  const int64_t nthr = (int64_t)gridDim.x * 256;
  const int64_t avail = a.hdr[HDR_NVALID];
  if (a.tokens_num_type == 2) {
    // key_value: (expert id, count) of the routed experts with a non-zero
    // count, in expert order, then zeros.  Thread t holds experts 4t..4t+3
    // (E <= 1024); a block scan of the non-zero flags places each pair.
    if (blockIdx.x == 0) {
      __shared__ int s_warp[8];
      const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
      int cnt[4], nz = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int e = 4 * tid + j;
        cnt[j] = e < a.E ? a.count[e] : 0;
        nz += cnt[j] > 0 ? 1 : 0;
      }
      int incl = nz;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
      }
      if (lane == 31) s_warp[warp] = incl;
      __syncthreads();
      int before = 0, n = 0;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        before += w < warp ? s_warp[w] : 0;
        n += s_warp[w];
      }
      int pos = before + incl - nz;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (cnt[j] > 0) {
          a.tokens_out[2 * pos] = a.id_base + 4 * tid + j;
          a.tokens_out[2 * pos + 1] = cnt[j];
          ++pos;
        }
      for (int64_t j = 2 * (int64_t)n + tid; j < 2 * (int64_t)a.E_all; j += 256) a.tokens_out[j] = 0;
    }
  } else {
    for (int64_t e = gtid; e < a.E; e += nthr) a.tokens_out[e] = a.tokens_num_type == 1 ? a.count[e] : a.cumsum[e];
  }
  if (gtid == 0 && a.available_out) *a.available_out = (int32_t)avail;
  if (a.row_idx_type == 1) {
    for (int64_t i = gtid; i < a.P; i += nthr) a.expanded_row_idx[i] = a.sorted_row[i];
  } else if (a.gather_idx) {
    const int64_t nmove = (!a.drop_pad && a.active_num > 0 && a.active_num < avail) ? a.active_num : avail;
    for (int64_t f = gtid; f < a.P; f += nthr) {
      const int g = a.gather[f];
      int d = -1;
      if (g >= 0) {
        if (!a.drop_pad) {
          d = g < nmove ? g : -1;
        } else {
          const int e = a.ids[f] - a.id_base;
          const int r = g - (a.cumsum[e] - a.count[e]);
          d = r < a.C ? e * a.C + r : -1;
        }
      }
      a.expanded_row_idx[f] = d;
    }
  }
  if (a.drop_pad) {
    const int lane = threadIdx.x & 31;
    const int64_t gw = gtid >> 5, nw = nthr >> 5;
    const int64_t nslot = (int64_t)a.E * a.C;
    const int64_t row_bytes = (int64_t)a.H * a.esize;
    for (int64_t s = gw; s < nslot; s += nw) {
      const int e = (int)(s / a.C), r = (int)(s % a.C);
      if (r < a.count[e]) continue;
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.expanded_x) + s * row_bytes);
      for (int64_t v = lane; v < row_bytes / 16; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
      if (lane == 0 && a.expanded_scale) a.expanded_scale[s] = 0.0f;
    }
  }
}

// ------------------------------------------------------------------ launchers
size_t route_small_smem(int E) { return (size_t)(32 * E + 3 * E + 256 + kRouteSmallMax) * 4; }
size_t route_big_smem(int E) { return (size_t)(8 * E + 3 * E + 256) * 4; }

cudaError_t launch_routing(const RouteArgs& a, cudaStream_t st, int* launches) {
  RouteArgs args = a;
  void* kargs[] = {&args};
  if (a.P <= kRouteSmallMax) {
    *launches = 1;
    return launch_with_pdl((const void*)route_small_kernel, dim3(1), dim3(1024), route_small_smem(a.E), st, kargs);
  }
  *launches = 2;
  cudaError_t err =
      launch_with_pdl((const void*)route_hist_kernel, dim3(a.nblk), dim3(256), route_big_smem(a.E), st, kargs);
  if (err != cudaSuccess) return err;
  return launch_with_pdl((const void*)route_rank_kernel, dim3(a.nblk), dim3(256), route_big_smem(a.E), st, kargs);
}

cudaError_t launch_init_move(const InitMoveArgs& a, cudaStream_t st) {
  InitMoveArgs args = a;
  void* kargs[] = {&args};
  const unsigned blocks = (unsigned)((a.T + 7) / 8);
  return launch_with_pdl((const void*)init_move_kernel, dim3(blocks ? blocks : 1), dim3(256), 0, st, kargs);
}

cudaError_t launch_init_rows(const InitRowsArgs& a, int64_t P, cudaStream_t st, int num_sms) {
  InitRowsArgs args = a;
  void* kargs[] = {&args};
  const int64_t want = (P + 7) / 8;
  const unsigned blocks = (unsigned)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  return launch_with_pdl((const void*)init_rows_kernel, dim3(blocks ? blocks : 1), dim3(256), 0, st, kargs);
}

cudaError_t launch_init_finish(const InitFinishArgs& a, cudaStream_t st, int num_sms) {
  InitFinishArgs args = a;
  void* kargs[] = {&args};
  return launch_with_pdl((const void*)init_finish_kernel, dim3(num_sms * 4), dim3(256), 0, st, kargs);
}

cudaError_t routing_set_attributes(int E) {
  cudaError_t err = cudaFuncSetAttribute((const void*)route_small_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)route_small_smem(E));
  if (err != cudaSuccess) return err;
  err = cudaFuncSetAttribute((const void*)route_hist_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)route_big_smem(E));
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute((const void*)route_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)route_big_smem(E));
}

}  // namespace moe
