// gemv.cu -- FC1 at decode batch sizes: weights streamed at HBM rate, the
// products on warp-level MMAs.
//
// ("Cake SiTU backend": FC1 over gate and up, SiTU, intermediate NVFP4
// requantization.)  With a handful of tokens per expert the block-scaled
// tcgen05 MMA spends most of its time on per-K-step scale copies into TMEM
// while the weights stream; here the weights stream through a bulk-copy
// ring, each weight code is decoded once, and the products run on
// mma.sync (m16n8k16, f16 operands, fp32 accumulation).
//
// A job is one token tile's W13 tile (64 intermediate features: 128 rows,
// gate and up interleaved, all H/256 k-blocks) and up to kGvTok of the
// tile's tokens; a tile with more tokens takes several jobs over the same
// weights (the later ones from L2).  The producer warp takes units (token
// tile, W13 tile) from the call's work counter, copies each job's X codes
// and block scales (token-major rows, 2 bulk copies per token) into one of
// two X slots and streams the W13 k-blocks (16 KB of codes by the tensor
// map of the tcgen05 path, 128-byte swizzled, + 2 KB of scale atoms by a bulk
// copy) through an 8-stage ring.
//
// Operands.  An E2M1 code times its E4M3 block scale is exact in f16 (at
// most 6 significant bits, magnitudes in [2^-10, 2688]), so both operands
// enter the MMA already scaled and the block structure disappears: X once
// per job (the job's tokens, into a shared f16 copy laid out for the B
// fragments), W as it is consumed (cvt.rn.f16x2.e2m1x2 and one f16x2
// multiply per code pair).  The f16 products are exact in fp32; a k-block's
// 16 MMA steps accumulate in a fresh fragment that is then added to the
// running fp32 sum.
//
// Fragments.  Sixteen consumer warps: warp w owns rows 16(w%8)..16(w%8)+15
// of the W13 tile (MMA rows g and g+8, g = lane/4) in the k-blocks of
// parity w/8, so the two halves of the warps take alternate ring stages and
// add their partial sums in the epilogue.  Thread t = lane%4 of a row group
// takes the bytes [32t, 32t+32) of each k-block row (4 block-scale groups;
// two 16-byte chunks, which the swizzle places in different banks for rows
// g and g+1).  MMA step s (of 16 per k-block) pairs its K indices 2t,2t+1
// with byte 32t+2s and 2t+8,2t+9 with byte 32t+2s+1 -- the same bytes of
// the token's X row in the B fragment (token g; lanes past the job's
// tokens read the first token, whose columns of the result are not used).
// The K order within a k-block is thus permuted, identically for both
// operands, which a dot product does not see.
//
// After the last k-block, z = sum * dX*dW13[e] goes through shared memory;
// one thread per (token, feature) applies SiTU to (z_gate, z_up) and 16
// lanes quantize a 16-feature group with qA[e] (the X quantizer's
// arithmetic) into the pair's padded row of A, codes and atom-layout scale,
// which FC2 reads unchanged.  Every wait is bounded.
#include <cuda_fp16.h>

#include "nvfp4.cuh"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

constexpr int kGvWarps = 16;                      // consumer warps: 16 W13 rows, alternate k-blocks
constexpr int kGvThreads = (kGvWarps + 1) * 32;   // + the producer warp
constexpr int kGvTok = 4;                         // tokens per job
constexpr int kGvStages = 8;
constexpr int kGvW = 16384;                       // one W13 k-block tile: 128 rows x 128 B
constexpr int kGvStage = kGvW + 2048;             // + its four scale atoms
constexpr int kGvSeg = 36;                        // words per (k-block, t) segment of X16: 32 + 4 of padding

struct GvBars {
  uint64_t full[kGvStages], empty[kGvStages];
  uint64_t xfull[2], xempty[2];     // raw X slots (producer -> consumers)
  uint64_t x16ready, x16free;       // the job's f16 X, between the consumer warps
  uint64_t zready[2], zfree[2];     // z slots (partial row sums of a job, between the consumer warps)
  int4 job[2];                      // {unit, expert, first padded row, m | token mask << 8 | W13 tile << 16}
  int32_t abort_flag;
};

// Words of one token's X16: NKB k-blocks x 4 segments of kGvSeg words, padded
// so that consecutive tokens start 16 banks apart (the B-fragment loads of
// two tokens in one quarter warp then hit disjoint banks).
__host__ __device__ inline int x16_token_words(int H) {
  const int w = (H / 256) * 4 * kGvSeg;
  return w + ((16 - w % 32) + 32) % 32;
}

// Shared memory: ring | raw X codes [2][kGvTok][H/2] | raw X scales
// [2][kGvTok][H/16] | X16 [kGvTok][token words] | z [2 slots][2 k-block
// parities][kGvTok][128] fp32 | barriers; plus 1 KB for the alignment of the
// base.
static size_t gv_smem_bytes(int H) {
  return (size_t)kGvStages * kGvStage + (size_t)2 * kGvTok * (H / 2) + (size_t)2 * kGvTok * (H / 16) +
         (size_t)kGvTok * x16_token_words(H) * 4 + (size_t)4 * kGvTok * 128 * 4 + sizeof(GvBars) + 1024;
}

// ----------------------------------------------------------- shared memory
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sts128(uint32_t a, uint32_t x, uint32_t y, uint32_t z, uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(x), "r"(y), "r"(z), "r"(w) : "memory");
}
__device__ __forceinline__ int32_t lds_volatile_s32(const void* p) {
  int32_t v;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
  return v;
}

// A job descriptor, stored before and read after the X slot's barrier
// (whose arrive / wait order them).
__device__ __forceinline__ void job_store(int4* slot, int4 v) {
  asm volatile("st.volatile.shared.v4.s32 [%0], {%1, %2, %3, %4};" ::"r"(smem_u32(slot)), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}
__device__ __forceinline__ int4 job_load(const int4* slot) {
  int4 v;
  asm volatile("ld.volatile.shared.v4.s32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(smem_u32(slot))
               : "memory");
  return v;
}

// Bounded wait; once any role of the CTA has given up, the others give up
// at their next wait that does not pass at once.
__device__ __forceinline__ bool gv_wait(uint64_t* bar, uint32_t parity, GvBars* bars, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  if (lds_volatile_s32(&bars->abort_flag)) return false;
  if (mbar_wait(bar, parity, status)) return true;
  asm volatile("st.volatile.shared.s32 [%0], 1;" ::"r"(smem_u32(&bars->abort_flag)) : "memory");
  return false;
}

// ------------------------------------------------------------- conversions
// One 32-bit word of E2M1 codes (element 2i in the low nibble of byte i) as
// four f16 pairs, exactly: pair i from byte i.
__device__ __forceinline__ void e2m1x8_to_h2(uint32_t w, uint32_t* h) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two E4M3 bytes (the low 16 bits of b, low byte first) as an f16 pair, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_h2(uint32_t b) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}" : "=r"(r) : "r"(b));
  return r;
}

// (lo, lo) and (hi, hi) of an f16 pair.
__device__ __forceinline__ uint32_t h2_lo2(uint32_t h) { return __byte_perm(h, 0, 0x1010); }
__device__ __forceinline__ uint32_t h2_hi2(uint32_t h) { return __byte_perm(h, 0, 0x3232); }

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// c = A * B + c, m16n8k16, f16 operands, fp32 accumulators.
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t lds8(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// ----------------------------------------------------------------- pieces
// One k-block of a job for thread (g, t) of a consumer warp: rows R0 and
// R0 + 8 of the stage's W13 tile (16-byte chunk c of row R at chunk c ^ (R%8),
// the 128-byte swizzle), bytes [32t, 32t+32); x16 is the thread's X16
// segment of this k-block.
__device__ __forceinline__ void gv_kblock(uint32_t st, uint32_t x16, int R0, int t, float (&sum)[4]) {
  const int R1 = R0 + 8, sw = R0 & 7;   // R1 % 8 == R0 % 8
  const uint32_t ra = st + R0 * 128, rb = st + R1 * 128;
  const uint32_t c0 = (uint32_t)(((2 * t) ^ sw) * 16), c1 = (uint32_t)(((2 * t + 1) ^ sw) * 16);
  const uint4 a0 = lds128(ra + c0), a1 = lds128(ra + c1), b0 = lds128(rb + c0), b1 = lds128(rb + c1);
  // block scales of groups 4t..4t+3 (atom t): row R at (R%32)*16 + (R/32)*4
  const uint32_t sa = lds32(st + kGvW + t * 512 + (R0 & 31) * 16 + (R0 >> 5) * 4);
  const uint32_t sb = lds32(st + kGvW + t * 512 + (R1 & 31) * 16 + (R1 >> 5) * 4);
  uint32_t xw[32];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint4 v = lds128(x16 + 16 * j);
    xw[4 * j] = v.x;
    xw[4 * j + 1] = v.y;
    xw[4 * j + 2] = v.z;
    xw[4 * j + 3] = v.w;
  }
  const uint32_t sa01 = e4m3x2_to_h2(sa), sa23 = e4m3x2_to_h2(sa >> 16);
  const uint32_t sb01 = e4m3x2_to_h2(sb), sb23 = e4m3x2_to_h2(sb >> 16);
  const uint32_t SA[4] = {h2_lo2(sa01), h2_hi2(sa01), h2_lo2(sa23), h2_hi2(sa23)};
  const uint32_t SB[4] = {h2_lo2(sb01), h2_hi2(sb01), h2_lo2(sb23), h2_hi2(sb23)};
  const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
  // four accumulation chains (MMA step s into chain s % 4)
  float cc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) cc[j][i] = 0.0f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    // word q: bytes 4q..4q+3 of the segment, block-scale group q/2; MMA steps 2q and 2q+1
    uint32_t ha[4], hb[4];
    e2m1x8_to_h2(wa[q], ha);
    e2m1x8_to_h2(wb[q], hb);
    const uint32_t sA = SA[q >> 1], sB = SB[q >> 1];
    mma16816(cc[(2 * q) & 3], hmul2(ha[0], sA), hmul2(hb[0], sB), hmul2(ha[1], sA), hmul2(hb[1], sB), xw[4 * q],
             xw[4 * q + 1]);
    mma16816(cc[(2 * q + 1) & 3], hmul2(ha[2], sA), hmul2(hb[2], sB), hmul2(ha[3], sA), hmul2(hb[3], sB),
             xw[4 * q + 2], xw[4 * q + 3]);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sum[i] += (cc[0][i] + cc[1][i]) + (cc[2][i] + cc[3][i]);
}

// The job's tokens from the raw X slot (codes, block scales) into X16: each
// code pair times its block scale as an f16 pair, byte 32t+e of k-block kb
// at word (kb*4 + t)*kGvSeg + e of the token's X16.  Thread i of the
// consumer warps takes 4-byte words i, i + 256, ...
__device__ __forceinline__ void gv_fill_x16(uint32_t xs, uint32_t xsc, uint32_t x16, int m, int H, int tid) {
  const int H2 = H / 2, G = H / 16, H8 = H / 8, TW = x16_token_words(H);
  for (int wi = tid; wi < m * H8; wi += kGvWarps * 32) {
    const int j = wi / H8, ww = wi - j * H8;
    const uint32_t codes = lds32(xs + j * H2 + 4 * ww);
    const uint32_t s2 = h2_lo2(e4m3x2_to_h2(lds8(xsc + j * G + (ww >> 1))));
    uint32_t h[4];
    e2m1x8_to_h2(codes, h);
    const int seg = (ww >> 5) * 4 + ((ww & 31) >> 3);
    sts128(x16 + 4 * (j * TW + seg * kGvSeg + 4 * (ww & 7)), hmul2(h[0], s2), hmul2(h[1], s2), hmul2(h[2], s2),
           hmul2(h[3], s2));
  }
}

// Tile descriptor of unit u (nit units per tile), or an invalid one.
__device__ __forceinline__ int4 gv_tile(const int4* tiles, int u, int nit) {
  return u >= 0 ? tiles[u / nit] : make_int4(-1, 0, 0, 0);
}

__device__ __forceinline__ bool gv_tile_ok(const int4& t, int E, int64_t max_rows) {
  return t.x >= 0 && t.x < E && t.y >= 0 && (t.y & (kTileRows - 1)) == 0 && t.z >= 1 && t.z <= kTileRows &&
         (int64_t)t.y + t.z <= max_rows;
}

// Flat pair indices of rows r0 .. r0 + kGvTok - 1 of a tile (-1 past its fill
// or for an invalid tile).
__device__ __forceinline__ void gv_pairs(const Fc1Args& p, const int4& t, int r0, int (&f)[kGvTok]) {
  const bool ok = gv_tile_ok(t, p.E, p.max_rows);
#pragma unroll
  for (int j = 0; j < kGvTok; ++j) f[j] = (ok && r0 + j < t.z) ? __ldg(p.prow_pair + t.y + r0 + j) : -1;
}

// ============================================================ FC1 (decode)
__global__ void __launch_bounds__(kGvThreads, 1)
    fc1_gemv_kernel(const __grid_constant__ CUtensorMap tm_w13, const Fc1Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int H2 = p.H / 2, G = p.H / 16, NIT = p.I / 64, NKB = p.H / 256, I2 = p.I / 2, KC = p.I / 16;
  uint8_t* xcodes = ring + kGvStages * kGvStage;
  uint8_t* xscales = xcodes + 2 * kGvTok * H2;
  uint8_t* x16 = xscales + 2 * kGvTok * G;
  float* zbuf = reinterpret_cast<float*>(x16 + (size_t)kGvTok * x16_token_words(p.H) * 4);
  GvBars* bars = reinterpret_cast<GvBars*>(zbuf + 4 * kGvTok * 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGvStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kGvWarps / 2);   // the warps of the k-block's parity
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->xfull[b], 1);
      mbar_init(&bars->xempty[b], kGvWarps);
      mbar_init(&bars->zready[b], kGvWarps);
      mbar_init(&bars->zfree[b], kGvWarps);
    }
    mbar_init(&bars->x16ready, kGvWarps);
    mbar_init(&bars->x16free, kGvWarps);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();   // routing's tiles and the quantized X
  pdl_launch_dependents();
  const int num_units = min(max(p.hdr[HDR_NUM_TT], 0), p.max_tiles) * NIT;   // (token tile, W13 tile)
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == kGvWarps) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      tma_prefetch_desc(&tm_w13);
      uint32_t stage = 0, phase = 0, xb = 0, xph = 0;
      uint32_t armed = 0, last_phase = 0;      // ring stages with copies issued; parity of each one's last use
      uint32_t xarmed = 0, xlast = 0;          // the same for the X slots
      bool ok = true;
      int taken = 0;
      auto take = [&]() -> int {
        const int u = p.dynamic ? atomicAdd(p.next, 1) : (int)blockIdx.x + taken * (int)gridDim.x;
        ++taken;
        return (u >= 0 && u < num_units) ? u : -1;
      };
      // Three units in flight, so no dependent load stalls the stream: the
      // unit being streamed (u0: tile, pairs of its first job), the next one
      // (u1: tile) and the one after (u2: taken).
      int u0 = take();
      int4 t0 = gv_tile(tiles, u0, NIT);
      int f0[kGvTok];
      gv_pairs(p, t0, 0, f0);
      int u1 = u0 >= 0 ? take() : -1;
      int4 t1 = gv_tile(tiles, u1, NIT);
      int u2 = u1 >= 0 ? take() : -1;
      while (ok && u0 >= 0) {
        int f1[kGvTok];
        gv_pairs(p, t1, 0, f1);
        const int4 t2 = gv_tile(tiles, u2, NIT);
        const int u3 = u2 >= 0 ? take() : -1;
        if (!gv_tile_ok(t0, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
        } else {
          const int e = t0.x, it = u0 % NIT;
          const int tile0 = (e * NIT + it) * NKB;   // the W13 tensor map's tile index of k-block 0
          const uint8_t* ssrc = p.sf13p + (size_t)tile0 * 2048;
          for (int r0 = 0; r0 < t0.z && ok; r0 += kGvTok) {
            int f[kGvTok];
            if (r0 == 0) {
#pragma unroll
              for (int j = 0; j < kGvTok; ++j) f[j] = f0[j];
            } else {
              gv_pairs(p, t0, r0, f);
            }
            const int m = min(kGvTok, t0.z - r0);
            int tok[kGvTok];
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < kGvTok; ++j) {
              tok[j] = (j < m && f[j] >= 0 && f[j] < p.num_pairs) ? f[j] / p.k : -1;
              if (tok[j] >= 0) mask |= 1u << j;
            }
            if (!gv_wait(&bars->xempty[xb], xph ^ 1u, bars, p.status)) {
              ok = false;
              break;
            }
            job_store(&bars->job[xb], make_int4(u0, e, t0.y + r0, m | (int)(mask << 8) | (it << 16)));
            mbar_arrive_expect_tx(&bars->xfull[xb], (uint32_t)__popc(mask) * (uint32_t)(H2 + G));
            xarmed |= 1u << xb;
            xlast = (xlast & ~(1u << xb)) | (xph << xb);
#pragma unroll
            for (int j = 0; j < kGvTok; ++j) {
              if (tok[j] < 0) continue;
              bulk_g2s(xcodes + (xb * kGvTok + j) * H2, p.xq + (size_t)tok[j] * H2, (uint32_t)H2, &bars->xfull[xb]);
              bulk_g2s(xscales + (xb * kGvTok + j) * G, p.sft + (size_t)tok[j] * G, (uint32_t)G, &bars->xfull[xb]);
            }
            xb ^= 1u;
            if (xb == 0) xph ^= 1u;
            for (int kb = 0; kb < NKB; ++kb) {
              if (!gv_wait(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
                ok = false;
                break;
              }
              uint8_t* st = ring + stage * kGvStage;
              mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)kGvStage);
              armed |= 1u << stage;
              last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
              tma_load_3d(st, &tm_w13, 0, 0, tile0 + kb, &bars->full[stage]);
              bulk_g2s(st + kGvW, ssrc + (size_t)kb * 2048, 2048u, &bars->full[stage]);
              if (++stage == kGvStages) {
                stage = 0;
                phase ^= 1u;
              }
            }
          }
        }
        u0 = u1;
        t0 = t1;
#pragma unroll
        for (int j = 0; j < kGvTok; ++j) f0[j] = f1[j];
        u1 = u2;
        t1 = t2;
        u2 = u3;
      }
      // the end of the sequence (its arrival completes a phase of the slot's
      // barrier too, so the drain below waits for that one)
      if (ok && gv_wait(&bars->xempty[xb], xph ^ 1u, bars, p.status)) {
        job_store(&bars->job[xb], make_int4(-1, 0, 0, 0));
        xarmed |= 1u << xb;
        xlast = (xlast & ~(1u << xb)) | (xph << xb);
        mbar_arrive(&bars->xfull[xb]);
      }
      // every issued copy has landed before the CTA may exit
      for (int s = 0; s < kGvStages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
      for (int b = 0; b < 2; ++b)
        if (xarmed & (1u << b)) mbar_wait(&bars->xfull[b], (xlast >> b) & 1u, p.status);
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3, R0 = 16 * (warp & 7) + g, kp = warp >> 3;
    const int tid = threadIdx.x, ej = tid >> 6, ef = tid & 63;   // epilogue (tid < 256): token ej, feature ef
    const int TW = x16_token_words(p.H);
    const uint32_t ring_s = smem_u32(ring), x16_s = smem_u32(x16);
    uint32_t kbase = 0;   // ring position of the job's k-block 0 (ring stage n % kGvStages, pass n / kGvStages)
    uint32_t xb = 0, xph = 0, x16ph = 0, zb = 0, zph = 0;
    while (true) {
      if (!gv_wait(&bars->xfull[xb], xph, bars, p.status)) break;
      const int4 jb = job_load(&bars->job[xb]);
      if (jb.x < 0) break;
      const int e = jb.y, m = jb.w & 0xFF, mask = (jb.w >> 8) & 0xFF, it = jb.w >> 16;
      const int64_t row = jb.z;
      // the expert's scalars, needed after the k-blocks
      const float s13 = __ldg(p.dXdW13 + e), qa = __ldg(p.qA + e), be = __ldg(p.beta + e), la = __ldg(p.lam + e);
      // X16 is free once every warp has finished the previous job's k-blocks
      if (!gv_wait(&bars->x16free, x16ph ^ 1u, bars, p.status)) break;
      gv_fill_x16(smem_u32(xcodes + xb * kGvTok * H2), smem_u32(xscales + xb * kGvTok * G), x16_s, m, p.H, tid);
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars->xempty[xb]);
        mbar_arrive(&bars->x16ready);
      }
      xb ^= 1u;
      if (xb == 0) xph ^= 1u;
      if (!gv_wait(&bars->x16ready, x16ph, bars, p.status)) break;
      // this thread's X16 segment of k-block 0: token g (the first token in
      // lanes past the job's tokens), segment t
      const uint32_t x16_lane = x16_s + 4 * (min(g, m - 1) * TW + t * kGvSeg);
      float sum[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      bool ok = true;
      for (int kb = kp; kb < NKB; kb += 2) {
        const uint32_t n = kbase + (uint32_t)kb, stage = n % kGvStages, phase = (n / kGvStages) & 1u;
        if (!gv_wait(&bars->full[stage], phase, bars, p.status)) {
          ok = false;
          break;
        }
        gv_kblock(ring_s + stage * kGvStage, x16_lane + 4 * kb * 4 * kGvSeg, R0, t, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[stage]);
      }
      kbase += (uint32_t)NKB;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->x16free);
      x16ph ^= 1u;
      if (!ok) break;
      // partial z[token][row] of this k-block parity: thread (g, t) holds rows
      // R0, R0 + 8 of tokens 2t, 2t + 1
      const uint32_t z = smem_u32(zbuf + zb * 2 * kGvTok * 128);
      const uint32_t zp = z + 4 * kp * kGvTok * 128;
      if (!gv_wait(&bars->zfree[zb], zph ^ 1u, bars, p.status)) break;
      if (2 * t < m) {
        sts_f32(zp + 4 * (2 * t * 128 + R0), sum[0]);
        sts_f32(zp + 4 * (2 * t * 128 + R0 + 8), sum[2]);
      }
      if (2 * t + 1 < m) {
        sts_f32(zp + 4 * ((2 * t + 1) * 128 + R0), sum[1]);
        sts_f32(zp + 4 * ((2 * t + 1) * 128 + R0 + 8), sum[3]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->zready[zb]);
      if (!gv_wait(&bars->zready[zb], zph, bars, p.status)) break;
      // SiTU of feature ef for token ej (rows 2ef = gate, 2ef+1 = up), then
      // 16 lanes quantize a 16-feature group (the first 8 warps)
      float a = 0.0f;
      if (tid < 256 && ej < m) {
        const uint32_t z1 = z + 4 * kGvTok * 128;
        const float zg = lds_f32(z + 4 * (ej * 128 + 2 * ef)) + lds_f32(z1 + 4 * (ej * 128 + 2 * ef));
        const float zu = lds_f32(z + 4 * (ej * 128 + 2 * ef + 1)) + lds_f32(z1 + 4 * (ej * 128 + 2 * ef + 1));
        a = situ_f32(__fmul_rn(zg, s13), __fmul_rn(zu, s13), be, 1.0f / be, la, 1.0f / la);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->zfree[zb]);
      zb ^= 1u;
      if (zb == 0) zph ^= 1u;
      if (tid < 256) {
        uint32_t word;
        const uint32_t sf = nvfp4_quant_lanes16(a, qa, word);
        if (ej < m && ((mask >> ej) & 1)) {
          const int64_t prow = row + ej;
          if ((lane & 7) == 0)
            *reinterpret_cast<uint32_t*>(p.aq + (size_t)prow * I2 + it * 32 + (ef >> 4) * 8 + ((ef >> 3) & 1) * 4) =
                word;
          if ((lane & 15) == 0) p.sfa[atom_offset(prow, it * 4 + (ef >> 4), KC)] = (uint8_t)sf;
        }
      }
    }
  }
}

size_t fc1_gemv_smem(int H) { return gv_smem_bytes(H); }

cudaError_t gemv_set_attributes() {
  return cudaFuncSetAttribute((const void*)fc1_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemOptin);
}

cudaError_t launch_fc1_gemv(const CUtensorMap& w13, const Fc1Args& a, int grid, cudaStream_t st) {
  CUtensorMap m0 = w13;
  Fc1Args args = a;
  void* kargs[] = {&m0, &args};
  return launch_with_pdl((const void*)fc1_gemv_kernel, dim3(grid), dim3(kGvThreads), gv_smem_bytes(a.H), st, kargs);
}

}  // namespace moe
