// gemv.cu -- FC1 and FC2 at decode batch sizes: weights streamed at HBM rate, the
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

constexpr int kGvWarps = 16;                      // FC2 consumer warps: 16 W2 rows, alternate output tiles
constexpr int kG1Par = 2;                         // FC1: k-block classes (k-block % kG1Par), 8 warps each
constexpr int kG1Warps = 8 * kG1Par;              // FC1 consumer warps: 16 W13 rows each
constexpr int kGvThreads = (kG1Warps + 1) * 32;   // FC1: + the producer warp
constexpr int kGvTok = 4;                         // tokens (FC1) or pairs (FC2) per job
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
// [2][kGvTok][H/16] | X16 [kGvTok][token words] | z [2 slots][kG1Par k-block
// classes][kGvTok][128] fp32 | barriers; plus 1 KB for the alignment of the
// base.
static size_t gv_smem_bytes(int H) {
  return (size_t)kGvStages * kGvStage + (size_t)2 * kGvTok * (H / 2) + (size_t)2 * kGvTok * (H / 16) +
         (size_t)kGvTok * x16_token_words(H) * 4 + (size_t)2 * kG1Par * kGvTok * 128 * 4 + sizeof(GvBars) + 1024;
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
  for (int wi = tid; wi < m * H8; wi += kG1Warps * 32) {
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
  GvBars* bars = reinterpret_cast<GvBars*>(zbuf + 2 * kG1Par * kGvTok * 128);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kGvStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 8);   // the warps of the k-block's class
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->xfull[b], 1);
      mbar_init(&bars->xempty[b], kG1Warps);
      mbar_init(&bars->zready[b], kG1Warps);
      mbar_init(&bars->zfree[b], kG1Warps);
    }
    mbar_init(&bars->x16ready, kG1Warps);
    mbar_init(&bars->x16free, kG1Warps);
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();   // routing's tiles and the quantized X
  pdl_launch_dependents();
  const int num_units = min(max(p.hdr[HDR_NUM_TT], 0), p.max_tiles) * NIT;   // (token tile, W13 tile)
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == kG1Warps) {
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
    const int g = lane >> 2, t = lane & 3, R0 = 16 * (warp & 7) + g, kp = warp >> 3;   // k-block class kp
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
      for (int kb = kp; kb < NKB; kb += kG1Par) {
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
      const uint32_t z = smem_u32(zbuf + zb * kG1Par * kGvTok * 128);
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
        float zg = lds_f32(z + 4 * (ej * 128 + 2 * ef)), zu = lds_f32(z + 4 * (ej * 128 + 2 * ef + 1));
#pragma unroll
        for (int c = 1; c < kG1Par; ++c) {
          const uint32_t zc = z + 4 * c * kGvTok * 128;
          zg += lds_f32(zc + 4 * (ej * 128 + 2 * ef));
          zu += lds_f32(zc + 4 * (ej * 128 + 2 * ef + 1));
        }
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

// ============================================================ FC2 (decode)
// ("Cake SiTU backend": FC2, BF16 weighted finalization.)  The same scheme
// for FC2: a unit is one token tile and a group of `group` consecutive
// 128-feature output tiles of its expert; a job is a unit and up to kGvTok
// of the tile's pairs.  Each ring stage holds one whole output tile (I/128
// k-blocks of 128 rows x 64 B, plain bulk copies, + its I/64 scale atoms).
// The sixteen consumer warps take alternate output tiles of the whole
// sequence of jobs (warps 0-7 the even ring positions, 8-15 the odd ones),
// warp w%8 the rows 16(w%8)..16(w%8)+15.  A converter warp turns each
// job's A rows (codes by bulk copy, block scales from their atoms by 4-byte
// cp.async) into pre-scaled f16 pairs in one of two A16 slots, one 20-word
// segment per (k-block, t), so the consumers never wait for one another
// between jobs.  Each output tile's sums are scaled by dA*dW2[e] and the
// pair's route weight and added into the token's fp32 accumulator row (L2
// reductions), as the tcgen05 FC2 does.
constexpr int kG2Stages = 6;
constexpr int kG2Seg = 20;                        // words per (k-block, t) segment of A16: 16 + 4 of padding

constexpr int kG2Threads = (kGvWarps + 2) * 32;  // consumers, the producer warp, the converter warp

struct G2Bars {
  uint64_t full[kG2Stages], empty[kG2Stages];
  uint64_t xfull[2], xempty[2];     // raw A slots (producer -> converter)
  uint64_t aready[2], afree[2];     // A16 slots (converter -> consumers)
  int4 job[2][3];                   // raw slot: {unit, expert, first padded row, m | mask << 8 | first output tile
                                    // << 16}, the pairs' tokens, their route weights (fp32 bits)
  int4 meta[2][4];                  // A16 slot: the same three, then {ring position of its first tile, 0, 0, 0}
  int32_t abort_flag;
};

__host__ __device__ inline int a16_pair_words(int I) {
  const int w = (I / 128) * 4 * kG2Seg;
  return w + ((16 - w % 32) + 32) % 32;
}
__host__ __device__ inline int g2_stage_bytes(int I) { return (I / 128) * 8192 + (I / 64) * 512; }

// Shared memory: ring | raw A codes [2][kGvTok][I/2] | raw A scales
// [2][kGvTok][I/16] | A16 [2][kGvTok][pair words] | barriers; + 1 KB of alignment.
static size_t g2_smem_bytes(int I) {
  return (size_t)kG2Stages * g2_stage_bytes(I) + (size_t)2 * kGvTok * (I / 2) + (size_t)2 * kGvTok * (I / 16) +
         (size_t)2 * kGvTok * a16_pair_words(I) * 4 + sizeof(G2Bars) + 1024;
}

__device__ __forceinline__ bool g2_wait(uint64_t* bar, uint32_t parity, G2Bars* bars, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  if (lds_volatile_s32(&bars->abort_flag)) return false;
  if (mbar_wait(bar, parity, status)) return true;
  asm volatile("st.volatile.shared.s32 [%0], 1;" ::"r"(smem_u32(&bars->abort_flag)) : "memory");
  return false;
}

__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}

// The job's pairs from the raw slot into A16 (by one warp): byte 16t+e of
// k-block kb at word (kb*4 + t)*kG2Seg + e of the pair's A16.
__device__ __forceinline__ void g2_fill_a16(uint32_t as, uint32_t asc, uint32_t a16, int m, int I, int lane) {
  const int I2 = I / 2, I16 = I / 16, I8 = I / 8, PW = a16_pair_words(I);
  for (int wi = lane; wi < m * I8; wi += 32) {
    const int j = wi / I8, ww = wi - j * I8;
    const uint32_t codes = lds32(as + j * I2 + 4 * ww);
    const uint32_t s2 = h2_lo2(e4m3x2_to_h2(lds8(asc + j * I16 + (ww >> 1))));
    uint32_t h[4];
    e2m1x8_to_h2(codes, h);
    const int seg = (ww >> 4) * 4 + ((ww & 15) >> 2);
    sts128(a16 + 4 * (j * PW + seg * kG2Seg + 4 * (ww & 3)), hmul2(h[0], s2), hmul2(h[1], s2), hmul2(h[2], s2),
           hmul2(h[3], s2));
  }
}

// One output tile for thread (g, t): rows R0, R0 + 8, all I/128 k-blocks
// (thread t's 16 bytes of each 64-byte k-block row); a16 is the thread's A16
// segment of k-block 0.
__device__ __forceinline__ void g2_tile(uint32_t st, uint32_t a16, int R0, int t, int NKB2, float (&sum)[4]) {
  const int R1 = R0 + 8;
  float cc[4][4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int i = 0; i < 4; ++i) cc[j][i] = 0.0f;
  const uint32_t sfb = st + NKB2 * 8192;
  for (int kb = 0; kb < NKB2; ++kb) {
    const uint4 a = lds128(st + kb * 8192 + R0 * 64 + 16 * t), b = lds128(st + kb * 8192 + R1 * 64 + 16 * t);
    // block scales of chunks 8kb+2t, 8kb+2t+1: atom 2kb + t/2, bytes 2(t%2), 2(t%2)+1 of row R
    const uint32_t at = sfb + (2 * kb + (t >> 1)) * 512 + 2 * (t & 1);
    const uint32_t sa = e4m3x2_to_h2(lds16(at + (R0 & 31) * 16 + (R0 >> 5) * 4));
    const uint32_t sb = e4m3x2_to_h2(lds16(at + (R1 & 31) * 16 + (R1 >> 5) * 4));
    const uint32_t SA[2] = {h2_lo2(sa), h2_hi2(sa)}, SB[2] = {h2_lo2(sb), h2_hi2(sb)};
    uint32_t xw[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint4 v = lds128(a16 + 4 * kb * 4 * kG2Seg + 16 * j);
      xw[4 * j] = v.x;
      xw[4 * j + 1] = v.y;
      xw[4 * j + 2] = v.z;
      xw[4 * j + 3] = v.w;
    }
    const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t ha[4], hb[4];
      e2m1x8_to_h2(wa[q], ha);
      e2m1x8_to_h2(wb[q], hb);
      const uint32_t sA = SA[q >> 1], sB = SB[q >> 1];
      mma16816(cc[(2 * q) & 3], hmul2(ha[0], sA), hmul2(hb[0], sB), hmul2(ha[1], sA), hmul2(hb[1], sB), xw[4 * q],
               xw[4 * q + 1]);
      mma16816(cc[(2 * q + 1) & 3], hmul2(ha[2], sA), hmul2(hb[2], sB), hmul2(ha[3], sA), hmul2(hb[3], sB),
               xw[4 * q + 2], xw[4 * q + 3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) sum[i] = (cc[0][i] + cc[1][i]) + (cc[2][i] + cc[3][i]);
}

// 4-byte asynchronous global->shared copy (completion counted by
// cp.async.mbarrier.arrive).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

__global__ void __launch_bounds__(kG2Threads, 1) fc2_gemv_kernel(const Fc2Args p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int I2 = p.I / 2, I16 = p.I / 16, NKB2 = p.I / 128, NMT = p.H / 128, SB = g2_stage_bytes(p.I);
  const int G = max(1, min(p.group, NMT)), NG = (NMT + G - 1) / G;
  uint8_t* acodes = ring + kG2Stages * SB;
  uint8_t* ascales = acodes + 2 * kGvTok * I2;
  uint8_t* a16 = ascales + 2 * kGvTok * I16;
  const int PW = a16_pair_words(p.I);
  G2Bars* bars = reinterpret_cast<G2Bars*>(a16 + (size_t)2 * kGvTok * PW * 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kG2Stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], kGvWarps / 2);   // the warps of the output tile's parity
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->xfull[b], 2);   // the producer's arrival (bulk copies) and its block-scale cp.asyncs'
      mbar_init(&bars->xempty[b], 1);
      mbar_init(&bars->aready[b], 1);
      mbar_init(&bars->afree[b], kGvWarps);
    }
    bars->abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait();   // FC1's A and everything before it
  pdl_launch_dependents();
  const int num_units = min(max(p.hdr[HDR_NUM_TT], 0), p.max_tiles) * NG;   // (token tile, group of output tiles)
  const int4* tiles = reinterpret_cast<const int4*>(p.tt_list);

  if (warp == kGvWarps) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      uint32_t stage = 0, phase = 0, xb = 0, xph = 0;
      uint32_t armed = 0, last_phase = 0;
      uint32_t xarmed = 0, xlast = 0;
      bool ok = true;
      int taken = 0;
      auto take = [&]() -> int {
        const int u = p.dynamic ? atomicAdd(p.next, 1) : (int)blockIdx.x + taken * (int)gridDim.x;
        ++taken;
        return (u >= 0 && u < num_units) ? u : -1;
      };
      auto pairs = [&](const int4& t, int r0, int (&f)[kGvTok], float (&w)[kGvTok]) {
        const bool okt = gv_tile_ok(t, p.E, p.max_rows);
#pragma unroll
        for (int j = 0; j < kGvTok; ++j) {
          const bool in = okt && r0 + j < t.z;
          f[j] = in ? __ldg(p.prow_pair + t.y + r0 + j) : -1;
          w[j] = in ? __ldg(p.wrow + t.y + r0 + j) : 0.0f;
        }
      };
      // One unit ahead, taken late: while the last job of the current unit
      // issues its stages, one step per stage takes the next unit from the
      // counter, loads its tile descriptor and then its first job's pairs,
      // so each step's latency hides under the stream and a CTA holds at most
      // one unit it has not started (the units are few and long here, and
      // units reserved early would stay with CTAs that fall behind).
      int u0 = take();
      int4 t0 = gv_tile(tiles, u0, NG);
      int f0[kGvTok];
      float w0[kGvTok];
      pairs(t0, 0, f0, w0);
      int nu = -1, step = 0;
      int4 nt = make_int4(-1, 0, 0, 0);
      int nf[kGvTok];
      float nw[kGvTok];
      auto advance = [&]() {
        if (step == 0) {
          nu = take();
        } else if (step == 1) {
          nt = gv_tile(tiles, nu, NG);
        } else if (step == 2) {
          pairs(nt, 0, nf, nw);
        }
        if (step < 3) ++step;
      };
      while (ok && u0 >= 0) {
        if (!gv_tile_ok(t0, p.E, p.max_rows)) {
          set_status(p.status, DEVSTAT_BAD_TILE);
        } else {
          const int e = t0.x, mt0 = (u0 % NG) * G, cnt = min(G, NMT - mt0);
          for (int r0 = 0; r0 < t0.z && ok; r0 += kGvTok) {
            const bool last_job = r0 + kGvTok >= t0.z;
            int f[kGvTok];
            float w[kGvTok];
            if (r0 == 0) {
#pragma unroll
              for (int j = 0; j < kGvTok; ++j) {
                f[j] = f0[j];
                w[j] = w0[j];
              }
            } else {
              pairs(t0, r0, f, w);
            }
            const int m = min(kGvTok, t0.z - r0);
            int tok[kGvTok];
            uint32_t mask = 0;
#pragma unroll
            for (int j = 0; j < kGvTok; ++j) {
              tok[j] = (j < m && f[j] >= 0 && f[j] < p.num_pairs) ? f[j] / p.k : -1;
              if (tok[j] >= 0) mask |= 1u << j;
            }
            if (!g2_wait(&bars->xempty[xb], xph ^ 1u, bars, p.status)) {
              ok = false;
              break;
            }
            job_store(&bars->job[xb][0], make_int4(u0, e, t0.y + r0, m | (int)(mask << 8) | (mt0 << 16)));
            job_store(&bars->job[xb][1], make_int4(tok[0], tok[1], tok[2], tok[3]));
            job_store(&bars->job[xb][2], make_int4(__float_as_int(w[0]), __float_as_int(w[1]), __float_as_int(w[2]),
                                                   __float_as_int(w[3])));
            // the pairs' block-scale words (4 chunks each) from their atoms
            const uint32_t asc = smem_u32(ascales + xb * kGvTok * I16);
            for (int j = 0; j < m; ++j) {
              const int64_t row = (int64_t)t0.y + r0 + j;
              for (int a = 0; a < I16 / 4; ++a)
                cp_async4(asc + j * I16 + 4 * a, p.sfa + ((size_t)(row >> 7) * (I16 / 4) + a) * 512 + (row & 31) * 16 +
                                                     ((row >> 5) & 3) * 4);
            }
            cp_async_mbar_arrive(&bars->xfull[xb]);
            mbar_arrive_expect_tx(&bars->xfull[xb], (uint32_t)m * (uint32_t)I2);
            xarmed |= 1u << xb;
            xlast = (xlast & ~(1u << xb)) | (xph << xb);
            for (int j = 0; j < m; ++j)
              bulk_g2s(acodes + (xb * kGvTok + j) * I2, p.aq + (size_t)(t0.y + r0 + j) * I2, (uint32_t)I2,
                       &bars->xfull[xb]);
            xb ^= 1u;
            if (xb == 0) xph ^= 1u;
            for (int i = 0; i < cnt; ++i) {
              if (!g2_wait(&bars->empty[stage], phase ^ 1u, bars, p.status)) {
                ok = false;
                break;
              }
              uint8_t* st = ring + stage * SB;
              const size_t tile = (size_t)e * NMT + mt0 + i;
              mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)SB);
              armed |= 1u << stage;
              last_phase = (last_phase & ~(1u << stage)) | (phase << stage);
              bulk_g2s(st, p.w2p + tile * NKB2 * 8192, (uint32_t)(NKB2 * 8192), &bars->full[stage]);
              bulk_g2s(st + NKB2 * 8192, p.sf2p + tile * (p.I / 64) * 512, (uint32_t)(NKB2 * 1024),
                       &bars->full[stage]);
              if (++stage == kG2Stages) {
                stage = 0;
                phase ^= 1u;
              }
              if (last_job) advance();
            }
          }
        }
        while (step < 3) advance();
        u0 = nu;
        t0 = nt;
#pragma unroll
        for (int j = 0; j < kGvTok; ++j) {
          f0[j] = nf[j];
          w0[j] = nw[j];
        }
        step = 0;
      }
      if (ok && g2_wait(&bars->xempty[xb], xph ^ 1u, bars, p.status)) {
        job_store(&bars->job[xb][0], make_int4(-1, 0, 0, 0));
        xarmed |= 1u << xb;
        xlast = (xlast & ~(1u << xb)) | (xph << xb);
        cp_async_mbar_arrive(&bars->xfull[xb]);
        mbar_arrive(&bars->xfull[xb]);
      }
      cp_async_wait_all();
      for (int s = 0; s < kG2Stages; ++s)
        if (armed & (1u << s)) mbar_wait(&bars->full[s], (last_phase >> s) & 1u, p.status);
      for (int b = 0; b < 2; ++b)
        if (xarmed & (1u << b)) mbar_wait(&bars->xfull[b], (xlast >> b) & 1u, p.status);
    }
  } else if (warp == kGvWarps + 1) {
    // --------------------------------------------------------- converter
    uint32_t xb = 0, xph = 0, ab = 0, aph = 0, base = 0;
    while (true) {
      if (!g2_wait(&bars->xfull[xb], xph, bars, p.status)) break;
      const int4 jb = job_load(&bars->job[xb][0]);
      if (!g2_wait(&bars->afree[ab], aph ^ 1u, bars, p.status)) break;
      if (jb.x < 0) {
        __syncwarp();
        if (lane == 0) {
          job_store(&bars->meta[ab][0], jb);
          mbar_arrive(&bars->aready[ab]);
        }
        break;
      }
      const int m = jb.w & 0xFF, cnt = min(G, NMT - (jb.w >> 16));
      g2_fill_a16(smem_u32(acodes + xb * kGvTok * I2), smem_u32(ascales + xb * kGvTok * I16),
                  smem_u32(a16 + (size_t)ab * kGvTok * PW * 4), m, p.I, lane);
      __syncwarp();
      if (lane == 0) {
        job_store(&bars->meta[ab][0], jb);
        job_store(&bars->meta[ab][1], job_load(&bars->job[xb][1]));
        job_store(&bars->meta[ab][2], job_load(&bars->job[xb][2]));
        job_store(&bars->meta[ab][3], make_int4((int)base, 0, 0, 0));
        mbar_arrive(&bars->xempty[xb]);
        mbar_arrive(&bars->aready[ab]);
      }
      base += (uint32_t)cnt;
      xb ^= 1u;
      if (xb == 0) xph ^= 1u;
      ab ^= 1u;
      if (ab == 0) aph ^= 1u;
    }
  } else {
    // ------------------------------------------------------------ consumers
    const int g = lane >> 2, t = lane & 3, R0 = 16 * (warp & 7) + g, wp = warp >> 3;
    const uint32_t ring_s = smem_u32(ring);
    uint32_t ab = 0, aph = 0;
    while (true) {
      if (!g2_wait(&bars->aready[ab], aph, bars, p.status)) break;
      const int4 jb = job_load(&bars->meta[ab][0]);
      if (jb.x < 0) break;
      const int4 tk = job_load(&bars->meta[ab][1]);
      const int4 wq = job_load(&bars->meta[ab][2]);
      const uint32_t base = (uint32_t)job_load(&bars->meta[ab][3]).x;
      const int e = jb.y, m = jb.w & 0xFF, mask = (jb.w >> 8) & 0xFF, mt0 = jb.w >> 16;
      const int cnt = min(G, NMT - mt0);
      const float s2 = __ldg(p.dAdW2 + e);
      // this thread's pairs 2t, 2t + 1 (their tokens, -1 if none, and route weights)
      const int tok0 = (t == 0) ? tk.x : (t == 1) ? tk.z : -1, tok1 = (t == 0) ? tk.y : (t == 1) ? tk.w : -1;
      const float wt0 = __int_as_float((t == 0) ? wq.x : wq.z), wt1 = __int_as_float((t == 0) ? wq.y : wq.w);
      const bool use0 = 2 * t < m && ((mask >> (2 * t)) & 1) && tok0 >= 0;
      const bool use1 = 2 * t + 1 < m && ((mask >> (2 * t + 1)) & 1) && tok1 >= 0;
      const uint32_t a16_lane = smem_u32(a16) + 4 * (((int)ab * kGvTok + min(g, m - 1)) * PW + t * kG2Seg);
      bool ok = true;
      // the job's ring positions of this warp's parity
      for (uint32_t n = base + ((base & 1u) != (uint32_t)wp ? 1u : 0u); n < base + (uint32_t)cnt; n += 2) {
        const uint32_t stage = n % kG2Stages, phase = (n / kG2Stages) & 1u;
        if (!g2_wait(&bars->full[stage], phase, bars, p.status)) {
          ok = false;
          break;
        }
        float sum[4];
        g2_tile(ring_s + stage * SB, a16_lane, R0, t, NKB2, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->empty[stage]);
        float* accr = p.acc + (size_t)(mt0 + (int)(n - base)) * 128 + R0;
        if (use0) {
          atomicAdd(accr + (size_t)tok0 * p.H, __fmul_rn(__fmul_rn(sum[0], s2), wt0));
          atomicAdd(accr + (size_t)tok0 * p.H + 8, __fmul_rn(__fmul_rn(sum[2], s2), wt0));
        }
        if (use1) {
          atomicAdd(accr + (size_t)tok1 * p.H, __fmul_rn(__fmul_rn(sum[1], s2), wt1));
          atomicAdd(accr + (size_t)tok1 * p.H + 8, __fmul_rn(__fmul_rn(sum[3], s2), wt1));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->afree[ab]);
      ab ^= 1u;
      if (ab == 0) aph ^= 1u;
      if (!ok) break;
    }
  }
}

size_t fc1_gemv_smem(int H) { return gv_smem_bytes(H); }

size_t fc2_gemv_smem(int I) { return g2_smem_bytes(I); }

cudaError_t gemv_set_attributes() {
  const cudaError_t err = cudaFuncSetAttribute((const void*)fc1_gemv_kernel,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemOptin);
  if (err != cudaSuccess) return err;
  return cudaFuncSetAttribute((const void*)fc2_gemv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kSmemOptin);
}

cudaError_t launch_fc2_gemv(const Fc2Args& a, int grid, cudaStream_t st) {
  Fc2Args args = a;
  void* kargs[] = {&args};
  return launch_with_pdl((const void*)fc2_gemv_kernel, dim3(grid), dim3(kG2Threads), g2_smem_bytes(a.I), st, kargs);
}

cudaError_t launch_fc1_gemv(const CUtensorMap& w13, const Fc1Args& a, int grid, cudaStream_t st) {
  CUtensorMap m0 = w13;
  Fc1Args args = a;
  void* kargs[] = {&m0, &args};
  return launch_with_pdl((const void*)fc1_gemv_kernel, dim3(grid), dim3(kGvThreads), gv_smem_bytes(a.H), st, kargs);
}

}  // namespace moe
