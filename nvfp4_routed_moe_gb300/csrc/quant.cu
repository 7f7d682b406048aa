// quant.cu -- activation quantization (token-major codes, block scales laid
// out for the padded expanded rows), the BF16 finalize, weight preparation
// into the kernel layout, and the test kernels that expose the device
// quantizer and codecs.
#include <cuda_bf16.h>

#include "nvfp4.cuh"
#include "plan.h"

namespace moe {

cudaError_t launch_with_pdl(const void* fn, dim3 grid, dim3 block, size_t smem, cudaStream_t st, void** args);

// ------------------------------------------------------------ X quantization
// Each lane quantizes one 16-element group of a token ("Cake SiTU backend":
// group-16 NVFP4 input quantization with qX) once and writes the codes once,
// to the token's row of the token-major codes; FC1 gathers them per tile row
// ("npu_moe_init_routing_v2", formula 5, gather form: expandedX[gatherRowIdx[i]]
// = quantResult[i // k], carried out as the GEMM's operand load).  The block
// scales go to the padded expanded row of every pair the token is routed to,
// in the atom layout the MMA's scale copies take.  It also
// stores each pair's route weight (fp32) at the pair's padded row for FC2,
// and zeroes the token's fp32 combine accumulator row, into which FC2 adds
// the token's route-weighted expert outputs.  Block scales go straight into
// the atom layout of every routed row (up to 4096 routed pairs), or, above that,
// once per token into token-major rows that sf_atoms_kernel then lays out
// with whole-atom writes (a token's scales land in 56 different atoms, and
// scattered 4-byte writes cost more than the extra pass).  When FC1 runs on
// the decode kernel (small batches) it reads the token-major scales itself:
// then no atoms are written and this kernel stores the route weights.
__global__ void __launch_bounds__(256) quant_x_kernel(const QuantXArgs a) {
  // Warp w takes 32 groups (512 elements) of token w / S, S = ceil(H/512)
  // slices per token, so a token's slices run in parallel warps.
  const int lane = threadIdx.x & 31;
  const int H = a.H, G = H / 16, KC = H / 16, S = (G + 31) / 32;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t t = w / S;
  const int sl = (int)(w - t * S);
  // The token-major work (codes, token-major scales, the accumulator row)
  // needs nothing from routing, so it does not wait for it: the routing
  // kernel before this one starts only once the previous forward has
  // completed, so nothing still reads the codes or the accumulator.  Only
  // the row-position work below waits.  With token-major scales the route
  // weights are placed by the scale-atom kernel, and one thread waits so
  // that this kernel still completes after routing.
  const bool atom_pass = a.sft && a.sfx;   // token-major scales, laid out by sf_atoms_kernel
  pdl_launch_dependents();
  if (atom_pass && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
  if (t >= a.T) return;
  const float q = __ldg(a.qX);
  // this slice's share of the token's accumulator row
  float4* accr = reinterpret_cast<float4*>(a.acc + t * H);
  for (int i = sl * 32 * 4 + lane; i < min(H / 4, (sl + 1) * 32 * 4); i += 32) accr[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  const uint4* xr = reinterpret_cast<const uint4*>(a.x + t * H);
  const int g = sl * 32 + lane;
  const bool valid = g < G;
  float v[16];
  if (valid) {
    const uint4 u0 = __ldg(xr + 2 * g), u1 = __ldg(xr + 2 * g + 1);
    const uint32_t wd[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[2 * i] = bf16_bits_to_f32(wd[i] & 0xFFFFu);
      v[2 * i + 1] = bf16_bits_to_f32(wd[i] >> 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = 0.f;
  }
  uint2 packed;
  const uint32_t sf = nvfp4_quant16(v, q, packed);
  // four consecutive groups share one 32-bit word of a scale atom row
  uint32_t word = sf << (8 * (lane & 3));
  word |= __shfl_xor_sync(0xffffffffu, word, 1);
  word |= __shfl_xor_sync(0xffffffffu, word, 2);
  if (a.sft && valid && (lane & 3) == 0) *reinterpret_cast<uint32_t*>(a.sft + t * G + g) = word;
  if (valid) *reinterpret_cast<uint2*>(a.xq + (size_t)t * (H / 2) + g * 8) = packed;
  if (atom_pass) return;
  pdl_wait();   // routing's row positions
  const int rp = (lane < a.k) ? a.row_pos[t * a.k + lane] : -1;
  if (sl == 0 && rp >= 0 && rp < a.max_rows) a.wrow[rp] = bf16_bits_to_f32(a.route_w[t * a.k + lane]);
  if (!a.sfx) return;
  for (int j = 0; j < a.k; ++j) {
    const int row = __shfl_sync(0xffffffffu, rp, j);
    if (row < 0 || row >= a.max_rows || !valid) continue;
    if ((lane & 3) == 0) *reinterpret_cast<uint32_t*>(a.sfx + atom_offset(row, g, KC)) = word;
  }
}

// ------------------------------------------------------------ scale atoms
// One warp per 128-row tile ("Nvfp4 Tensor", block-scale atom: the scale of
// padded row r, 16-element group g sits at byte (r%32)*16 + ((r%128)/32)*4 +
// g%4 of atom (r/128, g/4)): lane l owns rows l, l+32, l+64, l+96 of the
// tile.  Per step it loads 16 scale bytes (groups 16m..16m+15) of each of
// its four rows' tokens from the token-major scales and writes the 16-byte
// chunk l of atoms 4m..4m+3, word c of a chunk from row l + 32c, so a warp
// store covers one whole 512-byte atom.  Rows past a tile's fill are zero.
__global__ void __launch_bounds__(256, 4) sf_atoms_kernel(const SfAtomArgs a) {
  pdl_wait();
  pdl_launch_dependents();
  const int ntiles = min(a.hdr[HDR_NUM_TT], a.max_tiles);
  const int lane = threadIdx.x & 31, NA4 = a.H / 64, G = a.H / 16, NM = a.H / 256;
  const int4* tiles = reinterpret_cast<const int4*>(a.tt_list);
  uint4* atoms = reinterpret_cast<uint4*>(a.sfx);
  // Warp w takes the 256-column steps [kB * (w % NH), + kB) of tile w / NH:
  // a tile's steps are shared by NH warps with few registers each, so that
  // many warps, and their loads, are in flight on every SM.
  constexpr int kB = 2;
  const int NH = (NM + kB - 1) / kB;
  const int64_t nwarps = (int64_t)gridDim.x * 8;
  for (int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5); w < (int64_t)ntiles * NH; w += nwarps) {
    const int64_t tile = w / NH;
    const int m0 = (int)(w - tile * NH) * kB;
    const int rows = __ldg(&tiles[tile].z);
    const uint4* src[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int r = lane + 32 * c;
      const int f = r < rows ? __ldg(a.prow_pair + tile * kTileRows + r) : -1;
      const bool ok = f >= 0 && f < a.num_pairs;
      src[c] = ok ? reinterpret_cast<const uint4*>(a.sft + (int64_t)(f / a.k) * G) : nullptr;
      if (ok && m0 == 0) a.wrow[tile * kTileRows + r] = bf16_bits_to_f32(__ldg(a.route_w + f));
    }
    uint4* dst = atoms + tile * NA4 * 32 + lane;
    // kB 256-column steps (4 kB gathered 16-byte loads per lane) in flight
    // before their atoms are written
    uint4 v[kB][4];
#pragma unroll
    for (int i = 0; i < kB; ++i)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        v[i][c] = (m0 + i < NM && src[c]) ? __ldg(src[c] + m0 + i) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int i = 0; i < kB; ++i) {
      if (m0 + i >= NM) break;
      uint4* d = dst + 4 * (m0 + i) * 32;
      d[0] = make_uint4(v[i][0].x, v[i][1].x, v[i][2].x, v[i][3].x);
      d[32] = make_uint4(v[i][0].y, v[i][1].y, v[i][2].y, v[i][3].y);
      d[64] = make_uint4(v[i][0].z, v[i][1].z, v[i][2].z, v[i][3].z);
      d[96] = make_uint4(v[i][0].w, v[i][1].w, v[i][2].w, v[i][3].w);
    }
  }
}

// ------------------------------------------------------------------ finalize
// out[t, h] = bf16_rn(acc[t, h]) ("Cake SiTU backend": BF16 weighted
// finalization).  FC2 has added every routed pair's route-weighted output
// into acc in fp32; this rounds once.  One thread per 8 consecutive outputs.
__global__ void __launch_bounds__(256) finalize_kernel(const float* __restrict__ acc, uint16_t* __restrict__ out,
                                                       int64_t n8) {
  pdl_wait();
  pdl_launch_dependents();
  const float4* src = reinterpret_cast<const float4*>(acc);
  uint4* dst = reinterpret_cast<uint4*>(out);
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n8; i += (int64_t)gridDim.x * 256) {
    const float4 a = __ldcs(src + 2 * i), b = __ldcs(src + 2 * i + 1);
    uint32_t w[4];
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
      w[j] = *reinterpret_cast<const uint32_t*>(&h);
    }
    dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// --------------------------------------------------------- weight preparation
// Kernel layout of the prepared weights:
//   W13 codes  [E][I/64][H/256][128 rows][128 B]: tile row 2i is the gate row
//              of feature it*64 + i, row 2i+1 the matching up row;
//   W13 scales [E][I/64][H/256][4 atoms][512 B] over the same tile rows;
//   W2 codes   [E][H/128][I/128][128 rows][64 B];
//   W2 scales  [E][H/128][I/64 atoms][512 B];
// atoms in the 128x4 layout of the "Nvfp4 Tensor" page (block_scale).
__global__ void __launch_bounds__(256) prep_w13_codes_kernel(const PrepArgs a) {
  const int NIT = a.I / 64, NKB = a.H / 256;
  const int64_t units = (int64_t)a.E * 2 * a.I * (a.H / 2) / 16;
  for (int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x; u < units; u += (int64_t)gridDim.x * 256) {
    const int64_t o = u * 16;
    const int64_t tile = o / 16384;            // (e*NIT + it)*NKB + kb
    const int r = (int)((o / 128) % 128), byte = (int)(o % 128);
    const int kb = (int)(tile % NKB), it = (int)((tile / NKB) % NIT);
    const int64_t e = tile / ((int64_t)NKB * NIT);
    const int64_t src_row = e * 2 * a.I + (r & 1) * a.I + it * 64 + (r >> 1);
    const uint4 v = *reinterpret_cast<const uint4*>(a.w13 + src_row * (a.H / 2) + kb * 128 + byte);
    *reinterpret_cast<uint4*>(a.w13o + o) = v;
  }
}

__global__ void __launch_bounds__(256) prep_w13_sf_kernel(const PrepArgs a) {
  const int NIT = a.I / 64, NKB = a.H / 256;
  const int64_t n = (int64_t)a.E * 2 * a.I * (a.H / 16);
  for (int64_t o = (int64_t)blockIdx.x * 256 + threadIdx.x; o < n; o += (int64_t)gridDim.x * 256) {
    const int within = (int)(o % 512);
    const int64_t atom = o / 512;             // ((e*NIT + it)*NKB + kb)*4 + kt
    const int kt = (int)(atom % 4);
    const int64_t tile = atom / 4;
    const int kb = (int)(tile % NKB), it = (int)((tile / NKB) % NIT);
    const int64_t e = tile / ((int64_t)NKB * NIT);
    const int r = (within & 15) / 4 * 32 + within / 16;   // tile row: innerM*32 + outerM
    const int c = kb * 16 + kt * 4 + (within & 3);
    const int64_t src_row = e * 2 * a.I + (r & 1) * a.I + it * 64 + (r >> 1);
    a.sf13o[o] = a.sf13[src_row * (a.H / 16) + c];
  }
}

__global__ void __launch_bounds__(256) prep_w2_codes_kernel(const PrepArgs a) {
  const int NMT = a.H / 128, NKB2 = a.I / 128;
  const int64_t units = (int64_t)a.E * a.H * (a.I / 2) / 16;
  for (int64_t u = (int64_t)blockIdx.x * 256 + threadIdx.x; u < units; u += (int64_t)gridDim.x * 256) {
    const int64_t o = u * 16;
    const int64_t tile = o / 8192;            // (e*NMT + mt)*NKB2 + kb
    const int r = (int)((o / 64) % 128), byte = (int)(o % 64);
    const int kb = (int)(tile % NKB2), mt = (int)((tile / NKB2) % NMT);
    const int64_t e = tile / ((int64_t)NKB2 * NMT);
    const int64_t src_row = e * a.H + mt * 128 + r;
    const uint4 v = *reinterpret_cast<const uint4*>(a.w2 + src_row * (a.I / 2) + kb * 64 + byte);
    *reinterpret_cast<uint4*>(a.w2o + o) = v;
  }
}

__global__ void __launch_bounds__(256) prep_w2_sf_kernel(const PrepArgs a) {
  const int NMT = a.H / 128, NA = a.I / 64;
  const int64_t n = (int64_t)a.E * a.H * (a.I / 16);
  for (int64_t o = (int64_t)blockIdx.x * 256 + threadIdx.x; o < n; o += (int64_t)gridDim.x * 256) {
    const int within = (int)(o % 512);
    const int64_t atom = o / 512;             // (e*NMT + mt)*NA + a
    const int at = (int)(atom % NA);
    const int64_t tile = atom / NA;
    const int mt = (int)(tile % NMT);
    const int64_t e = tile / NMT;
    const int rr = (within & 15) / 4 * 32 + within / 16;
    const int c = at * 4 + (within & 3);
    const int64_t src_row = e * a.H + mt * 128 + rr;
    a.sf2o[o] = a.sf2[src_row * (a.I / 16) + c];
  }
}

// --------------------------------------------------------------- test kernels
__global__ void __launch_bounds__(256) codec_sweep_kernel(uint32_t start, int64_t n, uint8_t* lo, uint8_t* hi,
                                                          uint8_t* e4) {
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const float v = __uint_as_float(start + (uint32_t)i);
    if (lo) lo[i] = (uint8_t)(cvt_e2m1x2(0.0f, v) & 0xFu);
    if (hi) hi[i] = (uint8_t)(cvt_e2m1x2(v, 0.0f) >> 4);
    if (e4) e4[i] = (uint8_t)cvt_e4m3(v);
  }
}

__global__ void __launch_bounds__(256) quant_rows_kernel(const float* x, int64_t rows, int cols, const float* qpr,
                                                         uint8_t* packed, uint8_t* sf) {
  const int G = cols / 16;
  const int64_t n = rows * G;
  for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
    const int64_t r = i / G;
    const int g = (int)(i % G);
    float v[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = x[r * cols + g * 16 + j];
    uint2 p;
    sf[i] = (uint8_t)nvfp4_quant16(v, qpr[r], p);
    *reinterpret_cast<uint2*>(packed + r * (cols / 2) + g * 8) = p;
  }
}

// One warp per (row, 32 features): the FC1 epilogue's per-lane SiTU and
// 16-lane requant, written in the canonical layout.
__global__ void __launch_bounds__(256) situ_requant_kernel(const float* z, int64_t rows, int I, float qA, float beta,
                                                           float lam, float* a_out, uint8_t* packed, uint8_t* sf) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int per_row = I / 32;
  if (w >= rows * per_row) return;
  const int64_t r = w / per_row;
  const int f = (int)(w % per_row) * 32 + lane;
  const float g = z[r * 2 * I + f], u = z[r * 2 * I + I + f];
  const float act = situ_f32(g, u, beta, 1.0f / beta, lam, 1.0f / lam);
  a_out[r * I + f] = act;
  uint32_t word;
  const uint32_t s = nvfp4_quant_lanes16(act, qA, word);
  if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(packed + r * (I / 2) + f / 2) = word;
  if ((lane & 15) == 0) sf[r * (I / 16) + f / 16] = (uint8_t)s;
}

// The FC1 epilogue's 16-lane requant alone, on given activations.
__global__ void __launch_bounds__(256) requant_lanes_kernel(const float* act, int64_t rows, int I, float qA,
                                                            uint8_t* packed, uint8_t* sf) {
  const int lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int per_row = I / 32;
  if (w >= rows * per_row) return;
  const int64_t r = w / per_row;
  const int f = (int)(w % per_row) * 32 + lane;
  uint32_t word;
  const uint32_t s = nvfp4_quant_lanes16(act[r * I + f], qA, word);
  if ((lane & 7) == 0) *reinterpret_cast<uint32_t*>(packed + r * (I / 2) + f / 2) = word;
  if ((lane & 15) == 0) sf[r * (I / 16) + f / 16] = (uint8_t)s;
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_quant_x(const QuantXArgs& a, cudaStream_t st) {
  QuantXArgs args = a;
  void* kargs[] = {&args};
  const int64_t warps = a.T * ((a.H / 16 + 31) / 32);
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  return launch_with_pdl((const void*)quant_x_kernel, dim3(blocks), dim3(256), 0, st, kargs);
}

cudaError_t launch_sf_atoms(const SfAtomArgs& a, int64_t max_tiles, int num_sms, cudaStream_t st) {
  SfAtomArgs args = a;
  void* kargs[] = {&args};
  const int64_t want = (max_tiles * ((a.H / 256 + 1) / 2) + 7) / 8;   // a warp per 2 column steps of a tile
  const unsigned blocks = (unsigned)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  return launch_with_pdl((const void*)sf_atoms_kernel, dim3(blocks ? blocks : 1), dim3(256), 0, st, kargs);
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t T, int H, int num_sms, cudaStream_t st) {
  int64_t n8 = T * (H / 8);
  void* kargs[] = {(void*)&acc, (void*)&out, (void*)&n8};
  const int64_t want = (n8 + 255) / 256;
  const unsigned blocks = (unsigned)(want < (int64_t)num_sms * 8 ? want : (int64_t)num_sms * 8);
  return launch_with_pdl((const void*)finalize_kernel, dim3(blocks ? blocks : 1), dim3(256), 0, st, kargs);
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t st, int num_sms) {
  PrepArgs args = a;
  dim3 grid(num_sms * 8), block(256);
  prep_w13_codes_kernel<<<grid, block, 0, st>>>(args);
  prep_w13_sf_kernel<<<grid, block, 0, st>>>(args);
  prep_w2_codes_kernel<<<grid, block, 0, st>>>(args);
  prep_w2_sf_kernel<<<grid, block, 0, st>>>(args);
  return cudaGetLastError();
}

cudaError_t launch_codec_sweep(uint32_t start, int64_t n, uint8_t* lo, uint8_t* hi, uint8_t* e4, cudaStream_t st,
                               int num_sms) {
  codec_sweep_kernel<<<num_sms * 16, 256, 0, st>>>(start, n, lo, hi, e4);
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const float* x, int64_t rows, int cols, const float* qpr, uint8_t* packed, uint8_t* sf,
                              cudaStream_t st, int num_sms) {
  quant_rows_kernel<<<num_sms * 8, 256, 0, st>>>(x, rows, cols, qpr, packed, sf);
  return cudaGetLastError();
}

cudaError_t launch_situ_requant(const float* z, int64_t rows, int I, float qA, float beta, float lam, float* a_out,
                                uint8_t* packed, uint8_t* sf, cudaStream_t st) {
  const int64_t warps = rows * (I / 32);
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  situ_requant_kernel<<<blocks ? blocks : 1, 256, 0, st>>>(z, rows, I, qA, beta, lam, a_out, packed, sf);
  return cudaGetLastError();
}

cudaError_t launch_requant_lanes(const float* act, int64_t rows, int I, float qA, uint8_t* packed, uint8_t* sf,
                                 cudaStream_t st) {
  const int64_t warps = rows * (I / 32);
  const unsigned blocks = (unsigned)((warps + 7) / 8);
  requant_lanes_kernel<<<blocks ? blocks : 1, 256, 0, st>>>(act, rows, I, qA, packed, sf);
  return cudaGetLastError();
}

}  // namespace moe
