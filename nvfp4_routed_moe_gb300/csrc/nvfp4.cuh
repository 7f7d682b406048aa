// nvfp4.cuh -- device-side NVFP4 group quantizer and SiTU, used by the X
// quantization kernel, the FC1 epilogue and the test kernels alike.
//
// Group-16 quantization with encode scale q ("Cake SiTU backend": group-16
// NVFP4, qX = 1/dX, qA = 1/dA; "Nvfp4 Tensor": the global scale is applied
// after block dequantization):
//   amax = max |v_j|;  sf = E4M3_rn_sat((amax * q) / 6);  S = value(sf);
//   r = (S == 0) ? 0 : q / S;  code_j = E2M1_rn_sat(v_j * r).
// Every fp32 step is a separately rounded intrinsic (no contraction), so the
// codes are a deterministic function of the fp32 inputs.
#pragma once
#include "ptx.cuh"

namespace moe {

__device__ __forceinline__ uint32_t nvfp4_scale(float amax, float q, float& r) {
  const float t = __fmul_rn(amax, q);
  const float t6 = __fdiv_rn(t, 6.0f);
  const uint32_t sf = cvt_e4m3(t6);
  const float S = e4m3_to_f32(sf);
  r = (S == 0.0f) ? 0.0f : __fdiv_rn(q, S);
  return sf;
}

// One thread quantizes 16 values held in registers: 8 packed bytes (element
// 2i in the low nibble of byte i) and the E4M3 block-scale byte.
__device__ __forceinline__ uint32_t nvfp4_quant16(const float (&v)[16], float q, uint2& packed) {
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  float r;
  const uint32_t sf = nvfp4_scale(amax, q, r);
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const uint32_t b = cvt_e2m1x2(__fmul_rn(v[2 * i + 1], r), __fmul_rn(v[2 * i], r));
    w[i >> 2] |= b << (8 * (i & 3));
  }
  packed = make_uint2(w[0], w[1]);
  return sf;
}

// Lane-distributed form: each 16-lane half of the warp holds one group, one
// value per lane (lane l holds element l % 16).  Returns the block-scale byte
// (same in all 16 lanes of the group); `word` receives, in lanes with
// lane % 8 == 0, the 4 packed bytes of elements lane .. lane+7.
__device__ __forceinline__ uint32_t nvfp4_quant_lanes16(float a, float q, uint32_t& word) {
  float amax = fabsf(a);
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  float r;
  const uint32_t sf = nvfp4_scale(amax, q, r);
  uint32_t v = cvt_e2m1x2(0.0f, __fmul_rn(a, r)) & 0xFu;
  v |= (__shfl_down_sync(0xffffffffu, v, 1) & 0xFu) << 4;
  v = (v & 0xFFu) | ((__shfl_down_sync(0xffffffffu, v, 2) & 0xFFu) << 8);
  v = (v & 0xFFFFu) | ((__shfl_down_sync(0xffffffffu, v, 4) & 0xFFFFu) << 16);
  word = v;
  return sf;
}

// tanh from its definition: the odd Taylor series to y^9 for |y| < 1/4
// (truncation below 1e-8 relative there), else (1 - e^{-2|y|}) / (1 + e^{-2|y|})
// with the hardware exponential (relative error below 1e-6 for the result).
__device__ __forceinline__ float tanh_dev(float y) {
  const float a = fabsf(y);
  float t;
  if (a < 0.25f) {
    const float a2 = a * a;
    t = a * (1.0f + a2 * (-1.0f / 3.0f + a2 * (2.0f / 15.0f + a2 * (-17.0f / 315.0f + a2 * (62.0f / 2835.0f)))));
  } else {
    const float e = __expf(-2.0f * a);
    t = __fdividef(1.0f - e, 1.0f + e);
  }
  return copysignf(t, y);
}

// e^x by Cody-Waite range reduction (W. J. Cody and W. Waite, "Software
// Manual for the Elementary Functions", 1980): x log2(e) = n + f with n an
// integer and f in [-1/2, 1/2] computed with log2(e) split into two fp32
// parts, so the error of f no longer grows with |x|; e^x = 2^f 2^n, 2^f from
// the hardware base-2 exponential and 2^n from exponent bits.  Relative error
// a few 1e-7 (the hardware exponential's) over the whole fp32 range; +inf
// above about 88.7, 0 below about -87.3 (flushed), NaN for NaN.
__device__ __forceinline__ float exp_cw(float x) {
  constexpr float kLog2eHi = 1.44269502162933349609375f;   // fp32 nearest to log2(e)
  constexpr float kLog2eLo = 1.92596298909109e-08f;        // log2(e) - kLog2eHi
  const float t = fminf(fmaxf(x * kLog2eHi, -126.0f), 128.0f);
  const float n = rintf(t);
  const float f = fmaf(x, kLog2eHi, -n) + x * kLog2eLo;
  float p;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(p) : "f"(f));
  return p * __int_as_float(((int)n + 127) << 23);
}

// SiTU ("Cake SiTU backend": default (4*tanh(g/4)*sigmoid(g))*(25*tanh(u/25)),
// per-expert gate and linear smoothing parameters beta, lambda), with the
// reciprocals 1/beta and 1/lambda supplied by the caller.  The sigmoid divides
// approximately (2 ulp; exactly 0 once 1 + e^{-g} passes 2^126, where the
// sigmoid is below 1e-38).
__device__ __forceinline__ float situ_f32(float g, float u, float beta, float inv_beta, float lam, float inv_lam) {
  const float sig = __fdividef(1.0f, 1.0f + exp_cw(-g));
  const float gate = beta * tanh_dev(g * inv_beta) * sig;
  const float lin = lam * tanh_dev(u * inv_lam);
  return gate * lin;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// Byte offset of the block scale of (row, chunk) in the 128x4 atom layout
// ("Nvfp4 Tensor", block_scale) for a matrix with `kchunks` 16-element chunks
// per row (kchunks % 4 == 0).
__device__ __forceinline__ size_t atom_offset(int64_t row, int chunk, int kchunks) {
  return ((size_t)(row >> 7) * (size_t)(kchunks >> 2) + (size_t)(chunk >> 2)) * 512u + (size_t)(row & 31) * 16u +
         (size_t)((row >> 5) & 3) * 4u + (size_t)(chunk & 3);
}

}  // namespace moe
