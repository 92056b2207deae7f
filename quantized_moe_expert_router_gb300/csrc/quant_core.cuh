// quant_core.cuh -- NVFP4 quantization of activations with a static
// per-tensor input scale (the W4A4 numerics).
//
// The NVFP4 checkpoint of "Kimi-K3 on the same pod, two engines" (section
// "Same hardware, same weights") stores, beside each matrix's codes and e4m3
// block scales, two fp32 scalars: the weight scale and the input scale a.
// With W4A4 numerics the matrix's input is quantized the same way as the
// weights, with a in the role of the tensor scale:
//   per block of 16 consecutive elements:
//     s    = e4m3(max|v| / (6 a))        round to nearest even, saturating at 448
//     code = e2m1(v / (e4m3value(s) a))  round to nearest even, saturating at 6
//   (an all-zero block, or one whose s rounds to zero, gets zero codes), and
//   the quantized value is e2m1value(code) * e4m3value(s) * a.
// Every step is one correctly rounded fp32 operation (6 a, the quotient, the
// product s a, the quotient v / (s a)) or a rounding to a small format, so the
// bytes are a pure function of v and a.
//
// e2m1value(code) * e4m3value(s) has at most 2 + 4 significant bits and lies
// in [2^-10, 2688]: exact in f16.  The tensor-core paths feed that f16 value
// (not multiplied by a) to the MMA and apply a in the fp32 epilogue.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

// The block scale from the block's largest magnitude: returns the e4m3 byte,
// writes its value (f16, exact) and m = value * a (fp32), the divisor of the
// elements.
__device__ __forceinline__ uint8_t nvfp4_block_scale(float amax, float a, __half &sh, float &m) {
  const float denom = 6.0f * a;
  const float t = __fdiv_rn(amax, denom);
  const uint8_t sb = (uint8_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
  sh = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb, __NV_E4M3));
  m = __fmul_rn(__half2float(sh), a);
  return sb;
}

// One element: its e2m1 code and the value e2m1 * e4m3 (f16, exact); a zero
// block scale gives code 0.
__device__ __forceinline__ uint32_t nvfp4_element(float v, float m, __half sh, __half &val) {
  uint32_t c = 0u;
  val = __float2half_rn(0.f);
  if (__half2float(sh) > 0.f) {
    c = (uint32_t)__nv_cvt_float_to_fp4(__fdiv_rn(v, m), __NV_E2M1, cudaRoundNearest) & 0xFu;
    val = __hmul(__half(__nv_cvt_fp4_to_halfraw((__nv_fp4_storage_t)c, __NV_E2M1)), sh);
  }
  return c;
}

// Quantizes v[16] with input scale a: returns the e4m3 scale byte, writes the
// 16 codes (low nibble = even element, elements 0..7 in codes[0]) and the 16
// values e2m1 * e4m3 as f16 pairs (vals[j] = elements 2j, 2j+1; low half =
// even element).
__device__ __forceinline__ uint8_t nvfp4_quant_block(const float (&v)[16], float a, uint32_t (&codes)[2],
                                                     uint32_t (&vals)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
  __half sh;
  float m;
  const uint8_t sb = nvfp4_block_scale(amax, a, sh, m);
  codes[0] = codes[1] = 0u;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    __half h0, h1;
    const uint32_t c0 = nvfp4_element(v[2 * j], m, sh, h0);
    const uint32_t c1 = nvfp4_element(v[2 * j + 1], m, sh, h1);
    codes[j >> 2] |= (c0 | (c1 << 4)) << (8 * (j & 3));
    const __half2 hv = __halves2half2(h0, h1);
    vals[j] = *reinterpret_cast<const uint32_t *>(&hv);
  }
  return sb;
}

// The same quantization spread over the four lanes q = 0..3 of an MMA
// fragment quad: this lane holds elements 2q, 2q+1 (v0, v1) and 2q+8, 2q+9
// (v2, v3) of a 16-element block, the quad together the whole block.  Writes
// this lane's four values as two f16 pairs (the B fragment registers).  All
// 32 lanes of the warp must call it.
__device__ __forceinline__ void nvfp4_quant_quad(float v0, float v1, float v2, float v3, float a, uint32_t &b0,
                                                 uint32_t &b1) {
  float amax = fmaxf(fmaxf(fabsf(v0), fabsf(v1)), fmaxf(fabsf(v2), fabsf(v3)));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  __half sh;
  float m;
  nvfp4_block_scale(amax, a, sh, m);
  __half h0, h1, h2, h3;
  nvfp4_element(v0, m, sh, h0);
  nvfp4_element(v1, m, sh, h1);
  nvfp4_element(v2, m, sh, h2);
  nvfp4_element(v3, m, sh, h3);
  const __half2 p0 = __halves2half2(h0, h1), p1 = __halves2half2(h2, h3);
  b0 = *reinterpret_cast<const uint32_t *>(&p0);
  b1 = *reinterpret_cast<const uint32_t *>(&p1);
}

}  // namespace moe
