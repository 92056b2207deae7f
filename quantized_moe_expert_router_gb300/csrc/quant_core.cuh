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

// Quantizes v[16] with input scale a: returns the e4m3 scale byte, writes the
// 16 codes (low nibble = even element, elements 0..7 in codes[0]) and the 16
// values e2m1 * e4m3 as f16 pairs (vals[j] = elements 2j, 2j+1; low half =
// even element).
__device__ __forceinline__ uint8_t nvfp4_quant_block(const float (&v)[16], float a, uint32_t (&codes)[2],
                                                     uint32_t (&vals)[8]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[i]));
  const float denom = 6.0f * a;
  const float t = __fdiv_rn(amax, denom);
  const uint8_t sb = (uint8_t)__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
  const __half sh = __half(__nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sb, __NV_E4M3));
  const float sv = __half2float(sh);
  const float m = __fmul_rn(sv, a);
  codes[0] = codes[1] = 0u;
#pragma unroll
  for (int j = 0; j < 8; j++) {
    uint32_t c2[2] = {0u, 0u};
    __half h2[2] = {__float2half_rn(0.f), __float2half_rn(0.f)};
#pragma unroll
    for (int b = 0; b < 2; b++) {
      if (sv > 0.f) {
        const uint32_t c = (uint32_t)__nv_cvt_float_to_fp4(__fdiv_rn(v[2 * j + b], m), __NV_E2M1, cudaRoundNearest) & 0xFu;
        c2[b] = c;
        h2[b] = __hmul(__half(__nv_cvt_fp4_to_halfraw((__nv_fp4_storage_t)c, __NV_E2M1)), sh);
      }
    }
    codes[j >> 2] |= (c2[0] | (c2[1] << 4)) << (8 * (j & 3));
    const __half2 hv = __halves2half2(h2[0], h2[1]);
    vals[j] = *reinterpret_cast<const uint32_t *>(&hv);
  }
  return sb;
}

}  // namespace moe
