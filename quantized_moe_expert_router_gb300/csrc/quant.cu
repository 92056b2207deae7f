// quant.cu -- the W4A4 activation quantizer as a standalone call
// (moe_quantize_nvfp4): one thread per block of 16 elements, the block
// quantized by nvfp4_quant_block (quant_core.cuh), the code a W4A4 layer's
// kernels run on x and h.
#include <math.h>

#include "moe.h"
#include "quant_core.cuh"

namespace moe {

template <bool F32>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(const void *src, long long blocks, float a,
                                                              uint8_t *codes, uint8_t *scales) {
  for (long long b = blockIdx.x * (long long)blockDim.x + threadIdx.x; b < blocks;
       b += (long long)gridDim.x * blockDim.x) {
    float v[16];
    if constexpr (F32) {
      const float4 *p = reinterpret_cast<const float4 *>(src) + 4 * b;
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float4 f = __ldg(p + i);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
    } else {
      const uint4 *p = reinterpret_cast<const uint4 *>(src) + 2 * b;
      const uint4 u0 = __ldg(p), u1 = __ldg(p + 1);
      const uint32_t w[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
      for (int i = 0; i < 8; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
    uint32_t c[2], vals[8];
    scales[b] = nvfp4_quant_block(v, a, c, vals);
    reinterpret_cast<uint2 *>(codes)[b] = make_uint2(c[0], c[1]);
  }
}

}  // namespace moe

extern "C" moe_status moe_quantize_nvfp4(const void *src, int32_t src_dtype, int64_t rows, int32_t n, float a,
                                         uint8_t *codes, uint8_t *scales, cudaStream_t stream) {
  if (!src || !codes || !scales || rows < 1 || n < 16 || n % 16) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(codes)) & 15u) return MOE_ERR_INVALID_ARG;
  if (src_dtype != MOE_ACT_BF16 && src_dtype != MOE_ACT_F32) return MOE_ERR_INVALID_ARG;
  if (!(a > 0.f) || !isfinite(a)) return MOE_ERR_INVALID_ARG;
  const long long blocks = rows * (long long)(n / 16);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ERR_CUDA;
  long long grid = (blocks + 255) / 256;
  if (grid > 8LL * sms) grid = 8LL * sms;
  if (src_dtype == MOE_ACT_F32)
    moe::quantize_nvfp4_kernel<true><<<(unsigned)grid, 256, 0, stream>>>(src, blocks, a, codes, scales);
  else
    moe::quantize_nvfp4_kernel<false><<<(unsigned)grid, 256, 0, stream>>>(src, blocks, a, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
