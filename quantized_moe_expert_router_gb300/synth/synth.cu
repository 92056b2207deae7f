// synth.cu -- device twin of the host weight generator in synth/__init__.py.
//
// Generates canonical NVFP4 and MXFP4 expert matrices (codes, scales) from the same
// SplitMix64 counter streams, the same Irwin-Hall(8) normal deviates and the
// same NVFP4 / MXFP4 encoders, bit for bit: every step is an integer operation, a
// comparison, or one correctly rounded float64 operation (built with
// -fmad=false so no multiply-add is fused).  Input generation only: nothing
// here decodes weights or computes any part of the MoE layer.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t splitmix64(uint64_t z) {
  z += kGolden;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ int64_t ih8_sum(uint64_t key, uint64_t i) {
  int64_t s = 0;
  for (int j = 0; j < 2; j++) {
    const uint64_t d = splitmix64(key + (2 * i + j) * kGolden);
    s += (int64_t)(d & 0xFFFF) + (int64_t)((d >> 16) & 0xFFFF) + (int64_t)((d >> 32) & 0xFFFF) +
         (int64_t)(d >> 48);
  }
  return s;
}

// e4m3 round-to-nearest-even of v >= 0, saturating at 448; returns the code
// and its exact value.
__device__ void e4m3_encode(double v, uint32_t *code, double *val) {
  if (v >= 448.0) { *code = 0x7E; *val = 448.0; return; }
  if (v < 0.015625) {                      // below 2^-6: multiples of 2^-9
    const double q = rint(v * 512.0);
    if (q >= 8.0) { *code = 0x08; *val = 0.015625; }
    else { *code = (uint32_t)q; *val = q * 0.001953125; }
    return;
  }
  int ex;
  const double m = frexp(v, &ex);          // v = m 2^ex, m in [0.5, 1)
  int e = ex - 1;
  double q = rint((2.0 * m - 1.0) * 8.0);
  if (q >= 8.0) { e += 1; q = 0.0; }
  if (e > 8) { *code = 0x7E; *val = 448.0; return; }
  *code = (uint32_t)(((e + 7) << 3) | (int)q);
  *val = ldexp(1.0 + q / 8.0, e);
}

__device__ __forceinline__ uint32_t e2m1_encode(double w, double sg) {
  const double a = fabs(w);
  uint32_t mag = 7;
  if (a <= 5.0 * sg) mag = 6;
  if (a < 3.5 * sg) mag = 5;
  if (a <= 2.5 * sg) mag = 4;
  if (a < 1.75 * sg) mag = 3;
  if (a <= 1.25 * sg) mag = 2;
  if (a < 0.75 * sg) mag = 1;
  if (a <= 0.25 * sg) mag = 0;
  return (w < 0.0 && mag != 0) ? (mag | 8u) : mag;
}

// One thread per 16-element block of one matrix of one expert.
__global__ void gen_matrix_kernel(const uint64_t *keys, const float *g, int n, int rows, int K,
                                  double w_coef, uint8_t *codes, uint8_t *scales) {
  const int64_t blocks_per_row = K / 16;
  const int64_t per_expert = (int64_t)rows * blocks_per_row;
  const int64_t total = per_expert * n;
  for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < total;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = blk / per_expert, rb = blk % per_expert;
    const int64_t r = rb / blocks_per_row, bb = rb % blocks_per_row;
    const uint64_t key = keys[e];
    const uint64_t i0 = (uint64_t)(r * K + bb * 16);
    double w[16];
    double amax = 0.0;
    for (int j = 0; j < 16; j++) {
      w[j] = ((double)ih8_sum(key, i0 + j) - 262140.0) * w_coef;
      amax = fmax(amax, fabs(w[j]));
    }
    uint32_t scode = 0;
    double sval = 0.0;
    if (amax != 0.0) e4m3_encode(amax / (6.0 * (double)g[e]), &scode, &sval);
    const double sg = sval * (double)g[e];
    uint32_t c[16];
    for (int j = 0; j < 16; j++) c[j] = (sg > 0.0) ? e2m1_encode(w[j], sg) : 0u;
    uint2 out;
    out.x = c[0] | (c[1] << 4) | (c[2] << 8) | (c[3] << 12) | (c[4] << 16) | (c[5] << 20) |
            (c[6] << 24) | (c[7] << 28);
    out.y = c[8] | (c[9] << 4) | (c[10] << 8) | (c[11] << 12) | (c[12] << 16) | (c[13] << 20) |
            (c[14] << 24) | (c[15] << 28);
    *reinterpret_cast<uint2 *>(codes + e * (per_expert * 8) + rb * 8) = out;
    scales[e * per_expert + rb] = (uint8_t)scode;
  }
}

// One thread per 32-element block (MXFP4, OCP MX): shared exponent
// e = floor(log2 amax) - 2 clamped to [-127, 127] (-127 for an all-zero
// block), scale byte e + 127, codes = nearest e2m1 of w / 2^e.
__global__ void gen_matrix_mx_kernel(const uint64_t *keys, int n, int rows, int K, double w_coef, uint8_t *codes,
                                     uint8_t *scales) {
  const int64_t blocks_per_row = K / 32;
  const int64_t per_expert = (int64_t)rows * blocks_per_row;
  const int64_t total = per_expert * n;
  for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < total;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = blk / per_expert, rb = blk % per_expert;
    const int64_t r = rb / blocks_per_row, bb = rb % blocks_per_row;
    const uint64_t key = keys[e];
    const uint64_t i0 = (uint64_t)(r * K + bb * 32);
    double w[32];
    double amax = 0.0;
    for (int j = 0; j < 32; j++) {
      w[j] = ((double)ih8_sum(key, i0 + j) - 262140.0) * w_coef;
      amax = fmax(amax, fabs(w[j]));
    }
    int ex = 0;
    if (amax > 0.0) frexp(amax, &ex);
    int sh = amax > 0.0 ? ex - 1 - 2 : -127;
    sh = sh < -127 ? -127 : (sh > 127 ? 127 : sh);
    const double sc = ldexp(1.0, sh);
    uint32_t c[32];
    for (int j = 0; j < 32; j++) c[j] = e2m1_encode(w[j], sc);
    uint32_t out[4];
    for (int q = 0; q < 4; q++) {
      out[q] = 0;
      for (int j = 0; j < 8; j++) out[q] |= c[8 * q + j] << (4 * j);
    }
    *reinterpret_cast<uint4 *>(codes + e * (per_expert * 16) + rb * 16) = make_uint4(out[0], out[1], out[2], out[3]);
    scales[e * per_expert + rb] = (uint8_t)(sh + 127);
  }
}

}  // namespace

extern "C" {

// Canonical MXFP4 [n][rows][K/2] codes and [n][rows][K/32] e8m0 scales of one
// matrix kind for n experts (the same weight draws as the NVFP4 generator).
int synth_generate_matrices_mx(const uint64_t *keys, int n, int rows, int K, double w_coef, uint8_t *codes,
                               uint8_t *scales, cudaStream_t stream) {
  if (n <= 0 || rows <= 0 || K <= 0 || K % 32) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  gen_matrix_mx_kernel<<<sms * 8, 256, 0, stream>>>(keys, n, rows, K, w_coef, codes, scales);
  return (int)cudaGetLastError();
}


// Canonical NVFP4 [n][rows][K/2] codes and [n][rows][K/16] scales of one
// matrix kind for n experts; keys[n] (device) are the per-expert stream keys,
// g[n] (device) the fp32 global scales, w_coef the float64 factor that turns
// a centred Irwin-Hall sum into a weight.  Returns a cudaError_t value.
int synth_generate_matrices(const uint64_t *keys, const float *g, int n, int rows, int K,
                            double w_coef, uint8_t *codes, uint8_t *scales, cudaStream_t stream) {
  if (n <= 0 || rows <= 0 || K <= 0 || K % 16) return (int)cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  gen_matrix_kernel<<<sms * 8, 256, 0, stream>>>(keys, g, n, rows, K, w_coef, codes, scales);
  return (int)cudaGetLastError();
}

}  // extern "C"
