// pack_core.cuh -- the byte moves of one K-slice of one pair row of a packed
// tile (see pack.cu for the layout), shared by the expert packer and the
// packer of the dense matrices around the routed sum.
#pragma once

#include "moe_internal.cuh"

namespace moe {

__device__ __forceinline__ bool e4m3_is_nan(uint32_t b) { return (b & 0x7F) == 0x7F; }

// Slice w (k-steps 32w .. 32w + 31) of the source rows, written as slice wd
// of pair row g of a tile starting at tb (W slices): rowA codes/scales
// ca/sa, rowB cb/sb, real K (zero codes and scales past it).  NVFP4 (mx
// false): e4m3 scales per 16 elements; MXFP4: e8m0 per 32.  Returns 1 if a
// NaN scale byte was seen.
__device__ __forceinline__ int pack_pair_slice(const uint8_t *ca, const uint8_t *cb, const uint8_t *sa,
                                               const uint8_t *sb, int K, bool mx, int w, int wd, int g, int W,
                                               uint8_t *tb) {
  int nan_seen = 0;
  // code bytes of this slice (k-steps 32w .. 32w+31), zero past K
  const int kstep0 = 32 * w, ksteps = K / 16;
#pragma unroll 1
  for (int qg = 0; qg < 8; qg++) {                     // groups of 4 k-steps
    uint32_t words[4][4];                              // [lane q][k-step j]
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
      const int s = kstep0 + 4 * qg + jj;
      uint2 A = make_uint2(0, 0), B = make_uint2(0, 0);
      if (s < ksteps) {
        A = *reinterpret_cast<const uint2 *>(ca + 8 * s);
        B = *reinterpret_cast<const uint2 *>(cb + 8 * s);
      }
      const uint8_t *ab = reinterpret_cast<const uint8_t *>(&A);
      const uint8_t *bb = reinterpret_cast<const uint8_t *>(&B);
#pragma unroll
      for (int q = 0; q < 4; q++)
        words[q][jj] = (uint32_t)ab[q] | ((uint32_t)bb[q] << 8) | ((uint32_t)ab[q + 4] << 16) |
                       ((uint32_t)bb[q + 4] << 24);
    }
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int lane = 4 * g + q;
      *reinterpret_cast<uint4 *>(tb + (size_t)wd * 4096 + ((size_t)qg * 32 + lane) * 16) =
          make_uint4(words[q][0], words[q][1], words[q][2], words[q][3]);
    }
  }
  uint8_t *sbase = tb + (size_t)W * 4096;
  if (mx) {
    // MXFP4: per slice 2 units (k-steps 16u .. 16u + 15 = k-step pairs
    // 8u .. 8u + 7) of [8 rows g][16 bytes]: (rowA, rowB) e8m0 bytes of
    // each pair
    const int pair0 = kstep0 / 2, npairs = K / 32;
#pragma unroll 1
    for (int u = 0; u < 2; u++) {
      uint32_t sw[4];
#pragma unroll
      for (int h = 0; h < 4; h++) {
        uint32_t v = 0;
#pragma unroll
        for (int i2 = 0; i2 < 2; i2++) {
          const int P = pair0 + 8 * u + 2 * h + i2;
          uint32_t xa = 0, xb = 0;
          if (P < npairs) {
            xa = sa[P];
            xb = sb[P];
            nan_seen |= (xa == 0xFFu) | (xb == 0xFFu);
          }
          v |= (xa | (xb << 8)) << (16 * i2);
        }
        sw[h] = v;
      }
      *reinterpret_cast<uint4 *>(sbase + (size_t)wd * 256 + ((size_t)u * 8 + g) * 16) =
          make_uint4(sw[0], sw[1], sw[2], sw[3]);
    }
    return nan_seen;
  }
#pragma unroll 1
  for (int q8 = 0; q8 < 4; q8++) {
    uint32_t sw[4];
#pragma unroll
    for (int h = 0; h < 4; h++) {
      uint32_t v = 0;
#pragma unroll
      for (int i2 = 0; i2 < 2; i2++) {
        const int s = kstep0 + 8 * q8 + 2 * h + i2;
        uint32_t xa = 0, xb = 0;
        if (s < ksteps) {
          xa = sa[s];
          xb = sb[s];
          nan_seen |= e4m3_is_nan(xa) | e4m3_is_nan(xb);
        }
        v |= (xa | (xb << 8)) << (16 * i2);
      }
      sw[h] = v;
    }
    *reinterpret_cast<uint4 *>(sbase + (size_t)wd * 512 + ((size_t)q8 * 8 + g) * 16) =
        make_uint4(sw[0], sw[1], sw[2], sw[3]);
  }
  return nan_seen;
}

}  // namespace moe
