// pack.cu -- canonical NVFP4 expert weights -> the packed layout the expert
// kernels stream (byte moves only; no value changes).
//
// Packed expert e (at e * expert_bytes):
//   gate/up pair rows r = 0 .. I-1, each gu_pair_bytes = tpr_gu * 18 bytes:
//     codes : for block b < tpr_gu, 16 bytes = gate row r block b (8 bytes)
//             followed by up row r block b (8 bytes)
//     scales: for block b, 2 bytes = gate scale (r, b), up scale (r, b)
//   down pair rows p = 0 .. H/2-1 (at dn_region_off), each dn_pair_bytes:
//     codes : block b: down row 2p block b (8 bytes), down row 2p+1 block b
//     scales: block b: scale (2p, b), scale (2p+1, b)
//   Blocks past the real K (padding to a multiple of 512 elements) are zero.
// After all experts: float [E][6] = g_gate a_gate g_up a_up g_down a_down,
// then a 16-byte trailer whose first int32 is set when a NaN scale is seen.
//
// One thread moves one 16-byte code word and its two scale bytes, so
// consecutive threads read consecutive 8-byte canonical chunks and write
// consecutive 16-byte packed words.
#include "moe_internal.cuh"
#include "kernels.h"

namespace moe {

__device__ __forceinline__ bool e4m3_is_nan(uint32_t b) { return (b & 0x7F) == 0x7F; }

__global__ void pack_kernel(const PackArgs a) {
  const int64_t gu_items = (int64_t)a.E * a.I * a.tpr_gu;
  const int64_t dn_items = (int64_t)a.E * (a.H / 2) * a.tpr_dn;
  const int64_t total = gu_items + dn_items + a.E;
  const int gu_blocks = a.H / 16, dn_blocks = a.I / 16;
  int nan_seen = 0;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    if (it < gu_items) {
      const int b = (int)(it % a.tpr_gu);
      const int64_t er = it / a.tpr_gu;              // e * I + r
      const int64_t e = er / a.I, r = er % a.I;
      uint8_t *dst = a.packed + e * a.expert_bytes + r * a.gu_pair_bytes;
      uint4 w = make_uint4(0, 0, 0, 0);
      uint32_t s = 0;
      if (b < gu_blocks) {
        const uint2 g = *reinterpret_cast<const uint2 *>(a.gate_codes + er * (a.H / 2) + b * 8);
        const uint2 u = *reinterpret_cast<const uint2 *>(a.up_codes + er * (a.H / 2) + b * 8);
        const uint32_t gs = a.gate_scales[er * gu_blocks + b];
        const uint32_t us = a.up_scales[er * gu_blocks + b];
        nan_seen |= e4m3_is_nan(gs) | e4m3_is_nan(us);
        w = make_uint4(g.x, g.y, u.x, u.y);
        s = gs | (us << 8);
      }
      *reinterpret_cast<uint4 *>(dst + b * 16) = w;
      *reinterpret_cast<uint16_t *>(dst + (size_t)a.tpr_gu * 16 + b * 2) = (uint16_t)s;
    } else if (it < gu_items + dn_items) {
      const int64_t j = it - gu_items;
      const int b = (int)(j % a.tpr_dn);
      const int64_t ep = j / a.tpr_dn;               // e * (H/2) + p
      const int64_t e = ep / (a.H / 2), p = ep % (a.H / 2);
      uint8_t *dst = a.packed + e * a.expert_bytes + a.dn_region_off + p * a.dn_pair_bytes;
      uint4 w = make_uint4(0, 0, 0, 0);
      uint32_t s = 0;
      if (b < dn_blocks) {
        const int64_t row0 = e * a.H + 2 * p;        // global row index of down row 2p
        const uint2 c0 = *reinterpret_cast<const uint2 *>(a.down_codes + row0 * (a.I / 2) + b * 8);
        const uint2 c1 = *reinterpret_cast<const uint2 *>(a.down_codes + (row0 + 1) * (a.I / 2) + b * 8);
        const uint32_t s0 = a.down_scales[row0 * dn_blocks + b];
        const uint32_t s1 = a.down_scales[(row0 + 1) * dn_blocks + b];
        nan_seen |= e4m3_is_nan(s0) | e4m3_is_nan(s1);
        w = make_uint4(c0.x, c0.y, c1.x, c1.y);
        s = s0 | (s1 << 8);
      }
      *reinterpret_cast<uint4 *>(dst + b * 16) = w;
      *reinterpret_cast<uint16_t *>(dst + (size_t)a.tpr_dn * 16 + b * 2) = (uint16_t)s;
    } else {
      const int64_t e = it - gu_items - dn_items;
      float *dst = reinterpret_cast<float *>(a.packed + a.scalars_off) + e * 6;
      dst[0] = a.gate_g[e];
      dst[1] = a.gate_a[e];
      dst[2] = a.up_g[e];
      dst[3] = a.up_a[e];
      dst[4] = a.down_g[e];
      dst[5] = a.down_a[e];
    }
  }
  if (nan_seen) atomicOr(a.status, 1);
}

cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream) {
  pack_kernel<<<num_sms * 8, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
