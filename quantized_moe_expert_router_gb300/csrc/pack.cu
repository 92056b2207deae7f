// pack.cu -- canonical NVFP4 / MXFP4 expert weights -> the packed "tile" layout the
// expert kernels stream (byte moves only; no value changes).
//
// A pair row is two matrix rows that share K: gate row r with up row r
// (region 0, I pair rows per expert), or down rows 2p and 2p+1 (region 1, H/2
// pair rows).  A tile is 8 consecutive pair rows over the whole K, padded
// with zero codes and zero scales to Kp (a multiple of 512), split into
// W = Kp/512 slices of 32 k-steps of 16 elements.  Inside a tile:
//
//   codes  [W][8 groups of 4 k-steps][32 lanes][16 bytes]   (W * 4096 bytes)
//   scales [W][4 groups of 8 k-steps][8 rows g][16 bytes]   (W * 512 bytes)
//
// Lane l = 4g + q (g = l / 4 is the pair row in the tile, q = l % 4) holds for
// k-step s one 32-bit word of four code bytes: rowA byte 8s+q, rowB byte
// 8s+q, rowA byte 8s+q+4, rowB byte 8s+q+4, which are the elements
// (16s+2q, 16s+2q+1) and (16s+2q+8, 16s+2q+9) of the two rows.  That is the
// register fragment of operand A of mma.m16n8k16 (row g = rowA, row g+8 =
// rowB), so a warp loads a 16x16 weight block per k-step with one 4-byte
// share of a 16-byte shared-memory load.  The scale unit of row g holds, for
// 8 k-steps, the two e4m3 bytes (rowA scale, rowB scale) of each k-step.
//
// MXFP4 (one e8m0 scale per 32 elements) keeps the code units and halves the
// scale region of a slice: [2 units of 8 k-step pairs][8 rows g][16 bytes],
// the (rowA, rowB) bytes of each pair (W * 256 bytes); a NaN is the byte 0xFF.
//
// Packed expert e (at e * expert_bytes): I/8 gate/up tiles, then H/16 down
// tiles.  After all experts: float [E][6] = g_gate a_gate g_up a_up g_down
// a_down, then a 16-byte trailer whose first int32 is set when a NaN scale
// byte is seen.  The packed size equals the canonical size plus the trailer.
#include "moe_internal.cuh"
#include "kernels.h"
#include "pack_core.cuh"

namespace moe {

// One thread per (expert, region, tile, slice w, pair row g): reads the two
// rows' 256 code bytes and 32 scale bytes of the slice, writes 8 code units
// for each of the 4 lanes of row g and 4 scale units.
__global__ void pack_kernel(const PackArgs a) {
  const int64_t gu_items = (int64_t)a.E * (a.I / 8) * a.w_gu * 8;
  const int64_t dn_items = (int64_t)a.E * (a.H / 16) * a.w_dn * 8;
  const int64_t total = gu_items + dn_items + a.E;
  int nan_seen = 0;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < total;
       it += (int64_t)gridDim.x * blockDim.x) {
    if (it >= gu_items + dn_items) {
      const int64_t e = it - gu_items - dn_items;
      float *dst = reinterpret_cast<float *>(a.packed + a.scalars_off) + e * 6;
      dst[0] = a.gate_g[e]; dst[1] = a.gate_a[e];
      dst[2] = a.up_g[e];   dst[3] = a.up_a[e];
      dst[4] = a.down_g[e]; dst[5] = a.down_a[e];
      continue;
    }
    const bool gu = it < gu_items;
    const int64_t j = gu ? it : it - gu_items;
    const int W = gu ? a.w_gu : a.w_dn;
    const int g = (int)(j % 8);
    const int w = (int)((j / 8) % W);
    const int64_t et = j / (8 * (int64_t)W);             // e * tiles + tile
    const int64_t tiles = gu ? a.I / 8 : a.H / 16;
    const int64_t e = et / tiles, tile = et % tiles;
    const int K = gu ? a.H : a.I;                        // real K of the rows
    const int64_t p = tile * 8 + g;                      // pair row
    const bool mx = a.fmt == kFmtMxfp4;
    const int SB = mx ? 32 : 16;                         // elements per scale byte
    const uint8_t *ca, *cb, *sa, *sb;
    if (gu) {
      const int64_t row = e * a.I + p;
      ca = a.gate_codes + row * (K / 2); cb = a.up_codes + row * (K / 2);
      sa = a.gate_scales + row * (K / SB); sb = a.up_scales + row * (K / SB);
    } else {
      const int64_t row = e * a.H + 2 * p;
      ca = a.down_codes + row * (K / 2); cb = ca + K / 2;
      sa = a.down_scales + row * (K / SB); sb = sa + K / SB;
    }
    uint8_t *tb = a.packed + e * a.expert_bytes + (gu ? 0 : a.dn_region_off) +
                  tile * (size_t)W * (mx ? kTileSliceBytesMx : kTileSliceBytes);
    nan_seen |= pack_pair_slice(ca, cb, sa, sb, K, mx, w, w, g, W, tb);
  }
  if (nan_seen) atomicOr(a.status, 1);
}

cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream) {
  pack_kernel<<<num_sms * 8, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
