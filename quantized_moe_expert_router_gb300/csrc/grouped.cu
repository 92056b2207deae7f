// grouped.cu -- the routed expert FFN for C > 8 tokens, expert-major, on the
// 5th-generation tensor cores (tcgen05).
//
// Same definition as the decode path (expert_gemv.cu, combine.cu; the
// "MUL_MAT_ID" step of "Kimi-K3 on 2x A40 - measured findings", section "Why
// the placement experiments all looked the same", with the routed sum of
// "SparkInfer-K3", "How the TP module works"), organised as one grouped GEMM
// per projection: the rows of every distinct selected expert multiply the
// x (or h) rows of all the (token, slot) pairs that chose it.
//
//   group_dispatch_kernel   ids -> distinct experts (ascending) and, per
//                           expert, its (token, slot) pairs in ascending order
//   group_xprep_kernel      per token: the power of two 2^s that puts max|x|
//                           in [2^14, 2^15) (f16 x is then exact for bf16 x)
//   group_xgather_kernel    xg = the pairs' x rows in dispatch order, f16,
//                           laid out k-group major (see below)
//   group_tc_kernel<0>      gate/up + SwiGLU -> h per pair (fp32)
//   group_hprep_kernel      per pair: 2^s from max|h|, h * 2^s split into f16
//                           hi and lo rows (h to 2^-22 of the pair's max |h|)
//   group_tc_kernel<1>      down -> per-pair partial outputs
//   group_combine_kernel    y[t] = sum of t's pairs in ascending expert id
//
// group_tc_kernel.  A unit is (expert d, pair of 128-row m-tiles, chunk of
// the expert's pairs: 64 for gate/up, one B row each; 32 for down, their hi
// and lo B rows) over the whole K, so every unit is a complete dot product and
// units are independent.  Units are weighted (12 + one per 16 B rows) and cut
// into one contiguous range per CTA.  One CTA per SM, 16 warps:
//   warp 0      the weights: each 256-k half slice of the unit's 16 packed
//               tiles (36 KB) by two 4-D tensor-map loads (codes, scales) into
//               a 3-stage ring; evict-first on the last pass over an m-tile
//               pair, normal L2 priority while later chunks will read it again;
//   warp 1      the B rows for the same 256 k by one 3-D box into a 3-stage
//               ring (evict-last: every m-tile pair reads them): the global B
//               buffers are [K/8][rows][8] f16, so a box (8, R, 32) lands as
//               32 k-groups of R rows of 16 bytes, the K-major, unswizzled
//               core-matrix layout of the MMA's B operand;
//   warps 2, 3  MMA issuers, one per m-tile: tcgen05.mma kind::f16 (M=128,
//               N = the unit's B rows rounded up to 16, K=16), A from tensor
//               memory, B from shared memory, fp32 D in tensor memory (two
//               buffers of 64 columns per issuer, so the epilogue of a unit
//               overlaps the MMAs of the next); warp 2 owns tensor memory;
//   warps 4-11  decode: set j (4 warps; warp w reaches tensor-memory lanes
//               32 (w % 4) ..) feeds m-tile j; a thread owns one weight row,
//               turns 64 k of e2m1 codes into f16 (cvt.rn.f16x2.e2m1x2),
//               multiplies by the e4m3 block scales (exact: at most 6
//               significant bits) and stores them with tcgen05.st into its
//               m-tile's A buffers (two halves of 128 k per stage);
//   warps 12-15 epilogue: read D with tcgen05.ld, apply the tensor scale, the
//               2^-s of x or h and (gate/up) SwiGLU and the router weight, and
//               store per-pair rows with streaming stores.
// Weight row to tensor-memory lane: lane 32 q + l (warp quadrant q, lane l)
// holds row 8 (l & 1) + ((l >> 1) & 7) of packed tile 2 q + (l >> 4) of the
// m-tile: rowA (gate; down row 2p) for even l, rowB (up; down row 2p + 1) for
// odd l, so a gate row's up partner is the neighbouring lane and a warp's
// down outputs are 32 consecutive rows.
// Every wait is bounded (about two seconds of %globaltimer): on expiry the
// waiting role sets MOE_FLAG_TIMEOUT and stops; the producers then wait
// (bounded) for their copies in flight and each MMA warp for its MMAs before
// tensor memory is released.  The sums over K run in the MMA's fixed order
// and over a token's experts in ascending id order, so results are bitwise
// reproducible.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "moe_internal.cuh"
#include "kernels.h"
#include "gemv_core.cuh"
#include "quant_core.cuh"

namespace moe {

constexpr int kGDispatchThreads = 1024;
constexpr int kTcTiles = 8;                    // packed tiles of 16 rows per m-tile: M = 128
constexpr int kTcIssuers = 2;                  // MMA warps: issuer j owns m-tile j of a unit
constexpr int kTcUnitTiles = kTcTiles * kTcIssuers;   // packed tiles (256 weight rows) per unit
constexpr int kTcColsGU = 64;                  // pairs per unit, gate/up (one B row each)
constexpr int kTcColsDN = 32;                  // pairs per unit, down (hi and lo B rows)
constexpr int kTcBRows = 64;                   // B rows per stage at most
constexpr int kTcBoxes = 3;                    // B boxes of 16, 32 and 64 rows
constexpr int kTcStageK = 256;                 // k per stage (a half slice); the A and B rings advance together
constexpr int kTcAStageBytes = kTcUnitTiles * (2048 + 256);   // codes of 16 tiles, then their scales
constexpr int kTcBStageBytes = kTcBRows * kTcStageK * 2;
constexpr int kTcAStages = 3;
constexpr int kTcBStages = 3;
constexpr int kTcDCol0 = 0;                    // D: [issuer][2 buffers] of 64 columns
constexpr int kTcACol0 = 256;                  // A: [issuer][2 halves of a stage][2 sub-chunks of 64 k] of 32 columns
constexpr uint32_t kTcTmemCols = 512;
constexpr int kTcUnitBase = 12;                // work weight of a unit: 12 + one per 16 B rows
constexpr int kTcThreads = 512;
constexpr int kTcWProdA = 0, kTcWProdB = 1, kTcWMma = 2, kTcWDec0 = 4, kTcWEpi0 = 12;   // MMA warps 2, 3
constexpr int kTcEpiBar = 1;                   // named barrier of the 4 epilogue warps
constexpr int kTcSmemBytes = kTcBStages * kTcBStageBytes + kTcAStages * kTcAStageBytes + 1024;
static_assert(kTcSmemBytes <= kGroupSmemBytes, "grouped ring exceeds its shared-memory budget");

// gd layout (ints): [0] n, [16, 16 + E) expert of rank d, [16 + E, 17 + 2E) off, then pairs
__device__ __forceinline__ int *gd_expert(int *gd) { return gd + 16; }
__device__ __forceinline__ int *gd_off(int *gd, int E) { return gd + 16 + E; }
__device__ __forceinline__ int *gd_pairs(int *gd, int E) { return gd + 17 + 2 * E; }
__device__ __forceinline__ const int *gd_pairs(const int *gd, int E) { return gd + 17 + 2 * E; }

// Exclusive scan of v over a CTA of up to 1024 threads; `wsum` is 32 ints of
// shared memory; returns the prefix and writes the total.
__device__ __forceinline__ int cta_scan_excl(int v, int *wsum, int &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = (blockDim.x + 31) >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) wsum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const int c = lane < nw ? wsum[lane] : 0;
    int ic = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFull, ic, o);
      if (lane >= o) ic += t;
    }
    wsum[lane] = ic - c;                          // exclusive prefix of warp totals
    if (lane == 31) wsum[32] = ic;
  }
  __syncthreads();
  const int r = wsum[warp] + incl - v;
  total = wsum[32];
  __syncthreads();                                 // wsum may be reused
  return r;
}

// ---------------------------------------------------------------- dispatch
// One CTA of 1024 threads.  A slot is kept when its id is in [0, E) and not a
// repeat of a lower slot of the same token (negative ids: absent, silently;
// ids >= E and repeats: flagged).  The position of a kept pair inside its
// expert's list is the number of earlier tokens that chose the expert (a
// per-expert token bit mask), so the lists are in ascending pair order.
__global__ void __launch_bounds__(kGDispatchThreads) group_dispatch_kernel(const GroupArgs a) {
  extern __shared__ __align__(16) uint32_t gsm[];
  constexpr int MW = kGroupTokens / 32;           // mask words per expert
  uint32_t *mask = gsm;                           // [E][MW]
  int *cnt = reinterpret_cast<int *>(mask + (size_t)a.E * MW);   // [E]
  int *eoff = cnt + a.E;                          // [E]
  int *wsum = eoff + a.E;                         // [33]
  const int tid = threadIdx.x, nt = blockDim.x, P = a.C * a.k;
  for (int i = tid; i < a.E * MW; i += nt) mask[i] = 0u;
  for (int i = tid; i < a.E; i += nt) cnt[i] = 0;
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = a.ids[p];
    if (e < 0) continue;
    if (e >= a.E) {
      atomicOr(a.flags, MOE_FLAG_BAD_EXPERT_ID);
      continue;
    }
    const int t = p / a.k, slot = p - t * a.k;
    bool dup = false;
    for (int j = 0; j < slot; j++) dup |= a.ids[t * a.k + j] == e;
    if (dup) {
      atomicOr(a.flags, MOE_FLAG_DUPLICATE_ID);
      continue;
    }
    atomicOr(&mask[e * MW + (t >> 5)], 1u << (t & 31));
    atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  // pair offsets by expert id, and the ranks of the experts that were chosen
  int total = 0, ndist = 0;
  for (int e0 = 0; e0 < a.E; e0 += nt) {          // E <= 1024 = nt: one round
    const int e = e0 + tid;
    const int c = e < a.E ? cnt[e] : 0;
    int t1, t2;
    const int o = cta_scan_excl(c, wsum, t1) + total;
    const int r = cta_scan_excl(c > 0 ? 1 : 0, wsum, t2) + ndist;
    if (e < a.E) {
      eoff[e] = o;
      if (c > 0) {
        gd_expert(a.gd)[r] = e;
        gd_off(a.gd, a.E)[r] = o;
      }
    }
    total += t1;
    ndist += t2;
  }
  if (tid == 0) {
    a.gd[0] = ndist;
    gd_off(a.gd, a.E)[ndist] = total;
  }
  __syncthreads();
  int *pairs = gd_pairs(a.gd, a.E);
  for (int p = tid; p < P; p += nt) {
    const int e = a.ids[p];
    if ((unsigned)e >= (unsigned)a.E) continue;
    const int t = p / a.k, slot = p - t * a.k;
    bool dup = false;
    for (int j = 0; j < slot; j++) dup |= a.ids[t * a.k + j] == e;
    if (dup) continue;
    const uint32_t *m = mask + e * MW;
    int before = __popc(m[t >> 5] & ((1u << (t & 31)) - 1u));
    for (int w = 0; w < (t >> 5); w++) before += __popc(m[w]);
    pairs[eoff[e] + before] = p;
  }
}

// ---------------------------------------------------------------- x rows
// One CTA per token: xinv[t] = 2^-s_t with max|x_t| 2^s_t in [2^14, 2^15).
__global__ void __launch_bounds__(128) group_xprep_kernel(const GroupArgs a) {
  __shared__ float red[4];
  const int t = blockIdx.x, tid = threadIdx.x;
  const uint16_t *xr = a.x + (size_t)t * a.H;
  float m = 0.f;
  for (int j = tid; j < a.H / 8; j += blockDim.x) {
    const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr) + j);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++)
      m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    float inv;
    f16_range_scale(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), &inv);
    a.xinv[t] = inv;
  }
}

// xg[kg][j][0..7] = x[t_j][8 kg .. 8 kg + 7] * 2^s_t as f16 (zero past H) for
// every dispatched pair j (token t_j); rows of the buffer are the C * k pair
// positions, of which the first `total` are written.
__global__ void __launch_bounds__(256) group_xgather_kernel(const GroupArgs a) {
  const int n = a.gd[0];
  const int total = gd_off(a.gd, a.E)[n];
  const int *pairs = gd_pairs(a.gd, a.E);
  const int P = a.C * a.k, KG = a.Hp / 8;
  const int items = total * KG;
  for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < items; it += gridDim.x * blockDim.x) {
    const int kg = it / total, j = it - kg * total;
    const int t = __ldg(pairs + j) / a.k;
    uint4 out = make_uint4(0u, 0u, 0u, 0u);
    if (8 * kg < a.H) {
      const float up = __frcp_rn(__ldg(a.xinv + t));   // exact: a power of two
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + 8 * kg));
      out.x = pack_half2(__uint_as_float(v.x << 16) * up, __uint_as_float(v.x & 0xFFFF0000u) * up);
      out.y = pack_half2(__uint_as_float(v.y << 16) * up, __uint_as_float(v.y & 0xFFFF0000u) * up);
      out.z = pack_half2(__uint_as_float(v.z << 16) * up, __uint_as_float(v.z & 0xFFFF0000u) * up);
      out.w = pack_half2(__uint_as_float(v.w << 16) * up, __uint_as_float(v.w & 0xFFFF0000u) * up);
    }
    reinterpret_cast<uint4 *>(a.xg)[(size_t)kg * P + j] = out;
  }
}

// ---------------------------------------------------------------- h rows
// One CTA of 128 threads per dispatched pair j (pair p): the pair's max |h|
// sets 2^s (max|h| 2^s in [2^14, 2^15)); hg rows 2j and 2j + 1 get the f16
// hi part of h 2^s and the f16 rest (zero past I); hinv[p] = 2^-s.
constexpr int kHprepThreads = 128;
constexpr int kHprepGroups = 4;                 // k-groups of 8 per thread: Ip <= 4096
__global__ void __launch_bounds__(kHprepThreads) group_hprep_kernel(const GroupArgs a) {
  __shared__ float red[kHprepThreads / 32];
  const int n = a.gd[0];
  const int total = gd_off(a.gd, a.E)[n];
  const int *pairs = gd_pairs(a.gd, a.E);
  const int R2 = 2 * a.C * a.k, KG = a.Ip / 8, tid = threadIdx.x;
  for (int j = blockIdx.x; j < total; j += gridDim.x) {
    const int p = __ldg(pairs + j);
    const float4 *hr = reinterpret_cast<const float4 *>(a.hbuf + (size_t)p * a.I);
    float4 v[kHprepGroups][2];
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < kHprepGroups; i++) {
      const int kg = tid + kHprepThreads * i;
      v[i][0] = v[i][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (kg < KG && 8 * kg < a.I) {
        v[i][0] = __ldcg(hr + 2 * kg);
        v[i][1] = __ldcg(hr + 2 * kg + 1);
      }
#pragma unroll
      for (int hh = 0; hh < 2; hh++)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v[i][hh].x), fabsf(v[i][hh].y)), fmaxf(fabsf(v[i][hh].z), fabsf(v[i][hh].w))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if ((tid & 31) == 0) red[tid >> 5] = m;
    __syncthreads();
    float inv;
    const float up = f16_range_scale(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), &inv);
    __syncthreads();                               // red is reused by the next pair
#pragma unroll
    for (int i = 0; i < kHprepGroups; i++) {
      const int kg = tid + kHprepThreads * i;
      if (kg >= KG) continue;
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int hh = 0; hh < 2; hh++) {
        const float x0 = v[i][hh].x * up, x1 = v[i][hh].y * up, x2 = v[i][hh].z * up, x3 = v[i][hh].w * up;
        const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        hi[2 * hh] = *reinterpret_cast<const uint32_t *>(&h01);
        hi[2 * hh + 1] = *reinterpret_cast<const uint32_t *>(&h23);
        lo[2 * hh] = pack_half2(x0 - f01.x, x1 - f01.y);
        lo[2 * hh + 1] = pack_half2(x2 - f23.x, x3 - f23.y);
      }
      uint4 *dst = reinterpret_cast<uint4 *>(a.hg) + (size_t)kg * R2 + 2 * j;
      dst[0] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      dst[1] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    if (tid == 0) a.hinv[p] = inv;
  }
}

// ---------------------------------------------------------------- W4A4 rows
// W4A4: the B rows hold the NVFP4-quantized activations of each dispatched
// pair, e2m1 * e4m3 in f16 (exact); the input scale a is applied in the
// epilogue.  One item per (block of 16 elements, pair): 16 inputs, one
// quantized block, two 16-byte stores (k-groups 2 kb and 2 kb + 1).
//   x rows: token t_j's x quantized with its expert's gate/up input scale
//           max(a_gate, a_up) (gate and up read one quantized x);
//   h rows: pair p's h quantized with its expert's down input scale a_down.
__device__ __forceinline__ void store_quant_block(uint16_t *buf, int R, int kb, int j, const uint32_t (&vals)[8]) {
  uint4 *dst = reinterpret_cast<uint4 *>(buf);
  dst[(size_t)(2 * kb) * R + j] = make_uint4(vals[0], vals[1], vals[2], vals[3]);
  dst[(size_t)(2 * kb + 1) * R + j] = make_uint4(vals[4], vals[5], vals[6], vals[7]);
}

__global__ void __launch_bounds__(256) group_xquant_kernel(const GroupArgs a) {
  const int n = a.gd[0];
  const int total = gd_off(a.gd, a.E)[n];
  const int *pairs = gd_pairs(a.gd, a.E);
  const int P = a.C * a.k, KB = a.Hp / 16;
  const int items = total * KB;
  for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < items; it += gridDim.x * blockDim.x) {
    const int kb = it / total, j = it - kb * total;
    const int p = __ldg(pairs + j), t = p / a.k, e = __ldg(a.ids + p);
    uint32_t vals[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (16 * kb < a.H) {
      const float ain = fmaxf(__ldg(a.scalars + (size_t)e * 6 + 1), __ldg(a.scalars + (size_t)e * 6 + 3));
      const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + 16 * kb);
      const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      float v[16];
#pragma unroll
      for (int i = 0; i < 8; i++) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
      uint32_t codes[2];
      nvfp4_quant_block(v, ain, codes, vals);
    }
    store_quant_block(a.xg, P, kb, j, vals);
  }
}

__global__ void __launch_bounds__(256) group_hquant_kernel(const GroupArgs a) {
  const int n = a.gd[0];
  const int total = gd_off(a.gd, a.E)[n];
  const int *pairs = gd_pairs(a.gd, a.E);
  const int P = a.C * a.k, KB = a.Ip / 16;
  const int items = total * KB;
  for (int it = blockIdx.x * blockDim.x + threadIdx.x; it < items; it += gridDim.x * blockDim.x) {
    const int kb = it / total, j = it - kb * total;
    const int p = __ldg(pairs + j), e = __ldg(a.ids + p);
    uint32_t vals[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
    if (16 * kb < a.I) {
      const float adn = __ldg(a.scalars + (size_t)e * 6 + 5);
      const float4 *src = reinterpret_cast<const float4 *>(a.hbuf + (size_t)p * a.I + 16 * kb);
      float v[16];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const float4 f = __ldcg(src + i);
        v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
      }
      uint32_t codes[2];
      nvfp4_quant_block(v, adn, codes, vals);
    }
    store_quant_block(a.hg, P, kb, j, vals);
  }
}

// ---------------------------------------------------------------- tensor-core GEMM
struct GroupTcArgs {
  CUtensorMap bmap[kTcBoxes];   // B rows: boxes of (8, 16 << i, 32) over [K/8][rows][8] f16
  CUtensorMap amap[2];          // weights of the region, 8-byte elements: codes (256, 1, 16, 1) and
                                // scales (32, 1, 16, 1) boxes over [E][tiles][half slices][..]
  const float *scalars;
  const int *gd;
  const float *weights;         // [C][k] router weights (gate/up)
  const float *colscale;        // gate/up: xinv per token; down: hinv per pair
  float *out;                   // gate/up: hbuf [C*k][I]; down: ypair [C*k][H]
  int32_t *flags;
  int k, E, H, I;
  int Kp;                       // padded K of the weight rows
  int tiles;                    // packed tiles of 16 rows per expert in this region
  int cols;                     // pairs per unit
};

struct TcSmem {
  uint64_t a_full[kTcAStages], a_empty[kTcAStages];
  uint64_t b_full[kTcBStages], b_empty[kTcBStages];
  uint64_t a_ready[kTcIssuers][2], a_free[kTcIssuers][2];   // per issuer and half of a stage
  uint64_t d_full[2], d_free[2];
  uint64_t drain[kTcIssuers];
  uint32_t tmem_base;
  int n;
  int d_ok;                     // epilogue: the D wait succeeded
  int range[6];                 // first unit (d, mt, nc) of this CTA and the end
  int wsum[33];
  int colp[kTcBRows];           // epilogue: pair of each column of the unit
  float colw[kTcBRows], cols[kTcBRows];
  int16_t expert[kMaxExperts];
  int off[kMaxExperts + 1];
  int pre[kMaxExperts + 1];     // work prefix over experts
};

struct TcUnit {
  int d, mt, nc;
};
// Units are ordered m-tile pair first, then expert, then column chunk: the
// CTAs' contiguous ranges then cover every m-tile pair of an expert at about
// the same time (an expert's B rows, which all its m-tile pairs read, are
// fetched from DRAM once and then hit L2), while consecutive chunks of one
// m-tile pair stay together in a CTA (its weights are re-read from L2).
__device__ __forceinline__ bool unit_before(const TcUnit &u, const TcUnit &e) {
  return u.mt != e.mt ? u.mt < e.mt : (u.d != e.d ? u.d < e.d : u.nc < e.nc);
}
__device__ __forceinline__ int unit_nch(const TcSmem &s, int d, int cols) {
  return (s.off[d + 1] - s.off[d] + cols - 1) / cols;
}
__device__ __forceinline__ void unit_next(const TcSmem &s, TcUnit &u, int MT, int cols) {
  if (++u.nc == unit_nch(s, u.d, cols)) {
    u.nc = 0;
    if (++u.d == s.n) {
      u.d = 0;
      u.mt++;
    }
  }
}
// Work weight of a unit with `rows` B rows, and of one m-tile of an expert
// with cnt pairs (its column chunks: all full but the last).
__device__ __forceinline__ int unit_cost(int rows) { return kTcUnitBase + (rows + 15) / 16; }
__device__ __forceinline__ int mtile_cost(int cnt, int cols, int rf, int &cfull) {
  const int nch = (cnt + cols - 1) / cols;
  cfull = unit_cost(cols * rf);
  return (nch - 1) * cfull + unit_cost((cnt - (nch - 1) * cols) * rf);
}
// First unit whose work start is >= c; pre[d] is the work of the m-tile
// pairs of experts 0..d-1 in one m-tile row, pre[n] that of a whole row.
__device__ __forceinline__ TcUnit unit_at(const TcSmem &s, int MT, int cols, int rf, long long c) {
  const long long row = s.pre[s.n];
  TcUnit u = {0, MT, 0};
  if (row <= 0) return u;                          // no units
  u.mt = (int)(c / row);
  if (u.mt >= MT) return u;
  const int r = (int)(c - (long long)u.mt * row);
  int lo = 0, hi = s.n - 1;                        // largest d with pre[d] <= r
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.pre[mid] <= r) lo = mid; else hi = mid - 1;
  }
  u.d = lo;
  const int cnt = s.off[lo + 1] - s.off[lo], nch = (cnt + cols - 1) / cols;
  int cf;
  mtile_cost(cnt, cols, rf, cf);
  u.nc = (r - s.pre[lo] + cf - 1) / cf;
  if (u.nc >= nch) {
    u.nc = 0;
    if (++u.d == s.n) {
      u.d = 0;
      u.mt++;
    }
  }
  return u;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync %0, %1;" ::"n"(kTcEpiBar), "n"(128) : "memory"); }

// 32 columns of this warp's 32 tensor-memory lanes: store / load.
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}
// Shared-memory descriptor of a K-major, unswizzled operand: start address,
// byte offset between core matrices adjacent in K (leading) and in N
// (stride), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}
__device__ __forceinline__ void tc_mma(uint32_t d_t, uint32_t a_t, uint64_t b_desc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_t),
      "r"(a_t), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar,
                                            uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, int c3,
                                            uint64_t *bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3, %4, %5}], [%6], %7;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}
// Elements (0, 1) and (8, 9) of a code word's two rowA bytes (bytes 0, 2)
// as f16x2.
__device__ __forceinline__ void e2m1_bytes02(uint32_t w, uint32_t &lo, uint32_t &hi) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b2;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
  return *reinterpret_cast<const uint32_t *>(&r);
}
// Number of B rows, MMA N and box index of a unit with np pairs.
__device__ __forceinline__ void unit_shape(int np, int rf, int &rows, int &N, int &bi) {
  rows = np * rf;
  N = (rows + 15) & ~15;
  bi = N <= 16 ? 0 : (N <= 32 ? 1 : 2);
}

// MODE 0: gate/up + SwiGLU (x rows f16, per-token 2^-s, router weight folded
// into h); 1: down (hi and lo rows of h, per-pair 2^-s); 2: gate/up with W4A4
// rows (x quantized, the input scale applied here, h without the router
// weight); 3: down with W4A4 rows (one row per pair; input scale and router
// weight applied here).
template <int MODE>
__global__ void __launch_bounds__(kTcThreads, 1) group_tc_kernel(const __grid_constant__ GroupTcArgs a) {
  extern __shared__ uint8_t dsm[];
  __shared__ TcSmem s;
  constexpr bool GU = MODE == 0 || MODE == 2;
  constexpr int rf = MODE == 1 ? 2 : 1;            // B rows per pair
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int E = a.E, cols = a.cols;
  const int MP = (a.tiles + kTcUnitTiles - 1) / kTcUnitTiles;   // m-tile pairs per expert
  const int HS = a.Kp / kTcStageK;
  uint8_t *ring_b = dsm + ((1024u - (smem_u32(dsm) & 1023u)) & 1023u);   // 1024-byte aligned
  uint8_t *ring_a = ring_b + kTcBStages * kTcBStageBytes;

  if (tid == 0) {
    for (int i = 0; i < kTcAStages; i++) {
      mbar_init(&s.a_full[i], 1);
      mbar_init(&s.a_empty[i], 8);                 // the 8 decode warps
    }
    for (int i = 0; i < kTcBStages; i++) {
      mbar_init(&s.b_full[i], 1);
      mbar_init(&s.b_empty[i], kTcIssuers);
    }
    for (int j = 0; j < kTcIssuers; j++)
      for (int p = 0; p < 2; p++) {
        mbar_init(&s.a_ready[j][p], 4);            // the 4 warps of decode set j
        mbar_init(&s.a_free[j][p], 1);
      }
    for (int i = 0; i < 2; i++) {
      mbar_init(&s.d_full[i], kTcIssuers);
      mbar_init(&s.d_free[i], 4);                  // the 4 epilogue warps
    }
    for (int i = 0; i < kTcIssuers; i++) mbar_init(&s.drain[i], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    s.n = a.gd[0];
  }
  if (warp == kTcWMma) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s.tmem_base)),
                 "r"(kTcTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int n = s.n;
  {
    // experts, pair offsets and the work prefix (every CTA computes the same)
    int run = 0;
    for (int d0 = 0; d0 < n; d0 += blockDim.x) {
      const int d = d0 + tid;
      int cost = 0;
      if (d < n) {
        s.expert[d] = (int16_t)a.gd[16 + d];
        const int o = a.gd[16 + E + d], o1 = a.gd[17 + E + d];
        s.off[d] = o;
        int cf;
        cost = mtile_cost(o1 - o, cols, rf, cf);    // one m-tile pair of the expert
      }
      int t1;
      const int pre = cta_scan_excl(cost, s.wsum, t1) + run;
      if (d < n) s.pre[d] = pre;
      run += t1;
    }
    if (tid == 0) {
      s.off[n] = a.gd[16 + E + n];
      s.pre[n] = run;
    }
    __syncthreads();
    if (tid == 0) {
      const long long total = (long long)MP * s.pre[n];
      const TcUnit u0 = unit_at(s, MP, cols, rf, total * blockIdx.x / gridDim.x);
      const TcUnit u1 = unit_at(s, MP, cols, rf, total * (blockIdx.x + 1) / gridDim.x);
      s.range[0] = u0.d; s.range[1] = u0.mt; s.range[2] = u0.nc;
      s.range[3] = u1.d; s.range[4] = u1.mt; s.range[5] = u1.nc;
    }
    __syncthreads();
  }
  const TcUnit beg = {s.range[0], s.range[1], s.range[2]}, end = {s.range[3], s.range[4], s.range[5]};
  const uint32_t tbase = s.tmem_base;
  const int *pairs = gd_pairs(a.gd, E);

  if (warp == kTcWProdA) {
    // ------------------------------------------------ weights: a half slice of 16 tiles per stage
    if (lane == 0) {
      // the weights of an m-tile pair are read once per column chunk, one
      // chunk after the other: all but the last pass leave them in L2
      const uint64_t pol_last = l2_evict_first_policy(), pol_again = l2_evict_normal_policy();
      int ia = 0;
      bool ok = true;
      for (TcUnit u = beg; ok && unit_before(u, end); unit_next(s, u, MP, cols)) {
        const int e = s.expert[u.d], t0 = kTcUnitTiles * u.mt;
        const uint64_t pol = u.nc + 1 < unit_nch(s, u.d, cols) ? pol_again : pol_last;
        for (int hs = 0; hs < HS; hs++, ia++) {
          const int slot = ia % kTcAStages;
          if (ia >= kTcAStages && !mbar_wait_bounded(&s.a_empty[slot], (uint32_t)(ia / kTcAStages - 1) & 1u)) {
            atomicOr(a.flags, MOE_FLAG_TIMEOUT);
            ok = false;
            break;
          }
          uint8_t *dst = ring_a + (size_t)slot * kTcAStageBytes;
          // tiles past the region's last read as zeros
          mbar_arrive_expect_tx(&s.a_full[slot], (uint32_t)kTcAStageBytes);
          tma_load_4d(dst, &a.amap[0], 0, hs, t0, e, &s.a_full[slot], pol);
          tma_load_4d(dst + kTcUnitTiles * 2048, &a.amap[1], 0, hs, t0, e, &s.a_full[slot], pol);
        }
      }
      for (int j = (ia > kTcAStages ? ia - kTcAStages : 0); j < ia; j++)
        mbar_wait_bounded(&s.a_full[j % kTcAStages], (uint32_t)(j / kTcAStages) & 1u);
    }
  } else if (warp == kTcWProdB) {
    // ------------------------------------------------ B rows: 256 k per stage
    if (lane == 0) {
      // every m-tile pair of an expert reads the same B rows: keep them in L2
      const uint64_t pol = l2_evict_last_policy();
      int gb = 0;
      bool ok = true;
      for (TcUnit u = beg; ok && unit_before(u, end); unit_next(s, u, MP, cols)) {
        const int off = s.off[u.d], np = min(cols, s.off[u.d + 1] - off - u.nc * cols);
        int rows, N, bi;
        unit_shape(np, rf, rows, N, bi);
        const int row0 = rf * (off + u.nc * cols);
        for (int hs = 0; hs < HS; hs++, gb++) {
          const int slot = gb % kTcBStages;
          if (gb >= kTcBStages && !mbar_wait_bounded(&s.b_empty[slot], (uint32_t)(gb / kTcBStages - 1) & 1u)) {
            atomicOr(a.flags, MOE_FLAG_TIMEOUT);
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&s.b_full[slot], (uint32_t)((16 << bi) * kTcStageK * 2));
          tma_load_3d(ring_b + (size_t)slot * kTcBStageBytes, &a.bmap[bi], 0, row0, (kTcStageK / 8) * hs,
                      &s.b_full[slot], pol);
        }
      }
      for (int j = (gb > kTcBStages ? gb - kTcBStages : 0); j < gb; j++)
        mbar_wait_bounded(&s.b_full[j % kTcBStages], (uint32_t)(j / kTcBStages) & 1u);
    }
  } else if (warp == kTcWMma || warp == kTcWMma + 1) {
    // ------------------------------------------------ MMA issue: issuer j computes m-tile j of each unit
    const int j = warp - kTcWMma;
    if (lane == 0) {
      const uint32_t bring = smem_u32(ring_b);
      int gs = 0, ud = 0;                            // global stage, unit
      bool ok = true;
      for (TcUnit u = beg; ok && unit_before(u, end); unit_next(s, u, MP, cols), ud++) {
        const int off = s.off[u.d], np = min(cols, s.off[u.d + 1] - off - u.nc * cols);
        int rows, N, bi;
        unit_shape(np, rf, rows, N, bi);
        const uint32_t br = 16u << bi;
        const int db = ud & 1;
        if (ud >= 2 && !mbar_wait_bounded(&s.d_free[db], (uint32_t)((ud >> 1) - 1) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          break;
        }
        tc_fence_after();
        // D f32, A and B f16, both K-major, N, M = 128
        const uint32_t idesc = (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((128u >> 4) << 24);
        const uint32_t dt = tbase + (uint32_t)(kTcDCol0 + 128 * j + 64 * db);
        const uint64_t bd_lo = smem_desc(0u, br * 16u, 128u);   // LBO / SBO fields; start added per step
        for (int hs = 0; hs < HS && ok; hs++, gs++) {
          const int bs = gs % kTcBStages;
          if (!mbar_wait_bounded(&s.b_full[bs], (uint32_t)(gs / kTcBStages) & 1u)) {
            atomicOr(a.flags, MOE_FLAG_TIMEOUT);
            ok = false;
            break;
          }
          const uint32_t bstage = bring + (uint32_t)(bs * kTcBStageBytes);
#pragma unroll
          for (int p = 0; p < 2; p++) {
            if (!mbar_wait_bounded(&s.a_ready[j][p], (uint32_t)gs & 1u)) {
              atomicOr(a.flags, MOE_FLAG_TIMEOUT);
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; h++) {
              // sub-chunk 2p + h of the stage: k-groups 8 (2p + h) ..
              const uint64_t bd0 = bd_lo | (uint64_t)(((bstage + 128u * (2 * p + h) * br) >> 4) & 0x3FFFu);
              const uint32_t at = tbase + (uint32_t)(kTcACol0 + 128 * j + 64 * p + 32 * h);
#pragma unroll
              for (int kk = 0; kk < 4; kk++)
                tc_mma(dt, at + 8u * kk, bd0 + (uint64_t)(2u * kk * br), idesc, (uint32_t)(hs | p | h | kk));
            }
            tc_commit(&s.a_free[j][p]);
          }
          if (ok) tc_commit(&s.b_empty[bs]);
        }
        if (ok) tc_commit(&s.d_full[db]);
      }
      // every MMA issued has completed before tensor memory is released
      tc_commit(&s.drain[j]);
      mbar_wait_bounded(&s.drain[j], 0u);
    }
    __syncwarp();
  } else if (warp >= kTcWDec0 && warp < kTcWEpi0) {
    // ------------------------------------------------ decode into tensor memory: set j feeds issuer j
    const int set = (warp - kTcWDec0) >> 2, wq = warp & 3;
    const int Tl = kTcTiles * set + 2 * wq + (lane >> 4), g = (lane >> 1) & 7, hi = lane & 1;
    const uint32_t trow = tbase + ((uint32_t)(32 * wq) << 16) + (uint32_t)(kTcACol0 + 128 * set);
    const uint32_t sel = hi ? 0x3232u : 0x1010u;  // this row's scale in both halves
    int gs = 0;
    bool ok = true;
    for (TcUnit u = beg; ok && unit_before(u, end); unit_next(s, u, MP, cols)) {
      for (int hs = 0; hs < HS; hs++, gs++) {
        const int slot = gs % kTcAStages;
        if (!mbar_wait_bounded(&s.a_full[slot], (uint32_t)(gs / kTcAStages) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          ok = false;
          break;
        }
        const uint8_t *stg = ring_a + (size_t)slot * kTcAStageBytes;
#pragma unroll 1
        for (int p = 0; p < 2; p++) {
          if (gs > 0 && !mbar_wait_bounded(&s.a_free[set][p], (uint32_t)(gs - 1) & 1u)) {
            atomicOr(a.flags, MOE_FLAG_TIMEOUT);
            ok = false;
            break;
          }
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int sc = 2 * p + h;                // 64-k sub-chunk of the stage
            // lanes 4g + q of the sub-chunk's code group hold this row pair's
            // words of its 4 k-steps; the scale unit of row pair g holds the
            // (rowA, rowB) e4m3 bytes of each k-step
            const uint8_t *cp = stg + Tl * 2048 + sc * 512 + g * 64;
            uint4 cw[4];
#pragma unroll
            for (int q = 0; q < 4; q++) cw[q] = *reinterpret_cast<const uint4 *>(cp + 16 * q);
            const uint2 sw = *reinterpret_cast<const uint2 *>(stg + kTcUnitTiles * 2048 + Tl * 256 + (sc >> 1) * 128 +
                                                              g * 16 + (sc & 1) * 8);
            uint32_t r[32];
#pragma unroll
            for (int jj = 0; jj < 4; jj++) {
              const uint32_t s2 =
                  __byte_perm(e4m3x2_to_f16x2(((jj < 2 ? sw.x : sw.y) >> (16 * (jj & 1))) & 0xFFFFu), 0u, sel);
#pragma unroll
              for (int q = 0; q < 4; q++) {
                const uint32_t wv = (jj == 0 ? cw[q].x : jj == 1 ? cw[q].y : jj == 2 ? cw[q].z : cw[q].w) >> (8 * hi);
                uint32_t c01, c89;
                e2m1_bytes02(wv, c01, c89);
                r[8 * jj + q] = hmul2_u32(c01, s2);      // elements 2q, 2q+1 of k-step jj
                r[8 * jj + 4 + q] = hmul2_u32(c89, s2);  // elements 2q+8, 2q+9
              }
            }
            tc_st32(trow + (uint32_t)(64 * p + 32 * h), r);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&s.a_ready[set][p]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&s.a_empty[slot]);
      }
    }
  } else if (warp >= kTcWEpi0) {
    // ------------------------------------------------ epilogue
    const int wq = warp & 3, et = tid - 32 * kTcWEpi0;
    const int g = (lane >> 1) & 7, hi = lane & 1;
    const uint32_t trow = tbase + ((uint32_t)(32 * wq) << 16);
    int ud = 0, cur = -1;
    float sc0 = 0.f, sc1 = 0.f, xa = 1.f;            // tensor scales; W4A4: the input scale
    for (TcUnit u = beg; unit_before(u, end); unit_next(s, u, MP, cols), ud++) {
      const int off = s.off[u.d], np = min(cols, s.off[u.d + 1] - off - u.nc * cols);
      const int j0 = off + u.nc * cols;
      if (u.d != cur) {
        cur = u.d;
        const float *sc = a.scalars + (size_t)s.expert[u.d] * 6;
        sc0 = GU ? sc[0] : sc[4];
        sc1 = sc[2];
        if constexpr (MODE == 2) xa = fmaxf(sc[1], sc[3]);
        if constexpr (MODE == 3) xa = sc[5];
      }
      epi_sync();                                    // the previous unit's column data is read
      if (et < np) {
        const int p = __ldg(pairs + j0 + et);
        s.colp[et] = p;
        if constexpr (MODE == 0) {
          s.colw[et] = __ldg(a.weights + p);
          s.cols[et] = __ldg(a.colscale + p / a.k);
        } else if constexpr (MODE == 1) {
          s.cols[et] = __ldcg(a.colscale + p);
        } else if constexpr (MODE == 3) {
          s.colw[et] = __ldg(a.weights + p);
        }
      }
      const int db = ud & 1;
      if (et == 0) s.d_ok = mbar_wait_bounded(&s.d_full[db], (uint32_t)(ud >> 1) & 1u) ? 1 : 0;
      epi_sync();
      if (!s.d_ok) {
        if (et == 0) atomicOr(a.flags, MOE_FLAG_TIMEOUT);
        break;
      }
      tc_fence_after();
      const int ncol = np * rf;
#pragma unroll 1
      for (int mj = 0; mj < kTcIssuers; mj++) {
        const int T = kTcUnitTiles * u.mt + kTcTiles * mj + 2 * wq + (lane >> 4);   // packed tile of this lane's row
        const uint32_t dt = trow + (uint32_t)(kTcDCol0 + 128 * mj + 64 * db);
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          float v[32];
          tc_ld32(dt + (uint32_t)c0, v);
          if (mj == kTcIssuers - 1 && c0 + 32 >= ncol) {   // the last read of this D buffer
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.d_free[db]);
          }
          if constexpr (MODE == 0) {
#pragma unroll
            for (int i = 0; i < 32; i++) {
              const int nn = c0 + i;
              if (nn >= np) break;
              const float up = __shfl_xor_sync(kFull, v[i], 1);
              if (!hi && T < a.tiles) {
                const float xs = s.cols[nn];
                const float gg = v[i] * xs * sc0, uu = up * xs * sc1;
                __stcs(a.out + (size_t)s.colp[nn] * a.I + 8 * T + g, s.colw[nn] * silu(gg) * uu);
              }
            }
          } else if constexpr (MODE == 2) {
#pragma unroll
            for (int i = 0; i < 32; i++) {
              const int nn = c0 + i;
              if (nn >= np) break;
              const float up = __shfl_xor_sync(kFull, v[i], 1);
              if (!hi && T < a.tiles) {
                const float gg = v[i] * xa * sc0, uu = up * xa * sc1;
                __stcs(a.out + (size_t)s.colp[nn] * a.I + 8 * T + g, silu(gg) * uu);
              }
            }
          } else if constexpr (MODE == 3) {
#pragma unroll
            for (int i = 0; i < 32; i++) {
              const int nn = c0 + i;
              if (nn >= np) break;
              if (T < a.tiles)
                __stcs(a.out + (size_t)s.colp[nn] * a.H + 16 * T + (lane & 15), v[i] * xa * sc0 * s.colw[nn]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; i++) {
              const int nn = (c0 >> 1) + i;
              if (nn >= np) break;
              if (T < a.tiles)
                __stcs(a.out + (size_t)s.colp[nn] * a.H + 16 * T + (lane & 15), (v[2 * i] + v[2 * i + 1]) * s.cols[nn] * sc0);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kTcWMma) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTcTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------- combine
// One CTA per token: its kept slots ordered by expert id, then the partial
// outputs summed in that order (float4 columns).
__global__ void __launch_bounds__(128) group_combine_kernel(const GroupArgs a) {
  __shared__ int order[kMaxTopK];
  __shared__ int cnt;
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  if (tid < 32) {
    const int e = lane < a.k ? a.ids[(size_t)t * a.k + lane] : -1;
    bool valid = lane < a.k && (unsigned)e < (unsigned)a.E;
    for (int j = 0; j < a.k; j++) {
      const int ej = __shfl_sync(kFull, e, j);
      if (j < lane && ej == e) valid = false;
    }
    int rank = 0;
    for (int j = 0; j < a.k; j++) {
      const int ej = __shfl_sync(kFull, e, j);
      const int vj = __shfl_sync(kFull, (int)valid, j);
      rank += (vj && ej < e);
    }
    const unsigned vm = __ballot_sync(kFull, valid);
    if (valid) order[rank] = t * a.k + lane;
    if (lane == 0) cnt = __popc(vm);
  }
  __syncthreads();
  const int n = cnt, H4 = a.H / 4;
  for (int c4 = tid; c4 < H4; c4 += blockDim.x) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < n; j++) {
      const float4 v = __ldcg(reinterpret_cast<const float4 *>(a.ypair + (size_t)order[j] * a.H) + c4);
      s.x += v.x; s.y += v.y; s.z += v.z; s.w += v.w;
    }
    reinterpret_cast<float4 *>(a.y + (size_t)t * a.H)[c4] = s;
  }
}

// ------------------------------------------------------------------ host side
using TensorMapEncodeFn = PFN_cuTensorMapEncodeTiled_v12000;

static TensorMapEncodeFn tensor_map_encoder() {
  static const TensorMapEncodeFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<TensorMapEncodeFn>(p);
  }();
  return fn;
}

// Tensor maps of a B buffer [Kp/8][rows][8] f16: boxes of 32 k-groups of
// 16, 32 and 64 rows of 8 elements.
static cudaError_t encode_b_maps(CUtensorMap (&maps)[kTcBoxes], const void *base, int rows, int Kp) {
  const TensorMapEncodeFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  for (int i = 0; i < kTcBoxes; i++) {
    const cuuint64_t dims[3] = {8, (cuuint64_t)rows, (cuuint64_t)(Kp / 8)};
    const cuuint64_t strides[2] = {16, (cuuint64_t)rows * 16};
    const cuuint32_t box[3] = {8, (cuuint32_t)(16 << i), kTcStageK / 8};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

// Tensor maps of one weight region (gate/up or down) of every expert, in
// 8-byte elements: the codes [E][tiles][half slices][2048 B] and the scales
// [E][tiles][half slices][256 B] of the packed tiles; a box is one half slice
// of 16 consecutive tiles.
static cudaError_t encode_a_maps(CUtensorMap (&maps)[2], const uint8_t *packed, size_t region_off, int slices,
                                 int tiles, int tile_bytes, int E, size_t expert_bytes) {
  const TensorMapEncodeFn enc = tensor_map_encoder();
  if (!enc) return cudaErrorNotSupported;
  for (int i = 0; i < 2; i++) {
    const cuuint64_t inner = i == 0 ? 256 : 32;              // 2048 or 256 bytes
    const cuuint64_t dims[4] = {inner, (cuuint64_t)(2 * slices), (cuuint64_t)tiles, (cuuint64_t)E};
    const cuuint64_t strides[3] = {inner * 8, (cuuint64_t)tile_bytes, (cuuint64_t)expert_bytes};
    const cuuint32_t box[4] = {(cuuint32_t)inner, 1, kTcUnitTiles, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const uint8_t *base = packed + region_off + (i == 0 ? 0 : (size_t)slices * 4096);
    const CUresult r = enc(&maps[i], CU_TENSOR_MAP_DATA_TYPE_UINT64, 4, const_cast<uint8_t *>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t group_setup() {
  cudaError_t err =
      cudaFuncSetAttribute(group_tc_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_tc_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTcSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)group_dispatch_smem(kMaxExperts));
  return err;
}

size_t group_dispatch_smem(int E) { return (size_t)E * (kGroupTokens / 32) * 4 + 2 * (size_t)E * 4 + 33 * 4; }

cudaError_t launch_group_forward(GroupArgs a, int num_sms, int w_gu, int w_dn, size_t gu_tile_bytes,
                                 size_t dn_tile_bytes, size_t dn_region_off, cudaStream_t stream,
                                 cudaEvent_t after_gate_up) {
  const int P = a.C * a.k;
  GroupTcArgs t;
  memset(&t, 0, sizeof(t));
  cudaError_t err = encode_b_maps(t.bmap, a.xg, P, a.Hp);
  if (err != cudaSuccess) return err;
  group_dispatch_kernel<<<1, kGDispatchThreads, group_dispatch_smem(a.E), stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (a.w4a4) {
    group_xquant_kernel<<<num_sms * 4, 256, 0, stream>>>(a);
  } else {
    group_xprep_kernel<<<a.C, 128, 0, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    group_xgather_kernel<<<num_sms * 4, 256, 0, stream>>>(a);
  }
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // gate/up + SwiGLU
  t.scalars = a.scalars;
  t.gd = a.gd;
  t.weights = a.weights;
  t.flags = a.flags;
  t.k = a.k; t.E = a.E; t.H = a.H; t.I = a.I;
  t.colscale = a.xinv;
  t.out = a.hbuf;
  t.Kp = a.Hp;
  t.tiles = a.I / 8;
  t.cols = kTcColsGU;
  if ((err = encode_a_maps(t.amap, a.packed, 0, w_gu, t.tiles, (int)gu_tile_bytes, a.E, a.expert_bytes)) !=
      cudaSuccess)
    return err;
  if (a.w4a4) group_tc_kernel<2><<<num_sms, kTcThreads, kTcSmemBytes, stream>>>(t);
  else group_tc_kernel<0><<<num_sms, kTcThreads, kTcSmemBytes, stream>>>(t);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (after_gate_up && (err = cudaEventRecord(after_gate_up, stream)) != cudaSuccess) return err;
  if (a.w4a4) group_hquant_kernel<<<num_sms * 4, 256, 0, stream>>>(a);
  else group_hprep_kernel<<<num_sms * 8, kHprepThreads, 0, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // down
  if ((err = encode_b_maps(t.bmap, a.hg, a.w4a4 ? P : 2 * P, a.Ip)) != cudaSuccess) return err;
  t.colscale = a.hinv;
  t.out = a.ypair;
  t.Kp = a.Ip;
  t.tiles = a.H / 16;
  t.cols = a.w4a4 ? kTcColsGU : kTcColsDN;
  if ((err = encode_a_maps(t.amap, a.packed, dn_region_off, w_dn, t.tiles, (int)dn_tile_bytes, a.E, a.expert_bytes)) !=
      cudaSuccess)
    return err;
  if (a.w4a4) group_tc_kernel<3><<<num_sms, kTcThreads, kTcSmemBytes, stream>>>(t);
  else group_tc_kernel<1><<<num_sms, kTcThreads, kTcSmemBytes, stream>>>(t);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  group_combine_kernel<<<a.C, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
