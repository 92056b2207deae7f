// grouped.cu -- the routed expert FFN for C > 8 tokens, expert-major.
//
// Same definition as the decode path (expert_gemv.cu, combine.cu; the
// "MUL_MAT_ID" step of "Kimi-K3 on 2x A40 - measured findings", section "Why
// the placement experiments all looked the same", with the routed sum of
// "SparkInfer-K3", "How the TP module works"), organised for many tokens per
// expert (prefill, large batches): each distinct selected expert's weights
// are streamed once per pass of up to kGroupTokens tokens, whatever number of
// them chose it, and each consumer warp decodes its part of a weight tile
// into registers once and multiplies it with every token block of that
// expert.
//
//   group_dispatch_kernel   ids -> distinct experts (ascending) and, per
//                           expert, its (token, slot) pairs in ascending order
//   group_xprep_kernel      x -> f16 B fragments, scaled by a power of two per
//                           token (exact for bf16 input)
//   group_gemv_kernel<0>    gate/up + SwiGLU per (expert, tile of 8 pair rows,
//                           block of 8 pairs) -> h per pair, max |h| per pair
//   group_hprep_kernel      h -> f16 hi/lo B fragments scaled per pair by a
//                           power of two (h to 2^-22 of the pair's max |h|)
//   group_gemv_kernel<1>    down per (expert, tile, block of 4 pairs) ->
//                           per-pair partial outputs
//   group_combine_kernel    y[t] = sum of t's pairs in ascending expert id
//
// The decode and MMA arithmetic are those of the decode path (gemv_core.cuh);
// sums over warps and over a token's experts run in a fixed order, so results
// are bitwise reproducible.  The work split weighs each (expert, tile) unit
// by the streaming of the tile plus its token blocks, so hot experts (the
// one nearly every token of a Zipf-routed prefill picks) are spread over
// many SMs.
#include "moe_internal.cuh"
#include "kernels.h"
#include "gemv_core.cuh"

namespace moe {

constexpr int kGBlkGU = 8;       // pairs per token block, gate/up: one MMA column each
constexpr int kGBlkDN = 4;       // pairs per token block, down: hi and lo columns
constexpr int kGRedSlots = 4;    // consumer -> epilogue reduction ring
constexpr int kGUnitBase = 1;    // work split weight of streaming + decoding a tile ...
constexpr int kGBlockCost = 2;   // ... and of one token block of it (measured: a block costs about twice a tile)
constexpr int kGDispatchThreads = 1024;

// gd layout (ints): [0] n, [16, 16 + E) expert of rank d, [16 + E, 17 + 2E) off, then pairs
__device__ __forceinline__ int *gd_expert(int *gd) { return gd + 16; }
__device__ __forceinline__ int *gd_off(int *gd, int E) { return gd + 16 + E; }
__device__ __forceinline__ int *gd_pairs(int *gd, int E) { return gd + 17 + 2 * E; }

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

// ---------------------------------------------------------------- x fragments
// One CTA per token: xf[t][s][q] = (x[16s+2q], x[16s+2q+1]) and (x[16s+2q+8],
// x[16s+2q+9]) as f16, times 2^s_t with max|x_t| 2^s_t in [2^14, 2^15).
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
  m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float inv;
  const float up = f16_range_scale(m, &inv);
  if (tid == 0) a.xinv[t] = inv;
  const int S = a.Hp / 16;
  uint2 *out = a.xf + (size_t)t * S * 4;
  for (int i = tid; i < S * 4; i += blockDim.x) {
    const int s = i >> 2, q = i & 3, k0 = 16 * s + 2 * q;
    uint32_t v0 = 0, v1 = 0;
    if (k0 < a.H) {
      v0 = *reinterpret_cast<const uint32_t *>(xr + k0);
      v1 = *reinterpret_cast<const uint32_t *>(xr + k0 + 8);
    }
    out[i] = make_uint2(pack_half2(__uint_as_float(v0 << 16) * up, __uint_as_float(v0 & 0xFFFF0000u) * up),
                        pack_half2(__uint_as_float(v1 << 16) * up, __uint_as_float(v1 & 0xFFFF0000u) * up));
  }
}

// ---------------------------------------------------------------- h fragments
// Per kept pair p (from the dispatch lists): hf[p][s][q] = hi and lo f16x2
// pairs of h * 2^s_p (elements 2q, 2q+1 and 2q+8, 2q+9 of k-step s, read as
// one float4 from the operand-ordered hbuf), hinv[p] = 2^-s_p; the max |h|
// word is reset for the next call.
__global__ void __launch_bounds__(256) group_hprep_kernel(const GroupArgs a) {
  const int n = a.gd[0];
  const int total = gd_off(a.gd, a.E)[n];
  const int *pairs = gd_pairs(a.gd, a.E);
  const int S = a.Ip / 16;
  for (int j = blockIdx.x; j < total; j += gridDim.x) {
    const int p = pairs[j];
    const float am = __uint_as_float(__ldcg(a.hamax + p));
    float inv;
    const float up = f16_range_scale(am, &inv);
    const float4 *hr4 = reinterpret_cast<const float4 *>(a.hbuf + (size_t)p * a.I);
    uint2 *out = a.hf + (size_t)p * S * 8;
    for (int i = threadIdx.x; i < S * 4; i += blockDim.x) {
      const int s = i >> 2;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (16 * s < a.I) v = __ldcg(hr4 + i);
      const float x0 = v.x * up, x1 = v.y * up, x2 = v.z * up, x3 = v.w * up;
      const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      out[2 * i] = make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
      out[2 * i + 1] = make_uint2(pack_half2(x0 - f01.x, x1 - f01.y), pack_half2(x2 - f23.x, x3 - f23.y));
    }
    if (threadIdx.x == 0) {
      a.hinv[p] = inv;
      a.hamax[p] = 0u;
    }
  }
}

// ---------------------------------------------------------------- GEMV
struct GroupSmem {
  int16_t expert[kMaxExperts];
  int off[kMaxExperts + 1];
  int pre[kMaxExperts + 1];                        // cost prefix over experts
  int wsum[33];
  int n;
  int range[4];                                    // d0, tile0, d1, tile1 of this CTA
};

// Start (d, tile) of the first unit whose cost start is >= c (units of expert
// d cost cost_d each and start at pre[d] + tile * cost_d).
__device__ __forceinline__ void unit_at(const GroupSmem &s, int tiles, int blk, int c, int &d, int &tile) {
  int lo = 0, hi = s.n;                             // largest d with pre[d] <= c
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s.pre[mid] <= c) lo = mid; else hi = mid - 1;
  }
  d = lo;
  if (d >= s.n) { tile = 0; return; }
  const int nb = (s.off[d + 1] - s.off[d] + blk - 1) / blk;
  const int cost = kGUnitBase + kGBlockCost * nb;
  tile = (c - s.pre[d] + cost - 1) / cost;
  if (tile >= tiles) { d++; tile = 0; }
}

// Decode a warp's 16 k-steps of one tile into A fragments (f16, scaled).
__device__ __forceinline__ void decode_half_slice(const uint8_t *codes, const uint8_t *scales, uint32_t (&A)[kWarpSteps][4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  uint4 sc = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int qg = 0; qg < kWarpSteps / 4; qg++) {
    const uint4 cw = *reinterpret_cast<const uint4 *>(codes + ((size_t)qg * 32 + lane) * 16);
    if ((qg & 1) == 0) sc = *reinterpret_cast<const uint4 *>(scales + ((size_t)(qg >> 1) * 8 + g) * 16);
    const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
    const uint32_t scs[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
      const int s = 4 * qg + jj;
      const int ks = (qg & 1) * 4 + jj;
      const uint32_t s2 = e4m3x2_to_f16x2(scs[ks >> 1] >> (16 * (ks & 1)));
      e2m1x8_to_f16x2(cws[jj], A[s]);
      A[s][0] = hmul2_lo(A[s][0], s2);
      A[s][1] = hmul2_hi(A[s][1], s2);
      A[s][2] = hmul2_lo(A[s][2], s2);
      A[s][3] = hmul2_hi(A[s][3], s2);
    }
  }
}

// WIDE = 1 for tiles of 8 K-slices (18 warps): the register file is split over
// the four SM sub-partitions, so a 5th warp on one of them caps a thread at 96
// registers; with at most 16 warps a thread may use 128, which holds a tile's
// decoded weights (64 registers) and a token block's B fragments (32) at once.
template <int MODE, int WIDE>
__global__ void __launch_bounds__(WIDE ? kMaxCtaThreads : 512, 1) group_gemv_kernel(const GroupArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];   // [S][stage_bytes] then the reduction slots
  __shared__ GroupSmem gs;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t red_full[kGRedSlots];
  __shared__ __align__(8) uint64_t red_empty[kGRedSlots];
  constexpr int BLK = MODE == 0 ? kGBlkGU : kGBlkDN;

  const int NS = a.slices, W = 2 * NS, S = a.stages;
  float4 *red = reinterpret_cast<float4 *>(ring + (size_t)S * a.stage_bytes);   // [slots][W][32]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int slice = warp >> 1, half = warp & 1;
  const int ks0 = kSliceSteps * slice + kWarpSteps * half;
  const int g = lane >> 2, q = lane & 3;
  const int E = a.E;

  if (tid == 0) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], W);
    }
    for (int s = 0; s < kGRedSlots; s++) {
      mbar_init(&red_full[s], W);
      mbar_init(&red_empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    gs.n = a.gd[0];
  }
  __syncthreads();
  const int n = gs.n;
  // experts, pair offsets and the cost prefix (every CTA computes the same)
  {
    int run = 0;
    for (int d0 = 0; d0 < n; d0 += blockDim.x) {
      const int d = d0 + tid;
      int cost = 0;
      if (d < n) {
        gs.expert[d] = (int16_t)gd_expert(a.gd)[d];
        const int o = gd_off(a.gd, E)[d], o1 = gd_off(a.gd, E)[d + 1];
        gs.off[d] = o;
        cost = a.tiles * (kGUnitBase + kGBlockCost * ((o1 - o + BLK - 1) / BLK));
      }
      int t1;
      const int pre = cta_scan_excl(cost, gs.wsum, t1) + run;
      if (d < n) gs.pre[d] = pre;
      run += t1;
    }
    if (tid == 0) {
      gs.off[n] = gd_off(a.gd, E)[n];
      gs.pre[n] = run;
    }
    __syncthreads();
    if (tid == 0) {
      const int total = gs.pre[n];
      int d0, t0, d1, t1;
      // total * grid can exceed 32 bits here (once per CTA: 64-bit is fine)
      const int c0 = (int)((long long)total * blockIdx.x / gridDim.x);
      const int c1 = (int)((long long)total * (blockIdx.x + 1) / gridDim.x);
      unit_at(gs, a.tiles, BLK, c0, d0, t0);
      unit_at(gs, a.tiles, BLK, c1, d1, t1);
      gs.range[0] = d0; gs.range[1] = t0; gs.range[2] = d1; gs.range[3] = t1;
    }
    __syncthreads();
  }
  const int ud0 = gs.range[0], ut0 = gs.range[1], ud1 = gs.range[2], ut1 = gs.range[3];
  const int nunit = (ud1 - ud0) * a.tiles + (ut1 - ut0);
  const int *pairs = gd_pairs(a.gd, E);

  if (warp == W) {
    // ------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int i = 0;
      bool ok = true;
      int d = ud0, tile = ut0;
      for (; i < nunit; i++, tile++) {
        if (tile == a.tiles) { tile = 0; d++; }
        const int slot = i % S;
        const uint32_t use = (uint32_t)(i / S);
        if (use > 0 && !mbar_wait_bounded(&empty_bar[slot], (use - 1) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          ok = false;
          break;
        }
        const uint8_t *src = a.packed + (size_t)gs.expert[d] * a.expert_bytes + a.region_off +
                             (size_t)tile * a.tile_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)a.tile_bytes);
        bulk_copy_g2s(ring + (size_t)slot * a.stage_bytes, src, (uint32_t)a.tile_bytes, &full_bar[slot], pol);
      }
      if (!ok)
        for (int j = (i > S ? i - S : 0); j < i; j++) mbar_wait_bounded(&full_bar[j % S], (uint32_t)(j / S) & 1u);
    }
    return;
  }

  if (warp == W + 1) {
    // ------------------------------------------------ epilogue warp
    int d = ud0, tile = ut0, item = 0, cur = -1;
    float sc0 = 0.f, sc1 = 0.f, sc2 = 0.f;
    bool ok = true;
    for (int i = 0; i < nunit && ok; i++, tile++) {
      if (tile == a.tiles) { tile = 0; d++; }
      if (d != cur) {
        cur = d;
        const float *sc = a.scalars + (size_t)gs.expert[d] * 6;
        sc0 = sc[0]; sc1 = sc[2]; sc2 = sc[4];
      }
      const int o = gs.off[d], cnt = gs.off[d + 1] - o;
      for (int b = 0; b * BLK < cnt; b++, item++) {
        const int rs = item % kGRedSlots;
        if (!mbar_wait_bounded(&red_full[rs], (uint32_t)(item / kGRedSlots) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          ok = false;
          break;
        }
        if constexpr (MODE == 0) {
          const float4 *pr4 = red + (size_t)rs * W * 32 + lane;
          float4 sum = pr4[0];
          for (int ww = 1; ww < W; ww++) {
            const float4 v = pr4[ww * 32];
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
          float hm0 = 0.f, hm1 = 0.f;
#pragma unroll
          for (int c2 = 0; c2 < 2; c2++) {
            const int j = b * BLK + 2 * q + c2;
            if (j < cnt) {
              const int p = pairs[o + j];
              const float gg = (c2 ? sum.y : sum.x) * sc0;
              const float uu = (c2 ? sum.w : sum.z) * sc1;
              const float h = __ldg(a.weights + p) * silu(gg) * uu;
              a.hbuf[(size_t)p * a.I + operand_order(tile * 8 + g)] = h;
              if (c2) hm1 = fabsf(h); else hm0 = fabsf(h);
            }
          }
          // max |h| of the block's pairs over the tile's 8 pair rows
#pragma unroll
          for (int sh = 4; sh < 32; sh <<= 1) {
            hm0 = fmaxf(hm0, __shfl_xor_sync(kFull, hm0, sh));
            hm1 = fmaxf(hm1, __shfl_xor_sync(kFull, hm1, sh));
          }
          if (g == 0) {
            const int j0 = b * BLK + 2 * q;
            if (j0 < cnt) atomicMax(a.hamax + pairs[o + j0], __float_as_uint(hm0));
            if (j0 + 1 < cnt) atomicMax(a.hamax + pairs[o + j0 + 1], __float_as_uint(hm1));
          }
        } else {
          const float2 *pr2 = reinterpret_cast<const float2 *>(red + (size_t)rs * W * 32) + lane;
          float2 sum = pr2[0];
          for (int ww = 1; ww < W; ww++) {
            const float2 v = pr2[ww * 32];
            sum.x += v.x; sum.y += v.y;
          }
          const int j = b * BLK + q;
          if (j < cnt)
            *reinterpret_cast<float2 *>(a.ypair + (size_t)pairs[o + j] * a.H + 2 * (tile * 8 + g)) =
                make_float2(sum.x * sc2, sum.y * sc2);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[rs]);
      }
    }
    return;
  }

  // ---------------------------------------------------- consumers
  const int HS = (MODE == 0 ? a.Hp : a.Ip) / 16;   // k-steps of this region's B rows
  int d = ud0, tile = ut0, item = 0;
  bool ok = true;
  for (int i = 0; i < nunit && ok; i++, tile++) {
    if (tile == a.tiles) { tile = 0; d++; }
    const int slot = i % S;
    if (!mbar_wait_bounded(&full_bar[slot], (uint32_t)(i / S) & 1u)) {
      atomicOr(a.flags, MOE_FLAG_TIMEOUT);
      break;
    }
    uint32_t A[kWarpSteps][4];
    {
      const uint8_t *stg = ring + (size_t)slot * a.stage_bytes;
      decode_half_slice(stg + (size_t)slice * 4096 + (size_t)half * 2048,
                        stg + (size_t)NS * 4096 + (size_t)slice * 512 + (size_t)half * 256, A);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);   // the weights are in registers: refill the stage
    const int o = gs.off[d], cnt = gs.off[d + 1] - o;
    // this lane's pairs in a block: the one of its B column, and the two (or
    // one, down) of its accumulator columns; fetched one block ahead
    const int colj = MODE == 0 ? g : (g >> 1), accj = MODE == 0 ? 2 * q : q;
    auto pair_at = [&](int j) { return j < cnt ? __ldg(pairs + o + j) : -1; };
    int n_col = pair_at(colj), n_a0 = pair_at(accj), n_a1 = MODE == 0 ? pair_at(accj + 1) : -1;
    for (int b = 0; b * BLK < cnt; b++, item++) {
      const int p_col = n_col, p_a0 = n_a0, p_a1 = n_a1;
      n_col = pair_at((b + 1) * BLK + colj);
      n_a0 = pair_at((b + 1) * BLK + accj);
      if constexpr (MODE == 0) n_a1 = pair_at((b + 1) * BLK + accj + 1);
      const int rs = item % kGRedSlots;
      const uint32_t ruse = (uint32_t)(item / kGRedSlots);
      if (ruse > 0 && !mbar_wait_bounded(&red_empty[rs], (ruse - 1) & 1u)) {
        atomicOr(a.flags, MOE_FLAG_TIMEOUT);
        ok = false;
        break;
      }
      // B fragments of this lane's column and the 2^-s of its accumulator columns
      const uint2 *bsrc;
      float ci0, ci1;
      if constexpr (MODE == 0) {
        bsrc = p_col >= 0 ? a.xf + ((size_t)(p_col / a.k) * HS + ks0) * 4 + q : nullptr;
        ci0 = p_a0 >= 0 ? __ldg(a.xinv + p_a0 / a.k) : 0.f;
        ci1 = p_a1 >= 0 ? __ldg(a.xinv + p_a1 / a.k) : 0.f;
      } else {
        bsrc = p_col >= 0 ? a.hf + (((size_t)p_col * HS + ks0) * 4 + q) * 2 + (g & 1) : nullptr;
        ci0 = ci1 = p_a0 >= 0 ? __ldcg(a.hinv + p_a0) : 0.f;
      }
      // two accumulator chains; all B loads of the block issued together
      // (eight k-steps at a time where registers are short)
      float acc2[2][4] = {};
      constexpr int BB = WIDE ? 8 : 16;
#pragma unroll
      for (int h8 = 0; h8 < kWarpSteps / BB; h8++) {
        uint2 bv[BB];
#pragma unroll
        for (int s = 0; s < BB; s++) {
          const int ss = BB * h8 + s;
          bv[s] = bsrc ? __ldcg(bsrc + (size_t)ss * (MODE == 0 ? 4 : 8)) : make_uint2(0u, 0u);
        }
#pragma unroll
        for (int s = 0; s < BB; s++) mma16816(acc2[s & 1], A[BB * h8 + s], bv[s].x, bv[s].y);
      }
      float acc[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; c4++) acc[c4] = acc2[0][c4] + acc2[1][c4];
      if constexpr (MODE == 0)
        red[((size_t)rs * W + warp) * 32 + lane] = make_float4(acc[0] * ci0, acc[1] * ci1, acc[2] * ci0, acc[3] * ci1);
      else
        reinterpret_cast<float2 *>(red + (size_t)rs * W * 32)[(size_t)warp * 32 + lane] =
            make_float2((acc[0] + acc[1]) * ci0, (acc[2] + acc[3]) * ci0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[rs]);
    }
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
cudaError_t group_setup() {
  cudaError_t err = cudaFuncSetAttribute(group_gemv_kernel<0, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kGroupSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_gemv_kernel<1, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_gemv_kernel<0, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_gemv_kernel<1, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGroupSmemBytes);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(group_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)group_dispatch_smem(kMaxExperts));
  return err;
}

size_t group_dispatch_smem(int E) { return (size_t)E * (kGroupTokens / 32) * 4 + 2 * (size_t)E * 4 + 33 * 4; }

void group_geometry(int slices, int tile_bytes, int *stages, int *smem_bytes) {
  const int red = kGRedSlots * 2 * slices * 32 * (int)sizeof(float4);
  int s = (kGroupSmemBytes - red) / tile_bytes;
  if (s > kMaxStages) s = kMaxStages;
  if (s < 2) s = 2;
  *stages = s;
  *smem_bytes = s * tile_bytes + red;
}

cudaError_t launch_group_forward(GroupArgs a, int num_sms, int w_gu, int w_dn, size_t gu_tile_bytes,
                                 size_t dn_tile_bytes, size_t dn_region_off, cudaStream_t stream,
                                 cudaEvent_t after_gate_up) {
  group_dispatch_kernel<<<1, kGDispatchThreads, group_dispatch_smem(a.E), stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  group_xprep_kernel<<<a.C, 128, 0, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // gate/up
  a.region_off = 0;
  a.tiles = a.I / 8;
  a.tile_bytes = a.stage_bytes = (int)gu_tile_bytes;
  a.slices = w_gu;
  group_geometry(a.slices, a.stage_bytes, &a.stages, &a.smem_bytes);
  if (2 * w_gu + 2 > 16)
    group_gemv_kernel<0, 1><<<num_sms, 32 * (2 * w_gu + 2), a.smem_bytes, stream>>>(a);
  else
    group_gemv_kernel<0, 0><<<num_sms, 32 * (2 * w_gu + 2), a.smem_bytes, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (after_gate_up && (err = cudaEventRecord(after_gate_up, stream)) != cudaSuccess) return err;
  group_hprep_kernel<<<num_sms * 4, 256, 0, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  // down
  a.region_off = dn_region_off;
  a.tiles = a.H / 16;
  a.tile_bytes = a.stage_bytes = (int)dn_tile_bytes;
  a.slices = w_dn;
  group_geometry(a.slices, a.stage_bytes, &a.stages, &a.smem_bytes);
  if (2 * w_dn + 2 > 16)
    group_gemv_kernel<1, 1><<<num_sms, 32 * (2 * w_dn + 2), a.smem_bytes, stream>>>(a);
  else
    group_gemv_kernel<1, 0><<<num_sms, 32 * (2 * w_dn + 2), a.smem_bytes, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  group_combine_kernel<<<a.C, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
