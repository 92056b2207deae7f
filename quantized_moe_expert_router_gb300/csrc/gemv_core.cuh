// gemv_core.cuh -- the pieces shared by the expert kernels: warp-role
// constants, mbarrier and bulk-copy helpers, the e2m1/e4m3 decode and MMA
// step, the B-operand fragment builders and the dispatch of a token group's
// selected experts.  See expert_gemv.cu for the packed tile layout and the
// work split these serve.
#pragma once

#include "moe_internal.cuh"
#include "quant_core.cuh"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kSliceSteps = 32;                  // k-steps of one 512-element K-slice of a tile
constexpr int kWarpSteps = 16;                   // k-steps per consumer warp (half a slice)
constexpr int kMaxKWarps = 16;                   // consumer warps: K <= 4096
constexpr int kMaxCtaThreads = 32 * (kMaxKWarps + 2);   // + producer and epilogue warps
constexpr int kMaxStages = 8;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

struct DispatchSmem {
  uint32_t bitmap[kMaxExperts / 32];
  int base[kMaxExperts / 32];
  int n;
  int16_t expert[kMaxPairs];
  uint32_t tokmask[kMaxPairs];
  int pair[kMaxPairs][kGemvTokens];            // by token (lowest slot of a repeated id)
  int16_t slot_pair[kMaxPairs][kGemvTokens];   // by slot (tokens in ascending order)
  uint8_t nslot[kMaxPairs];
  int32_t ids[kMaxPairs];                      // the group's ids, pair p = t*k + slot
  float wt[kMaxPairs];                         // router weight of pair p
  float scal[kMaxPairs][3];                    // tensor scales g_gate, g_up, g_down of rank d (load_dispatch_scales)
};

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with `parity` to complete; false on expiry.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t it = 1;; it++) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) return false;
  }
}
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// e4m3 pair (low byte: rowA scale, high byte: rowB scale) -> f16x2.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t v16) {
  uint32_t r;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(r) : "r"(v16));
  return r;
}
// a * (s.lo, s.lo) and a * (s.hi, s.hi) in f16x2 (exact for code x scale).
__device__ __forceinline__ uint32_t hmul2_lo(uint32_t a, uint32_t s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), __low2half2(*reinterpret_cast<const __half2 *>(&s)));
  return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t hmul2_hi(uint32_t a, uint32_t s) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2 *>(&a), __high2half2(*reinterpret_cast<const __half2 *>(&s)));
  return *reinterpret_cast<const uint32_t *>(&r);
}
__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}
// silu(v) = v / (1 + e^-v), with the SFU exponential and reciprocal (relative
// error ~2^-21, far below the output tolerance).
__device__ __forceinline__ float silu(float g) { return g * __frcp_rn(1.f + __expf(-g)); }

// Power of two 2^s with amax * 2^s in [2^14, 2^15) (s clamped to +-120);
// returns 2^s and writes 2^-s.
__device__ __forceinline__ float f16_range_scale(float amax, float *inv) {
  int s = 0;
  if (amax > 0.f) s = 14 - ((int)((__float_as_uint(amax) >> 23) & 0xFF) - 127);
  s = max(-120, min(120, s));
  *inv = __uint_as_float((uint32_t)(127 - s) << 23);
  return __uint_as_float((uint32_t)(127 + s) << 23);
}

// Position of element k of an h vector in hbuf: each 16-element block is
// stored in the order the down kernel's B operand reads it, so that lane
// (g, q) finds elements 2q, 2q+1, 2q+8, 2q+9 of a k-step as one float4.
__device__ __forceinline__ int operand_order(int k) {
  const int r = k & 15;
  return (k & ~15) + 4 * ((r & 7) >> 1) + 2 * (r >> 3) + (r & 1);
}

// ---------------------------------------------------------------- dispatch
// Distinct selected experts of this token group in ascending id order, with
// for each the tokens that chose it (mask, and the (token, slot) pair index
// p = t*k + slot both by token and in ascending token order).  A negative id
// is an absent slot (skipped: a caller evaluating a band of experts marks the
// others so); ids >= E are flagged and skipped; an id repeated inside a token
// is flagged and only its lowest slot is used (the combine kernel applies the
// same rules).
// The inputs are read from global memory once, together (one round trip on
// the path to the first weight copy); all else is shared memory.
__device__ __forceinline__ void build_dispatch(DispatchSmem &s, const int32_t *ids, const float *weights, int C, int k,
                                               int E, int32_t *flags) {
  const int tid = threadIdx.x, nt = blockDim.x, P = C * k;
  if (C == 1) {
    // one token: warp 0 alone, slot i in lane i (k <= 32); the same tables
    // as below with one CTA barrier instead of five
    if (tid < 32) {
      int e = -1;
      if (tid < k) {
        e = ids[tid];
        s.ids[tid] = e;
        s.wt[tid] = weights[tid];
      }
      const bool inr = tid < k && (unsigned)e < (unsigned)E;
      if (tid < k && e >= E) atomicOr(flags, MOE_FLAG_BAD_EXPERT_ID);
      bool first = inr;                          // the lowest slot holding this id
      for (int j = 0; j < k; j++) {
        const int ej = __shfl_sync(kFull, e, j);
        if (j < tid && ej == e) first = false;
      }
      if (inr && !first) atomicOr(flags, MOE_FLAG_DUPLICATE_ID);
      const uint32_t fm = __ballot_sync(kFull, first);
      int r = 0;                                 // rank by ascending expert id
      for (int j = 0; j < k; j++) {
        const int ej = __shfl_sync(kFull, e, j);
        r += ((fm >> j) & 1u) && ej < e;
      }
      if (first) {
        s.expert[r] = (int16_t)e;
        s.tokmask[r] = 1u;
        s.pair[r][0] = tid;
        s.slot_pair[r][0] = (int16_t)tid;
        s.nslot[r] = 1;
      }
      if (tid == 0) s.n = __popc(fm);
    }
    __syncthreads();
    return;
  }
  for (int p = tid; p < P; p += nt) {
    s.ids[p] = ids[p];
    s.wt[p] = weights[p];
  }
  for (int i = tid; i < kMaxExperts / 32; i += nt) s.bitmap[i] = 0u;
  for (int i = tid; i < P; i += nt) s.tokmask[i] = 0u;
  for (int i = tid; i < P * kGemvTokens; i += nt) (&s.pair[0][0])[i] = 0x7FFFFFFF;
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = s.ids[p];
    if ((unsigned)e < (unsigned)E)
      atomicOr(&s.bitmap[e >> 5], 1u << (e & 31));
    else if (e >= E)                             // negative ids are absent slots, not errors
      atomicOr(flags, MOE_FLAG_BAD_EXPERT_ID);
  }
  __syncthreads();
  if (tid < 32) {
    const int c = __popc(s.bitmap[tid]);
    int incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (tid >= o) incl += v;
    }
    s.base[tid] = incl - c;
    if (tid == 31) s.n = incl;
  }
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = s.ids[p];
    if ((unsigned)e >= (unsigned)E) continue;
    const int w = e >> 5;
    const int r = s.base[w] + __popc(s.bitmap[w] & ((1u << (e & 31)) - 1u));
    const int t = p / k;
    const uint32_t old = atomicOr(&s.tokmask[r], 1u << t);
    if ((old >> t) & 1u) atomicOr(flags, MOE_FLAG_DUPLICATE_ID);
    atomicMin(&s.pair[r][t], p);
    s.expert[r] = (int16_t)e;
  }
  __syncthreads();
  for (int r = tid; r < s.n; r += nt) {
    uint32_t m = s.tokmask[r];
    int j = 0;
    while (m) {
      const int t = __ffs(m) - 1;
      m &= m - 1u;
      s.slot_pair[r][j++] = (int16_t)s.pair[r][t];
    }
    s.nslot[r] = (uint8_t)j;
  }
  __syncthreads();
}

// Tensor scales g_gate, g_up, g_down of the dispatched experts of ranks
// [r0, r1), loaded by one warp (the only one that applies them), off the
// path to the first weight copy.
__device__ __forceinline__ void load_dispatch_scales(DispatchSmem &s, const float *scalars, int r0, int r1) {
  for (int r = r0 + (int)(threadIdx.x & 31); r < r1; r += 32) {
    const float *sc = scalars + (size_t)s.expert[r] * 6;
    s.scal[r][0] = sc[0];
    s.scal[r][1] = sc[2];
    s.scal[r][2] = sc[4];
  }
  __syncwarp();
}

// ---------------------------------------------------------------- fragments
// B fragments of x for a consumer warp's 16 k-steps starting at k-step ks0
// (gate/up): column n = token n of the group (zero beyond C), lane (g, q)
// holds x[g][16 s + 2q, +1] and x[g][16 s + 2q + 8, +9] as f16, scaled by a
// power of two per token and warp K range (exact for bf16 input).  Returns
// in colinv0/colinv1 the 2^-s of accumulator columns 2q and 2q + 1.
__device__ __forceinline__ void build_x_fragments(const uint16_t *x, int C, int H, int ks0, uint32_t (&bf)[kWarpSteps][2],
                                                  float &colinv0, float &colinv1) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  float am = 0.f;
  const bool tok = g < C;
  const uint16_t *xr = x + (size_t)(tok ? g : 0) * H;
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++) {
    const int k0 = 16 * (ks0 + s) + 2 * q;
    uint32_t v0 = 0, v1 = 0;
    if (tok && k0 < H) {
      v0 = *reinterpret_cast<const uint32_t *>(xr + k0);
      v1 = *reinterpret_cast<const uint32_t *>(xr + k0 + 8);
    }
    bf[s][0] = v0;
    bf[s][1] = v1;
    am = fmaxf(am, fmaxf(fmaxf(fabsf(__uint_as_float(v0 << 16)), fabsf(__uint_as_float(v0 & 0xFFFF0000u))),
                         fmaxf(fabsf(__uint_as_float(v1 << 16)), fabsf(__uint_as_float(v1 & 0xFFFF0000u)))));
  }
  am = fmaxf(am, __shfl_xor_sync(kFull, am, 1));
  am = fmaxf(am, __shfl_xor_sync(kFull, am, 2));
  float inv;
  const float up = f16_range_scale(am, &inv);
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++)
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const uint32_t v = bf[s][h];
      bf[s][h] = pack_half2(__uint_as_float(v << 16) * up, __uint_as_float(v & 0xFFFF0000u) * up);
    }
  colinv0 = __shfl_sync(kFull, inv, (2 * q) * 4);
  colinv1 = __shfl_sync(kFull, inv, (2 * q + 1) * 4);
}

// W4A4: the raw bf16 pairs of x for the same fragment positions (quantized
// per expert by quant_x_fragments once the stage's expert is known).
__device__ __forceinline__ void load_x_raw(const uint16_t *x, int C, int H, int ks0, uint32_t (&bf)[kWarpSteps][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const bool tok = g < C;
  const uint16_t *xr = x + (size_t)(tok ? g : 0) * H;
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++) {
    const int k0 = 16 * (ks0 + s) + 2 * q;
    uint32_t v0 = 0, v1 = 0;
    if (tok && k0 < H) {
      v0 = *reinterpret_cast<const uint32_t *>(xr + k0);
      v1 = *reinterpret_cast<const uint32_t *>(xr + k0 + 8);
    }
    bf[s][0] = v0;
    bf[s][1] = v1;
  }
}
// W4A4: the raw bf16 fragments of x quantized in place to NVFP4 values
// e2m1 * e4m3 (f16, exact) with the input scale a; each k-step is one
// 16-element block, held by the lane quad of the token.
__device__ __forceinline__ void quant_x_fragments(uint32_t (&bf)[kWarpSteps][2], float a) {
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++) {
    const uint32_t w0 = bf[s][0], w1 = bf[s][1];
    nvfp4_quant_quad(__uint_as_float(w0 << 16), __uint_as_float(w0 & 0xFFFF0000u), __uint_as_float(w1 << 16),
                     __uint_as_float(w1 & 0xFFFF0000u), a, bf[s][0], bf[s][1]);
  }
}
// W4A4 B fragments of h (down): column g = slot g of the expert (pair = that
// slot's (token, slot) index or -1), h quantized to NVFP4 values with the
// down input scale a; one MMA column per slot, so 8 slots in one pass.
__device__ __forceinline__ void build_h_fragments_a4(const float *hbuf, int I, int ks0, int pair, float a,
                                                     uint32_t (&bf)[kWarpSteps][2]) {
  const int lane = threadIdx.x & 31, q = lane & 3;
  const bool have = pair >= 0;
  const float4 *hr4 = reinterpret_cast<const float4 *>(hbuf + (size_t)(have ? pair : 0) * I) + q;
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++) {
    const int ks = ks0 + s;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (have && 16 * ks < I) v = __ldcg(hr4 + 4 * ks);
    nvfp4_quant_quad(v.x, v.y, v.z, v.w, a, bf[s][0], bf[s][1]);
  }
}

// B fragments of h for a consumer warp's 16 k-steps starting at ks0 (down):
// column g = slot 4 pass + g / 2 of the expert, the hi (g even) or lo (g odd)
// f16 part of h * 2^s with 2^s set by that slot's max |h|.  Lane (g, q) reads
// the four values of each k-step it needs as one float4 (hbuf keeps every
// 16-element block in operand order).  pair_of_col = the (token, slot) pair of
// this lane's column or -1.  Returns 2^-s of this lane's accumulator columns.
__device__ __forceinline__ float build_h_fragments(const float *hbuf, const uint32_t *hamax, int I, int ks0, int pair,
                                                   uint32_t (&bf)[kWarpSteps][2]) {
  const int lane = threadIdx.x & 31, g = lane >> 2, q = lane & 3;
  const bool have = pair >= 0;
  const float4 *hr4 = reinterpret_cast<const float4 *>(hbuf + (size_t)(have ? pair : 0) * I) + q;
  const float am = have ? __uint_as_float(__ldcg(hamax + (have ? pair : 0))) : 0.f;
  float inv;
  const float up = f16_range_scale(am, &inv);
  const bool lo = (g & 1) != 0;
#pragma unroll
  for (int s = 0; s < kWarpSteps; s++) {
    const int ks = ks0 + s;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (have && 16 * ks < I) v = __ldcg(hr4 + 4 * ks);
    const float x0 = v.x * up, x1 = v.y * up, x2 = v.z * up, x3 = v.w * up;
    const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
    if (lo) {
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      bf[s][0] = pack_half2(x0 - f01.x, x1 - f01.y);
      bf[s][1] = pack_half2(x2 - f23.x, x3 - f23.y);
    } else {
      bf[s][0] = *reinterpret_cast<const uint32_t *>(&h01);
      bf[s][1] = *reinterpret_cast<const uint32_t *>(&h23);
    }
  }
  // columns 2q (hi) and 2q+1 (lo) of this lane belong to slot q
  return __shfl_sync(kFull, inv, (2 * q) * 4);
}

// ---------------------------------------------------------------- MMA step
// One consumer warp's 16 k-steps of one tile: codes/scales point at the
// warp's half slice inside the staged tile.  The 16x16 block of decoded
// weights is the A fragment of mma.m16n8k16; four independent accumulator
// chains (k-step s feeds chain s % 4) keep consecutive MMAs of the warp from
// waiting on each other.  acc = the four chains summed.
__device__ __forceinline__ void mma_half_slice(const uint8_t *codes, const uint8_t *scales,
                                               const uint32_t (&bf)[kWarpSteps][2], float (&acc)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  float acc4[4][4] = {};
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
      const int ks = (qg & 1) * 4 + jj;              // k-step inside the 8-step scale unit
      const uint32_t s2 = e4m3x2_to_f16x2(scs[ks >> 1] >> (16 * (ks & 1)));
      uint32_t A[4];
      e2m1x8_to_f16x2(cws[jj], A);
      A[0] = hmul2_lo(A[0], s2);
      A[1] = hmul2_hi(A[1], s2);
      A[2] = hmul2_lo(A[2], s2);
      A[3] = hmul2_hi(A[3], s2);
      mma16816(acc4[jj], A, bf[s][0], bf[s][1]);
    }
  }
#pragma unroll
  for (int c4 = 0; c4 < 4; c4++) acc[c4] = (acc4[0][c4] + acc4[1][c4]) + (acc4[2][c4] + acc4[3][c4]);
}

// The same step for two tiles that share the B fragments (the down
// projection stages two tiles at a time): per k-step both tiles' 16x16
// weight blocks are decoded and multiplied, two accumulator chains per tile.
// accA/accB = each tile's chains summed.
__device__ __forceinline__ void mma_half_slice_x2(const uint8_t *codesA, const uint8_t *scalesA, const uint8_t *codesB,
                                                  const uint8_t *scalesB, const uint32_t (&bf)[kWarpSteps][2],
                                                  float (&accA)[4], float (&accB)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  float ca[2][4] = {}, cb[2][4] = {};
  uint4 sa = make_uint4(0, 0, 0, 0), sb = make_uint4(0, 0, 0, 0);
#pragma unroll
  for (int qg = 0; qg < kWarpSteps / 4; qg++) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(codesA + ((size_t)qg * 32 + lane) * 16);
    const uint4 wb = *reinterpret_cast<const uint4 *>(codesB + ((size_t)qg * 32 + lane) * 16);
    if ((qg & 1) == 0) {
      sa = *reinterpret_cast<const uint4 *>(scalesA + ((size_t)(qg >> 1) * 8 + g) * 16);
      sb = *reinterpret_cast<const uint4 *>(scalesB + ((size_t)(qg >> 1) * 8 + g) * 16);
    }
    const uint32_t was[4] = {wa.x, wa.y, wa.z, wa.w}, wbs[4] = {wb.x, wb.y, wb.z, wb.w};
    const uint32_t sas[4] = {sa.x, sa.y, sa.z, sa.w}, sbs[4] = {sb.x, sb.y, sb.z, sb.w};
#pragma unroll
    for (int jj = 0; jj < 4; jj++) {
      const int s = 4 * qg + jj;
      const int ks = (qg & 1) * 4 + jj;
      const uint32_t s2a = e4m3x2_to_f16x2(sas[ks >> 1] >> (16 * (ks & 1)));
      const uint32_t s2b = e4m3x2_to_f16x2(sbs[ks >> 1] >> (16 * (ks & 1)));
      uint32_t A[4], B[4];
      e2m1x8_to_f16x2(was[jj], A);
      e2m1x8_to_f16x2(wbs[jj], B);
      A[0] = hmul2_lo(A[0], s2a); A[1] = hmul2_hi(A[1], s2a); A[2] = hmul2_lo(A[2], s2a); A[3] = hmul2_hi(A[3], s2a);
      B[0] = hmul2_lo(B[0], s2b); B[1] = hmul2_hi(B[1], s2b); B[2] = hmul2_lo(B[2], s2b); B[3] = hmul2_hi(B[3], s2b);
      mma16816(ca[jj & 1], A, bf[s][0], bf[s][1]);
      mma16816(cb[jj & 1], B, bf[s][0], bf[s][1]);
    }
  }
#pragma unroll
  for (int c4 = 0; c4 < 4; c4++) {
    accA[c4] = ca[0][c4] + ca[1][c4];
    accB[c4] = cb[0][c4] + cb[1][c4];
  }
}

// ---------------------------------------------------------------- MXFP4
// e8m0 scale byte -> fp32 2^(b - 127) (b = 0 gives the subnormal 2^-127; the
// packer rejects the NaN byte 0xFF).
__device__ __forceinline__ float e8m0_to_float(uint32_t b) { return __uint_as_float(b ? (b << 23) : 0x00400000u); }

// The MXFP4 forms of the two steps above.  A block scale covers 32 elements
// (two k-steps), a power of two that f16 cannot always hold, so it is applied
// in fp32 after the MMA: the two k-steps of a pair are multiplied with the
// raw e2m1 codes (exact in f16) into a fresh accumulator, which is then
// scaled by the rowA / rowB e8m0 values and added to the running sum.  The
// scale unit of row pair g for the warp's 16 k-steps is 16 bytes: the (rowA,
// rowB) bytes of its 8 k-step pairs.
__device__ __forceinline__ void mx_pair_step(const uint32_t cw0, const uint32_t cw1, const uint32_t (&b0)[2],
                                             const uint32_t (&b1)[2], uint32_t sab, float (&c)[4]) {
  float t[4] = {0.f, 0.f, 0.f, 0.f};
  uint32_t A[4];
  e2m1x8_to_f16x2(cw0, A);
  mma16816(t, A, b0[0], b0[1]);
  e2m1x8_to_f16x2(cw1, A);
  mma16816(t, A, b1[0], b1[1]);
  const float fa = e8m0_to_float(sab & 0xFFu), fb = e8m0_to_float((sab >> 8) & 0xFFu);
  c[0] = fmaf(t[0], fa, c[0]);
  c[1] = fmaf(t[1], fa, c[1]);
  c[2] = fmaf(t[2], fb, c[2]);
  c[3] = fmaf(t[3], fb, c[3]);
}

__device__ __forceinline__ void mma_half_slice_mx(const uint8_t *codes, const uint8_t *scales,
                                                  const uint32_t (&bf)[kWarpSteps][2], float (&acc)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const uint4 sc = *reinterpret_cast<const uint4 *>(scales + g * 16);
  const uint32_t scs[4] = {sc.x, sc.y, sc.z, sc.w};
  float c2[2][4] = {};
#pragma unroll
  for (int qg = 0; qg < kWarpSteps / 4; qg++) {
    const uint4 cw = *reinterpret_cast<const uint4 *>(codes + ((size_t)qg * 32 + lane) * 16);
    const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int pp = 0; pp < 2; pp++) {
      const int P = 2 * qg + pp;                       // k-step pair of the warp's 8
      mx_pair_step(cws[2 * pp], cws[2 * pp + 1], bf[2 * P], bf[2 * P + 1], scs[P >> 1] >> (16 * (P & 1)), c2[pp]);
    }
  }
#pragma unroll
  for (int c4 = 0; c4 < 4; c4++) acc[c4] = c2[0][c4] + c2[1][c4];
}

__device__ __forceinline__ void mma_half_slice_x2_mx(const uint8_t *codesA, const uint8_t *scalesA, const uint8_t *codesB,
                                                     const uint8_t *scalesB, const uint32_t (&bf)[kWarpSteps][2],
                                                     float (&accA)[4], float (&accB)[4]) {
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const uint4 sa = *reinterpret_cast<const uint4 *>(scalesA + g * 16);
  const uint4 sb = *reinterpret_cast<const uint4 *>(scalesB + g * 16);
  const uint32_t sas[4] = {sa.x, sa.y, sa.z, sa.w}, sbs[4] = {sb.x, sb.y, sb.z, sb.w};
  float ca[4] = {}, cb[4] = {};
#pragma unroll
  for (int qg = 0; qg < kWarpSteps / 4; qg++) {
    const uint4 wa = *reinterpret_cast<const uint4 *>(codesA + ((size_t)qg * 32 + lane) * 16);
    const uint4 wb = *reinterpret_cast<const uint4 *>(codesB + ((size_t)qg * 32 + lane) * 16);
    const uint32_t was[4] = {wa.x, wa.y, wa.z, wa.w}, wbs[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
    for (int pp = 0; pp < 2; pp++) {
      const int P = 2 * qg + pp;
      mx_pair_step(was[2 * pp], was[2 * pp + 1], bf[2 * P], bf[2 * P + 1], sas[P >> 1] >> (16 * (P & 1)), ca);
      mx_pair_step(wbs[2 * pp], wbs[2 * pp + 1], bf[2 * P], bf[2 * P + 1], sbs[P >> 1] >> (16 * (P & 1)), cb);
    }
  }
#pragma unroll
  for (int c4 = 0; c4 < 4; c4++) {
    accA[c4] = ca[c4];
    accB[c4] = cb[c4];
  }
}

}  // namespace moe
