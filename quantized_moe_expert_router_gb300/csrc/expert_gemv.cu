// expert_gemv.cu -- dequant-fused expert GEMV for decode batches (C <= 8):
//
//   mode 0 (gate/up):  for every selected expert e and token t that chose it,
//       g = G_e x_t, u = U_e x_t,  hbuf[(t,slot)] = w[t][slot] * silu(g) * u
//   mode 1 (down):     ypair[(t,slot)] = D_e hbuf[(t,slot)]
//
// The definition is the "MUL_MAT_ID" step of "Kimi-K3 on 2x A40 - measured
// findings" (section "Why the placement experiments all looked the same") with
// the routed sum of "SparkInfer-K3" ("How the TP module works"): each token's
// output is the router-weighted sum of its selected experts' FFN outputs.
// Folding the router weight into h before the down projection is the same sum
// (D is linear).
//
// Work split.  The selected experts are de-duplicated in every CTA (a bitmap
// over expert ids; popcount ranks give ascending expert order), so each
// expert's bytes are streamed once whatever number of tokens chose it.  The
// flattened list (distinct expert, tile of 8 pair rows) is cut into equal
// contiguous ranges, one CTA per SM, so every SM streams the same bytes to
// within one tile.  Tiles are contiguous in the packed layout (pack.cu).
//
// Streaming.  The CTA is warp-specialised and its warps never meet at a
// CTA-wide barrier after the dispatch: one producer lane copies each tile with
// one bulk copy (cp.async.bulk, global -> shared, completion counted on an
// mbarrier) into a ring of S stage buffers, up to S tiles ahead.  The W
// consumer warps all work on the same tile, each on its own 256-element
// K range (16 k-steps: half of one of the tile's 512-element slices), and hand
// their partials to one epilogue warp through a ring of reduction slots, also
// tracked by mbarriers (one item per tile and token pass).  Every wait is
// bounded (about two seconds of %globaltimer): on expiry the waiting warp sets
// MOE_FLAG_TIMEOUT and leaves, and the producer waits (bounded) for its copies
// still in flight before exiting.
//
// Compute.  Decoding stays in registers: per k-step a lane converts its 4
// code bytes with cvt.rn.f16x2.e2m1x2 and multiplies them by the row's e4m3
// block scale in f16 (exact: at most 2+4 significant bits, |value| <= 2688,
// no subnormals).  The 16x16 block of decoded weights is the A fragment of
// mma.m16n8k16 (rows g and g+8 = the two rows of pair row g of the tile), and
// the MMA accumulates in fp32 across the warp's K range; the eight MMA columns
// carry the decode batch:
//   gate/up: column n = token n of the group (x in f16, scaled by a power of
//            two per token and warp K range: exact for bf16 input);
//   down:    columns 2j, 2j+1 = the hi and lo f16 parts of h for the j-th
//            token that chose the expert (scaled by a power of two set by
//            that token slot's max |h|), so hi + lo carries h to 2^-22 of
//            its largest element.
// The partials (each rescaled by 2^-s) are summed over the W warps in a fixed
// order by the epilogue warp, which applies the tensor scale and writes hbuf
// (plus the running max |h| per token slot, which sets the down kernel's
// power-of-two scale) or ypair.
//
// The weighted sum over a token's experts is the separate combine kernel
// (combine.cu), which reads ypair in ascending expert order: no float atomics,
// bitwise reproducible.
#include "moe_internal.cuh"
#include "kernels.h"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kSliceSteps = 32;                  // k-steps of one 512-element K-slice of a tile
constexpr int kWarpSteps = 16;                   // k-steps per consumer warp (half a slice)
constexpr int kMaxKWarps = 16;                   // consumer warps: K <= 4096
constexpr int kMaxCtaThreads = 32 * (kMaxKWarps + 2);   // + producer and epilogue warps
constexpr int kRedSlots = 4;                     // consumer -> epilogue reduction ring
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
  float wt[kMaxPairs];                         // router weight of pair p
  float scal[kMaxPairs][3];                    // tensor scales g_gate, g_up, g_down of rank d
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
// p = t*k + slot both by token and in ascending token order).  Ids outside
// [0,E) are flagged and skipped; an id repeated inside a token is flagged and
// only its lowest slot is used (the combine kernel applies the same rule).
__device__ void build_dispatch(DispatchSmem &s, const int32_t *ids, const float *weights,
                               const float *scalars, int C, int k, int E, int32_t *flags) {
  const int tid = threadIdx.x, nt = blockDim.x, P = C * k;
  for (int i = tid; i < kMaxExperts / 32; i += nt) s.bitmap[i] = 0u;
  for (int i = tid; i < P; i += nt) s.tokmask[i] = 0u;
  for (int i = tid; i < P * kGemvTokens; i += nt) (&s.pair[0][0])[i] = 0x7FFFFFFF;
  __syncthreads();
  for (int p = tid; p < P; p += nt) {
    const int e = ids[p];
    if ((unsigned)e < (unsigned)E)
      atomicOr(&s.bitmap[e >> 5], 1u << (e & 31));
    else
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
    const int e = ids[p];
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
  for (int p = tid; p < P; p += nt) s.wt[p] = weights[p];
  for (int r = tid; r < s.n; r += nt) {
    const float *sc = scalars + (size_t)s.expert[r] * 6;
    s.scal[r][0] = sc[0];
    s.scal[r][1] = sc[2];
    s.scal[r][2] = sc[4];
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

template <int MODE>
__global__ void __launch_bounds__(kMaxCtaThreads, 1) expert_gemv_kernel(const GemvArgs a) {
  extern __shared__ __align__(128) uint8_t ring[];   // [S][stage_bytes] then the reduction slots
  __shared__ DispatchSmem ds;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t red_full[kRedSlots];
  __shared__ __align__(8) uint64_t red_empty[kRedSlots];

  const int NS = a.slices, W = 2 * NS, S = a.stages;
  // reduction slots [kRedSlots][W][32 lanes] of float4, after the ring
  float4 *red = reinterpret_cast<float4 *>(ring + (size_t)S * a.stage_bytes);
  const int red_slot_f4 = W * 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_producer = warp == W;
  const bool is_epilogue = warp == W + 1;
  const bool is_consumer = warp < W;
  const int slice = warp >> 1, half = warp & 1;  // consumer: k-steps 32*slice + 16*half + [0, 16)
  const int ks0 = kSliceSteps * slice + kWarpSteps * half;
  const int g = lane >> 2, q = lane & 3;
  const int K = MODE == 0 ? a.H : a.I;          // real K of this region's rows

  if (tid == 32 * W) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], W);
    }
    for (int s = 0; s < kRedSlots; s++) {
      mbar_init(&red_full[s], W);
      mbar_init(&red_empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---------------- B fragments of x (gate/up), independent of the router
  uint32_t bf[kWarpSteps][2];
  float colinv0 = 1.f, colinv1 = 1.f;           // 2^-s of accumulator columns 2q, 2q+1
  if constexpr (MODE == 0) {
    if (is_consumer) {
      float am = 0.f;
      const bool tok = g < a.C;
      const uint16_t *xr = a.x + (size_t)(tok ? g : 0) * a.H;
#pragma unroll
      for (int s = 0; s < kWarpSteps; s++) {
        const int k0 = 16 * (ks0 + s) + 2 * q;
        uint32_t v0 = 0, v1 = 0;
        if (tok && k0 < K) {
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
  }

  if constexpr (MODE == 0) pdl_wait();           // ids/weights come from the router
  build_dispatch(ds, a.ids, a.weights, a.scalars, a.C, a.k, a.E, a.flags);
  pdl_launch_dependents();

  const int n = ds.n;
  const long long T = (long long)n * a.tiles;
  const long long t0 = T * blockIdx.x / gridDim.x, t1 = T * (blockIdx.x + 1) / gridDim.x;
  const int nstage = (int)(t1 - t0);

  if (is_producer) {
    // ------------------------------------------------ producer: bulk copies
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int i = 0;
      bool ok = true;
      int d = (int)(t0 / a.tiles), tile = (int)(t0 - (long long)d * a.tiles);
      for (; i < nstage; i++, tile++) {
        if (tile == a.tiles) { tile = 0; d++; }
        const int slot = i % S;
        const uint32_t use = (uint32_t)(i / S);
        if (use > 0 && !mbar_wait_bounded(&empty_bar[slot], (use - 1) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          ok = false;
          break;
        }
        const uint8_t *src = a.packed + (size_t)ds.expert[d] * a.expert_bytes + a.region_off +
                             (size_t)tile * a.tile_bytes;
        mbar_arrive_expect_tx(&full_bar[slot], (uint32_t)a.tile_bytes);
        bulk_copy_g2s(ring + (size_t)slot * a.stage_bytes, src, (uint32_t)a.tile_bytes, &full_bar[slot], pol);
      }
      if (!ok) {
        // leave no copy in flight: wait (bounded) for the last use of each slot
        for (int j = (i > S ? i - S : 0); j < i; j++)
          mbar_wait_bounded(&full_bar[j % S], (uint32_t)(j / S) & 1u);
      }
    }
    return;
  }

  // Items of the reduction ring: one per (stage, pass), in stage order; the
  // down kernel makes one pass per 4 token slots of the tile's expert.
  if (is_epilogue) {
    // ------------------------------------------------ epilogue warp
    if constexpr (MODE == 1) pdl_wait();
    // (expert rank, tile) of stage i, advanced incrementally (no 64-bit division)
    int d = (int)(t0 / a.tiles), tile = (int)(t0 - (long long)d * a.tiles);
    // gate/up: running max |h| of tokens 2q, 2q+1 for expert rank d, merged
    // into hamax when d changes and at the end
    float hm0 = 0.f, hm1 = 0.f;
    auto flush_hmax = [&](int dd) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        hm0 = fmaxf(hm0, __shfl_xor_sync(kFull, hm0, o));
        hm1 = fmaxf(hm1, __shfl_xor_sync(kFull, hm1, o));
      }
      if (g == 0) {
        const uint32_t mask = ds.tokmask[dd];
        if ((mask >> (2 * q)) & 1u) atomicMax(a.hamax + ds.pair[dd][2 * q], __float_as_uint(hm0));
        if ((mask >> (2 * q + 1)) & 1u) atomicMax(a.hamax + ds.pair[dd][2 * q + 1], __float_as_uint(hm1));
      }
      hm0 = hm1 = 0.f;
    };
    int cur_d = d;
    int item = 0;
    bool ok = true;
    for (int i = 0; i < nstage && ok; i++) {
      if constexpr (MODE == 0) {
        if (d != cur_d) {
          flush_hmax(cur_d);
          cur_d = d;
        }
      }
      const int npass = MODE == 0 ? 1 : (ds.nslot[d] + 3) / 4;
      for (int pass = 0; pass < npass; pass++, item++) {
        const int rs = item % kRedSlots;
        if (!mbar_wait_bounded(&red_full[rs], (uint32_t)(item / kRedSlots) & 1u)) {
          atomicOr(a.flags, MOE_FLAG_TIMEOUT);
          ok = false;
          break;
        }
        const float4 *pr4 = red + (size_t)rs * red_slot_f4 + lane;
        float4 sum = pr4[0];
#pragma unroll
        for (int ww = 1; ww < kMaxKWarps; ww++) {
          if (ww < W) {
            const float4 v = pr4[ww * 32];
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
        }
        if constexpr (MODE == 0) {
          const uint32_t mask = ds.tokmask[d];
          float *hrow = a.hbuf + operand_order(tile * 8 + g);
#pragma unroll
          for (int c2 = 0; c2 < 2; c2++) {
            const int t = 2 * q + c2;
            if ((mask >> t) & 1u) {
              const int p = ds.pair[d][t];
              const float gg = (c2 ? sum.y : sum.x) * ds.scal[d][0];
              const float uu = (c2 ? sum.w : sum.z) * ds.scal[d][1];
              const float h = ds.wt[p] * silu(gg) * uu;
              hrow[(size_t)p * a.I] = h;
              if (c2) hm1 = fmaxf(hm1, fabsf(h)); else hm0 = fmaxf(hm0, fabsf(h));
            }
          }
        } else {
          const int sl = 4 * pass + q;
          if (sl < ds.nslot[d]) {
            const float gd = ds.scal[d][2];
            *reinterpret_cast<float2 *>(a.ypair + (size_t)ds.slot_pair[d][sl] * a.H + 2 * (tile * 8 + g)) =
                make_float2((sum.x + sum.y) * gd, (sum.z + sum.w) * gd);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&red_empty[rs]);
      }
      if (++tile == a.tiles) { tile = 0; d++; }
    }
    if constexpr (MODE == 0) {
      if (nstage > 0) flush_hmax(cur_d);
    }
    return;
  }

  // ---------------------------------------------------- consumers
  if constexpr (MODE == 1) pdl_wait();           // hbuf comes from the gate/up kernel
  int cur_key = -1;                              // (expert rank, pass) of bf
  int d = (int)(t0 / a.tiles), tile = (int)(t0 - (long long)d * a.tiles);
  int item = 0;
  bool ok = true;
  for (int i = 0; i < nstage && ok; i++) {
    const int slot = i % S;
    const int npass = MODE == 0 ? 1 : (ds.nslot[d] + 3) / 4;
    if (!mbar_wait_bounded(&full_bar[slot], (uint32_t)(i / S) & 1u)) {
      atomicOr(a.flags, MOE_FLAG_TIMEOUT);
      break;
    }
    const uint8_t *codes = ring + (size_t)slot * a.stage_bytes + (size_t)slice * 4096 + (size_t)half * 2048;
    const uint8_t *scales =
        ring + (size_t)slot * a.stage_bytes + (size_t)NS * 4096 + (size_t)slice * 512 + (size_t)half * 256;

    for (int pass = 0; pass < npass; pass++, item++) {
      const int rs = item % kRedSlots;
      const uint32_t ruse = (uint32_t)(item / kRedSlots);
      if (ruse > 0 && !mbar_wait_bounded(&red_empty[rs], (ruse - 1) & 1u)) {
        atomicOr(a.flags, MOE_FLAG_TIMEOUT);
        ok = false;
        break;
      }
      if constexpr (MODE == 1) {
        const int key = d * 2 + pass;
        if (key != cur_key) {
          // B fragments of h: column g = slot 4*pass + g/2, hi (g even) / lo
          // (g odd) f16 part of h * 2^s, with 2^s set by the slot's max |h|.
          // Lane (g, q) reads the four values of each k-step it needs as one
          // float4 (hbuf keeps every 16-element block in operand order).
          cur_key = key;
          const int sl = 4 * pass + (g >> 1);
          const bool have = sl < ds.nslot[d];
          const int pr = have ? ds.slot_pair[d][sl] : 0;
          const float4 *hr4 = reinterpret_cast<const float4 *>(a.hbuf + (size_t)pr * a.I) + q;
          const float am = have ? __uint_as_float(__ldcg(a.hamax + pr)) : 0.f;
          float inv;
          const float up = f16_range_scale(am, &inv);
          const bool lo = (g & 1) != 0;
#pragma unroll
          for (int s = 0; s < kWarpSteps; s++) {
            const int ks = ks0 + s;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (have && 16 * ks < K) v = __ldcg(hr4 + 4 * ks);
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
          colinv0 = colinv1 = __shfl_sync(kFull, inv, (2 * q) * 4);
        }
      }

      // four independent accumulator chains (k-step s feeds chain s % 4) so
      // consecutive MMAs of a warp do not wait on each other's results
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
      float acc[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; c4++) acc[c4] = (acc4[0][c4] + acc4[1][c4]) + (acc4[2][c4] + acc4[3][c4]);
      red[(size_t)rs * red_slot_f4 + (size_t)warp * 32 + lane] =
          make_float4(acc[0] * colinv0, acc[1] * colinv1, acc[2] * colinv0, acc[3] * colinv1);
      __syncwarp();
      if (lane == 0) mbar_arrive(&red_full[rs]);     // this warp's partials are in the reduction slot
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty_bar[slot]);    // stage buffer may be refilled
    if (++tile == a.tiles) { tile = 0; d++; }
  }
}

// ------------------------------------------------------------------ host side
// Ring geometry: as many tile stages as fit beside the reduction slots.
void gemv_geometry(int slices, int *stages, int *stage_bytes, int *smem_bytes) {
  const int tile = slices * kTileSliceBytes;
  const int red = kRedSlots * 2 * slices * 32 * (int)sizeof(float4);
  int s = (kGemvSmemBytes - red) / tile;
  if (s > kMaxStages) s = kMaxStages;
  if (s < 2) s = 2;
  *stage_bytes = tile;
  *stages = s;
  *smem_bytes = s * tile + red;
}

template <int MODE>
static cudaError_t launch_one(const GemvArgs &a, int grid, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(32 * (2 * a.slices + 2));   // consumers + producer + epilogue warps
  cfg.dynamicSmemBytes = (size_t)a.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, expert_gemv_kernel<MODE>, a);
}

cudaError_t launch_expert_gemv(int mode, const GemvArgs &a, int grid, bool pdl, cudaStream_t stream) {
  return mode == 0 ? launch_one<0>(a, grid, pdl, stream) : launch_one<1>(a, grid, pdl, stream);
}

cudaError_t gemv_setup() {
  // the largest dynamic shared memory any geometry requests (the attribute is
  // per kernel and device, so it must not depend on the layer that sets it)
  const int smem = kGemvSmemBytes;
  cudaError_t err = cudaFuncSetAttribute(expert_gemv_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(expert_gemv_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return err;
}

}  // namespace moe
