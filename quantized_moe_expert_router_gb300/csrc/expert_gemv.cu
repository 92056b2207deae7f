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
// flattened list of (distinct expert, stage unit) is cut into equal contiguous
// ranges, one CTA per SM, so every SM streams the same bytes to within one
// unit.  A stage unit is one tile of 8 pair rows (gate/up) or two consecutive
// tiles (down: the smaller tiles need twice the work per synchronisation);
// tiles are contiguous in the packed layout (pack.cu).
//
// Streaming.  The CTA is warp-specialised and its warps never meet at a
// CTA-wide barrier after the dispatch: one producer lane copies each stage
// unit with one bulk copy (cp.async.bulk, global -> shared, completion counted
// on an mbarrier) into a ring of S stage buffers, up to S units ahead.  The W
// consumer warps all work on the same unit, each on its own 256-element K
// range (16 k-steps: half of one of the tile's 512-element slices), write
// their partials into the reduction slots that belong to the stage buffer and
// arrive on the stage's "reduced" mbarrier; the epilogue warp sums them and
// only then releases the stage buffer to the producer, so a consumer waits on
// nothing but the arrival of its data.  Every wait is bounded (about two
// seconds of %globaltimer): on expiry the waiting warp sets MOE_FLAG_TIMEOUT
// and leaves, and the producer waits (bounded) for its copies still in flight
// before exiting.
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
#include "gemv_core.cuh"

namespace moe {

constexpr int kDnTilesPerStage = 2;             // down projection: two tiles of 8 pair rows per stage

// MODE 0: gate/up, one tile per stage; MODE 2: gate/up, two tiles per stage
// (decode groups of at most 2 tokens: their partials are 1/4 of a warp's
// accumulators, so a stage's reduction slots stay small); MODE 1: down, two
// tiles per stage.
template <int MODE, int FMT, bool A4>
__global__ void __launch_bounds__(kMaxCtaThreads, 1) expert_gemv_kernel(const GemvArgs a) {
  constexpr bool GU = MODE != 1;
  constexpr bool MX = FMT == kFmtMxfp4;
  extern __shared__ __align__(128) uint8_t ring[];   // [S][stage_bytes] then the reduction slots
  __shared__ DispatchSmem ds;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ __align__(8) uint64_t red_full[kMaxStages];

  const int NS = a.slices, W = 2 * NS, S = a.stages;
  // reduction slots after the ring, a.red_stage_f4 float4 per stage:
  //   MODE 0: [W warps][32 lanes] float4
  //   MODE 2: [2 tiles][W warps][8 pair rows] float4 (tokens 0, 1 only)
  //   MODE 1: [2 passes][2 tiles][W warps][32 lanes] float2 (one pass per 4 token slots, C <= 8)
  constexpr int NP = MODE == 1 ? 2 : 1;
  float4 *red = reinterpret_cast<float4 *>(ring + (size_t)S * a.stage_bytes);
  const int red_slot_f4 = a.red_stage_f4 / NP;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool is_producer = warp == W;
  const bool is_epilogue = warp == W + 1;
  const bool is_consumer = warp < W;
  const int slice = warp >> 1, half = warp & 1;  // consumer: k-steps 32*slice + 16*half + [0, 16)
  const int ks0 = kSliceSteps * slice + kWarpSteps * half;
  const int g = lane >> 2, q = lane & 3;

  if (tid == 32 * W) {
    for (int s = 0; s < S; s++) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&red_full[s], W);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }

  // ---------------- B fragments of x (gate/up), independent of the router
  uint32_t bf[kWarpSteps][2];
  float colinv0 = 1.f, colinv1 = 1.f;           // 2^-s of accumulator columns 2q, 2q+1
  if constexpr (GU) {
    if (is_consumer) {
      if constexpr (A4) load_x_raw(a.x, a.C, a.H, ks0, bf);   // quantized once the stage's expert is known
      else build_x_fragments(a.x, a.C, a.H, ks0, bf, colinv0, colinv1);
    }
  }

  if constexpr (GU) pdl_wait();                  // ids/weights come from the router
  build_dispatch(ds, a.ids, a.weights, a.C, a.k, a.E, a.flags);
  pdl_launch_dependents();

  const int n = ds.n;
  const int T = n * a.tiles;
  const int t0 = split_point(T, blockIdx.x, gridDim.x), t1 = split_point(T, blockIdx.x + 1, gridDim.x);
  const int nstage = t1 - t0;

  if (is_producer) {
    // ------------------------------------------------ producer: bulk copies
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int i = 0;
      bool ok = true;
      int d = t0 / a.tiles, tile = t0 - d * a.tiles;
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
    // (expert rank, tile) of stage i, advanced incrementally
    int d = t0 / a.tiles, tile = t0 - d * a.tiles;
    if (nstage > 0) load_dispatch_scales(ds, a.scalars, d, (t1 - 1) / a.tiles + 1);
    if constexpr (MODE == 1) pdl_wait();
    // gate/up: running max |h| of tokens 2q, 2q+1 for expert rank d, merged
    // into hamax when d changes and at the end
    float hm0 = 0.f, hm1 = 0.f;
    auto flush_hmax = [&](int dd) {
#pragma unroll
      for (int o = MODE == 2 ? 1 : 4; o < 32; o <<= 1) {   // MODE 2: tokens 0, 1 in every lane
        hm0 = fmaxf(hm0, __shfl_xor_sync(kFull, hm0, o));
        hm1 = fmaxf(hm1, __shfl_xor_sync(kFull, hm1, o));
      }
      if (g == 0 && (MODE != 2 || q == 0)) {
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
      if constexpr (GU) {
        if (d != cur_d) {
          flush_hmax(cur_d);
          cur_d = d;
        }
      }
      const int npass = (GU || A4) ? 1 : (ds.nslot[d] + 3) / 4;
      const int eslot = i % S;
      if (!mbar_wait_bounded(&red_full[eslot], (uint32_t)(i / S) & 1u)) {
        atomicOr(a.flags, MOE_FLAG_TIMEOUT);
        ok = false;
        break;
      }
      for (int pass = 0; pass < npass; pass++, item++) {
        const int rs = eslot * NP + pass;
        if constexpr (MODE == 0) {
          const float4 *pr4 = red + (size_t)rs * red_slot_f4 + lane;
          float4 sum = pr4[0];
          for (int ww = 1; ww < W; ww++) {
            const float4 v = pr4[ww * 32];
            sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
          }
          const uint32_t mask = ds.tokmask[d];
          float *hrow = a.hbuf + operand_order(tile * 8 + g);
#pragma unroll
          for (int c2 = 0; c2 < 2; c2++) {
            const int t = 2 * q + c2;
            if ((mask >> t) & 1u) {
              const int p = ds.pair[d][t];
              const float gg = (c2 ? sum.y : sum.x) * ds.scal[d][0];
              const float uu = (c2 ? sum.w : sum.z) * ds.scal[d][1];
              const float h = (A4 ? 1.f : ds.wt[p]) * silu(gg) * uu;   // W4A4: router weight after down
              hrow[(size_t)p * a.I] = h;
              if (c2) hm1 = fmaxf(hm1, fabsf(h)); else hm0 = fmaxf(hm0, fabsf(h));
            }
          }
        } else if constexpr (MODE == 2) {
          // lanes 0..15: pair row g2 of tile tt of the stage, tokens 0 and 1
          if (lane < 16) {
            const int tt = lane >> 3, g2 = lane & 7;
            const float4 *pr4 = red + (size_t)rs * red_slot_f4 + (size_t)tt * W * 8 + g2;
            float4 sum = pr4[0];
            for (int ww = 1; ww < W; ww++) {
              const float4 v = pr4[ww * 8];
              sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            const uint32_t mask = ds.tokmask[d];
            float *hrow = a.hbuf + operand_order((tile * 2 + tt) * 8 + g2);
#pragma unroll
            for (int t = 0; t < 2; t++) {
              if ((mask >> t) & 1u) {
                const int p = ds.pair[d][t];
                const float gg = (t ? sum.y : sum.x) * ds.scal[d][0];
                const float uu = (t ? sum.w : sum.z) * ds.scal[d][1];
                const float h = (A4 ? 1.f : ds.wt[p]) * silu(gg) * uu;
                hrow[(size_t)p * a.I] = h;
                if (t) hm1 = fmaxf(hm1, fabsf(h)); else hm0 = fmaxf(hm0, fabsf(h));
              }
            }
          }
        } else if constexpr (A4) {
          // one MMA column per slot: lane q holds slots 2q and 2q+1, rows A
          // and B; the router weight multiplies the expert's output here
          const float4 *pr4 = red + (size_t)eslot * a.red_stage_f4 + lane;
          const float gd = ds.scal[d][2];
          const int ns = ds.nslot[d];
#pragma unroll
          for (int tt = 0; tt < kDnTilesPerStage; tt++) {
            float4 sum = pr4[(size_t)tt * W * 32];
            for (int ww = 1; ww < W; ww++) {
              const float4 v = pr4[(size_t)(tt * W + ww) * 32];
              sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            const size_t col = 2 * ((tile * kDnTilesPerStage + tt) * 8 + g);
            if (2 * q < ns) {
              const int p0 = ds.slot_pair[d][2 * q];
              *reinterpret_cast<float2 *>(a.ypair + (size_t)p0 * a.H + col) =
                  make_float2(sum.x * gd * ds.wt[p0], sum.z * gd * ds.wt[p0]);
            }
            if (2 * q + 1 < ns) {
              const int p1 = ds.slot_pair[d][2 * q + 1];
              *reinterpret_cast<float2 *>(a.ypair + (size_t)p1 * a.H + col) =
                  make_float2(sum.y * gd * ds.wt[p1], sum.w * gd * ds.wt[p1]);
            }
          }
        } else {
          const float2 *pr2 = reinterpret_cast<const float2 *>(red + (size_t)rs * red_slot_f4) + lane;
          const int sl = 4 * pass + q;
          const float gd = ds.scal[d][2];
#pragma unroll
          for (int tt = 0; tt < kDnTilesPerStage; tt++) {
            float2 sum = pr2[(size_t)tt * W * 32];
            for (int ww = 1; ww < W; ww++) {
              const float2 v = pr2[(size_t)(tt * W + ww) * 32];
              sum.x += v.x; sum.y += v.y;
            }
            if (sl < ds.nslot[d])
              *reinterpret_cast<float2 *>(a.ypair + (size_t)ds.slot_pair[d][sl] * a.H +
                                          2 * ((tile * kDnTilesPerStage + tt) * 8 + g)) =
                  make_float2(sum.x * gd, sum.y * gd);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[eslot]);   // ring stage and its reduction slots are free
      if (++tile == a.tiles) { tile = 0; d++; }
    }
    if constexpr (GU) {
      if (nstage > 0) flush_hmax(cur_d);
    }
    return;
  }

  // ---------------------------------------------------- consumers
  if constexpr (MODE == 1) pdl_wait();           // hbuf comes from the gate/up kernel
  int cur_key = -1;                              // (expert rank, pass) of bf
  int d = t0 / a.tiles, tile = t0 - d * a.tiles;
  int item = 0;
  bool ok = true;
  int xq_d = -1;                                 // W4A4 gate/up: expert rank bf is quantized for
  float ascale = 1.f;                            // W4A4: that rank's input scale (gate/up) or down scale
  for (int i = 0; i < nstage && ok; i++) {
    const int slot = i % S;
    const int npass = (GU || A4) ? 1 : (ds.nslot[d] + 3) / 4;
    if (A4 && d != xq_d) {   // (A4 is a template constant)
      // the rank's input scale, loaded before the data wait: gate/up reads x
      // quantized with max(a_gate, a_up), down h with a_down
      const float *sc = a.scalars + (size_t)ds.expert[d] * 6;
      ascale = GU ? fmaxf(__ldg(sc + 1), __ldg(sc + 3)) : __ldg(sc + 5);
    }
    if (!mbar_wait_bounded(&full_bar[slot], (uint32_t)(i / S) & 1u)) {
      atomicOr(a.flags, MOE_FLAG_TIMEOUT);
      break;
    }
    if constexpr (GU) {
      if (A4 && d != xq_d) {
        if (xq_d >= 0) load_x_raw(a.x, a.C, a.H, ks0, bf);   // bf holds the previous rank's values
        quant_x_fragments(bf, ascale);
        colinv0 = colinv1 = ascale;
        xq_d = d;
      }
    }
    // scale units: NVFP4 256 B per half slice (8 rows x 8 k-steps x 2 rows x 2
    // groups), MXFP4 128 B (8 rows x 8 k-step pairs x 2 rows)
    constexpr int kHalfScaleBytes = MX ? 128 : 256;
    const uint8_t *codes = ring + (size_t)slot * a.stage_bytes + (size_t)slice * 4096 + (size_t)half * 2048;
    const uint8_t *scales = ring + (size_t)slot * a.stage_bytes + (size_t)NS * 4096 +
                            (size_t)(2 * slice + half) * kHalfScaleBytes;

    for (int pass = 0; pass < npass; pass++, item++) {
      const int rs = slot * NP + pass;
      if constexpr (MODE == 1) {
        const int key = d * 2 + pass;
        if (key != cur_key) {
          cur_key = key;
          if constexpr (A4) {
            build_h_fragments_a4(a.hbuf, a.I, ks0, g < ds.nslot[d] ? ds.slot_pair[d][g] : -1, ascale, bf);
            colinv0 = colinv1 = ascale;
            xq_d = d;
          } else {
            const int sl = 4 * pass + (g >> 1);
            colinv0 = colinv1 =
                build_h_fragments(a.hbuf, a.hamax, a.I, ks0, sl < ds.nslot[d] ? ds.slot_pair[d][sl] : -1, bf);
          }
        }
      }

      if constexpr (MODE == 0) {
        float acc[4];
        if constexpr (MX) mma_half_slice_mx(codes, scales, bf, acc);
        else mma_half_slice(codes, scales, bf, acc);
        red[(size_t)rs * red_slot_f4 + (size_t)warp * 32 + lane] =
            make_float4(acc[0] * colinv0, acc[1] * colinv1, acc[2] * colinv0, acc[3] * colinv1);
      } else if constexpr (MODE == 2) {
        // two tiles per stage; lanes q = 0 hold the columns of tokens 0 and 1
        const int tb = a.tile_bytes / 2;
        float accA[4], accB[4];
        if constexpr (MX) mma_half_slice_x2_mx(codes, scales, codes + tb, scales + tb, bf, accA, accB);
        else mma_half_slice_x2(codes, scales, codes + tb, scales + tb, bf, accA, accB);
        if (q == 0) {
          float4 *r4 = red + (size_t)rs * red_slot_f4;
          r4[(size_t)warp * 8 + g] = make_float4(accA[0] * colinv0, accA[1] * colinv1, accA[2] * colinv0, accA[3] * colinv1);
          r4[(size_t)(W + warp) * 8 + g] =
              make_float4(accB[0] * colinv0, accB[1] * colinv1, accB[2] * colinv0, accB[3] * colinv1);
        }
      } else {
        // two tiles per stage; the hi and lo columns of a slot are added here
        // (both carry the slot's 2^-s), so a partial is one float2 per tile
        const int tb = a.tile_bytes / kDnTilesPerStage;
        float accA[4], accB[4];
        if constexpr (MX) mma_half_slice_x2_mx(codes, scales, codes + tb, scales + tb, bf, accA, accB);
        else mma_half_slice_x2(codes, scales, codes + tb, scales + tb, bf, accA, accB);
        if constexpr (A4) {
          // columns 2q, 2q+1 are slots 2q, 2q+1: a partial is one float4 per tile
          float4 *r4 = red + (size_t)slot * a.red_stage_f4;
          r4[(size_t)warp * 32 + lane] = make_float4(accA[0] * colinv0, accA[1] * colinv0, accA[2] * colinv0, accA[3] * colinv0);
          r4[(size_t)(W + warp) * 32 + lane] =
              make_float4(accB[0] * colinv0, accB[1] * colinv0, accB[2] * colinv0, accB[3] * colinv0);
        } else {
          float2 *r2 = reinterpret_cast<float2 *>(red + (size_t)rs * red_slot_f4);
          r2[(size_t)warp * 32 + lane] = make_float2((accA[0] + accA[1]) * colinv0, (accA[2] + accA[3]) * colinv0);
          r2[(size_t)(W + warp) * 32 + lane] = make_float2((accB[0] + accB[1]) * colinv0, (accB[2] + accB[3]) * colinv0);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&red_full[slot]);     // this warp's partials of the stage are written
    if (++tile == a.tiles) { tile = 0; d++; }
  }
}

// ------------------------------------------------------------------ host side
// Ring geometry: as many stages (stage unit + its reduction slots) as fit.
void gemv_geometry(int stage_bytes, int red_stage_bytes, int *stages, int *smem_bytes) {
  int s = kGemvSmemBytes / (stage_bytes + red_stage_bytes);
  if (s > kMaxStages) s = kMaxStages;
  if (s < 2) s = 2;
  *stages = s;
  *smem_bytes = s * (stage_bytes + red_stage_bytes);
}

template <int MODE, int FMT, bool A4>
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
  return cudaLaunchKernelEx(&cfg, expert_gemv_kernel<MODE, FMT, A4>, a);
}

template <int FMT, bool A4>
static cudaError_t launch_fmt(int mode, const GemvArgs &a, int grid, bool pdl, cudaStream_t stream) {
  return mode == 0   ? launch_one<0, FMT, A4>(a, grid, pdl, stream)
         : mode == 2 ? launch_one<2, FMT, A4>(a, grid, pdl, stream)
                     : launch_one<1, FMT, A4>(a, grid, pdl, stream);
}

cudaError_t launch_expert_gemv(int mode, const GemvArgs &a, int grid, bool pdl, cudaStream_t stream) {
  if (a.fmt == kFmtMxfp4) return launch_fmt<kFmtMxfp4, false>(mode, a, grid, pdl, stream);   // W4A4 is NVFP4 only
  return a.w4a4 ? launch_fmt<kFmtNvfp4, true>(mode, a, grid, pdl, stream)
                : launch_fmt<kFmtNvfp4, false>(mode, a, grid, pdl, stream);
}

template <int MODE, int FMT, bool A4>
static cudaError_t allow_smem(int smem) {
  return cudaFuncSetAttribute(expert_gemv_kernel<MODE, FMT, A4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t gemv_setup() {
  // the largest dynamic shared memory any geometry requests (the attribute is
  // per kernel and device, so it must not depend on the layer that sets it)
  const int smem = kGemvSmemBytes;
  cudaError_t err = allow_smem<0, kFmtNvfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<1, kFmtNvfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<2, kFmtNvfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<0, kFmtMxfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<1, kFmtMxfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<2, kFmtMxfp4, false>(smem);
  if (err == cudaSuccess) err = allow_smem<0, kFmtNvfp4, true>(smem);
  if (err == cudaSuccess) err = allow_smem<1, kFmtNvfp4, true>(smem);
  if (err == cudaSuccess) err = allow_smem<2, kFmtNvfp4, true>(smem);
  return err;
}

}  // namespace moe
