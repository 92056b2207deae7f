// dense.cu -- the dense 4-bit GEMVs around the routed sum and the RMS norm
// between them ("SparkInfer-K3", section "How the TP module works":
// FfnPartial = router -> routed_down -> experts, FfnFinish = routed_norm ->
// routed_up -> shared experts; section "The model": hidden 7168, latent MoE
// at 3584, 2 shared experts).
//
//   routed_down   x[t] = D_lat u[t]            [latent][hidden], u bf16, x -> bf16
//   routed_norm   n[t] = y[t] / sqrt(mean y[t]^2 + eps) * gamma
//   routed_up     z[t] = U_lat n[t]            [hidden][latent], n fp32
//   shared s      z[t] += D_s (silu(G_s u[t]) * (U_s u[t]))
//
// A matrix is packed in the routed experts' tile layout (pack_core.cuh):
// pair rows (2p, 2p+1) for a plain matrix, (gate row p, up row p) for a
// shared expert's gate/up.  A GEMV runs in two kernels:
//   dense_partial_kernel  one warp per unit (tile of 16 rows, 512-element
//                         K-slice; units slice-major, an equal contiguous
//                         range per CTA, so a CTA builds the B fragments of
//                         only the one or two slices it covers): the unit's
//                         code and scale bytes come
//                         straight from global memory into registers (all
//                         twelve 16-byte loads of a lane in flight at once),
//                         the B operand (the C <= 8 input vectors as f16,
//                         scaled per token by a power of two; fp32 inputs as
//                         f16 hi + lo parts, two MMA columns per token) from
//                         shared memory, fp32 accumulation by mma.m16n8k16;
//                         the unit's partial goes to a workspace buffer;
//   dense_finish_kernel   one thread per (token, pair row): the partials of
//                         a tile summed over its slices in slice order, the
//                         tensor scale, then the epilogue (plain rows written
//                         or added to the output, or SwiGLU of a gate/up pair).
// No float atomics: results are bitwise reproducible.
#include <cuda_bf16.h>

#include "moe_internal.cuh"
#include "kernels.h"
#include "gemv_core.cuh"
#include "pack_core.cuh"

namespace moe {

constexpr int kDenseWarps = 16;

// ---------------------------------------------------------------- packing
// One thread per (source tile, source slice w, pair row g); the tile and
// slice land at tile0 + tile, wd0 + w of a destination of W slices per tile.
__global__ void pack_dense_kernel(const PackDenseArgs a) {
  const bool mx = a.fmt == kFmtMxfp4;
  const int SB = mx ? 32 : 16;
  const int64_t tiles = a.mode == 0 ? a.M / 16 : a.M / 8;
  const int64_t items = tiles * a.Wsrc * 8;
  const size_t slice_bytes = mx ? kTileSliceBytesMx : kTileSliceBytes;
  int nan_seen = 0;
  for (int64_t it = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; it < items; it += (int64_t)gridDim.x * blockDim.x) {
    const int g = (int)(it % 8);
    const int w = (int)((it / 8) % a.Wsrc);
    const int64_t tile = it / (8 * (int64_t)a.Wsrc);
    const int64_t p = tile * 8 + g;
    const uint8_t *ca, *cb, *sa, *sb;
    if (a.mode == 0) {                           // rows 2p and 2p + 1 of A
      ca = a.codesA + 2 * p * (a.K / 2); cb = ca + a.K / 2;
      sa = a.scalesA + 2 * p * (a.K / SB); sb = sa + a.K / SB;
    } else {                                     // row p of A and of B
      ca = a.codesA + p * (a.K / 2); cb = a.codesB + p * (a.K / 2);
      sa = a.scalesA + p * (a.K / SB); sb = a.scalesB + p * (a.K / SB);
    }
    nan_seen |= pack_pair_slice(ca, cb, sa, sb, a.K, mx, w, a.wd0 + w, g, a.W,
                                a.dst + (a.tile0 + tile) * a.W * slice_bytes);
  }
  if (nan_seen) atomicOr(a.status, 1);
}

// ---------------------------------------------------------------- partials
// XF32: fp32 input (hi / lo columns); NP: B-fragment passes (fp32: one per
// four tokens; bf16: one)
template <int FMT, bool XF32, int NP>
__global__ void __launch_bounds__(32 * kDenseWarps, 1) dense_partial_kernel(const DenseArgs a) {
  extern __shared__ uint2 frag[];                // [npass][KSL][32 lanes]: B fragments of this CTA's k-steps
  __shared__ float s_inv[kGemvTokens];           // 2^-s of each token's f16 scale
  __shared__ float s_max[kDenseWarps][kGemvTokens];
  constexpr bool MX = FMT == kFmtMxfp4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, q = lane & 3;
  const int NWL = a.w1 - a.w0;                   // this launch's slices
  // units slice-major (u = slice * tiles + tile): this CTA's contiguous range
  // spans one or two slices
  const int units = a.tiles * NWL;
  const int u0 = split_point(units, blockIdx.x, gridDim.x), u1 = split_point(units, blockIdx.x + 1, gridDim.x);
  if (u0 >= u1) return;
  const int wf = u0 / a.tiles, nsl = (u1 - 1) / a.tiles - wf + 1;
  const int KSL = 32 * nsl;                      // k-steps of the CTA's slices
  const int kbase = 512 * (a.w0 + wf);           // first element of their K range
  constexpr int npass = NP;
  const uint16_t *xb = static_cast<const uint16_t *>(a.x);
  const float *xf = static_cast<const float *>(a.x);
  auto xval = [&](int t, int k) -> float {
    if (k >= a.K) return 0.f;
    return XF32 ? __ldg(xf + (size_t)t * a.K + k) : __uint_as_float((uint32_t)__ldg(xb + (size_t)t * a.K + k) << 16);
  };
  // per-token max |x| over the whole K (fixed reduction tree): every CTA and
  // every launch of one GEMV scale a token alike; 16-byte loads (K % 64 == 0)
  for (int t = 0; t < a.C; t++) {
    float m = 0.f;
    if constexpr (XF32) {
      const float4 *r = reinterpret_cast<const float4 *>(xf + (size_t)t * a.K);
      for (int j = tid; j < a.K / 4; j += blockDim.x) {
        const float4 v = __ldg(r + j);
        m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
      }
    } else {
      const uint4 *r = reinterpret_cast<const uint4 *>(xb + (size_t)t * a.K);
      for (int j = tid; j < a.K / 8; j += blockDim.x) {
        const uint4 v = __ldg(r + j);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; e++)
          m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w4[e] << 16)), fabsf(__uint_as_float(w4[e] & 0xFFFF0000u))));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
    if (lane == 0) s_max[warp][t] = m;
  }
  __syncthreads();
  if (tid < a.C) {
    float m = 0.f;
    for (int w = 0; w < kDenseWarps; w++) m = fmaxf(m, s_max[w][tid]);
    float inv;
    f16_range_scale(m, &inv);
    s_inv[tid] = inv;
  }
  __syncthreads();
  // B fragments: lane (g, q) of k-step ks holds elements 16 ks + 2q, +1 and
  // 16 ks + 2q + 8, +9 of column g: token g (bf16 input), or the hi (g even)
  // / lo (g odd) part of token 4 pass + g / 2 (fp32 input)
  for (int i = tid; i < npass * KSL * 32; i += blockDim.x) {
    const int l = i & 31, ks = (i >> 5) % KSL, pass = (i >> 5) / KSL;
    const int gg = l >> 2, qq = l & 3;
    const int t = XF32 ? 4 * pass + (gg >> 1) : gg;
    uint2 v = make_uint2(0u, 0u);
    if (t < a.C) {
      const float up = __frcp_rn(s_inv[t]);      // exact: a power of two
      const int k0 = kbase + 16 * ks + 2 * qq;
      const float x0 = xval(t, k0) * up, x1 = xval(t, k0 + 1) * up, x2 = xval(t, k0 + 8) * up, x3 = xval(t, k0 + 9) * up;
      const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
      if (XF32 && (gg & 1)) {
        const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
        v = make_uint2(pack_half2(x0 - f01.x, x1 - f01.y), pack_half2(x2 - f23.x, x3 - f23.y));
      } else {
        v = make_uint2(*reinterpret_cast<const uint32_t *>(&h01), *reinterpret_cast<const uint32_t *>(&h23));
      }
    }
    frag[i] = v;
  }
  __syncthreads();
  // column scales of this lane's accumulator columns 2q, 2q + 1 (per pass)
  float cinv[NP][2];
#pragma unroll
  for (int pass = 0; pass < NP; pass++) {
    const int t0 = XF32 ? 4 * pass + q : 2 * q, t1 = XF32 ? t0 : 2 * q + 1;
    cinv[pass][0] = t0 < a.C ? s_inv[t0] : 0.f;
    cinv[pass][1] = t1 < a.C ? s_inv[t1] : 0.f;
  }
  const uint64_t pol = l2_evict_first_policy();
  for (int u = u0 + warp; u < u1; u += kDenseWarps) {
    const int wl = u / a.tiles, tile = u - wl * a.tiles, w = a.w0 + wl;
    const uint8_t *base = a.w + (size_t)tile * a.tile_bytes;
    uint4 cw[8], sc[4];
#pragma unroll
    for (int qg = 0; qg < 8; qg++) cw[qg] = ld_stream_v4(base + (size_t)w * 4096 + ((size_t)qg * 32 + lane) * 16, pol);
    if constexpr (MX) {
#pragma unroll
      for (int u2 = 0; u2 < 2; u2++)
        sc[u2] = ld_stream_v4(base + (size_t)a.W * 4096 + (size_t)w * 256 + ((size_t)u2 * 8 + g) * 16, pol);
    } else {
#pragma unroll
      for (int q8 = 0; q8 < 4; q8++)
        sc[q8] = ld_stream_v4(base + (size_t)a.W * 4096 + (size_t)w * 512 + ((size_t)q8 * 8 + g) * 16, pol);
    }
    float acc[NP][2][4] = {};                    // [pass][chain][fragment]
    const uint2 *fr = frag + (size_t)(32 * (wl - wf)) * 32 + lane;
    if constexpr (MX) {
#pragma unroll
      for (int P = 0; P < 16; P++) {             // k-step pairs 2P, 2P + 1
        const uint4 c4 = cw[P >> 1];
        const uint32_t w0 = (P & 1) ? c4.z : c4.x, w1 = (P & 1) ? c4.w : c4.y;
        const uint4 s4 = sc[P >> 3];
        const int wi = (P & 7) >> 1;
        const uint32_t sab = (wi == 0 ? s4.x : wi == 1 ? s4.y : wi == 2 ? s4.z : s4.w) >> (16 * (P & 1));
#pragma unroll
        for (int pass = 0; pass < npass; pass++) {
          const uint2 b0 = fr[(size_t)(pass * KSL + 2 * P) * 32], b1 = fr[(size_t)(pass * KSL + 2 * P + 1) * 32];
          const uint32_t bb0[2] = {b0.x, b0.y}, bb1[2] = {b1.x, b1.y};
          mx_pair_step(w0, w1, bb0, bb1, sab, acc[pass][P & 1]);
        }
      }
    } else {
#pragma unroll
      for (int s = 0; s < 32; s++) {
        const uint4 c4 = cw[s >> 2];
        const int j = s & 3;
        const uint32_t word = j == 0 ? c4.x : j == 1 ? c4.y : j == 2 ? c4.z : c4.w;
        const uint4 s4 = sc[s >> 3];
        const int k8 = s & 7;
        const uint32_t sw = (k8 >> 1) == 0 ? s4.x : (k8 >> 1) == 1 ? s4.y : (k8 >> 1) == 2 ? s4.z : s4.w;
        const uint32_t s2 = e4m3x2_to_f16x2(sw >> (16 * (k8 & 1)));
        uint32_t A[4];
        e2m1x8_to_f16x2(word, A);
        A[0] = hmul2_lo(A[0], s2);
        A[1] = hmul2_hi(A[1], s2);
        A[2] = hmul2_lo(A[2], s2);
        A[3] = hmul2_hi(A[3], s2);
#pragma unroll
        for (int pass = 0; pass < npass; pass++) {
          const uint2 b = fr[(size_t)(pass * KSL + s) * 32];
          mma16816(acc[pass][s & 1], A, b.x, b.y);
        }
      }
    }
#pragma unroll
    for (int pass = 0; pass < npass; pass++) {
      float r[4];
#pragma unroll
      for (int c4 = 0; c4 < 4; c4++) r[c4] = acc[pass][0][c4] + acc[pass][1][c4];
      reinterpret_cast<float4 *>(a.part)[(((size_t)tile * a.W + w) * npass + pass) * 32 + lane] =
          make_float4(r[0] * cinv[pass][0], r[1] * cinv[pass][1], r[2] * cinv[pass][0], r[3] * cinv[pass][1]);
    }
  }
}

// ---------------------------------------------------------------- finish
// One thread per (token t, pair row p) of the matrix: the slices' partials
// summed in slice order (each times its slice scale, if any), then the
// epilogue of the tile range (segment) the pair row is in.
__global__ void dense_finish_kernel(const DenseFinishArgs a) {
  const int pairs = a.tiles * 8;
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= a.C * pairs) return;
  const int t = i / pairs, p = i - t * pairs;
  const int tile = p >> 3, g = p & 7;
  const int npass = a.xf32 ? (a.C + 3) / 4 : 1;
  const int pass = a.xf32 ? t >> 2 : 0, q = a.xf32 ? (t & 3) : (t >> 1), c = a.xf32 ? 0 : (t & 1);
  const int lane = 4 * g + q;
  float sa = 0.f, sb = 0.f;
  // the slices' partials in batches whose loads are all in flight together,
  // then added in slice order
  constexpr int kBatch = 8;
  const float4 *pp = reinterpret_cast<const float4 *>(a.part) + ((size_t)tile * a.W * npass + pass) * 32 + lane;
  for (int w0 = 0; w0 < a.W; w0 += kBatch) {
    float4 v[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; j++)
      v[j] = w0 + j < a.W ? __ldcg(pp + (size_t)(w0 + j) * npass * 32) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kBatch; j++) {
      if (w0 + j >= a.W) break;
      float va, vb;
      if (a.xf32) {                              // hi + lo columns of the token
        va = v[j].x + v[j].y;
        vb = v[j].z + v[j].w;
      } else {
        va = c ? v[j].y : v[j].x;
        vb = c ? v[j].w : v[j].z;
      }
      if (a.slice_scale) {
        const float ss = a.slice_scale[w0 + j];
        va *= ss;
        vb *= ss;
      }
      sa += va;
      sb += vb;
    }
  }
  int si = 0;
  while (si + 1 < a.nseg && tile >= a.seg[si].tile1) si++;
  const DenseSeg &sg = a.seg[si];
  const int pl = p - 8 * sg.tile0;               // pair row within the segment
  const float ga = sg.ga ? *sg.ga : 1.f, gb = sg.gb ? *sg.gb : 1.f;
  if (sg.mode == 1) {                            // gate / up pair: h = silu(g) * u
    sg.out_f32[(size_t)t * sg.out_ld + sg.col0 + pl] = silu(sa * ga) * (sb * gb);
    return;
  }
  const float ra = sa * ga, rb = sb * ga;        // rows 2p, 2p + 1
  const size_t o = (size_t)t * sg.out_ld + sg.col0 + 2 * pl;
  if (sg.out_bf16) {
    sg.out_bf16[o] = __bfloat16_as_ushort(__float2bfloat16_rn(ra));
    sg.out_bf16[o + 1] = __bfloat16_as_ushort(__float2bfloat16_rn(rb));
  } else if (sg.accumulate) {
    sg.out_f32[o] += ra;
    sg.out_f32[o + 1] += rb;
  } else {
    sg.out_f32[o] = ra;
    sg.out_f32[o + 1] = rb;
  }
}

// ---------------------------------------------------------------- RMS norm
// One CTA of 256 threads per token: sum of squares (fixed tree), then
// out = y / sqrt(ss / n + eps) * gamma.
__global__ void __launch_bounds__(256) rms_norm_kernel(const float *y, const float *gamma, float eps, int n, float *out,
                                                       int out_ld) {
  __shared__ float wsum[8];
  const int t = blockIdx.x, tid = threadIdx.x;
  const float *yr = y + (size_t)t * n;
  float s = 0.f;
  for (int i = tid; i < n; i += blockDim.x) s = fmaf(yr[i], yr[i], s);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
  if ((tid & 31) == 0) wsum[tid >> 5] = s;
  __syncthreads();
  float ss = 0.f;
#pragma unroll
  for (int w = 0; w < 8; w++) ss += wsum[w];
  const float r = 1.f / sqrtf(ss / (float)n + eps);
  for (int i = tid; i < n; i += blockDim.x) out[(size_t)t * out_ld + i] = yr[i] * r * gamma[i];
}

// ------------------------------------------------------------------ host side
cudaError_t launch_pack_dense(const PackDenseArgs &a, int num_sms, cudaStream_t stream) {
  pack_dense_kernel<<<num_sms * 4, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

// Shared memory of the B fragments of `slices` K-slices.
static size_t frag_bytes(int slices, int C, bool xf32) {
  const int npass = xf32 ? (C + 3) / 4 : 1;
  return (size_t)npass * slices * 32 * 32 * sizeof(uint2);
}

template <int FMT, bool XF32, int NP>
static cudaError_t launch_partial(const DenseArgs &a, int grid, size_t smem, cudaStream_t stream) {
  static bool attr_set = false;   // one opt-in per instantiation (the largest size the library uses)
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(dense_partial_kernel<FMT, XF32, NP>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize, kDenseSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  dense_partial_kernel<FMT, XF32, NP><<<grid, 32 * kDenseWarps, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_partial_fmt(const DenseArgs &a, int grid, size_t smem, cudaStream_t stream) {
  if (!a.xf32) return launch_partial<FMT, false, 1>(a, grid, smem, stream);
  return a.C <= 4 ? launch_partial<FMT, true, 1>(a, grid, smem, stream) : launch_partial<FMT, true, 2>(a, grid, smem, stream);
}

// Grid of a launch over `slices` slices and the most slices one CTA's
// contiguous unit range spans (ceil(range / tiles) + 1).
static void partial_grid(int tiles, int slices, int num_sms, int *grid, int *span) {
  const int units = tiles * slices;
  int g = (units + kDenseWarps - 1) / kDenseWarps;
  if (g > num_sms) g = num_sms;
  const int per_cta = (units + g - 1) / g;
  int sp = (per_cta + tiles - 1) / tiles + 1;
  if (sp > slices) sp = slices;
  *grid = g;
  *span = sp;
}

cudaError_t launch_dense_gemv(const DenseArgs &a0, const DenseFinishArgs &f, int num_sms, cudaStream_t stream) {
  if (a0.C < 1 || a0.C > kGemvTokens || f.nseg < 1 || f.nseg > kMaxDenseSegs) return cudaErrorInvalidValue;
  // slices per launch: as many as keep the B fragments of the slices one CTA
  // spans within shared memory (normally all of them in one launch)
  int per = a0.W, grid = 1, span = 1;
  for (;;) {
    partial_grid(a0.tiles, per, num_sms, &grid, &span);
    if (per == 1 || frag_bytes(span, a0.C, a0.xf32 != 0) <= (size_t)kDenseSmemBytes) break;
    per = (per + 1) / 2;
  }
  cudaError_t err = cudaSuccess;
  for (int w0 = 0; w0 < a0.W && err == cudaSuccess; w0 += per) {
    DenseArgs a = a0;
    a.w0 = w0;
    a.w1 = w0 + per < a0.W ? w0 + per : a0.W;
    partial_grid(a.tiles, a.w1 - a.w0, num_sms, &grid, &span);
    const size_t smem = frag_bytes(span, a.C, a.xf32 != 0);
    err = a.fmt == kFmtMxfp4 ? launch_partial_fmt<kFmtMxfp4>(a, grid, smem, stream)
                             : launch_partial_fmt<kFmtNvfp4>(a, grid, smem, stream);
  }
  if (err != cudaSuccess) return err;
  const int items = f.C * f.tiles * 8;
  dense_finish_kernel<<<(items + 255) / 256, 256, 0, stream>>>(f);
  return cudaGetLastError();
}

cudaError_t launch_rms_norm(const float *y, const float *gamma, float eps, int C, int n, float *out, int out_ld,
                            cudaStream_t stream) {
  rms_norm_kernel<<<C, 256, 0, stream>>>(y, gamma, eps, n, out, out_ld);
  return cudaGetLastError();
}

}  // namespace moe
