// expert_gemv.cu -- dequant-fused expert GEMV for decode batches (C <= 8):
//
//   mode 0 (gate/up):  for every selected expert e and token t that chose it,
//       g = G_e x_t, u = U_e x_t,  hbuf[(t,slot)] = w[t][slot] * silu(g) * u
//   mode 1 (down):     ypair[(t,slot)] = D_e hbuf[(t,slot)], then
//       y[t] = sum over t's experts, ascending expert id, of ypair[(t,slot)]
//
// The definition is the "MUL_MAT_ID" step of "Kimi-K3 on 2x A40 - measured
// findings" (section "Why the placement experiments all looked the same") with
// the routed sum of "SparkInfer-K3" ("How the TP module works"): each token's
// output is the router-weighted sum of its selected experts' FFN outputs.
// Folding the router weight into h before the down projection is the same sum
// (D is linear).
//
// Work split.  The selected experts are de-duplicated in every CTA (a bitmap
// over expert ids, popcount ranks = ascending expert order), so each expert's
// bytes are streamed once whatever number of tokens chose it.  The flattened
// list (distinct expert, pair row) is cut into equal contiguous ranges, one
// per CTA, so every SM streams the same number of bytes (to one pair row).
// Inside a CTA, thread b owns 16-element block b of K for every pair row: per
// row it issues one 16-byte load of codes (two rows' blocks) and one 2-byte
// load of their two e4m3 scales, decodes in registers
// (cvt.rn.f16x2.e2m1x2) and accumulates in fp32.  Partial sums of 16/NT rows
// x NT tokens x 2 rows are reduced across the CTA with one warp transpose-
// reduction and one shared-memory pass.
//
// Gate/up uses x in f16 scaled by a power of two per token (exact: a bf16
// value has 8 significant bits; the scale puts max|x| in [2^14, 2^15)) and
// the sm_100 mixed-precision fma (f16 x f16 + fp32).  Down uses h in fp32
// and packed fp32x2 fmas on the decoded weights.  The block scale multiplies
// each 16-element partial sum in fp32; the tensor scale multiplies the row.
//
// The down kernel combines without float atomics: every CTA counts, per
// 64-row chunk, the pair rows it finished; the CTA that completes a chunk
// (count == experts x rows) sums that chunk's ypair rows for every token in
// ascending expert order and resets the count.  No CTA waits for another.
#include "moe_internal.cuh"
#include "kernels.h"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kMaxGemvThreads = 256;   // K <= 4096

struct DispatchSmem {
  uint32_t bitmap[kMaxExperts / 32];
  int base[kMaxExperts / 32];
  int n;
  int16_t expert[kMaxPairs];
  uint32_t tokmask[kMaxPairs];
  int16_t pair[kMaxPairs][kGemvTokens];
};

// Distinct selected experts of this token group in ascending id order, with
// for each the mask of tokens that chose it and the (token, slot) pair index
// p = t*k + slot.  Ids outside [0,E) and repeats inside a token are flagged
// and skipped.
__device__ void build_dispatch(DispatchSmem &s, const int32_t *ids, int C, int k, int E,
                               int32_t *flags) {
  const int tid = threadIdx.x, nt = blockDim.x, P = C * k;
  for (int i = tid; i < kMaxExperts / 32; i += nt) s.bitmap[i] = 0u;
  for (int i = tid; i < P; i += nt) s.tokmask[i] = 0u;
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
    if ((old >> t) & 1u)
      atomicOr(flags, MOE_FLAG_DUPLICATE_ID);
    else
      s.pair[r][t] = (int16_t)p;
    s.expert[r] = (int16_t)e;
  }
  __syncthreads();
}

// Sum 32 per-lane values over the warp; lane l returns the sum of value l.
// Five butterfly steps, each halving the values a lane keeps.
__device__ __forceinline__ float warp_transpose_reduce32(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; i++) {
      const float send = up ? v[i] : v[i + o];
      const float keep = up ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, o);
    }
  }
  return v[0];
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + expf(-g)); }

template <int MODE, int NT>
__global__ void __launch_bounds__(kMaxGemvThreads) expert_gemv_kernel(const GemvArgs a) {
  constexpr int R = 16 / NT;          // pair rows per batch
  constexpr int V = 2 * NT * R;       // partial sums per thread per batch
  static_assert(V == 32, "one value per lane after the transpose-reduction");
  __shared__ DispatchSmem ds;
  __shared__ float red[kMaxGemvThreads / 32][33];
  __shared__ float tok_inv[NT];
  __shared__ uint32_t tok_amax[kMaxGemvThreads / 32][NT];
  __shared__ int s_chunk;

  const int b = threadIdx.x, TPR = blockDim.x;
  const int lane = b & 31, warp = b >> 5, nwarps = TPR >> 5;
  const int kb = 16 * b;                          // first K element of this thread
  const uint64_t pol = l2_evict_first_policy();

  // ---------------- operand prologue (does not depend on the previous kernel)
  uint32_t xh[MODE == 0 ? NT : 1][8];
  float hv[MODE == 1 ? NT : 1][16];
  if constexpr (MODE == 0) {
    float xf[NT][16];
#pragma unroll
    for (int t = 0; t < NT; t++) {
      uint32_t am = 0;
      if (t < a.C && kb < a.H) {
        const uint4 *src = reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H + kb);
        const uint4 v0 = src[0], v1 = src[1];
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
          xf[t][2 * i] = __uint_as_float(w[i] << 16);
          xf[t][2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
#pragma unroll
        for (int i = 0; i < 16; i++) am = max(am, __float_as_uint(fabsf(xf[t][i])));
      } else {
#pragma unroll
        for (int i = 0; i < 16; i++) xf[t][i] = 0.f;
      }
      am = __reduce_max_sync(kFull, am);
      if (lane == 0) tok_amax[warp][t] = am;
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < NT; t++) {
      uint32_t am = 0;
      for (int w = 0; w < nwarps; w++) am = max(am, tok_amax[w][t]);
      // power of two putting max|x| in [2^14, 2^15): exact rescale into f16
      int s = 0;
      if (am != 0u) s = 14 - ((int)((am >> 23) & 0xFF) - 127);
      s = max(-126, min(126, s));
      const float up = __uint_as_float((uint32_t)(127 + s) << 23);
      if (b == 0) tok_inv[t] = __uint_as_float((uint32_t)(127 - s) << 23);
#pragma unroll
      for (int i = 0; i < 8; i++) {
        const __half2 h = __floats2half2_rn(xf[t][2 * i] * up, xf[t][2 * i + 1] * up);
        xh[t][i] = *reinterpret_cast<const uint32_t *>(&h);
      }
    }
  }

  pdl_wait();   // ids/weights (router) for gate/up; hbuf (gate/up) for down
  build_dispatch(ds, a.ids, a.C, a.k, a.E, a.flags);
  pdl_launch_dependents();

  const int n = ds.n;
  if (MODE == 1 && n == 0) {
    // nothing routed: the combine never triggers, so write zeros here
    if (blockIdx.x == 0)
      for (int i = b; i < a.C * a.H; i += TPR) a.y[i] = 0.f;
    return;
  }
  const long long Q = (long long)n * a.rows;
  long long q = Q * blockIdx.x / gridDim.x;
  const long long q1 = Q * (blockIdx.x + 1) / gridDim.x;
  int cur_d = -1;
  if (b == 0) s_chunk = -1;

  while (q < q1) {
    const int d = (int)(q / a.rows), r = (int)(q % a.rows);
    int nr = (int)min((long long)R, q1 - q);
    nr = min(nr, a.rows - r);
    if (MODE == 1) nr = min(nr, kChunkPairRows - (r % kChunkPairRows));
    const int e = ds.expert[d];
    const uint32_t mask = ds.tokmask[d];

    if constexpr (MODE == 1) {
      if (d != cur_d) {
        cur_d = d;
#pragma unroll
        for (int t = 0; t < NT; t++) {
          if (((mask >> t) & 1u) && kb < a.I) {
            const float4 *src = reinterpret_cast<const float4 *>(a.hbuf + (size_t)ds.pair[d][t] * a.I + kb);
#pragma unroll
            for (int i = 0; i < 4; i++) {
              const float4 v = __ldcg(src + i);
              hv[t][4 * i] = v.x; hv[t][4 * i + 1] = v.y; hv[t][4 * i + 2] = v.z; hv[t][4 * i + 3] = v.w;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 16; i++) hv[t][i] = 0.f;
          }
        }
      }
    }

    const uint8_t *rowp = a.packed + (size_t)e * a.expert_bytes + a.region_off + (size_t)r * a.pair_bytes;
    uint4 cw[R];
    uint32_t sw[R];
#pragma unroll
    for (int j = 0; j < R; j++) {
      if (j < nr) {
        const uint8_t *p = rowp + (size_t)j * a.pair_bytes;
        cw[j] = ld_stream_v4(p + b * 16, pol);
        sw[j] = ld_stream_u16(p + (size_t)TPR * 16 + b * 2, pol);
      } else {
        cw[j] = make_uint4(0, 0, 0, 0);
        sw[j] = 0u;
      }
    }

    float acc[V];
#pragma unroll
    for (int j = 0; j < R; j++) {
      const float2 sc = e4m3x2_to_float2(sw[j]);
      uint32_t hA[8], hB[8];
      {
        uint32_t t4[4];
        e2m1x8_to_f16x2(cw[j].x, t4);
        hA[0] = t4[0]; hA[1] = t4[1]; hA[2] = t4[2]; hA[3] = t4[3];
        e2m1x8_to_f16x2(cw[j].y, t4);
        hA[4] = t4[0]; hA[5] = t4[1]; hA[6] = t4[2]; hA[7] = t4[3];
        e2m1x8_to_f16x2(cw[j].z, t4);
        hB[0] = t4[0]; hB[1] = t4[1]; hB[2] = t4[2]; hB[3] = t4[3];
        e2m1x8_to_f16x2(cw[j].w, t4);
        hB[4] = t4[0]; hB[5] = t4[1]; hB[6] = t4[2]; hB[7] = t4[3];
      }
#pragma unroll
      for (int t = 0; t < NT; t++) {
        float dA = 0.f, dB = 0.f;
        if ((mask >> t) & 1u) {
          if constexpr (MODE == 0) {
#pragma unroll
            for (int i = 0; i < 8; i++) {
              dA = fma2_f16_f32(hA[i], xh[t][i], dA);
              dB = fma2_f16_f32(hB[i], xh[t][i], dB);
            }
          } else {
            float2 pA = make_float2(0.f, 0.f), pB = make_float2(0.f, 0.f);
#pragma unroll
            for (int i = 0; i < 8; i++) {
              const float2 hvi = make_float2(hv[t][2 * i], hv[t][2 * i + 1]);
              pA = ffma2(__half22float2(*reinterpret_cast<const __half2 *>(&hA[i])), hvi, pA);
              pB = ffma2(__half22float2(*reinterpret_cast<const __half2 *>(&hB[i])), hvi, pB);
            }
            dA = pA.x + pA.y;
            dB = pB.x + pB.y;
          }
        }
        acc[(j * NT + t) * 2] = dA * sc.x;
        acc[(j * NT + t) * 2 + 1] = dB * sc.y;
      }
    }

    const float val = warp_transpose_reduce32(acc, lane);
    red[warp][lane] = val;
    __syncthreads();
    if (warp == 0) {
      float s = 0.f;
      for (int w = 0; w < nwarps; w++) s += red[w][lane];
      const float other = __shfl_xor_sync(kFull, s, 1);
      const int jt = lane >> 1, j = jt / NT, t = jt % NT;
      if ((lane & 1) == 0 && j < nr && ((mask >> t) & 1u)) {
        const int p = ds.pair[d][t];
        const float *sc = a.scalars + (size_t)e * 6;
        if constexpr (MODE == 0) {
          const float inv = tok_inv[t];
          const float g = s * sc[0] * inv, u = other * sc[2] * inv;
          a.hbuf[(size_t)p * a.I + r + j] = a.weights[p] * silu(g) * u;
        } else {
          const float gd = sc[4];
          *reinterpret_cast<float2 *>(a.ypair + (size_t)p * a.H + 2 * (r + j)) = make_float2(s * gd, other * gd);
        }
      }
      if constexpr (MODE == 1) {
        __threadfence();
        __syncwarp();
        if (lane == 0) {
          const int c = r / kChunkPairRows;
          const int csize = min(kChunkPairRows, a.rows - c * kChunkPairRows);
          const unsigned old = atomicAdd(a.chunk_cnt + c, (unsigned)nr);
          s_chunk = (old + nr == (unsigned)(n * csize)) ? c : -1;
        }
      }
    }
    __syncthreads();
    if constexpr (MODE == 1) {
      const int c = s_chunk;
      if (c >= 0) {
        __threadfence();
        const int row0 = 2 * c * kChunkPairRows;
        const int nrow = min(2 * kChunkPairRows, a.H - row0);
        for (int it = b; it < nrow * a.C; it += TPR) {
          const int t = it / nrow, row = row0 + it % nrow;
          float sum = 0.f;
          for (int dd = 0; dd < n; dd++)
            if ((ds.tokmask[dd] >> t) & 1u) sum += __ldcg(a.ypair + (size_t)ds.pair[dd][t] * a.H + row);
          a.y[(size_t)t * a.H + row] = sum;
        }
        if (b == 0) a.chunk_cnt[c] = 0u;
      }
    }
    q += nr;
  }
}

template <int MODE, int NT>
static cudaError_t launch_one(const GemvArgs &a, int threads, int grid, bool pdl, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, expert_gemv_kernel<MODE, NT>, a);
}

cudaError_t launch_expert_gemv(int mode, int nt, const GemvArgs &a, int threads, int grid,
                               bool pdl, cudaStream_t stream) {
  if (mode == 0) {
    switch (nt) {
      case 1: return launch_one<0, 1>(a, threads, grid, pdl, stream);
      case 2: return launch_one<0, 2>(a, threads, grid, pdl, stream);
      case 4: return launch_one<0, 4>(a, threads, grid, pdl, stream);
      default: return launch_one<0, 8>(a, threads, grid, pdl, stream);
    }
  }
  switch (nt) {
    case 1: return launch_one<1, 1>(a, threads, grid, pdl, stream);
    case 2: return launch_one<1, 2>(a, threads, grid, pdl, stream);
    case 4: return launch_one<1, 4>(a, threads, grid, pdl, stream);
    default: return launch_one<1, 8>(a, threads, grid, pdl, stream);
  }
}

template <int MODE, int NT>
static int occ_one(int threads) {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, expert_gemv_kernel<MODE, NT>, threads, 0) != cudaSuccess)
    return 1;
  return occ > 0 ? occ : 1;
}

int gemv_occupancy(int mode, int nt, int threads) {
  if (mode == 0) {
    switch (nt) {
      case 1: return occ_one<0, 1>(threads);
      case 2: return occ_one<0, 2>(threads);
      case 4: return occ_one<0, 4>(threads);
      default: return occ_one<0, 8>(threads);
    }
  }
  switch (nt) {
    case 1: return occ_one<1, 1>(threads);
    case 2: return occ_one<1, 2>(threads);
    case 4: return occ_one<1, 4>(threads);
    default: return occ_one<1, 8>(threads);
  }
}

}  // namespace moe
