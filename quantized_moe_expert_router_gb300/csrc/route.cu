// route.cu -- router logits and top-k with renormalised softmax weights.
//
// Definition ("SparkInfer-K3", section "How the TP module works": one
// replicated router, every rank agrees on the same top-16):
//   l[t][e] = sum_j Wr[e][j] x[t][j] (+ bias[e])            (fp32 accumulate)
//   keep the k largest l[t][.], equal logits -> lower expert index first
//   w[t][i] = exp(l_i - l_max) / sum over kept exp(l_j - l_max)
// (a softmax over all experts renormalised over the kept ones; the full
// softmax denominator cancels).  ids are written in ascending expert order.
//
// Small C (decode): one kernel.  Each warp owns whole router rows and streams
// them once with 16-byte loads against x held in shared memory; every CTA
// then takes a ticket, and the last CTA to finish runs the top-k of each token
// in one warp (the ticket is reset for the next call).  No CTA ever waits for
// another.  Large C: a tiled fp32 logits kernel and a top-k kernel.
#include "moe_internal.cuh"
#include "kernels.h"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 is
// folded onto +0.  Key 0 (the image of one negative NaN pattern) marks
// "taken / absent".
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

// Top-k of one token's E logits by one warp.  Lane l holds experts l + 32 i.
// Each round takes the warp maximum key (redux.sync), breaks ties by the
// lowest expert index (redux.sync min), and removes the winner.
__device__ void warp_topk(const float *logits, int E, int k, int32_t *ids_out,
                          float *w_out) {
  const int lane = threadIdx.x & 31;
  uint32_t key[kMaxExperts / 32];
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; i++) {
    const int e = lane + 32 * i;
    key[i] = (e < E) ? order_key(__ldcg(logits + e)) : 0u;
  }
  uint32_t bk = 0;
  int bi = 0x7FFFFFFF;
#pragma unroll
  for (int i = 0; i < kMaxExperts / 32; i++)
    if (key[i] > bk) { bk = key[i]; bi = lane + 32 * i; }

  uint32_t my_key = 0;
  int my_idx = 0x7FFFFFFF;
  for (int r = 0; r < k; r++) {
    const uint32_t wmax = __reduce_max_sync(kFull, bk);
    const uint32_t cand = (bk == wmax) ? (uint32_t)bi : 0xFFFFFFFFu;
    const int widx = (int)__reduce_min_sync(kFull, cand);
    if (lane == r) { my_key = wmax; my_idx = widx; }
    if ((widx & 31) == lane) {
      const int slot = widx >> 5;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; i++)
        if (i == slot) key[i] = 0u;
      bk = 0;
      bi = 0x7FFFFFFF;
#pragma unroll
      for (int i = 0; i < kMaxExperts / 32; i++)
        if (key[i] > bk) { bk = key[i]; bi = lane + 32 * i; }
    }
  }
  // renormalised softmax over the kept logits; lane 0 holds the largest
  const float lmax = __shfl_sync(kFull, key_value(my_key), 0);
  const float ex = (lane < k) ? expf(key_value(my_key) - lmax) : 0.f;
  float sum = ex;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(kFull, sum, o);
  // rank in ascending expert order
  int rank = 0;
  for (int j = 0; j < k; j++) {
    const int other = __shfl_sync(kFull, my_idx, j);
    rank += (other < my_idx);
  }
  if (lane < k) {
    ids_out[rank] = my_idx;
    w_out[rank] = ex / sum;
  }
}

template <int CT>
__global__ void __launch_bounds__(256) route_fused_kernel(const RouteArgs a) {
  extern __shared__ float4 xs4[];          // [CT][H/4] float4
  float *xs = reinterpret_cast<float *>(xs4);
  __shared__ int s_last;
  pdl_wait();
  const int H4 = a.H / 4;
  for (int i = threadIdx.x; i < CT * a.H; i += blockDim.x) {
    const int t = i / a.H, j = i - t * a.H;
    xs[i] = (t < a.C) ? __uint_as_float((uint32_t)a.x[(size_t)t * a.H + j] << 16) : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const uint64_t pol = l2_evict_first_policy();
  for (int e = blockIdx.x * nwarps + warp; e < a.E; e += gridDim.x * nwarps) {
    const float4 *wrow = reinterpret_cast<const float4 *>(a.w_router + (size_t)e * a.H);
    float acc[CT];
#pragma unroll
    for (int t = 0; t < CT; t++) acc[t] = 0.f;
#pragma unroll 7
    for (int j = lane; j < H4; j += 32) {
      const uint4 wr = ld_stream_v4(wrow + j, pol);
      const float4 w = make_float4(__uint_as_float(wr.x), __uint_as_float(wr.y),
                                   __uint_as_float(wr.z), __uint_as_float(wr.w));
#pragma unroll
      for (int t = 0; t < CT; t++) {
        const float4 xv = xs4[t * H4 + j];
        acc[t] = fmaf(w.x, xv.x, acc[t]);
        acc[t] = fmaf(w.y, xv.y, acc[t]);
        acc[t] = fmaf(w.z, xv.z, acc[t]);
        acc[t] = fmaf(w.w, xv.w, acc[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < CT; t++)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc[t] += __shfl_xor_sync(kFull, acc[t], o);
    if (lane == 0) {
      const float b = a.bias ? a.bias[e] : 0.f;
#pragma unroll
      for (int t = 0; t < CT; t++)
        if (t < a.C) a.logits[(size_t)t * a.E + e] = acc[t] + b;
    }
  }
  // last CTA to finish runs the top-k
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t done = atomicAdd(a.ticket, 1u);
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  if (warp < a.C)
    warp_topk(a.logits + (size_t)warp * a.E, a.E, a.k, a.ids + (size_t)warp * a.k,
              a.weights + (size_t)warp * a.k);
  if (threadIdx.x == 0) *a.ticket = 0u;
}

// ------------------------------------------------------------ large C
// logits[C][E] = X[C][H] Wr^T + bias.  64 tokens x 64 experts per CTA,
// 256 threads with 4 x 4 outputs each, K tiles of 32 staged in shared memory.
__global__ void __launch_bounds__(256) route_logits_tiled_kernel(const RouteArgs a) {
  __shared__ float Xs[32][64 + 4];
  __shared__ float Ws[32][64 + 4];
  pdl_wait();
  const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < a.H; k0 += 32) {
    for (int i = tid; i < 64 * 32; i += 256) {
      const int r = i >> 5, c = i & 31;
      const int t = t0 + r, e = e0 + r;
      Xs[c][r] = (t < a.C) ? __uint_as_float((uint32_t)a.x[(size_t)t * a.H + k0 + c] << 16) : 0.f;
      Ws[c][r] = (e < a.E) ? a.w_router[(size_t)e * a.H + k0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < 32; c++) {
      float xv[4], wv[4];
#pragma unroll
      for (int i = 0; i < 4; i++) { xv[i] = Xs[c][ty * 4 + i]; wv[i] = Ws[c][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int t = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
      if (t < a.C && e < a.E) a.logits[(size_t)t * a.E + e] = acc[i][j] + (a.bias ? a.bias[e] : 0.f);
    }
}

__global__ void __launch_bounds__(256) route_topk_kernel(const RouteArgs a) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= a.C) return;
  warp_topk(a.logits + (size_t)t * a.E, a.E, a.k, a.ids + (size_t)t * a.k,
            a.weights + (size_t)t * a.k);
}

static size_t fused_smem(int ct, int H) { return sizeof(float) * (size_t)ct * H; }

// Opt-in shared memory for the largest hidden size the library accepts, so
// the attribute does not depend on which layer set it.
cudaError_t route_setup() {
  constexpr int kMaxHidden = 4096;
  cudaError_t err = cudaFuncSetAttribute(route_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused_smem(1, kMaxHidden));
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(route_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused_smem(2, kMaxHidden));
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(route_fused_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused_smem(4, kMaxHidden));
  if (err == cudaSuccess)
    err = cudaFuncSetAttribute(route_fused_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)fused_smem(8, kMaxHidden));
  return err;
}

cudaError_t launch_route_fused(const RouteArgs &a, int grid, cudaStream_t stream) {
  const int ct = a.C <= 1 ? 1 : a.C <= 2 ? 2 : a.C <= 4 ? 4 : 8;
  const size_t smem = fused_smem(ct, a.H);
  switch (ct) {
    case 1: route_fused_kernel<1><<<grid, 256, smem, stream>>>(a); break;
    case 2: route_fused_kernel<2><<<grid, 256, smem, stream>>>(a); break;
    case 4: route_fused_kernel<4><<<grid, 256, smem, stream>>>(a); break;
    default: route_fused_kernel<8><<<grid, 256, smem, stream>>>(a); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_route_batched(const RouteArgs &a, cudaStream_t stream) {
  dim3 g1((a.E + 63) / 64, (a.C + 63) / 64);
  route_logits_tiled_kernel<<<g1, 256, 0, stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  route_topk_kernel<<<(a.C + 7) / 8, 256, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
