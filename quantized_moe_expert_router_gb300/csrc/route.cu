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
// Small C (decode): one kernel.  Each CTA streams a contiguous range of
// router rows into shared memory with bulk copies, and each warp multiplies
// its rows by x (fp32, in shared memory) as soon as they are in.  Every CTA
// then takes a ticket, and the last CTA to finish runs the top-k of each
// token with all its warps (the ticket is reset for the next call).  No CTA
// ever waits for another.  A CTA whose rows do not arrive marks its logits
// NaN, which makes every token select nothing.  Large C: a tiled fp32 logits
// kernel and a top-k kernel with one CTA per token.
#include "moe_internal.cuh"
#include "kernels.h"
#include "topk.cuh"

namespace moe {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kRouteWarps = 8;

// Shared memory of the fused router: x of up to CT tokens as fp32, then the
// CTA's router rows (one round of at most kRouteRowSmem bytes).
constexpr int kRouteSmemBytes = 200 * 1024;

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Bounded wait for phase `parity` of the rows barrier; false when `limit_ns`
// of %globaltimer pass first.
__device__ __forceinline__ bool rows_wait(uint64_t *bar, uint32_t parity, unsigned long long limit_ns) {
  unsigned long long t0 = 0;
  for (uint32_t it = 0;; it++) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}" : "=r"(done) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    if (done) return true;
    unsigned long long now;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
    if (it == 0) t0 = now;
    else if (now - t0 > limit_ns) return false;
  }
}

template <int CT>
__global__ void __launch_bounds__(kRouteWarps * 32) route_fused_kernel(const RouteArgs a) {
  extern __shared__ __align__(128) float4 xs4[];   // [CT][H/4] then [rows][H/4]
  __shared__ int s_last;
  __shared__ SelectSmem tk;
  __shared__ __align__(8) uint64_t rows_bar[kRouteWarps];   // round row r arrives on rows_bar[r % 8]
  pdl_wait();
  pdl_launch_dependents();                 // the expert kernel may start its prologue
  const int H4 = a.H / 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const size_t row_bytes = (size_t)a.H * sizeof(float);
  float4 *rows4 = xs4 + (size_t)CT * H4;
  const int max_rows = (kRouteSmemBytes - CT * a.H * (int)sizeof(float)) / (a.H * (int)sizeof(float));
  // this CTA's router rows: a contiguous range, streamed into shared memory
  // with bulk copies in rounds of at most max_rows rows; warp w takes rows
  // w, w + 8, ... of a round as soon as they are in (its own barrier)
  const int r0 = split_point(a.E, blockIdx.x, gridDim.x), r1 = split_point(a.E, blockIdx.x + 1, gridDim.x);
  const uint64_t pol = l2_evict_first_policy();
  if (threadIdx.x == 0) {
    for (int w = 0; w < kRouteWarps; w++)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&rows_bar[w])) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  bool ok = true;
  int round = 0;
  for (int rb = r0; rb < r1; rb += max_rows, round++) {
    const int nr = (r1 - rb) < max_rows ? (r1 - rb) : max_rows;
    if (threadIdx.x == 0) {
      // every barrier completes one phase per round (a warp without rows
      // expects 0 bytes); (a.stall_tx: test hook, bytes that no copy
      // delivers, so the waits below run out)
      for (int w = 0; w < kRouteWarps; w++) {
        const uint32_t nw = nr > w ? (uint32_t)((nr - 1 - w) / kRouteWarps + 1) : 0u;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&rows_bar[w])),
                     "r"(nw * (uint32_t)row_bytes + (round == 0 && w == 0 ? a.stall_tx : 0u)) : "memory");
      }
      for (int r = 0; r < nr; r++)
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;"
            ::"r"(smem_addr(rows4 + (size_t)r * H4)), "l"(a.w_router + (size_t)(rb + r) * a.H),
            "r"((uint32_t)row_bytes), "r"(smem_addr(&rows_bar[r % kRouteWarps])), "l"(pol) : "memory");
    }
    if (round == 0) {
      // x -> fp32 in shared memory, 8 bf16 per 16-byte load, all loads of a
      // thread issued together
      const int H8 = a.H / 8;
#pragma unroll 4
      for (int i = threadIdx.x; i < CT * H8; i += blockDim.x) {
        const int t = i / H8, j = i - t * H8;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < a.C) v = __ldg(reinterpret_cast<const uint4 *>(a.x + (size_t)t * a.H) + j);
        xs4[2 * i] = make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u),
                                 __uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u));
        xs4[2 * i + 1] = make_float4(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u),
                                     __uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u));
      }
      __syncthreads();
    }
    // bounded wait for this warp's rows of the round (a.wait_ns of
    // %globaltimer, about two seconds), then its dot products
    const bool mine = __all_sync(kFull, rows_wait(&rows_bar[warp], (uint32_t)(round & 1), a.wait_ns)) != 0;
    if (mine) {
      for (int r = warp; r < nr; r += kRouteWarps) {
        const float4 *wrow = rows4 + (size_t)r * H4;
        float acc[CT];
#pragma unroll
        for (int t = 0; t < CT; t++) acc[t] = 0.f;
        for (int j = lane; j < H4; j += 32) {
          const float4 w = wrow[j];
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
          const int e = rb + r;
          const float b = a.bias ? a.bias[e] : 0.f;
#pragma unroll
          for (int t = 0; t < CT; t++)
            if (t < a.C) a.logits[(size_t)t * a.E + e] = acc[t] + b;
        }
      }
    }
    // one decision for the CTA; the rows buffer is refilled by the next round
    ok = __syncthreads_and(mine) != 0;
    if (!ok) break;
  }
  if (!ok) {
    // Some rows of the round did not arrive in time: flag it, give each
    // warp's copies one more bounded wait so that none is left in flight when
    // the CTA exits, and write NaN over all this CTA's logits, so that the
    // selection finds no expert for any token (ids -1, weights 0).
    if (threadIdx.x == 0) atomicOr(a.flags, MOE_FLAG_TIMEOUT);
    if (lane == 0) rows_wait(&rows_bar[warp], (uint32_t)(round & 1), a.wait_ns);
    for (int i = threadIdx.x; i < a.C * (r1 - r0); i += blockDim.x) {
      const int t = i / (r1 - r0), e = r0 + (i - t * (r1 - r0));
      a.logits[(size_t)t * a.E + e] = __int_as_float(0x7FC00000);
    }
  }
  // Every CTA takes a ticket, failed or not, so the last one always resets
  // the counter for the next call.  Thread 0's acquire-release add publishes
  // this CTA's logits (ordered before it by the barrier) and, in the last
  // CTA, makes every other CTA's visible to the selection after the barrier.
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t done;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(done) : "l"(a.ticket) : "memory");
    s_last = (done == gridDim.x - 1);
  }
  __syncthreads();
  if (!s_last) return;
  for (int t = 0; t < a.C; t++)
    cta_select_topk<kRouteWarps * 32>(a.logits + (size_t)t * a.E, a.E, a.k, a.ids + (size_t)t * a.k,
                                      a.weights + (size_t)t * a.k, tk);
  if (threadIdx.x == 0) *a.ticket = 0u;
}

// ------------------------------------------------------------ large C
// Partial logits part[z][C][E] = X[C][K_z] Wr[E][K_z]^T over the z-th of
// kRouteSplits contiguous ranges of 32-wide K tiles.  64 tokens x 64
// experts per CTA, 256 threads with 4 x 4 outputs each, K tiles of 32 staged
// in shared memory (k-major, so a thread reads its 4 tokens and 4 experts of
// one k as two 16-byte loads).
__global__ void __launch_bounds__(256) route_logits_tiled_kernel(const RouteArgs a) {
  __shared__ __align__(16) float Xs[32][64 + 4];
  __shared__ __align__(16) float Ws[32][64 + 4];
  pdl_wait();
  const int t0 = blockIdx.y * 64, e0 = blockIdx.x * 64;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int KT = a.H / 32;
  const int kt0 = split_point(KT, blockIdx.z, gridDim.z), kt1 = split_point(KT, blockIdx.z + 1, gridDim.z);
  // tile loads: X row rx (8 bf16 at kx), W rows rw and rw + 32 (4 floats at kw);
  // the next tile's loads are in flight while the current one is multiplied
  const int rx = tid >> 2, kx = (tid & 3) * 8, rw = tid >> 3, kw = (tid & 7) * 4;
  const bool xin = t0 + rx < a.C, win0 = e0 + rw < a.E, win1 = e0 + rw + 32 < a.E;
  const uint16_t *xrow = a.x + (size_t)(t0 + rx) * a.H + kx;
  const float *wrow0 = a.w_router + (size_t)(e0 + rw) * a.H + kw, *wrow1 = wrow0 + (size_t)32 * a.H;
  uint4 xr = make_uint4(0u, 0u, 0u, 0u);
  float4 wr0 = make_float4(0.f, 0.f, 0.f, 0.f), wr1 = wr0;
  auto load = [&](int kt) {
    const int k0 = 32 * kt;
    if (xin) xr = __ldg(reinterpret_cast<const uint4 *>(xrow + k0));
    if (win0) wr0 = __ldg(reinterpret_cast<const float4 *>(wrow0 + k0));
    if (win1) wr1 = __ldg(reinterpret_cast<const float4 *>(wrow1 + k0));
  };
  if (kt0 < kt1) load(kt0);
  float acc[4][4] = {};
  for (int kt = kt0; kt < kt1; kt++) {
    const uint32_t xw[4] = {xr.x, xr.y, xr.z, xr.w};
#pragma unroll
    for (int j = 0; j < 4; j++) {
      Xs[kx + 2 * j][rx] = __uint_as_float(xw[j] << 16);
      Xs[kx + 2 * j + 1][rx] = __uint_as_float(xw[j] & 0xFFFF0000u);
    }
    Ws[kw][rw] = wr0.x; Ws[kw + 1][rw] = wr0.y; Ws[kw + 2][rw] = wr0.z; Ws[kw + 3][rw] = wr0.w;
    Ws[kw][rw + 32] = wr1.x; Ws[kw + 1][rw + 32] = wr1.y; Ws[kw + 2][rw + 32] = wr1.z; Ws[kw + 3][rw + 32] = wr1.w;
    __syncthreads();
    if (kt + 1 < kt1) load(kt + 1);
#pragma unroll 8
    for (int c = 0; c < 32; c++) {
      const float4 x4 = *reinterpret_cast<const float4 *>(&Xs[c][ty * 4]);
      const float4 w4 = *reinterpret_cast<const float4 *>(&Ws[c][tx * 4]);
      const float xv[4] = {x4.x, x4.y, x4.z, x4.w}, wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) acc[i][j] = fmaf(xv[i], wv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float *part = a.logits + (size_t)blockIdx.z * a.C * a.E;
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int t = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
      if (t < a.C && e < a.E) part[(size_t)t * a.E + e] = acc[i][j];
    }
}

// One CTA per token: logits = the partials summed in split order, plus the
// bias (written over partial 0), then the top-k of the row.
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(const RouteArgs a) {
  __shared__ SelectSmem tk;
  const int t = blockIdx.x;
  float *lg = a.logits + (size_t)t * a.E;
  for (int e = threadIdx.x; e < a.E; e += blockDim.x) {
    float v = lg[e];
    for (int z = 1; z < kRouteSplits; z++) v += lg[(size_t)z * a.C * a.E + e];
    lg[e] = v + (a.bias ? a.bias[e] : 0.f);
  }
  __syncthreads();
  cta_select_topk<kRouteWarps * 32>(lg, a.E, a.k, a.ids + (size_t)t * a.k, a.weights + (size_t)t * a.k, tk);
}

static size_t fused_smem(int ct, int H) { (void)ct; (void)H; return kRouteSmemBytes; }

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

void route_wait_policy(uint32_t config_flags, RouteArgs *a) {
  const bool stall = (config_flags & MOE_CONFIG_TEST_ROUTER_STALL) != 0;
  a->stall_tx = stall ? 16u : 0u;
  a->wait_ns = stall ? 20000000ull : 2000000000ull;   // 20 ms under the test hook, else ~2 s
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
  dim3 g1((a.E + 63) / 64, (a.C + 63) / 64, kRouteSplits);
  route_logits_tiled_kernel<<<g1, 256, 0, stream>>>(a);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  route_topk_kernel<<<a.C, kRouteWarps * 32, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
