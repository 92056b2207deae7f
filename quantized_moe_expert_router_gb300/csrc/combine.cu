// combine.cu -- the routed sum of one token group:
//   y[t] = sum over token t's selected experts, in ascending expert id, of
//          ypair[(t, slot)]  (= w[t][slot] * D_e silu(G_e x_t) * (U_e x_t))
// "SparkInfer-K3", section "How the TP module works": each token's output is
// the sum of its selected experts' weighted outputs (the router weight is
// already folded into ypair by the expert kernels).
//
// Slots follow the expert kernels' rules: an id outside [0, E) is skipped,
// and an id repeated inside a token counts once, with its lowest slot.  The
// fixed summation order makes y bitwise reproducible without float atomics.
// Every CTA first orders the slots of all tokens in shared memory (one warp
// per token), then threads sum float4 columns of ypair.
#include "moe_internal.cuh"
#include "kernels.h"

namespace moe {

constexpr int kCombineBatch = 16;
constexpr int kCombineThreads = 64;

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineArgs a) {
  __shared__ int order[kGemvTokens][kMaxTopK];
  __shared__ int cnt[kGemvTokens];
  __shared__ int s_live;                        // 0: instruction warm-up pass, 1: the sums
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int t = warp; t < a.C; t += kCombineThreads / 32) {
    const int e = lane < a.k ? a.ids[(size_t)t * a.k + lane] : -1;
    // valid: in range, and not a repeat of a lower slot's id
    bool valid = lane < a.k && (unsigned)e < (unsigned)a.E;
    for (int j = 0; j < a.k; j++) {
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      if (j < lane && ej == e) valid = false;
    }
    // rank among the valid slots by ascending expert id (ids are distinct there)
    int rank = 0;
    for (int j = 0; j < a.k; j++) {
      const int ej = __shfl_sync(0xFFFFFFFFu, e, j);
      const int vj = __shfl_sync(0xFFFFFFFFu, (int)valid, j);
      rank += (vj && ej < e);
    }
    const unsigned vm = __ballot_sync(0xFFFFFFFFu, valid);
    if (valid) order[t][rank] = t * a.k + lane;
    if (lane == 0) cnt[t] = __popc(vm);
  }
  // The sums run twice through the same instructions: first before the wait
  // with every memory access predicated off (the down grid is still running;
  // this only brings the code into the SM's instruction cache), then for
  // real.  The pass flag is read from shared memory in the loop, so the
  // compiler cannot split the loop into two copies.
  if (tid == 0) s_live = 0;
  __syncthreads();
  const int H4 = a.H / 4;
#pragma unroll 1
  for (int pass = 0; pass < 2; pass++) {
    if (pass == 1) {
      __syncthreads();                          // every thread is done with the warm-up pass
      pdl_wait();                               // ypair comes from the down kernel
      if (blockIdx.x == 0)                      // the down kernel has read every |h| maximum
        for (int i = tid; i < a.C * a.k; i += blockDim.x) a.hamax[i] = 0u;
      if (tid == 0) s_live = 1;
      __syncthreads();
    }
    for (int it = blockIdx.x * blockDim.x + tid; it < a.C * H4; it += gridDim.x * blockDim.x) {
      const bool live = *reinterpret_cast<volatile int *>(&s_live) != 0;
      const int t = it / H4, c4 = it - t * H4;
      const int n = cnt[t];
      float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
      // all loads of a batch in flight together, then summed in slot order
      for (int j0 = 0; j0 < n; j0 += kCombineBatch) {
        float4 v[kCombineBatch];
#pragma unroll
        for (int j = 0; j < kCombineBatch; j++)
          v[j] = live && j0 + j < n
                     ? __ldcg(reinterpret_cast<const float4 *>(a.ypair + (size_t)order[t][j0 + j] * a.H) + c4)
                     : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kCombineBatch; j++) {
          if (j0 + j < n) {
            s.x += v[j].x; s.y += v[j].y; s.z += v[j].z; s.w += v[j].w;
          }
        }
      }
      if (live) reinterpret_cast<float4 *>(a.y + (size_t)t * a.H)[c4] = s;
    }
  }
}

cudaError_t launch_combine(const CombineArgs &a, int num_sms, bool pdl, cudaStream_t stream) {
  const int items = a.C * (a.H / 4);
  int grid = (items + kCombineThreads - 1) / kCombineThreads;
  if (grid > num_sms) grid = num_sms;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCombineThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, a);
}

}  // namespace moe
