// topk.cuh -- top-k of one token's router logits by one CTA, with the
// renormalised softmax weights.
//
// Definition ("SparkInfer-K3", section "How the TP module works": one
// replicated router, every rank agrees on the same top-16): keep the k
// largest logits, equal logits -> lower expert index first, and weight them
// with w_i = exp(l_i - l_max) / sum over kept exp(l_j - l_max) (a softmax
// over all experts renormalised over the kept ones; the full denominator
// cancels).  ids are written in ascending expert order.
//
// Method: a threshold, then exact ranks among the few keys above it.  Keys
// are order-preserving 32-bit images of the logits, packed with the inverted
// expert id into one 64-bit value so that "precedes" is a single compare
// (larger logit first, then lower id).  Each thread holds a contiguous run of
// expert ids.  (1) The warps whose lanes all hold experts are cut into groups
// of lanes, enough groups to have at least k; the group maxima are distinct
// keys, so T, the k-th largest group maximum, has at least k keys at or above
// it.  (2) The keys >= T are compacted into shared memory in ascending id
// order (one CTA scan).  (3) Each candidate's rank, the number of candidates
// that precede it, is counted by a team of 4 lanes; ranks < k are kept, and
// their output slots in ascending id order come from a bit mask of the kept
// candidates.  With logits of distinct values there are about 2k candidates;
// ties only make the candidate list (and the rank loop) longer.  The
// selection is latency-bound: every step is a few warp-wide operations
// between CTA barriers.
//
// A token with a NaN among its logits selects nothing: ids -1 (absent
// slots) and weights 0.  The fused router marks the rows of a block whose
// copies did not arrive that way.
#pragma once

#include "moe_internal.cuh"

namespace moe {

// Order-preserving map fp32 -> uint32 (larger float -> larger key); -0 is
// folded onto +0.
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) == 0) u = 0;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
  return __uint_as_float(u);
}

struct SelectSmem {
  unsigned long long cand[kMaxExperts];   // (key << 32) | (1023 - id), ascending id order
  uint32_t kept[kMaxExperts / 32];        // bit c: candidate c has rank < k
  uint32_t wcnt[32];                      // per-warp candidate counts
  uint32_t gmax[64];                      // group maxima
  uint32_t wmax[32];                      // per-warp largest key
  uint32_t thr;                           // T
  float exs[32];                          // exp(l - l_max) of the kept, by output slot
};

__device__ __forceinline__ unsigned long long pack_key(uint32_t key, int e) {
  return ((unsigned long long)key << 32) | (uint32_t)(kMaxExperts - 1 - e);
}

// Top-k (1 <= k <= 32, k <= E <= 1024) of the E logits at lg, written to
// ids_out[k] (ascending expert id) and w_out[k].  Threads [0, NT) hold the
// keys (NT = 128 or 256, kMaxExperts / NT contiguous experts each); every
// thread of the CTA must call it (blockDim.x >= NT, a multiple of 32).  The
// logits are read with ld.global.cg, so values written by other CTAs before a
// grid-wide barrier are seen.
template <int NT>
__device__ __forceinline__ void cta_select_topk(const float *lg, int E, int k, int32_t *ids_out, float *w_out,
                                                SelectSmem &s) {
  static_assert(NT == 128 || NT == 256, "128 or 256 key threads");
  constexpr unsigned kAll = 0xFFFFFFFFu;
  constexpr int V = kMaxExperts / NT, NW = NT / 32;
  constexpr int kFast = 64;                      // candidate count of the unrolled paths
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int e0 = tid * V;
  const bool part = tid < NT;
  uint32_t key[V];
  uint32_t m = 0;
  bool nan_seen = false;
#pragma unroll
  for (int v = 0; v < V; v++) {
    const float l = (part && e0 + v < E) ? __ldcg(lg + e0 + v) : 0.f;
    nan_seen |= l != l;
    key[v] = (part && e0 + v < E) ? order_key(l) : 0u;
    m = max(m, key[v]);
  }
  for (int i = tid; i < kMaxExperts / 32; i += blockDim.x) s.kept[i] = 0u;
  // (1) group maxima of the warps whose lanes all hold experts (E / (32 V)
  // counts only such warps), 2^lg_gpw groups per warp: the fewest that give
  // k groups, so at most max(2k - 1, NW) <= 64 groups
  const int nfull = min(E / (32 * V), NW);
  int lg_gpw = 0;
  while (lg_gpw < 5 && (nfull << lg_gpw) < k) lg_gpw++;
  const int lg_g = 5 - lg_gpw;                   // lanes per group = 1 << lg_g
  const int ngroups = nfull << lg_gpw;
  uint32_t gm = m;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1)
    if (o < (1 << lg_g)) gm = max(gm, __shfl_xor_sync(kAll, gm, o));
  if (warp < nfull && (lane & ((1 << lg_g) - 1)) == 0) s.gmax[(warp << lg_gpw) + (lane >> lg_g)] = gm;
  const uint32_t wm = __reduce_max_sync(kAll, m);
  if (lane == 0) s.wmax[warp] = wm;
  if (__syncthreads_or(nan_seen)) {
    if (tid < k) {
      ids_out[tid] = -1;
      w_out[tid] = 0.f;
    }
    __syncthreads();                             // s is reused by the next call
    return;
  }
  // T = k-th largest group maximum (with multiplicity): the value v with
  // #(> v) < k <= #(>= v), found by warp 0 (lane l holds groups l and l + 32
  // and counts against all groups by shuffles).  T = 0 when there are fewer
  // than k groups (every key is then a candidate).
  if (warp == 0) {
    uint32_t t = 0u;
    if (ngroups >= k) {
      const uint32_t g0 = lane < ngroups ? s.gmax[lane] : 0u;
      const uint32_t g1 = lane + 32 < ngroups ? s.gmax[lane + 32] : 0u;
      uint32_t gt0 = 0, ge0 = 0, gt1 = 0, ge1 = 0;
#pragma unroll
      for (int i = 0; i < 32; i++) {
        const uint32_t x = __shfl_sync(kAll, g0, i);
        const bool in = i < ngroups;
        gt0 += in && x > g0; ge0 += in && x >= g0; gt1 += in && x > g1; ge1 += in && x >= g1;
      }
      if (ngroups > 32) {
#pragma unroll
        for (int i = 0; i < 32; i++) {
          const uint32_t x = __shfl_sync(kAll, g1, i);
          const bool in = i + 32 < ngroups;
          gt0 += in && x > g0; ge0 += in && x >= g0; gt1 += in && x > g1; ge1 += in && x >= g1;
        }
      }
      const bool hit0 = lane < ngroups && gt0 < (uint32_t)k && ge0 >= (uint32_t)k;
      const bool hit1 = lane + 32 < ngroups && gt1 < (uint32_t)k && ge1 >= (uint32_t)k;
      const unsigned b0 = __ballot_sync(kAll, hit0), b1 = __ballot_sync(kAll, hit1);
      t = b0 ? __shfl_sync(kAll, g0, __ffs(b0) - 1) : __shfl_sync(kAll, g1, __ffs(b1) - 1);
    }
    if (lane == 0) s.thr = t;
  }
  __syncthreads();
  const uint32_t T = s.thr;
  // (2) candidates, keys >= T, in ascending id order
  uint32_t nc = 0;
#pragma unroll
  for (int v = 0; v < V; v++) nc += (part && e0 + v < E && key[v] >= T) ? 1u : 0u;
  uint32_t incl = nc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kAll, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31 && warp < NW) s.wcnt[warp] = incl;
  __syncthreads();
  const uint32_t wc = lane < NW ? s.wcnt[lane] : 0u;
  uint32_t off = __reduce_add_sync(kAll, lane < warp ? wc : 0u) + incl - nc;
  const uint32_t ncand = __reduce_add_sync(kAll, wc);
  const uint32_t kmax = __reduce_max_sync(kAll, lane < NW ? s.wmax[lane] : 0u);
#pragma unroll
  for (int v = 0; v < V; v++)
    if (part && e0 + v < E && key[v] >= T) s.cand[off++] = pack_key(key[v], e0 + v);
  __syncthreads();
  // (3) rank = number of candidates preceding this one; keep ranks < k
  const int nteams = (int)(blockDim.x >> 2);
  if (ncand <= (uint32_t)kFast && (int)ncand <= nteams) {
    // one candidate per team of 4 lanes; lane j of a team compares candidates
    // j, j + 4, ... (all its loads issued together)
    const int c = tid >> 2, tl4 = tid & 3;
    const unsigned long long me = c < (int)ncand ? s.cand[c] : ~0ull;
    unsigned long long v[kFast / 4];
#pragma unroll
    for (int i = 0; i < kFast / 4; i++) v[i] = s.cand[4 * i + tl4];
    uint32_t rank = 0;
#pragma unroll
    for (int i = 0; i < kFast / 4; i++) rank += (4 * i + tl4 < (int)ncand && v[i] > me) ? 1u : 0u;
    rank += __shfl_xor_sync(kAll, rank, 1);
    rank += __shfl_xor_sync(kAll, rank, 2);
    if (c < (int)ncand && tl4 == 0 && rank < (uint32_t)k) atomicOr(&s.kept[c >> 5], 1u << (c & 31));
  } else {
    for (uint32_t c = tid; c < ncand; c += blockDim.x) {
      const unsigned long long me = s.cand[c];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < ncand; j++) rank += (s.cand[j] > me) ? 1u : 0u;
      if (rank < (uint32_t)k) atomicOr(&s.kept[c >> 5], 1u << (c & 31));
    }
  }
  __syncthreads();
  // (4) output by warp 0: lane l takes candidates l, l + 32, ...; slot = kept
  // candidates before it (ascending id).  The denominator is summed over the
  // slots by a fixed shuffle tree, so the weights do not depend on how the
  // candidates were found (bitwise identical in every CTA and for any NT).
  if (warp == 0) {
    const float lmax = key_value(kmax);
    const int nwords = (int)((ncand + 31) >> 5);
    uint32_t before = 0;
    for (int w = 0; w < nwords; w++) {
      const uint32_t bits = s.kept[w];
      if ((bits >> lane) & 1u) {
        const unsigned long long me = s.cand[32 * w + lane];
        const uint32_t slot = before + __popc(bits & ((1u << lane) - 1u));
        ids_out[slot] = kMaxExperts - 1 - (int)(uint32_t)(me & 0xFFFFFFFFull);
        s.exs[slot] = expf(key_value((uint32_t)(me >> 32)) - lmax);
      }
      before += __popc(bits);
    }
    __syncwarp();
    const float ex = lane < k ? s.exs[lane] : 0.f;
    float denom = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) denom += __shfl_xor_sync(kAll, denom, o);
    if (lane < k) w_out[lane] = ex / denom;
  }
  __syncthreads();                               // s is reused by the next call
}

}  // namespace moe
