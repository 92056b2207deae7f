// kernels.h -- argument blocks and launchers of the MoE kernels (host side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

struct PackArgs {
  const uint8_t *gate_codes, *gate_scales, *up_codes, *up_scales, *down_codes, *down_scales;
  const float *gate_g, *gate_a, *up_g, *up_a, *down_g, *down_a;
  uint8_t *packed;
  int32_t *status;   // in the packed trailer
  int E, H, I, tpr_gu, tpr_dn;
  size_t gu_pair_bytes, dn_pair_bytes, dn_region_off, expert_bytes, scalars_off;
};
cudaError_t launch_pack(const PackArgs &a, int num_sms, cudaStream_t stream);

struct RouteArgs {
  const uint16_t *x;     // bf16 bits [C][H]
  const float *w_router; // [E][H]
  const float *bias;     // [E] or null
  int32_t *ids;          // [C][k]
  float *weights;        // [C][k]
  float *logits;         // workspace [C][E]
  uint32_t *ticket;      // workspace counter (0 between calls)
  int C, E, H, k;
};
// Router GEMV fused with top-k (C <= 8): grid is fixed per layer.
cudaError_t launch_route_fused(const RouteArgs &a, int grid, cudaStream_t stream);
// Router for larger C: tiled logits kernel, then one warp per token for top-k.
cudaError_t launch_route_batched(const RouteArgs &a, cudaStream_t stream);
// Opt-in shared memory for the fused router; call once per device.
cudaError_t route_setup(int H);

struct GemvArgs {
  const uint8_t *packed;
  const float *scalars;      // packed + scalars_off: float [E][6]
  const uint16_t *x;         // bf16 bits [C][H]
  const int32_t *ids;        // [C][k]
  const float *weights;      // [C][k]
  float *hbuf;               // [C*k][I]
  float *ypair;              // [C*k][H]
  float *y;                  // [C][H]
  int32_t *flags;
  uint32_t *chunk_cnt;
  int C, k, E, H, I;
  size_t expert_bytes;
  size_t region_off;         // 0 (gate/up) or the down region offset
  int pair_bytes;            // bytes of one pair row of this region
  int rows;                  // pair rows per expert: I (gate/up) or H/2 (down)
};
// mode 0: gate/up + SwiGLU -> hbuf; mode 1: down -> ypair -> combine -> y.
// nt: tokens compiled for (1, 2, 4 or 8) >= C.
cudaError_t launch_expert_gemv(int mode, int nt, const GemvArgs &a, int threads, int grid,
                               bool pdl, cudaStream_t stream);
// CTAs per SM the gemv kernel reaches with `threads` threads.
int gemv_occupancy(int mode, int nt, int threads);

}  // namespace moe
