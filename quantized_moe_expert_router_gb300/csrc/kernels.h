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
  int E, H, I, w_gu, w_dn;
  int fmt;           // kFmtNvfp4: e4m3 scales per 16 elements; kFmtMxfp4: e8m0 per 32
  size_t dn_region_off, expert_bytes, scalars_off;
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
  int32_t *flags;        // workspace flag word (MOE_FLAG_TIMEOUT)
  int C, E, H, k;
  uint32_t stall_tx;     // test hook: extra bytes every CTA waits for and no copy delivers (0 = off)
  unsigned long long wait_ns;   // limit of a bounded wait
};
// Router GEMV fused with top-k (C <= 8): grid is fixed per layer.
cudaError_t launch_route_fused(const RouteArgs &a, int grid, cudaStream_t stream);
// Router for larger C: tiled logits kernel, then one warp per token for top-k.
cudaError_t launch_route_batched(const RouteArgs &a, cudaStream_t stream);
// Opt-in shared memory for the fused router (once per device; idempotent).
cudaError_t route_setup();
// Wait limit and test stall of the router from the layer's config flags.
void route_wait_policy(uint32_t config_flags, RouteArgs *a);

struct GemvArgs {
  const uint8_t *packed;
  const float *scalars;      // packed + scalars_off: float [E][6]
  const uint16_t *x;         // bf16 bits [C][H]
  const int32_t *ids;        // [C][k]
  const float *weights;      // [C][k]
  float *hbuf;               // [C*k][I], 16-element blocks in operand order
  uint32_t *hamax;           // [C*k] max |h| (float bits), zero outside a call
  float *ypair;              // [C*k][H]
  float *y;                  // [C][H]
  int32_t *flags;
  int C, k, E, H, I;
  size_t expert_bytes;
  size_t region_off;         // 0 (gate/up) or the down region offset
  int tiles;                 // stage units per expert: I/8 tiles (gate/up) or H/32 tile pairs (down)
  int tile_bytes;            // bytes of one stage unit: one tile (gate/up) or two (down) of slices * kTileSliceBytes
  int slices;                // 512-element K-slices per tile (padded K / 512); 2 consumer warps each
  int stages;                // shared-memory ring stages
  int stage_bytes;           // bytes of one ring stage (one stage unit)
  int red_stage_f4;          // reduction slots of one stage, in float4
  int smem_bytes;            // dynamic shared memory: ring + reduction slots
  int fmt;                   // kFmtNvfp4 or kFmtMxfp4 (scale unit layout and decode)
  int w4a4;                  // W4A4: x and h quantized to NVFP4 in the fragments, router weight after down
};
// Ring geometry and dynamic shared memory of one kernel.
void gemv_geometry(int stage_bytes, int red_stage_bytes, int *stages, int *smem_bytes);
// Opt-in shared memory of the expert kernels (once per device; idempotent).
cudaError_t gemv_setup();
// mode 0: gate/up + SwiGLU -> hbuf (one tile per stage); mode 2: the same, two
// tiles per stage (groups of at most 2 tokens); mode 1: down -> ypair.
cudaError_t launch_expert_gemv(int mode, const GemvArgs &a, int grid, bool pdl, cudaStream_t stream);

struct CombineArgs {
  const int32_t *ids;        // [C][k]
  const float *ypair;        // [C*k][H]
  uint32_t *hamax;           // [C*k], reset to zero once the down kernel is done
  float *y;                  // [C][H]
  int C, k, E, H;
};
// y[t] = sum of ypair over token t's valid slots in ascending expert id order.
cudaError_t launch_combine(const CombineArgs &a, int num_sms, bool pdl, cudaStream_t stream);

struct GroupArgs {
  const uint16_t *x;         // bf16 bits [C][H] of this pass
  const int32_t *ids;        // [C][k]
  const float *weights;      // [C][k]
  const uint8_t *packed;
  const float *scalars;      // packed + scalars_off: float [E][6]
  int *gd;                   // expert-major dispatch: n, expert [E], off [E + 1], pairs
  float *xinv;               // [C]             2^-s of each token's f16 scale
  uint16_t *xg;              // f16 [Hp/8][C*k][8]  x rows of the dispatched pairs, pair order
  float *hbuf;               // [C*k][I]        h per pair
  uint16_t *hg;              // f16 [Ip/8][2*C*k][8] hi / lo rows of h, pair order
  float *hinv;               // [C*k]           2^-s of each pair's h scale
  float *ypair;              // [C*k][H]
  float *y;                  // [C][H]
  int32_t *flags;
  int C, k, E, H, I, Hp, Ip;
  size_t expert_bytes;
  int w4a4;                  // W4A4 numerics: xg and hg hold NVFP4-quantized values, one hg row per pair
};
// Opt-in shared memory of the grouped kernels (once per device; idempotent).
cudaError_t group_setup();
size_t group_dispatch_smem(int E);
// The routed experts of one pass of up to kGroupTokens tokens, expert-major:
// dispatch, x rows, gate/up, h rows, down, combine.
cudaError_t launch_group_forward(GroupArgs a, int num_sms, int w_gu, int w_dn, size_t gu_tile_bytes,
                                 size_t dn_tile_bytes, size_t dn_region_off, cudaStream_t stream,
                                 cudaEvent_t after_gate_up);

// ------------------------------------------------ around the routed sum (dense.cu)
struct PackDenseArgs {
  const uint8_t *codesA, *scalesA;   // mode 0: the matrix [M][K]; mode 1: the gate matrix [M][K]
  const uint8_t *codesB, *scalesB;   // mode 1: the up matrix [M][K]
  uint8_t *dst;                      // packed tiles of the destination matrix
  int32_t *status;                   // set to 1 on a NaN scale byte
  int M, K, mode, fmt;               // mode 0: pair rows (2p, 2p+1); mode 1: (gate p, up p)
  int Wsrc;                          // 512-element K-slices of the source rows
  int W;                             // slices of a destination tile (its stride)
  int tile0, wd0;                    // first destination tile and slice
};
cudaError_t launch_pack_dense(const PackDenseArgs &a, int num_sms, cudaStream_t stream);

struct DenseArgs {
  const uint8_t *w;          // packed tiles of the matrix
  const void *x;             // input vectors [C][K]: bf16 bits (xf32 = 0) or fp32
  float *part;               // workspace: [tiles * W units][passes][32 lanes] float4
  int xf32, C, K, W, tiles, fmt;
  int w0, w1;                // slices of this launch (the B fragments of their K range fit shared memory)
  size_t tile_bytes;
};
// A range of tiles of a dense GEMV and what its finisher writes:
//   mode 0: plain pair rows (2p, 2p + 1) -> columns col0 + 2p, +1 (fp32
//           written or added, or bf16); mode 1: SwiGLU of a (gate p, up p)
//   pair -> column col0 + p (fp32).  p counts from the segment's first tile.
constexpr int kMaxDenseSegs = 5;
struct DenseSeg {
  int tile0, tile1, mode, accumulate, out_ld, col0;
  const float *ga, *gb;      // device tensor scales (null: 1)
  float *out_f32;
  uint16_t *out_bf16;
};
struct DenseFinishArgs {
  const float *part;
  const float *slice_scale;  // device [W] scale of each K-slice's partial, or null
  DenseSeg seg[kMaxDenseSegs];
  int nseg, xf32, C, W, tiles;
};
// Workspace bytes of a GEMV's partials and shared memory of its B fragments.
inline size_t dense_partial_bytes(int tiles, int W, int C, bool xf32) {
  return (size_t)tiles * W * (xf32 ? (C + 3) / 4 : 1) * 32 * 16;
}
cudaError_t launch_dense_gemv(const DenseArgs &a, const DenseFinishArgs &f, int num_sms, cudaStream_t stream);
cudaError_t launch_rms_norm(const float *y, const float *gamma, float eps, int C, int n, float *out, int out_ld,
                            cudaStream_t stream);

}  // namespace moe
