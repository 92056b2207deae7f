// moe_api.cu -- the extern "C" entry points declared in include/moe.h.
//
// Host-side only: argument validation, packed/workspace layout arithmetic and
// the launch sequence.  Every step of the computation runs in the kernels of
// pack.cu, route.cu and expert_gemv.cu; there is no host or CPU fallback.
#include <stdlib.h>
#include <string.h>

#include <new>

#include "kernels.h"
#include "moe_internal.cuh"

using moe::align_up;

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = false;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
  }
  ~DeviceGuard() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

int gemv_grid(const moe_layer &L, long long max_tiles) {
  long long g = L.num_sms;                 // one CTA per SM (the ring uses most of shared memory)
  if (g > max_tiles) g = max_tiles;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

extern "C" {

const char *moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MOE_ERR_INVALID_VALUE: return "invalid value (NaN e4m3 scale)";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_OUT_OF_MEMORY: return "out of memory";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BAD_EXPERT_ID: return "bad expert id";
  }
  return "unknown status";
}

moe_status moe_layer_create(const moe_config *cfg, int device, moe_layer_t *out) {
  if (!cfg || !out) return MOE_ERR_INVALID_ARG;
  const moe_config c = *cfg;
  if ((c.flags & ~(uint32_t)(MOE_CONFIG_TEST_ROUTER_STALL | MOE_CONFIG_MXFP4 | MOE_CONFIG_GROUPED_ABOVE_8 |
                             MOE_CONFIG_W4A4)) != 0 ||
      c.max_tokens < 1)
    return MOE_ERR_INVALID_ARG;
  if ((c.flags & MOE_CONFIG_MXFP4) && (c.flags & MOE_CONFIG_W4A4)) return MOE_ERR_INVALID_ARG;
  if (c.num_experts < 1 || c.num_experts > moe::kMaxExperts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.top_k < 1 || c.top_k > moe::kMaxTopK || c.top_k > c.num_experts) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.hidden < 64 || c.hidden % 64 || c.hidden > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.intermediate < 64 || c.intermediate % 64 || c.intermediate > 4096) return MOE_ERR_UNSUPPORTED_SHAPE;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(device);
  if (!guard.ok) return MOE_ERR_CUDA;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return MOE_ERR_CUDA;

  moe_layer *L = new (std::nothrow) moe_layer();
  if (!L) return MOE_ERR_OUT_OF_MEMORY;
  L->cfg = c;
  L->fmt = (c.flags & MOE_CONFIG_MXFP4) ? moe::kFmtMxfp4 : moe::kFmtNvfp4;
  L->w4a4 = (c.flags & MOE_CONFIG_W4A4) ? 1 : 0;
  L->device = device;
  L->num_sms = sms;
  L->Hp = (int)align_up(c.hidden, moe::kKAlign);
  L->Ip = (int)align_up(c.intermediate, moe::kKAlign);
  L->w_gu = L->Hp / moe::kKAlign;
  L->w_dn = L->Ip / moe::kKAlign;
  const size_t slice_bytes = L->fmt == moe::kFmtMxfp4 ? moe::kTileSliceBytesMx : moe::kTileSliceBytes;
  L->gu_tile_bytes = (size_t)L->w_gu * slice_bytes;
  L->dn_tile_bytes = (size_t)L->w_dn * slice_bytes;
  L->dn_region_off = (size_t)(c.intermediate / 8) * L->gu_tile_bytes;
  L->expert_bytes = L->dn_region_off + (size_t)(c.hidden / 16) * L->dn_tile_bytes;
  L->scalars_off = (size_t)c.num_experts * L->expert_bytes;
  L->trailer_off = align_up(L->scalars_off + (size_t)c.num_experts * 6 * sizeof(float), 16);
  L->packed_bytes = L->trailer_off + 16;
  L->stage_events_on = 0;
  // below the crossover the decode kernels (groups of 8 tokens, each expert
  // read once per group) beat the grouped GEMM, whose MMAs are mostly padding
  // when an expert has one or two tokens: measured with uniform routing at
  // 896 experts, top-16, the two paths meet between 24 and 32 tokens
  L->grouped_min_tokens = (c.flags & MOE_CONFIG_GROUPED_ABOVE_8) ? moe::kGemvTokens + 1 : moe::kGroupedMinTokens;
  if (moe::gemv_setup() != cudaSuccess) {
    delete L;
    return MOE_ERR_CUDA;
  }
  if (moe::route_setup() != cudaSuccess || moe::group_setup() != cudaSuccess) {
    delete L;
    return MOE_ERR_CUDA;
  }
  *out = L;
  return MOE_OK;
}

moe_status moe_layer_destroy(moe_layer_t L) {
  delete L;
  return MOE_OK;
}

moe_status moe_packed_bytes(moe_layer_t L, size_t *bytes) {
  if (!L || !bytes) return MOE_ERR_INVALID_ARG;
  *bytes = L->packed_bytes;
  return MOE_OK;
}

moe_status moe_workspace_bytes(moe_layer_t L, int num_tokens, size_t *bytes) {
  if (!L || !bytes || num_tokens < 1) return MOE_ERR_INVALID_ARG;
  *bytes = moe::ws_layout(*L, num_tokens).total;
  return MOE_OK;
}

moe_status moe_pack_weights(moe_layer_t L, const moe_canonical_weights *cw, void *packed,
                            cudaStream_t stream) {
  if (!L || !cw || !packed) return MOE_ERR_INVALID_ARG;
  const moe_fp4_tensor *ts[3] = {&cw->gate, &cw->up, &cw->down};
  for (const moe_fp4_tensor *t : ts) {
    if (!t->codes || !t->scales || !t->global_scale || !t->input_scale) return MOE_ERR_INVALID_ARG;
    if (!aligned16(t->codes)) return MOE_ERR_INVALID_ARG;
  }
  if (!aligned16(packed)) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  uint8_t *pk = static_cast<uint8_t *>(packed);
  int32_t *status = reinterpret_cast<int32_t *>(pk + L->trailer_off);
  cudaError_t err = cudaMemsetAsync(pk + L->trailer_off, 0, 16, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  moe::PackArgs a;
  a.gate_codes = cw->gate.codes; a.gate_scales = cw->gate.scales;
  a.up_codes = cw->up.codes; a.up_scales = cw->up.scales;
  a.down_codes = cw->down.codes; a.down_scales = cw->down.scales;
  a.gate_g = cw->gate.global_scale; a.gate_a = cw->gate.input_scale;
  a.up_g = cw->up.global_scale; a.up_a = cw->up.input_scale;
  a.down_g = cw->down.global_scale; a.down_a = cw->down.input_scale;
  a.packed = pk;
  a.status = status;
  a.E = L->cfg.num_experts; a.H = L->cfg.hidden; a.I = L->cfg.intermediate;
  a.w_gu = L->w_gu; a.w_dn = L->w_dn;
  a.fmt = L->fmt;
  a.dn_region_off = L->dn_region_off; a.expert_bytes = L->expert_bytes;
  a.scalars_off = L->scalars_off;
  err = moe::launch_pack(a, L->num_sms, stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  int32_t host_status = 0;
  err = cudaMemcpyAsync(&host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return host_status ? MOE_ERR_INVALID_VALUE : MOE_OK;
}

moe_status moe_route(moe_layer_t L, const uint16_t *x, int C, const float *w_router,
                     const float *bias, int32_t *ids, float *weights, void *ws,
                     size_t ws_bytes, cudaStream_t stream) {
  if (!L || !x || !w_router || !ids || !weights || !ws) return MOE_ERR_INVALID_ARG;
  if (C < 1 || C > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_router) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const moe::WsLayout wl = moe::ws_layout(*L, C);
  if (ws_bytes < wl.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DeviceGuard guard(L->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  uint8_t *w = static_cast<uint8_t *>(ws);
  moe::RouteArgs a;
  a.x = x; a.w_router = w_router; a.bias = bias; a.ids = ids; a.weights = weights;
  a.logits = reinterpret_cast<float *>(w + (C <= moe::kGemvTokens ? wl.logits : wl.glogits));
  a.ticket = &reinterpret_cast<moe::WsControl *>(w)->route_ticket;
  a.flags = &reinterpret_cast<moe::WsControl *>(w)->flags;
  a.C = C; a.E = L->cfg.num_experts; a.H = L->cfg.hidden; a.k = L->cfg.top_k;
  moe::route_wait_policy(L->cfg.flags, &a);
  cudaError_t err;
  if (C <= moe::kRouteFusedTokens) {
    const int grid = a.E < L->num_sms ? a.E : L->num_sms;   // router rows dealt round-robin
    err = moe::launch_route_fused(a, grid, stream);
  } else {
    err = moe::launch_route_batched(a, stream);
  }
  return cuda_status(err);
}

}  // extern "C"

namespace {

// moe_forward's work.  `after_router`: the fused router kernel was queued
// right before on `stream` (moe_route_forward), so the gate/up kernel may be
// launched as its programmatic dependent.  That kernel reads x before it
// waits for the preceding grid; x is then already visible, because the router
// (a normal launch) could only start once everything queued before it had
// finished.  A standalone call has no such guarantee for x written by the
// caller's last kernel, so there the gate/up kernel is a normal launch.
moe_status forward_impl(moe_layer_t L, const uint16_t *x, int C, const int32_t *ids, const float *weights,
                        const void *packed, float *y, void *ws, size_t ws_bytes, cudaStream_t stream,
                        bool after_router) {
  if (!L || !x || !ids || !weights || !packed || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (C < 1 || C > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(packed) || !aligned16(y) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  const moe::WsLayout wl = moe::ws_layout(*L, C);
  if (ws_bytes < wl.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  DeviceGuard guard(L->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  uint8_t *w = static_cast<uint8_t *>(ws);
  const uint8_t *pk = static_cast<const uint8_t *>(packed);
  const int H = L->cfg.hidden, I = L->cfg.intermediate, k = L->cfg.top_k;

  moe::GemvArgs a;
  a.packed = pk;
  a.scalars = reinterpret_cast<const float *>(pk + L->scalars_off);
  a.hbuf = reinterpret_cast<float *>(w + wl.hbuf);
  a.hamax = reinterpret_cast<uint32_t *>(w + wl.hamax);
  a.ypair = reinterpret_cast<float *>(w + wl.ypair);
  a.flags = &reinterpret_cast<moe::WsControl *>(w)->flags;
  a.k = k; a.E = L->cfg.num_experts; a.H = H; a.I = I;
  a.expert_bytes = L->expert_bytes;
  a.fmt = L->fmt;
  a.w4a4 = L->w4a4;

  cudaError_t err = cudaSuccess;
  if (L->stage_events_on) err = cudaEventRecord(L->stage_events[0], stream);
  // C >= grouped_min_tokens: the grouped tcgen05 path (NVFP4); MXFP4 layers
  // run every C on the decode kernels, in groups of 8
  if (C >= L->grouped_min_tokens && L->fmt == moe::kFmtNvfp4) {
    // expert-major passes of up to kGroupTokens tokens
    moe::GroupArgs g = {};
    g.packed = pk;
    g.scalars = a.scalars;
    g.gd = reinterpret_cast<int *>(w + wl.gd);
    g.xinv = reinterpret_cast<float *>(w + wl.xinv);
    g.xg = reinterpret_cast<uint16_t *>(w + wl.xg);
    g.hbuf = reinterpret_cast<float *>(w + wl.ghbuf);
    g.hg = reinterpret_cast<uint16_t *>(w + wl.hg);
    g.hinv = reinterpret_cast<float *>(w + wl.hinv);
    g.ypair = reinterpret_cast<float *>(w + wl.gypair);
    g.flags = a.flags;
    g.k = k; g.E = L->cfg.num_experts; g.H = H; g.I = I; g.Hp = L->Hp; g.Ip = L->Ip;
    g.expert_bytes = L->expert_bytes;
    g.w4a4 = L->w4a4;
    for (int t0 = 0; t0 < C && err == cudaSuccess; t0 += moe::kGroupTokens) {
      g.C = (C - t0) < moe::kGroupTokens ? (C - t0) : moe::kGroupTokens;
      g.x = x + (size_t)t0 * H;
      g.ids = ids + (size_t)t0 * k;
      g.weights = weights + (size_t)t0 * k;
      g.y = y + (size_t)t0 * H;
      err = moe::launch_group_forward(g, L->num_sms, L->w_gu, L->w_dn, L->gu_tile_bytes, L->dn_tile_bytes,
                                      L->dn_region_off, stream,
                                      (L->stage_events_on && t0 == 0) ? L->stage_events[1] : nullptr);
    }
    if (err == cudaSuccess && L->stage_events_on) err = cudaEventRecord(L->stage_events[2], stream);
    return cuda_status(err);
  }
  for (int t0 = 0; t0 < C && err == cudaSuccess; t0 += moe::kGemvTokens) {
    const int Cg = (C - t0) < moe::kGemvTokens ? (C - t0) : moe::kGemvTokens;
    a.C = Cg;
    a.x = x + (size_t)t0 * H;
    a.ids = ids + (size_t)t0 * k;
    a.weights = weights + (size_t)t0 * k;
    a.y = y + (size_t)t0 * H;
    const long long max_pairs = (long long)Cg * k;
    // gate/up + SwiGLU: two tiles per stage when the group has at most two
    // tokens (their partials fit small reduction slots), else one
    const int wq = 2 * L->w_gu;                // consumer warps
    const bool gu_pairs = Cg <= 2;
    a.region_off = 0;
    a.tiles = gu_pairs ? I / 16 : I / 8;       // I % 64 == 0
    a.tile_bytes = (gu_pairs ? 2 : 1) * (int)L->gu_tile_bytes;
    a.slices = L->w_gu;
    a.stage_bytes = a.tile_bytes;
    a.red_stage_f4 = gu_pairs ? 2 * wq * 8 : wq * 32;
    moe::gemv_geometry(a.stage_bytes, a.red_stage_f4 * 16, &a.stages, &a.smem_bytes);
    err = moe::launch_expert_gemv(gu_pairs ? 2 : 0, a, gemv_grid(*L, max_pairs * a.tiles), after_router && t0 == 0,
                                  stream);
    if (err != cudaSuccess) break;
    if (L->stage_events_on && t0 == 0) err = cudaEventRecord(L->stage_events[1], stream);
    if (err != cudaSuccess) break;
    // down: two tiles per stage, reduction slots for two passes of 4 token slots
    const int wd = 2 * L->w_dn;
    a.region_off = L->dn_region_off;
    a.tiles = H / 32;                          // H % 64 == 0
    a.tile_bytes = 2 * (int)L->dn_tile_bytes;
    a.slices = L->w_dn;
    a.stage_bytes = a.tile_bytes;
    a.red_stage_f4 = 2 * wd * 32;
    moe::gemv_geometry(a.stage_bytes, a.red_stage_f4 * 16, &a.stages, &a.smem_bytes);
    err = moe::launch_expert_gemv(1, a, gemv_grid(*L, max_pairs * a.tiles), true, stream);
    if (err != cudaSuccess) break;
    // weighted sum over each token's experts, ascending expert id
    moe::CombineArgs cb;
    cb.ids = a.ids; cb.ypair = a.ypair; cb.y = a.y; cb.hamax = a.hamax;
    cb.C = Cg; cb.k = k; cb.E = a.E; cb.H = H;
    err = moe::launch_combine(cb, L->num_sms, true, stream);
  }
  if (err == cudaSuccess && L->stage_events_on) err = cudaEventRecord(L->stage_events[2], stream);
  return cuda_status(err);
}

}  // namespace

extern "C" {

moe_status moe_forward(moe_layer_t L, const uint16_t *x, int C, const int32_t *ids, const float *weights,
                       const void *packed, float *y, void *ws, size_t ws_bytes, cudaStream_t stream) {
  return forward_impl(L, x, C, ids, weights, packed, y, ws, ws_bytes, stream, false);
}

moe_status moe_route_forward(moe_layer_t L, const uint16_t *x, int C, const float *w_router,
                             const float *bias, const void *packed, int32_t *ids, float *weights, float *y,
                             void *ws, size_t ws_bytes, cudaStream_t stream) {
  if (!L || !x || !w_router || !packed || !ids || !weights || !y || !ws) return MOE_ERR_INVALID_ARG;
  if (C < 1 || C > L->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(packed) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
  const moe_status st = moe_route(L, x, C, w_router, bias, ids, weights, ws, ws_bytes, stream);
  if (st != MOE_OK) return st;
  return forward_impl(L, x, C, ids, weights, packed, y, ws, ws_bytes, stream,
                      C <= moe::kRouteFusedTokens && !L->stage_events_on);
}

moe_status moe_get_device_status(moe_layer_t L, void *ws, cudaStream_t stream, int32_t *flags) {
  if (!L || !ws || !flags) return MOE_ERR_INVALID_ARG;
  DeviceGuard guard(L->device);
  if (!guard.ok) return MOE_ERR_CUDA;
  moe::WsControl *ctl = static_cast<moe::WsControl *>(ws);
  cudaError_t err = cudaStreamSynchronize(stream);
  if (err == cudaSuccess) err = cudaMemcpy(flags, &ctl->flags, sizeof(int32_t), cudaMemcpyDeviceToHost);
  // flags and router ticket (and the reserved word) back to zero: a router
  // grid that stopped early leaves the workspace as good as new
  static_assert(offsetof(moe::WsControl, reserved) == 8, "control words 0..11");
  if (err == cudaSuccess) err = cudaMemsetAsync(ctl, 0, 12, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  return cuda_status(err);
}

moe_status moe_set_stage_events(moe_layer_t L, cudaEvent_t *events, int n_events) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (!events) {
    L->stage_events_on = 0;
    return MOE_OK;
  }
  if (n_events != 3) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i < 3; i++) L->stage_events[i] = events[i];
  L->stage_events_on = 1;
  return MOE_OK;
}

}  // extern "C"
