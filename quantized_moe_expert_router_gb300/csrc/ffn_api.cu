// ffn_api.cu -- the extern "C" entry points of the FFN around the routed sum
// (moe_ffn_* in include/moe.h): host-side layout arithmetic, argument
// checks and the launch sequence of FfnPartial (routed_down, then the routed
// layer) and FfnFinish (routed_norm, routed_up, shared experts) as
// "SparkInfer-K3" splits them (section "How the TP module works").  Every
// step of the computation runs in the kernels of dense.cu and of the routed
// layer.
#include <string.h>

#include <new>

#include "kernels.h"
#include "moe_internal.cuh"

using moe::align_up;

struct moe_ffn {
  moe_ffn_config cfg;
  moe_layer_t routed;
  int hidden, latent, S, Is, fmt;
  int Wh, Wl, Wi;                   // 512-element K-slices of hidden, latent and Is
  size_t slice_bytes;
  // GEMV A, input u (bf16, K = hidden): tiles [routed_down (latent / 16) |
  // shared s gate/up pairs (Is / 8 each)]; GEMV B, input [n | h_0 | h_1 ...]
  // (fp32, K = KB, each part padded to whole slices): tiles hidden / 16 of
  // [routed_up | shared down 0 | shared down 1 ...] side by side along K
  int tilesA, rd_tiles, sgu_tiles, tilesB, WB, KB;
  size_t off_A, off_B, off_scal, off_sscale, off_gamma, off_trailer, packed_bytes;
};

namespace {

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

struct FfnWs {
  size_t routed, x_lat, y_r, xB, part, total;
};

FfnWs ffn_ws(const moe_ffn &F, int C) {
  FfnWs w = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  size_t routed_bytes = 0;
  moe_workspace_bytes(F.routed, C, &routed_bytes);
  w.routed = take(routed_bytes);
  w.x_lat = take(2 * (size_t)C * F.latent);
  w.y_r = take(4 * (size_t)C * F.latent);
  w.xB = take(4 * (size_t)C * F.KB);         // zero between the parts: the workspace is zero-filled once
  const size_t pa = moe::dense_partial_bytes(F.tilesA, F.Wh, C, false), pb = moe::dense_partial_bytes(F.tilesB, F.WB, C, true);
  w.part = take(pa > pb ? pa : pb);
  w.total = off;
  return w;
}

moe_status check_call(const moe_ffn *F, const uint16_t *u, int C, const void *ffn_packed, void *ws, size_t ws_bytes) {
  if (!F || !u || !ffn_packed || !ws) return MOE_ERR_INVALID_ARG;
  if (C < 1 || C > moe::kGemvTokens || C > F->routed->cfg.max_tokens) return MOE_ERR_INVALID_ARG;
  if (!aligned16(u) || !aligned16(ffn_packed) || !aligned16(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ffn_ws(*F, C).total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return MOE_OK;
}

// GEMV A over its tiles [t0, t1): routed_down -> x_lat (bf16), the shared
// experts' gate/up pairs -> h_s = silu(g) * u into xB (fp32).
cudaError_t gemv_A(const moe_ffn &F, const uint8_t *pk, const uint16_t *u, int C, uint8_t *w, const FfnWs &wl, int t0,
                   int t1, cudaStream_t stream) {
  const float *scal = reinterpret_cast<const float *>(pk + F.off_scal);
  moe::DenseArgs a = {};
  const size_t tile_bytes = (size_t)F.Wh * F.slice_bytes;
  a.w = pk + F.off_A + (size_t)t0 * tile_bytes;
  a.x = u;
  a.part = reinterpret_cast<float *>(w + wl.part);
  a.xf32 = 0; a.C = C; a.K = F.hidden; a.W = F.Wh; a.tiles = t1 - t0; a.fmt = F.fmt;
  a.tile_bytes = tile_bytes;
  moe::DenseFinishArgs f = {};
  f.part = a.part; f.xf32 = 0; f.C = C; f.W = F.Wh; f.tiles = t1 - t0;
  auto add_seg = [&](int s0, int s1, moe::DenseSeg sg) {    // absolute tiles [s0, s1) of A
    const int lo = s0 > t0 ? s0 : t0, hi = s1 < t1 ? s1 : t1;
    if (lo >= hi) return;
    sg.tile0 = lo - t0;
    sg.tile1 = hi - t0;
    // the segment's pair rows start (lo - s0) tiles into its matrix
    sg.col0 += (sg.mode == 1 ? 8 : 16) * (lo - s0);
    f.seg[f.nseg++] = sg;
  };
  moe::DenseSeg rd = {};
  rd.mode = 0; rd.ga = scal + 0; rd.out_bf16 = reinterpret_cast<uint16_t *>(w + wl.x_lat); rd.out_ld = F.latent;
  add_seg(0, F.rd_tiles, rd);
  for (int s = 0; s < F.S; s++) {
    moe::DenseSeg gu = {};
    gu.mode = 1; gu.ga = scal + 2 + 3 * s; gu.gb = scal + 3 + 3 * s;
    gu.out_f32 = reinterpret_cast<float *>(w + wl.xB); gu.out_ld = F.KB; gu.col0 = F.Wl * moe::kKAlign + s * F.Wi * moe::kKAlign;
    add_seg(F.rd_tiles + s * F.sgu_tiles, F.rd_tiles + (s + 1) * F.sgu_tiles, gu);
  }
  if (f.nseg == 0) return cudaSuccess;
  return moe::launch_dense_gemv(a, f, F.routed->num_sms, stream);
}

// GEMV B: out = routed_up n + sum_s down_s h_s, one matrix along K with a
// tensor scale per K-slice.
cudaError_t gemv_B(const moe_ffn &F, const uint8_t *pk, int C, uint8_t *w, const FfnWs &wl, float *out,
                   cudaStream_t stream) {
  moe::DenseArgs a = {};
  a.w = pk + F.off_B;
  a.x = w + wl.xB;
  a.part = reinterpret_cast<float *>(w + wl.part);
  a.xf32 = 1; a.C = C; a.K = F.KB; a.W = F.WB; a.tiles = F.tilesB; a.fmt = F.fmt;
  a.tile_bytes = (size_t)F.WB * F.slice_bytes;
  moe::DenseFinishArgs f = {};
  f.part = a.part; f.xf32 = 1; f.C = C; f.W = F.WB; f.tiles = F.tilesB;
  f.slice_scale = reinterpret_cast<const float *>(pk + F.off_sscale);
  f.nseg = 1;
  f.seg[0].tile0 = 0; f.seg[0].tile1 = F.tilesB; f.seg[0].mode = 0;
  f.seg[0].out_f32 = out; f.seg[0].out_ld = F.hidden;
  return moe::launch_dense_gemv(a, f, F.routed->num_sms, stream);
}

struct DeviceScope {
  int prev = -1;
  bool ok = false;
  explicit DeviceScope(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) return;
    ok = prev == dev || cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceScope() {
    if (ok && prev >= 0) cudaSetDevice(prev);
  }
};

}  // namespace

extern "C" {

moe_status moe_ffn_create(const moe_ffn_config *cfg, moe_layer_t routed, moe_ffn_t *out) {
  if (!cfg || !routed || !out) return MOE_ERR_INVALID_ARG;
  const moe_ffn_config c = *cfg;
  if (c.flags != 0 || !(c.eps > 0.f) || c.shared_experts < 0 || c.shared_experts > moe::kMaxDenseSegs - 1)
    return MOE_ERR_INVALID_ARG;
  if (routed->w4a4) return MOE_ERR_INVALID_ARG;     // the projections around the routed sum are W4A16
  if (c.hidden < 64 || c.hidden % 64 || c.hidden > 8192) return MOE_ERR_UNSUPPORTED_SHAPE;
  if (c.shared_experts > 0 && (c.shared_intermediate < 64 || c.shared_intermediate % 64 || c.shared_intermediate > 4096))
    return MOE_ERR_UNSUPPORTED_SHAPE;
  moe_ffn *F = new (std::nothrow) moe_ffn();
  if (!F) return MOE_ERR_OUT_OF_MEMORY;
  F->cfg = c;
  F->routed = routed;
  F->hidden = c.hidden;
  F->latent = routed->cfg.hidden;
  F->S = c.shared_experts;
  F->Is = c.shared_experts > 0 ? c.shared_intermediate : 0;
  F->fmt = routed->fmt;
  F->Wh = (int)(align_up(F->hidden, moe::kKAlign) / moe::kKAlign);
  F->Wl = (int)(align_up(F->latent, moe::kKAlign) / moe::kKAlign);
  F->Wi = F->Is > 0 ? (int)(align_up(F->Is, moe::kKAlign) / moe::kKAlign) : 0;
  F->slice_bytes = F->fmt == moe::kFmtMxfp4 ? moe::kTileSliceBytesMx : moe::kTileSliceBytes;
  F->rd_tiles = F->latent / 16;
  F->sgu_tiles = F->Is / 8;
  F->tilesA = F->rd_tiles + F->S * F->sgu_tiles;
  F->tilesB = F->hidden / 16;
  F->WB = F->Wl + F->S * F->Wi;
  F->KB = F->WB * moe::kKAlign;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  F->off_A = take((size_t)F->tilesA * F->Wh * F->slice_bytes);
  F->off_B = take((size_t)F->tilesB * F->WB * F->slice_bytes);
  F->off_scal = take(sizeof(float) * (2 + 3 * (size_t)F->S));
  F->off_sscale = take(sizeof(float) * (size_t)F->WB);
  F->off_gamma = take(sizeof(float) * (size_t)F->latent);
  F->off_trailer = take(16);
  F->packed_bytes = off;
  *out = F;
  return MOE_OK;
}

moe_status moe_ffn_destroy(moe_ffn_t F) {
  delete F;
  return MOE_OK;
}

moe_status moe_ffn_packed_bytes(moe_ffn_t F, size_t *bytes) {
  if (!F || !bytes) return MOE_ERR_INVALID_ARG;
  *bytes = F->packed_bytes;
  return MOE_OK;
}

moe_status moe_ffn_workspace_bytes(moe_ffn_t F, int num_tokens, size_t *bytes) {
  if (!F || !bytes || num_tokens < 1 || num_tokens > moe::kGemvTokens) return MOE_ERR_INVALID_ARG;
  *bytes = ffn_ws(*F, num_tokens).total;
  return MOE_OK;
}

moe_status moe_ffn_pack_weights(moe_ffn_t F, const moe_ffn_weights *w, void *packed, cudaStream_t stream) {
  if (!F || !w || !packed || !w->norm_gamma || !aligned16(packed)) return MOE_ERR_INVALID_ARG;
  const moe_fp4_tensor *ts[5] = {&w->routed_down, &w->routed_up, &w->shared.gate, &w->shared.up, &w->shared.down};
  for (int i = 0; i < (F->S > 0 ? 5 : 2); i++)
    if (!ts[i]->codes || !ts[i]->scales || !ts[i]->global_scale || !aligned16(ts[i]->codes)) return MOE_ERR_INVALID_ARG;
  DeviceScope dev(F->routed->device);
  if (!dev.ok) return MOE_ERR_CUDA;
  uint8_t *pk = static_cast<uint8_t *>(packed);
  int32_t *status = reinterpret_cast<int32_t *>(pk + F->off_trailer);
  const int SB = F->fmt == moe::kFmtMxfp4 ? 32 : 16;
  cudaError_t err = cudaMemsetAsync(pk, 0, F->packed_bytes, stream);   // padding slices stay zero
  auto pack = [&](const uint8_t *ca, const uint8_t *sa, const uint8_t *cb, const uint8_t *sb, int M, int K, int mode,
                  size_t off, int W, int tile0, int wd0) {
    if (err != cudaSuccess) return;
    moe::PackDenseArgs a = {};
    a.codesA = ca; a.scalesA = sa; a.codesB = cb; a.scalesB = sb;
    a.dst = pk + off; a.status = status;
    a.M = M; a.K = K; a.mode = mode; a.fmt = F->fmt;
    a.Wsrc = (int)(align_up(K, moe::kKAlign) / moe::kKAlign);
    a.W = W; a.tile0 = tile0; a.wd0 = wd0;
    err = moe::launch_pack_dense(a, F->routed->num_sms, stream);
  };
  const int H = F->hidden, L = F->latent, Is = F->Is;
  // GEMV A: routed_down pair rows, then each shared expert's (gate, up) pairs
  pack(w->routed_down.codes, w->routed_down.scales, nullptr, nullptr, L, H, 0, F->off_A, F->Wh, 0, 0);
  for (int s = 0; s < F->S; s++)
    pack(w->shared.gate.codes + (size_t)s * Is * (H / 2), w->shared.gate.scales + (size_t)s * Is * (H / SB),
         w->shared.up.codes + (size_t)s * Is * (H / 2), w->shared.up.scales + (size_t)s * Is * (H / SB), Is, H, 1,
         F->off_A, F->Wh, F->rd_tiles + s * F->sgu_tiles, 0);
  // GEMV B: routed_up in slices [0, Wl), shared down s in [Wl + s Wi, ...)
  pack(w->routed_up.codes, w->routed_up.scales, nullptr, nullptr, H, L, 0, F->off_B, F->WB, 0, 0);
  for (int s = 0; s < F->S; s++)
    pack(w->shared.down.codes + (size_t)s * H * (Is / 2), w->shared.down.scales + (size_t)s * H * (Is / SB), nullptr,
         nullptr, H, Is, 0, F->off_B, F->WB, 0, F->Wl + s * F->Wi);
  float *scal = reinterpret_cast<float *>(pk + F->off_scal);
  float *sscale = reinterpret_cast<float *>(pk + F->off_sscale);
  auto copy = [&](float *dst, const float *src, size_t n) {
    if (err == cudaSuccess) err = cudaMemcpyAsync(dst, src, n * sizeof(float), cudaMemcpyDeviceToDevice, stream);
  };
  copy(scal + 0, w->routed_down.global_scale, 1);
  copy(scal + 1, w->routed_up.global_scale, 1);
  for (int s = 0; s < F->S; s++) {
    copy(scal + 2 + 3 * s, w->shared.gate.global_scale + s, 1);
    copy(scal + 3 + 3 * s, w->shared.up.global_scale + s, 1);
    copy(scal + 4 + 3 * s, w->shared.down.global_scale + s, 1);
  }
  for (int j = 0; j < F->WB; j++)                        // GEMV B: the tensor scale of each K-slice
    copy(sscale + j, j < F->Wl ? w->routed_up.global_scale : w->shared.down.global_scale + (j - F->Wl) / F->Wi, 1);
  copy(reinterpret_cast<float *>(pk + F->off_gamma), w->norm_gamma, (size_t)L);
  int32_t host_status = 0;
  if (err == cudaSuccess) err = cudaMemcpyAsync(&host_status, status, sizeof(int32_t), cudaMemcpyDeviceToHost, stream);
  if (err == cudaSuccess) err = cudaStreamSynchronize(stream);
  if (err != cudaSuccess) return MOE_ERR_CUDA;
  return host_status ? MOE_ERR_INVALID_VALUE : MOE_OK;
}

moe_status moe_ffn_partial(moe_ffn_t F, const uint16_t *u, int C, const float *w_router, const float *bias,
                           const void *routed_packed, const void *ffn_packed, int32_t *ids, float *weights,
                           float *y_routed, void *ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_call(F, u, C, ffn_packed, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!w_router || !routed_packed || !ids || !weights || !y_routed || !aligned16(y_routed)) return MOE_ERR_INVALID_ARG;
  const FfnWs wl = ffn_ws(*F, C);
  uint8_t *w = static_cast<uint8_t *>(ws);
  {
    DeviceScope dev(F->routed->device);
    if (!dev.ok) return MOE_ERR_CUDA;
    // routed_down: x = D_lat u, rounded to bf16 (the routed layer's input type)
    if (gemv_A(*F, static_cast<const uint8_t *>(ffn_packed), u, C, w, wl, 0, F->rd_tiles, stream) != cudaSuccess)
      return MOE_ERR_CUDA;
  }
  size_t routed_bytes = 0;
  moe_workspace_bytes(F->routed, C, &routed_bytes);
  return moe_route_forward(F->routed, reinterpret_cast<const uint16_t *>(w + wl.x_lat), C, w_router, bias,
                           routed_packed, ids, weights, y_routed, w + wl.routed, routed_bytes, stream);
}

moe_status moe_ffn_finish(moe_ffn_t F, const uint16_t *u, int C, const float *y_routed, const void *ffn_packed,
                          float *out, void *ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_call(F, u, C, ffn_packed, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!y_routed || !out || !aligned16(out) || !aligned16(y_routed)) return MOE_ERR_INVALID_ARG;
  const FfnWs wl = ffn_ws(*F, C);
  uint8_t *w = static_cast<uint8_t *>(ws);
  const uint8_t *pk = static_cast<const uint8_t *>(ffn_packed);
  DeviceScope dev(F->routed->device);
  if (!dev.ok) return MOE_ERR_CUDA;
  // the shared experts' gate/up (GEMV A's last tiles), routed_norm into the
  // first columns of GEMV B's input, then GEMV B
  cudaError_t err = gemv_A(*F, pk, u, C, w, wl, F->rd_tiles, F->tilesA, stream);
  if (err == cudaSuccess)
    err = moe::launch_rms_norm(y_routed, reinterpret_cast<const float *>(pk + F->off_gamma), F->cfg.eps, C, F->latent,
                               reinterpret_cast<float *>(w + wl.xB), F->KB, stream);
  if (err == cudaSuccess) err = gemv_B(*F, pk, C, w, wl, out, stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_ffn_forward(moe_ffn_t F, const uint16_t *u, int C, const float *w_router, const float *bias,
                           const void *routed_packed, const void *ffn_packed, int32_t *ids, float *weights, float *out,
                           void *ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status st = check_call(F, u, C, ffn_packed, ws, ws_bytes);
  if (st != MOE_OK) return st;
  if (!w_router || !routed_packed || !ids || !weights || !out || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  const FfnWs wl = ffn_ws(*F, C);
  uint8_t *w = static_cast<uint8_t *>(ws);
  const uint8_t *pk = static_cast<const uint8_t *>(ffn_packed);
  float *y_r = reinterpret_cast<float *>(w + wl.y_r);
  {
    DeviceScope dev(F->routed->device);
    if (!dev.ok) return MOE_ERR_CUDA;
    // one GEMV for routed_down and every shared expert's gate/up (both read u)
    if (gemv_A(*F, pk, u, C, w, wl, 0, F->tilesA, stream) != cudaSuccess) return MOE_ERR_CUDA;
  }
  size_t routed_bytes = 0;
  moe_workspace_bytes(F->routed, C, &routed_bytes);
  st = moe_route_forward(F->routed, reinterpret_cast<const uint16_t *>(w + wl.x_lat), C, w_router, bias, routed_packed,
                         ids, weights, y_r, w + wl.routed, routed_bytes, stream);
  if (st != MOE_OK) return st;
  DeviceScope dev(F->routed->device);
  if (!dev.ok) return MOE_ERR_CUDA;
  cudaError_t err = moe::launch_rms_norm(y_r, reinterpret_cast<const float *>(pk + F->off_gamma), F->cfg.eps, C,
                                         F->latent, reinterpret_cast<float *>(w + wl.xB), F->KB, stream);
  if (err == cudaSuccess) err = gemv_B(*F, pk, C, w, wl, out, stream);
  return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
