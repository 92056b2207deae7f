// moe_internal.cuh -- layer handle, packed-layout arithmetic and PTX helpers
// shared by the kernels of the routed NVFP4 MoE library (sm_103a only).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "this library is written for Blackwell (sm_103a); build with -gencode arch=compute_103a,code=sm_103a"
#endif

namespace moe {

// ----------------------------------------------------------------- limits
constexpr int kMaxExperts = 1024;        // dispatch bitmap: 32 words of 32 bits
constexpr int kMaxTopK = 32;             // one top-k slot per lane
constexpr int kGemvTokens = 8;           // tokens per GEMV group (token mask bits)
constexpr int kGroupTokens = 512;        // tokens per pass of the grouped (expert-major) path
constexpr int kGroupedMinTokens = 28;    // calls of this many tokens or more take the grouped path (measured crossover)
constexpr int kMaxPairs = kGemvTokens * kMaxTopK;   // (token, slot) pairs per group
constexpr int kKAlign = 512;             // packed K is padded to this (32 lanes x 16)
constexpr int kRouteFusedTokens = 8;     // route: fused top-k in the last CTA up to this C
constexpr int kRouteSplits = 4;          // route, C > 8: K ranges of the logits GEMM (partials summed in order)
constexpr int kGemvSmemBytes = 211968;   // dynamic shared memory of one expert-GEMV CTA (+ ~20 KB static)
constexpr int kGroupSmemBytes = 212992;  // dynamic shared memory of one grouped-GEMM CTA at most (+ ~12 KB static)
constexpr int kTileSliceBytes = 4608;    // one 512-element K-slice of a tile: 4096 code + 512 scale bytes
constexpr int kTileSliceBytesMx = 4352;  // the same for MXFP4: 4096 code + 256 scale bytes (one per 32 elements)
constexpr int kFmtNvfp4 = 0, kFmtMxfp4 = 1;
constexpr int kDenseSmemBytes = 204800;  // B fragments of a dense GEMV: passes x K/16 k-steps x 256 bytes at most

// Workspace control block (first 256 bytes of the workspace).
struct WsControl {
  int32_t flags;          // MOE_FLAG_* bits, cleared by moe_get_device_status
  uint32_t route_ticket;  // CTAs of the router that finished their logits
  uint32_t reserved;       // zero
  uint32_t pad[61];
};
static_assert(sizeof(WsControl) == 256, "control block is 256 bytes");

// Byte offsets of the workspace regions.  The decode regions (token groups of
// at most kGemvTokens) sit at fixed offsets whatever C is; calls with C > 8
// add the router logits of all C tokens and the grouped path's buffers for
// passes of up to kGroupTokens tokens.
struct WsLayout {
  size_t logits;      // float  [kGemvTokens][E]        router logits, C <= 8
  size_t hbuf;        // float  [kGemvTokens * k][I]    w * silu(g) * u per (token, slot), each
                      //        16-element block stored in MMA operand order (see expert_gemv.cu)
  size_t hamax;       // uint32 [kGemvTokens * k]       max |h| per (token, slot) as float bits
  size_t ypair;       // float  [kGemvTokens * k][H]    D_e h per (token, slot)
  // C > 8 only (0 otherwise): Cg = min(C, kGroupTokens) tokens, Pg = Cg * k pairs
  size_t glogits;     // float  [kRouteSplits][C][E]    router logit partials; logits in partial 0
  size_t gd;          // int    n, then expert [E], off [E + 1], pairs [Pg]   expert-major dispatch
  size_t xinv;        // float  [Cg]                    2^-s of each token's f16 scale
  size_t xg;          // f16    [Hp / 8][Pg][8]         x rows of the pairs in dispatch order
  size_t ghbuf;       // float  [Pg][I]                 h per pair
  size_t hg;          // f16    [Ip / 8][2 Pg][8]       hi / lo rows of h in dispatch order
  size_t hinv;        // float  [Pg]                    2^-s of each pair's h scale
  size_t gypair;      // float  [Pg][H]                 D_e h per pair
  size_t total;
};

}  // namespace moe

// The handle.  Immutable after moe_layer_create except for the optional
// stage-event hook.
struct moe_layer {
  moe_config cfg;
  int fmt;                    // kFmtNvfp4 or kFmtMxfp4 (MOE_CONFIG_MXFP4)
  int w4a4;                   // MOE_CONFIG_W4A4: activations quantized to NVFP4 (decode and grouped paths)
  int device;
  int num_sms;
  int Hp, Ip;                 // K of gate/up and of down, padded to kKAlign
  int w_gu, w_dn;             // 512-element K-slices (= consumer warps of a group)
  size_t gu_tile_bytes;       // w_gu * slice bytes (kTileSliceBytes or kTileSliceBytesMx): 8 gate/up pair rows
  size_t dn_tile_bytes;       // w_dn * slice bytes: 8 down pair rows
  size_t dn_region_off;       // offset of the down tiles inside an expert
  size_t expert_bytes;        // packed bytes of one expert (without scalars)
  size_t scalars_off;         // float [E][6] : g_gate a_gate g_up a_up g_down a_down
  size_t trailer_off;         // 16-byte status trailer written by the packer
  size_t packed_bytes;
  cudaEvent_t stage_events[3];
  int stage_events_on;
  int grouped_min_tokens;     // calls of at least this many tokens take the grouped (tcgen05) path
};

namespace moe {

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(const moe_layer &L, int C) {
  WsLayout w = {};
  const size_t E = L.cfg.num_experts, H = L.cfg.hidden, I = L.cfg.intermediate, k = L.cfg.top_k;
  size_t off = sizeof(WsControl);
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, 256);
    return at;
  };
  const size_t pairs = (size_t)kGemvTokens * k;
  w.logits = take(sizeof(float) * kGemvTokens * E);
  w.hbuf = take(sizeof(float) * pairs * I);
  w.hamax = take(sizeof(uint32_t) * pairs);
  w.ypair = take(sizeof(float) * pairs * H);
  if (C > kGemvTokens) {
    const size_t Cg = C < kGroupTokens ? C : kGroupTokens, Pg = Cg * k;
    w.glogits = take(sizeof(float) * kRouteSplits * (size_t)C * E);
    w.gd = take(sizeof(int) * (16 + E + (E + 1) + Pg));
    w.xinv = take(sizeof(float) * Cg);
    w.xg = take(2 * Pg * (size_t)L.Hp);
    w.ghbuf = take(sizeof(float) * Pg * I);
    w.hg = take(2 * 2 * Pg * (size_t)L.Ip);
    w.hinv = take(sizeof(float) * Pg);
    w.gypair = take(sizeof(float) * Pg * H);
  }
  w.total = off;
  return w;
}

// ------------------------------------------------------------ PTX helpers
#ifdef __CUDACC__

// Streaming 16-byte load: no L1 allocation, L2 evict-first (the weights are
// read once per call; keep L2 for the activations and partial sums).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// Default L2 residency, for data read again soon.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 evict-last: data a kernel reads many times (the grouped path's B rows).
__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void *ptr, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr), "l"(pol));
  return v;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void *ptr, uint64_t pol) {
  unsigned short v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.u16 %0, [%1], %2;"
               : "=h"(v)
               : "l"(ptr), "l"(pol));
  return v;
}

// Four e2m1 pairs (one 32-bit word = 8 codes, low nibble first) -> four
// f16x2 words; word i holds elements 2i (low half) and 2i+1 (high half).
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

// Two e4m3 bytes (low byte first) -> two fp32 values.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two_bytes) {
  uint32_t h2;
  asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(two_bytes));
  __half2 hh = *reinterpret_cast<__half2 *>(&h2);
  return __half22float2(hh);
}

// acc += a.lo * b.lo + a.hi * b.hi with f16 inputs and fp32 accumulation
// (mixed-precision fma, sm_100+): each product of two f16 values is exact in
// fp32 and is rounded once when added.
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t"
      "mov.b32 {al, ah}, %1;\n\t"
      "mov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.f16 %0, al, bl, %0;\n\t"
      "fma.rn.f32.f16 %0, ah, bh, %0;\n\t}"
      : "+f"(acc)
      : "r"(a), "r"(b));
  return acc;
}

// Packed fp32x2 fma: (d.x, d.y) = (a.x*b.x + c.x, a.y*b.y + c.y).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  uint64_t ra = *reinterpret_cast<uint64_t *>(&a), rb = *reinterpret_cast<uint64_t *>(&b),
           rc = *reinterpret_cast<uint64_t *>(&c), rd;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  return *reinterpret_cast<float2 *>(&rd);
}

// Start of part `part` of `parts` equal contiguous parts of [0, total), in
// 32-bit arithmetic (total * parts < 2^32 for every use here: the 64-bit
// division is a long software routine that every thread would run).
__device__ __forceinline__ int split_point(int total, int part, int parts) {
  return (int)(((uint32_t)total * (uint32_t)part) / (uint32_t)parts);
}

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#endif  // __CUDACC__

}  // namespace moe
