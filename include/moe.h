/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed NVFP4 MoE FFN library.
 *
 * One MoE layer of a Kimi-K3-class model at decode ("MUL_MAT_ID"): router
 * scores, top-k of the routed experts with softmax weights renormalised over
 * the top-k, an NVFP4 SwiGLU FFN per selected expert, and the weighted sum of
 * the expert outputs.  Shapes and byte counts follow "SparkInfer-K3"
 * (sections "The model" and "How the TP module works") and "Kimi-K3 on the
 * same pod, two engines" (section "Same hardware, same weights": 896 routed
 * experts, top-16, 18,579,480 bytes per NVFP4 expert).
 *
 * Conventions for every entry point
 *   - All pointers named "device" are CUDA device pointers on the layer's
 *     device, owned by the caller, 16-byte aligned, and must stay valid until
 *     the work queued on `stream` has finished.  The library allocates no
 *     device memory and keeps no pointer after a call returns.
 *   - Argument and shape errors are returned synchronously before anything is
 *     queued.  A failed launch returns MOE_ERR_CUDA.  Errors found in the data
 *     on the device (an expert id out of range or repeated within a token) set
 *     bits in a flag word inside the workspace: read them with
 *     moe_get_device_status.  No kernel traps or asserts.
 *   - moe_route, moe_forward and moe_route_forward allocate nothing and never
 *     synchronise the host, so a sequence of them can be captured into a CUDA
 *     graph.
 *   - The handle is immutable after creation; concurrent calls on different
 *     streams need different workspaces and output buffers.
 *
 * Canonical NVFP4 matrix [rows][K] (the checkpoint's byte layout as read
 * here; it reproduces the 18,579,480 bytes per expert exactly):
 *   codes   uint8 [rows][K/2]  e2m1 codes, low nibble = element 2j, high = 2j+1
 *   scales  uint8 [rows][K/16] e4m3 scale of elements 16b .. 16b+15 of the row
 *   global_scale float         multiplies every element of the matrix
 *   input_scale  float         carried, not used (activations stay bf16/fp32)
 *   weight(r, k) = e2m1(code) * e4m3(scale) * global_scale
 * Expert e's FFN:  g = G x, u = U x (G, U: [I][H]);  a = silu(g) * u;
 *                  y_e = D a (D: [H][I]).
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,        /* null/misaligned pointer, bad count */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,  /* shape outside the supported range */
  MOE_ERR_INVALID_VALUE = 3,      /* a NaN e4m3 scale byte in the weights */
  MOE_ERR_WORKSPACE_TOO_SMALL = 4,
  MOE_ERR_OUT_OF_MEMORY = 5,
  MOE_ERR_CUDA = 6,               /* a CUDA runtime call or launch failed */
  MOE_ERR_DEVICE_TIMEOUT = 7,     /* reserved: a bounded device wait ran out */
  MOE_ERR_BAD_EXPERT_ID = 8       /* device flag: an id out of [0,E) or repeated */
} moe_status;

/* Device flag bits reported by moe_get_device_status. */
#define MOE_FLAG_BAD_EXPERT_ID 0x1   /* an id outside [0, num_experts): slot skipped */
#define MOE_FLAG_DUPLICATE_ID 0x2    /* an expert repeated within one token: one copy dropped */
#define MOE_FLAG_TIMEOUT 0x4         /* a bounded device wait ran out; outputs of that call are invalid */

/* moe_config.flags.  Test hook only, never set in use: every router CTA
 * (C <= 8) waits for 16 bytes that no copy delivers, with a 20 ms limit
 * instead of ~2 s, so the timeout path can be exercised without a GPU fault:
 * MOE_FLAG_TIMEOUT is raised and the call's ids are all -1. */
#define MOE_CONFIG_TEST_ROUTER_STALL 0x80000000u

/* moe_config.flags: the layer's weights are MXFP4 (OCP Microscaling: e2m1
 * codes as in NVFP4, one e8m0 scale byte per 32 elements along K, value
 * 2^(byte - 127), 0xFF = NaN), the format of the ggml MUL_MAT_ID microbench in
 * "Kimi-K3 on 2x A40 - measured findings" (section "Why the placement
 * experiments all looked the same").  moe_fp4_tensor.scales is then
 * [E][rows][K/32] and global_scale still multiplies the matrix (pass 1.0 for
 * plain MXFP4).  Every C runs on the decode kernels (groups of 8 tokens, each
 * expert read once per group); the tcgen05 grouped path is NVFP4 only. */
#define MOE_CONFIG_MXFP4 0x1u

/* moe_config.flags: take the grouped tcgen05 path for every call of more
 * than 8 tokens.  By default calls of 9 .. 27 tokens run on the decode
 * kernels in groups of 8, which are faster there (with uniform routing over
 * 896 experts each expert has one or two tokens, so the grouped GEMM's MMAs
 * are mostly padding); 28 tokens or more take the grouped path.  NVFP4
 * layers only. */
#define MOE_CONFIG_GROUPED_ABOVE_8 0x2u

/* moe_config.flags: W4A4 numerics (NVFP4 layers only).  Each matrix's input
 * is quantized to NVFP4 with that matrix's fp32 input scale a (the second of
 * its two scalars; "Kimi-K3 on the same pod, two engines", section "Same
 * hardware, same weights": 24 bytes of fp32 scalars per expert): per block of
 * 16 elements the e4m3 scale byte s = e4m3(max|v| / (6 a)) and the e2m1
 * codes e2m1(v / (s a)), both rounded to nearest even and saturating; the
 * quantized value is e2m1 * s * a.  x is quantized per (token, expert) with
 * max(a_gate, a_up) (gate and up read one quantized x); h = silu(g) * u per
 * (token, expert) with a_down; the router weight multiplies the expert's
 * output after the down projection.  Below 28 tokens the decode kernels
 * quantize x and h in their MMA fragments; from 28 tokens the grouped tcgen05
 * kernels quantize the gathered rows.  Results agree with the W4A16 ones only
 * to the activation quantization noise (a few per cent). */
#define MOE_CONFIG_W4A4 0x4u

typedef struct {
  int32_t num_experts;   /* E, 1 .. 1024 */
  int32_t top_k;         /* k, 1 .. min(32, E) */
  int32_t hidden;        /* H, expert input/output width, multiple of 64, <= 4096 */
  int32_t intermediate;  /* I, expert FFN width, multiple of 64, <= 4096 */
  int32_t max_tokens;    /* largest C passed to route/forward, >= 1 */
  uint32_t flags;        /* MOE_CONFIG_MXFP4 or MOE_CONFIG_W4A4, MOE_CONFIG_GROUPED_ABOVE_8, the test hook
                            MOE_CONFIG_TEST_ROUTER_STALL, or 0; MXFP4 with W4A4: MOE_ERR_INVALID_ARG */
} moe_config;

typedef struct {
  const uint8_t *codes;        /* device, [E][rows][K/2] */
  const uint8_t *scales;       /* device, [E][rows][K/16] e4m3 (NVFP4) or [E][rows][K/32] e8m0 (MXFP4) */
  const float *global_scale;   /* device, [E] */
  const float *input_scale;    /* device, [E] (copied into the packed buffer; read only by
                                  MOE_CONFIG_W4A4 layers, which quantise the matrix's input with it) */
} moe_fp4_tensor;

typedef struct {
  moe_fp4_tensor gate;  /* rows I, K H */
  moe_fp4_tensor up;    /* rows I, K H */
  moe_fp4_tensor down;  /* rows H, K I */
} moe_canonical_weights;

typedef struct moe_layer *moe_layer_t;

/* Validate `cfg` and create a host-side handle for `device` (queries its SM
 * count; allocates no device memory).  *out is set only on MOE_OK. */
moe_status moe_layer_create(const moe_config *cfg, int device, moe_layer_t *out);

/* Free the handle (host memory only).  NULL is accepted. */
moe_status moe_layer_destroy(moe_layer_t layer);

/* Bytes of the packed weight buffer moe_pack_weights writes.  For H and I
 * multiples of 512 it equals E * (bytes of one canonical expert) + 16: the
 * packer reorders bytes and adds nothing but a 16-byte status trailer (the
 * same holds for MXFP4 layers).  Smaller shapes are padded along K to a
 * multiple of 512 with zero codes. */
moe_status moe_packed_bytes(moe_layer_t layer, size_t *bytes);

/* Bytes of workspace route/forward need for up to `num_tokens` tokens.  The
 * workspace is caller-owned device memory that must be ZERO-FILLED once
 * before its first use; route and forward leave it in a reusable state. */
moe_status moe_workspace_bytes(moe_layer_t layer, int num_tokens, size_t *bytes);

/* Reorder canonical NVFP4 (or MXFP4) weights (all E experts) into the packed layout the
 * kernels stream.  The canonical form is the checkpoint's per matrix ("Kimi-K3
 * on the same pod, two engines", section "Same hardware, same weights": 4-bit
 * codes, an e4m3 scale per 16 elements, and two fp32 scalars -- the 24 bytes
 * per expert beside the codes and scales); MXFP4 is the ggml microbench format
 * of "Kimi-K3 on 2x A40 - measured findings" ("Why the placement experiments
 * all looked the same").  Per expert, I "gate/up pair rows" (gate row r and up row r
 * interleaved per 16-element block) then H/2 "down pair rows" (down rows 2p
 * and 2p+1 interleaved), each pair row holding its codes and then its scale
 * bytes; the 6 fp32 scalars of all experts follow.  Offline, once per layer:
 * this call synchronises `stream` and returns MOE_ERR_INVALID_VALUE if any
 * scale byte is a NaN (e4m3 0x7F or 0xFF; e8m0 0xFF).  `packed` (device,
 * moe_packed_bytes long) must not overlap the canonical buffers. */
moe_status moe_pack_weights(moe_layer_t layer, const moe_canonical_weights *canon,
                            void *packed, cudaStream_t stream);

/* Router and top-k for C tokens ("SparkInfer-K3", "How the TP module works":
 * one replicated router, all ranks agree on the same top-k):
 *   logits l[t][e] = sum_j w_router[e][j] * x[t][j] (+ bias[e]), fp32
 *   ids[t][0..k)     the k largest logits, equal logits -> lower index first,
 *                    written in ascending expert id order
 *   weights[t][i]    softmax over all experts renormalised over the k kept
 *                    = exp(l_i - l_max) / sum over kept of exp(l_j - l_max)
 * x: device bf16 bits [C][H]; w_router: device fp32 [E][H]; bias: device fp32
 * [E] or NULL; ids: device int32 [C][k]; weights: device fp32 [C][k];
 * ws: workspace of at least moe_workspace_bytes(C).  1 <= C <= max_tokens.
 * Failure: if a router block's bounded wait for its weight rows runs out
 * (C <= 8), MOE_FLAG_TIMEOUT is raised and every id of the call is written as
 * -1 (weight 0), which moe_forward treats as an absent slot; the workspace
 * stays usable for the next call.  A token whose logits include a NaN (from a
 * NaN in x, w_router or bias) selects nothing in the same way. */
moe_status moe_route(moe_layer_t layer, const uint16_t *x, int num_tokens,
                     const float *w_router, const float *bias, int32_t *ids,
                     float *weights, void *ws, size_t ws_bytes, cudaStream_t stream);

/* Routed expert FFN and combine for C tokens: the MUL_MAT_ID step of "Kimi-K3
 * on 2x A40 - measured findings" ("Why the placement experiments all looked
 * the same": each token's selected experts' 3584->3072->3584 FFNs) with the
 * routed sum of "SparkInfer-K3" ("How the TP module works"):
 *   y[t] = sum_i weights[t][i] * D_e (silu(G_e x[t]) * (U_e x[t])),  e = ids[t][i]
 * (MOE_CONFIG_W4A4: G_e and U_e see x quantised to NVFP4, D_e sees h
 * quantised, as that flag describes).  Below 28 tokens (MXFP4: every C) the
 * decode kernels run groups of 8 tokens; from 28 tokens the grouped tcgen05
 * kernels run passes of up to 512 tokens expert-major.
 * x: device bf16 bits [C][H]; ids: device int32 [C][k] (any order; each
 * token's ids must be distinct and < E -- offending slots are skipped and
 * flagged; a negative id marks an absent slot, skipped without a flag, which
 * is how one rank of an expert-parallel split evaluates only the experts it
 * holds: see quantized_moe_expert_router_gb300/partition.py); weights: device
 * fp32 [C][k]; packed: the buffer written by
 * moe_pack_weights; y: device fp32 [C][H] (overwritten).  Each selected
 * expert's packed bytes are read once per call whatever number of tokens
 * chose it.  The sum over a token's experts runs in ascending expert id
 * order, so results are bitwise reproducible. */
moe_status moe_forward(moe_layer_t layer, const uint16_t *x, int num_tokens,
                       const int32_t *ids, const float *weights, const void *packed,
                       float *y, void *ws, size_t ws_bytes, cudaStream_t stream);

/* The whole layer for C tokens: moe_route then moe_forward on `stream`
 * (ids and weights are written).  Arguments and errors as those two calls;
 * nothing is queued when an argument is rejected. */
moe_status moe_route_forward(moe_layer_t layer, const uint16_t *x, int num_tokens,
                             const float *w_router, const float *bias, const void *packed,
                             int32_t *ids, float *weights, float *y, void *ws, size_t ws_bytes,
                             cudaStream_t stream);

/* Synchronise `stream`, return the device flag bits accumulated in `ws` since
 * the last call (MOE_FLAG_*), and clear them together with the router's
 * completion counters (after a MOE_FLAG_TIMEOUT the workspace is then as good
 * as new).  No other call may be in flight on `ws`. */
moe_status moe_get_device_status(moe_layer_t layer, void *ws, cudaStream_t stream,
                                 int32_t *flags);

/* Optional timing hook: when `events` is non-NULL, moe_forward records
 * events[0] on its stream before its first kernel, events[1] after the
 * gate/up kernel and events[2] after the down/combine kernel (n_events must
 * be 3).  Pass NULL to switch it off.  Not thread-safe with respect to
 * concurrent moe_forward calls on the same handle. */
moe_status moe_set_stage_events(moe_layer_t layer, cudaEvent_t *events, int n_events);

/* moe_route without a workspace.  The pages have no counterpart: this entry
 * point exists for callers that cannot allocate device memory -- code running
 * while a stream is captured in a mode that forbids cudaMalloc, plug-ins whose
 * host framework owns every device buffer, and latency-critical loops that
 * must not pay cudaMalloc's implicit synchronisation.  It computes exactly
 * what moe_route computes (same kernel), keeping the router logits and its
 * completion counter in a fixed 32 KiB + 256 B array inside the library
 * (resident on every GPU that loads the library until the process exits).
 * Arguments as moe_route, minus the workspace.  Limits: C <= 8 and
 * C * num_experts <= 8192, otherwise MOE_ERR_WORKSPACE_TOO_SMALL and nothing
 * is queued.  The first call on a device looks up the array's address; make
 * it outside any stream capture.  All calls share the array, so calls that
 * overlap on the GPU race: serialise them on one stream.  Allocates nothing.
 * This entry point reports no device flags (it has no workspace to hold
 * them): a call whose bounded router wait ran out writes every id as -1 and
 * every weight as 0, which the caller can test.  The cached address of the
 * array is per device and becomes invalid after cudaDeviceReset. */
moe_status moe_route_noalloc(moe_layer_t layer, const uint16_t *x, int num_tokens,
                             const float *w_router, const float *bias, int32_t *ids,
                             float *weights, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * The FFN around the routed sum ("SparkInfer-K3", section "How the TP module
 * works": FfnPartial = router -> routed_down -> the experts, FfnFinish =
 * routed_norm -> routed_up -> shared experts; section "The model": hidden
 * 7168, latent MoE at 3584, 2 shared experts).  For C <= 8 tokens u (bf16,
 * [C][hidden]):
 *   x   = routed_down u                      [latent][hidden]; x rounded to bf16
 *   y_r = the routed layer on x (router, top-k, experts; moe_route_forward)
 *   n   = routed_norm(y_r) = y_r / sqrt(mean(y_r^2) + eps) * gamma
 *   out = routed_up n + sum over shared experts s of D_s (silu(G_s u) * (U_s u))
 * with latent = the routed layer's hidden size.  The partial / finish split
 * is where an expert-parallel caller sums the ranks' y_r (the reduce sits at
 * the latent width because the RMS norm is not linear).  Every matrix is in
 * the routed layer's format (NVFP4, or MXFP4 when the routed layer has
 * MOE_CONFIG_MXFP4), packed by moe_ffn_pack_weights. */
typedef struct moe_ffn *moe_ffn_t;

typedef struct {
  int32_t hidden;               /* the model width (7168 at the K3 shape); multiple of 64, <= 8192 */
  int32_t shared_experts;       /* S >= 0 (2 at the K3 shape) */
  int32_t shared_intermediate;  /* FFN width of a shared expert; multiple of 64, <= 4096 */
  float eps;                    /* routed_norm epsilon (> 0) */
  uint32_t flags;               /* must be 0 */
} moe_ffn_config;

typedef struct {
  moe_fp4_tensor routed_down;   /* one matrix [latent][hidden]: codes [latent][hidden/2], ... scalars [1] */
  moe_fp4_tensor routed_up;     /* one matrix [hidden][latent] */
  moe_canonical_weights shared; /* S experts: gate/up [S][shared_intermediate][hidden], down [S][hidden][shared_intermediate] */
  const float *norm_gamma;      /* device fp32 [latent] */
} moe_ffn_weights;

/* A host-side handle tied to `routed` (which must outlive it).  The dense
 * projections run W4A16 numerics; a routed layer created with
 * MOE_CONFIG_W4A4 is rejected (MOE_ERR_INVALID_ARG). */
moe_status moe_ffn_create(const moe_ffn_config *cfg, moe_layer_t routed, moe_ffn_t *out);
moe_status moe_ffn_destroy(moe_ffn_t ffn);
/* Bytes of the packed buffer of the FFN's own weights (not the routed ones). */
moe_status moe_ffn_packed_bytes(moe_ffn_t ffn, size_t *bytes);
/* Workspace for C tokens (it contains the routed layer's workspace); zero-filled once. */
moe_status moe_ffn_workspace_bytes(moe_ffn_t ffn, int num_tokens, size_t *bytes);
/* Pack routed_down, routed_up, the shared experts and gamma (synchronises
 * `stream`; MOE_ERR_INVALID_VALUE on a NaN scale byte). */
moe_status moe_ffn_pack_weights(moe_ffn_t ffn, const moe_ffn_weights *w, void *packed, cudaStream_t stream);
/* FfnPartial: x = routed_down u, then moe_route_forward on x: ids, weights
 * ([C][k]) and y_routed (device fp32 [C][latent]) are written.  1 <= C <=
 * min(8, the routed layer's max_tokens). */
moe_status moe_ffn_partial(moe_ffn_t ffn, const uint16_t *u, int num_tokens, const float *w_router,
                           const float *bias, const void *routed_packed, const void *ffn_packed, int32_t *ids,
                           float *weights, float *y_routed, void *ws, size_t ws_bytes, cudaStream_t stream);
/* FfnFinish: out (device fp32 [C][hidden]) = routed_up(routed_norm(y_routed))
 * + the shared experts on u. */
moe_status moe_ffn_finish(moe_ffn_t ffn, const uint16_t *u, int num_tokens, const float *y_routed,
                          const void *ffn_packed, float *out, void *ws, size_t ws_bytes, cudaStream_t stream);
/* Both phases (y_routed kept in the workspace). */
moe_status moe_ffn_forward(moe_ffn_t ffn, const uint16_t *u, int num_tokens, const float *w_router,
                           const float *bias, const void *routed_packed, const void *ffn_packed, int32_t *ids,
                           float *weights, float *out, void *ws, size_t ws_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------
 * The W4A4 activation quantizer (MOE_CONFIG_W4A4) as a call of its own.
 * Quantizes `rows` rows of n elements (n a multiple of 16) to NVFP4 with the
 * static input scale a (finite, > 0): per block of 16 elements the e4m3 scale
 * byte s = e4m3(max|v| / (6 a)) and the e2m1 codes e2m1(v / (e4m3(s) a)),
 * each step one correctly rounded fp32 operation, both roundings to nearest
 * even and saturating (an all-zero block, or one whose s underflows to 0,
 * gets zero codes); the input scale of "Kimi-K3 on the same pod, two
 * engines", section "Same hardware, same weights".  The kernels of the W4A4
 * layers quantize with the same device code.
 *   src     device, [rows][n], bf16 bits (src_dtype MOE_ACT_BF16) or fp32
 *           (MOE_ACT_F32), 16-byte aligned; read only
 *   codes   device, [rows][n/2], low nibble = even element, 16-byte aligned
 *   scales  device, [rows][n/16] e4m3 bytes
 * The caller owns every buffer.  Queued on `stream`; MOE_ERR_INVALID_ARG on a
 * null or misaligned pointer, rows < 1, n < 16, n % 16 != 0, an unknown
 * src_dtype or a not finite or not positive a; MOE_ERR_CUDA if the launch
 * fails. */
#define MOE_ACT_BF16 0
#define MOE_ACT_F32 1
moe_status moe_quantize_nvfp4(const void *src, int32_t src_dtype, int64_t rows, int32_t n, float a,
                              uint8_t *codes, uint8_t *scales, cudaStream_t stream);

/* Static, NUL-terminated description of a status code. */
const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
