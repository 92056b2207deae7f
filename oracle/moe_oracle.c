/*
 * moe_oracle.c -- plain, slow, float64 CPU oracle for the routed NVFP4 MoE FFN.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check of the
 * package entry module and the CPU-baseline leg of the benchmark may load this
 * file.  The product library never links it, calls it or falls back to it, and
 * this file shares no code, header, table or helper with the CUDA path.
 *
 * What it computes (one MoE layer of a Kimi-K3-class model at decode, the
 * "MUL_MAT_ID" step):
 *   1. router logits  l[t][e] = sum_j Wr[e][j] * x[t][j]  (+ bias[e])
 *   2. softmax over all E experts, the k largest logits kept (equal logits:
 *      lower expert index first), the kept probabilities renormalised to sum 1
 *   3. for every kept expert: g = G x, u = U x, a = silu(g) * u, y_e = D a,
 *      with G, U, D decoded exactly from NVFP4
 *   4. y[t] = sum_i w[t][i] * y_{e_i}
 * Sources: "SparkInfer-K3" README, sections "How the TP module works" (every
 * rank runs the same router and agrees on the same top-16; the partial expert
 * sums add up to the full 3584-wide output) and "The model" (896 routed
 * experts, top-16, experts in a 3584-wide latent space, expert FFN 3072);
 * "Kimi-K3 on 2x A40 - measured findings", section "Why the placement
 * experiments all looked the same" (MUL_MAT_ID over the selected experts'
 * 3584->3072 matrices); "Kimi-K3 on the same pod, two engines", section "Same
 * hardware, same weights" (NVFP4 checkpoint, 18,579,480 bytes per routed
 * expert).
 *
 * Readings taken where the pages are silent (each is listed in the design
 * notes):
 *   - router scoring is a softmax, renormalised over the top-k, with no extra
 *     routed scaling factor;
 *   - the expert activation is SwiGLU, silu(g) * u (the K3 page names a
 *     different activation, "situ", without a formula);
 *   - NVFP4 bytes per matrix [rows][K]: one e2m1 code per element, two per
 *     byte, the LOW nibble holding the even element; one e4m3 scale byte per
 *     16 consecutive elements along K; one fp32 tensor (global) scale that
 *     multiplies every element; one fp32 input scale that this path carries
 *     but does not use.  That reading is the only one that reproduces the
 *     page's 18,579,480 bytes for three 3072x3584 matrices exactly:
 *     3 * (3072*3584/2 + 3072*3584/16 + 2*4).
 *
 * Precision: every product and sum is float64.  A decoded weight
 * e2m1 * e4m3 * fp32 has at most 2 + 4 + 24 significant bits, so it is exact
 * in float64.  Build with -ffp-contract=off so the result does not depend on
 * whether the host compiler fuses multiply-adds.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NAN_SCALE 2
#define ORACLE_ERR_BAD_ID 3

/* ---------------------------------------------------------------- decode */

/* e2m1 (FP4): bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: value = mantissa * 0.5.
 * Otherwise value = 2^(exp-1) * (1 + mantissa/2). */
double oracle_e2m1_value(uint8_t nibble) {
  int sign = (nibble >> 3) & 1;
  int exp_field = (nibble >> 1) & 3;
  int mant = nibble & 1;
  double mag;
  if (exp_field == 0)
    mag = 0.5 * (double)mant;
  else
    mag = ldexp(1.0 + 0.5 * (double)mant, exp_field - 1);
  return sign ? -mag : mag;
}

/* e4m3 ("fn" variant): bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa.  Exponent field 0 is subnormal: value = mantissa/8 * 2^-6.
 * Exponent 15 with mantissa 7 (bytes 0x7F, 0xFF) is NaN; there are no
 * infinities, so the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_value(uint8_t byte) {
  int sign = (byte >> 7) & 1;
  int exp_field = (byte >> 3) & 15;
  int mant = byte & 7;
  double mag;
  if (exp_field == 15 && mant == 7) return NAN;
  if (exp_field == 0)
    mag = ldexp((double)mant / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)mant / 8.0, exp_field - 7);
  return sign ? -mag : mag;
}

/* e8m0 (the MX scale type, OCP Microscaling Formats spec): an unsigned
 * biased exponent, value = 2^(byte - 127); byte 0xFF is NaN. */
double oracle_e8m0_value(uint8_t byte) {
  if (byte == 0xFF) return NAN;
  return ldexp(1.0, (int)byte - 127);
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double oracle_bf16_value(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Bytes of one canonical NVFP4 expert (gate [I][H], up [I][H], down [H][I]):
 * codes + scale bytes + two fp32 per matrix.  The K3 shape (H 3584, I 3072)
 * must give the 18,579,480 bytes per routed expert printed in "Kimi-K3 on the
 * same pod, two engines", section "Same hardware, same weights". */
uint64_t oracle_expert_bytes(int64_t hidden, int64_t inter) {
  uint64_t per_matrix_elems = (uint64_t)hidden * (uint64_t)inter;
  uint64_t one = per_matrix_elems / 2 + per_matrix_elems / 16 + 2 * 4;
  return 3 * one;
}

/* Value tables filled from the two decode functions above (16 and 256
 * entries), so the matrix loops below look values up instead of calling
 * ldexp per element.  Same numbers, exactly. */
static double e2m1_table[16];
static double e4m3_table[256];
static int tables_ready = 0;

static void init_tables(void) {
  if (tables_ready) return;
  for (int i = 0; i < 16; i++) e2m1_table[i] = oracle_e2m1_value((uint8_t)i);
  for (int i = 0; i < 256; i++) e4m3_table[i] = oracle_e4m3_value((uint8_t)i);
  tables_ready = 1;
}

/* The two 4-bit weight formats.  Both store one e2m1 code per element, two
 * per byte, the low nibble holding the even element, and multiply the whole
 * matrix by the fp32 tensor scale g:
 *   NVFP4: one e4m3 scale per 16 consecutive elements along K
 *          (scales [rows][K/16]);
 *   MXFP4: one e8m0 scale per 32 consecutive elements along K
 *          (scales [rows][K/32]; OCP MX, the format of the ggml microbench in
 *          "Kimi-K3 on 2x A40 - measured findings", section "Why the
 *          placement experiments all looked the same"). */
#define ORACLE_FMT_NVFP4 0
#define ORACLE_FMT_MXFP4 1

static int fmt_block(int fmt) { return fmt == ORACLE_FMT_MXFP4 ? 32 : 16; }

static double fmt_scale(int fmt, uint8_t b) {
  return fmt == ORACLE_FMT_MXFP4 ? oracle_e8m0_value(b) : e4m3_table[b];
}

/* Weight (r, k) of one matrix [rows][K]:
 *   code  = nibble k%2 (low nibble for even k) of codes[r*K/2 + k/2]
 *   scale = scales[r*K/B + k/B]   (B = 16 for NVFP4, 32 for MXFP4)
 *   w     = e2m1(code) * scale * g                                           */
static double fp4_weight(int fmt, const uint8_t *codes, const uint8_t *scales, float g,
                         int64_t K, int64_t r, int64_t k) {
  const int B = fmt_block(fmt);
  uint8_t byte = codes[r * (K / 2) + k / 2];
  uint8_t nibble = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  uint8_t sbyte = scales[r * (K / B) + k / B];
  return e2m1_table[nibble] * fmt_scale(fmt, sbyte) * (double)g;
}

/* 1 if any of the n scale bytes is a NaN of the format. */
static int fmt_has_nan(int fmt, const uint8_t *scales, int64_t n) {
  for (int64_t i = 0; i < n; i++)
    if (isnan(fmt_scale(fmt, scales[i]))) return 1;
  return 0;
}

/* Dense float64 copy of one matrix: out[rows][K].  Returns
 * ORACLE_ERR_NAN_SCALE if any scale byte is NaN. */
int oracle_dequant_fmt(int fmt, const uint8_t *codes, const uint8_t *scales, float g,
                       int64_t rows, int64_t K, double *out) {
  if ((fmt != ORACLE_FMT_NVFP4 && fmt != ORACLE_FMT_MXFP4) || !codes || !scales || !out || rows < 0 || K <= 0 ||
      K % fmt_block(fmt) != 0)
    return ORACLE_ERR_ARG;
  init_tables();
  if (fmt_has_nan(fmt, scales, rows * (K / fmt_block(fmt)))) return ORACLE_ERR_NAN_SCALE;
  for (int64_t r = 0; r < rows; r++)
    for (int64_t k = 0; k < K; k++)
      out[r * K + k] = fp4_weight(fmt, codes, scales, g, K, r, k);
  return ORACLE_OK;
}

int oracle_dequant(const uint8_t *codes, const uint8_t *scales, float g,
                   int64_t rows, int64_t K, double *out) {
  return oracle_dequant_fmt(ORACLE_FMT_NVFP4, codes, scales, g, rows, K, out);
}

/* ---------------------------------------------------------------- router */

/* Router logits l[t][e] = sum_j Wr[e][j] * x[t][j] (+ bias[e]); Wr is fp32
 * [E][H], x is bf16 [C][H], bias is fp32 [E] or NULL.  The router is
 * replicated and identical on every rank ("SparkInfer-K3", "How the TP module
 * works"). */
int oracle_router_logits(int C, int E, int H, const float *Wr,
                         const uint16_t *x, const float *bias,
                         double *logits) {
  if (C < 0 || E <= 0 || H <= 0 || !Wr || !x || !logits) return ORACLE_ERR_ARG;
  for (int t = 0; t < C; t++)
    for (int e = 0; e < E; e++) {
      double s = 0.0;
      for (int j = 0; j < H; j++)
        s += (double)Wr[(int64_t)e * H + j] *
             oracle_bf16_value(x[(int64_t)t * H + j]);
      if (bias) s += (double)bias[e];
      logits[(int64_t)t * E + e] = s;
    }
  return ORACLE_OK;
}

/* Top-k routing of one token's logits l[0..E-1]:
 *   p = softmax(l) over all E experts (computed as exp(l - max l) / sum);
 *   the k experts with the largest logits are kept, equal logits ranked by
 *   lower expert index first;
 *   w_i = p_i / sum over the kept experts of p_j.
 * Output: ids in ascending expert order with their weights, and the boundary
 * gap l_(k) - l_(k+1) between the k-th and (k+1)-th ranked logits (+inf when
 * k == E).  The kept set is plain selection: k passes, each taking the best
 * remaining expert by (logit descending, index ascending). */
int oracle_route(int C, int E, int k, const double *logits, int32_t *ids,
                 double *weights, double *gap) {
  if (C < 0 || E <= 0 || k <= 0 || k > E || !logits || !ids || !weights)
    return ORACLE_ERR_ARG;
  unsigned char *taken = (unsigned char *)malloc((size_t)E);
  double *p = (double *)malloc(sizeof(double) * (size_t)E);
  if (!taken || !p) {
    free(taken);
    free(p);
    return ORACLE_ERR_ARG;
  }
  for (int t = 0; t < C; t++) {
    const double *l = logits + (int64_t)t * E;
    double lmax = l[0];
    for (int e = 1; e < E; e++)
      if (l[e] > lmax) lmax = l[e];
    double z = 0.0;
    for (int e = 0; e < E; e++) {
      p[e] = exp(l[e] - lmax);
      z += p[e];
    }
    for (int e = 0; e < E; e++) p[e] /= z;

    memset(taken, 0, (size_t)E);
    double kth = 0.0;
    for (int r = 0; r < k; r++) {
      int best = -1;
      for (int e = 0; e < E; e++) {
        if (taken[e]) continue;
        if (best < 0 || l[e] > l[best]) best = e; /* strict '>' keeps the lower index on ties */
      }
      taken[best] = 1;
      kth = l[best];
    }
    if (gap) {
      if (k == E) {
        gap[t] = INFINITY;
      } else {
        int next = -1;
        for (int e = 0; e < E; e++) {
          if (taken[e]) continue;
          if (next < 0 || l[e] > l[next]) next = e;
        }
        gap[t] = kth - l[next];
      }
    }
    double psel = 0.0;
    for (int e = 0; e < E; e++)
      if (taken[e]) psel += p[e];
    int n = 0;
    for (int e = 0; e < E; e++) /* ascending expert id */
      if (taken[e]) {
        ids[(int64_t)t * k + n] = e;
        weights[(int64_t)t * k + n] = p[e] / psel;
        n++;
      }
  }
  free(taken);
  free(p);
  return ORACLE_OK;
}

/* ------------------------------------------------------------ expert FFN */

static double silu(double v) { return v / (1.0 + exp(-v)); }

/* One expert's SwiGLU FFN on a float64 input vector x[H]:
 *   g = G x, u = U x         (G, U: [I][H])
 *   a = silu(g) * u
 *   y = D a                  (D: [H][I])
 * with the matrices in format `fmt`.  Shapes from "SparkInfer-K3", "The
 * model": the expert reads and writes the 3584-wide latent space and is 3072
 * wide inside. */
int oracle_expert_ffn_fmt(int fmt, int H, int I,
                          const uint8_t *gate_codes, const uint8_t *gate_scales, float gate_g,
                          const uint8_t *up_codes, const uint8_t *up_scales, float up_g,
                          const uint8_t *down_codes, const uint8_t *down_scales, float down_g,
                          const double *x, double *y) {
  if (fmt != ORACLE_FMT_NVFP4 && fmt != ORACLE_FMT_MXFP4) return ORACLE_ERR_ARG;
  const int B = fmt_block(fmt);
  if (H <= 0 || I <= 0 || H % B || I % B || !x || !y) return ORACLE_ERR_ARG;
  init_tables();
  if (fmt_has_nan(fmt, gate_scales, (int64_t)I * (H / B)) || fmt_has_nan(fmt, up_scales, (int64_t)I * (H / B)) ||
      fmt_has_nan(fmt, down_scales, (int64_t)H * (I / B)))
    return ORACLE_ERR_NAN_SCALE;
  double *a = (double *)malloc(sizeof(double) * (size_t)I);
  if (!a) return ORACLE_ERR_ARG;
  for (int r = 0; r < I; r++) {
    double g = 0.0, u = 0.0;
    for (int k = 0; k < H; k++) {
      g += fp4_weight(fmt, gate_codes, gate_scales, gate_g, H, r, k) * x[k];
      u += fp4_weight(fmt, up_codes, up_scales, up_g, H, r, k) * x[k];
    }
    a[r] = silu(g) * u;
  }
  for (int r = 0; r < H; r++) {
    double s = 0.0;
    for (int k = 0; k < I; k++)
      s += fp4_weight(fmt, down_codes, down_scales, down_g, I, r, k) * a[k];
    y[r] = s;
  }
  free(a);
  return ORACLE_OK;
}

int oracle_expert_ffn(int H, int I,
                      const uint8_t *gate_codes, const uint8_t *gate_scales, float gate_g,
                      const uint8_t *up_codes, const uint8_t *up_scales, float up_g,
                      const uint8_t *down_codes, const uint8_t *down_scales, float down_g,
                      const double *x, double *y) {
  return oracle_expert_ffn_fmt(ORACLE_FMT_NVFP4, H, I, gate_codes, gate_scales, gate_g, up_codes, up_scales, up_g,
                               down_codes, down_scales, down_g, x, y);
}

int oracle_expert_ffn_w4a4(int H, int I,
                           const uint8_t *gate_codes, const uint8_t *gate_scales, float gate_g,
                           const uint8_t *up_codes, const uint8_t *up_scales, float up_g,
                           const uint8_t *down_codes, const uint8_t *down_scales, float down_g,
                           float a_in, float a_dn, const double *x, double *y, double *act_out);

/* Everything one token needs: the arguments of oracle_moe_forward.  With
 * down_a set the experts run with W4A4 numerics (oracle_expert_ffn_w4a4):
 * x is quantized with max(gate_a[e], up_a[e]) and h with down_a[e]; act, when
 * set, receives every pair's float64 activation [C * k][I]. */
typedef struct {
  int fmt;
  int C, E, k, H, I;
  const uint8_t *gate_codes, *gate_scales;
  const float *gate_g;
  const uint8_t *up_codes, *up_scales;
  const float *up_g;
  const uint8_t *down_codes, *down_scales;
  const float *down_g;
  const uint16_t *x;
  const int32_t *ids;
  const double *w;
  double *y;
  const float *gate_a, *up_a, *down_a;
  double *act;
} forward_args;

/* The FFN of expert e on x, in the numerics the arguments select; pair is
 * the (token, slot) index that names the act row. */
static int run_expert(const forward_args *a, int e, int64_t pair, const double *x, double *y) {
  const int H = a->H, I = a->I, B = fmt_block(a->fmt);
  const int64_t gu_codes = (int64_t)I * H / 2, gu_scales = (int64_t)I * H / B;
  const int64_t dn_codes = (int64_t)H * I / 2, dn_scales = (int64_t)H * I / B;
  if (a->down_a) {
    const float ain = a->gate_a[e] > a->up_a[e] ? a->gate_a[e] : a->up_a[e];
    return oracle_expert_ffn_w4a4(H, I, a->gate_codes + e * gu_codes, a->gate_scales + e * gu_scales, a->gate_g[e],
                                  a->up_codes + e * gu_codes, a->up_scales + e * gu_scales, a->up_g[e],
                                  a->down_codes + e * dn_codes, a->down_scales + e * dn_scales, a->down_g[e],
                                  ain, a->down_a[e], x, y, a->act ? a->act + pair * I : NULL);
  }
  return oracle_expert_ffn_fmt(a->fmt, H, I, a->gate_codes + e * gu_codes, a->gate_scales + e * gu_scales,
                               a->gate_g[e], a->up_codes + e * gu_codes, a->up_scales + e * gu_scales, a->up_g[e],
                               a->down_codes + e * dn_codes, a->down_scales + e * dn_scales, a->down_g[e], x, y);
}

/* y[t] of one token, with the scratch vectors xt[H] and ye[H]. */
static int forward_token(const forward_args *a, int t, double *xt, double *ye) {
  const int H = a->H, k = a->k;
  for (int j = 0; j < H; j++) xt[j] = oracle_bf16_value(a->x[(int64_t)t * H + j]);
  for (int j = 0; j < H; j++) a->y[(int64_t)t * H + j] = 0.0;
  for (int i = 0; i < k; i++) {
    int e = a->ids[(int64_t)t * k + i];
    if (e < 0 || e >= a->E) return ORACLE_ERR_BAD_ID;
    int rc = run_expert(a, e, (int64_t)t * k + i, xt, ye);
    if (rc != ORACLE_OK) return rc;
    double wi = a->w[(int64_t)t * k + i];
    for (int j = 0; j < H; j++) a->y[(int64_t)t * H + j] += wi * ye[j];
  }
  return ORACLE_OK;
}

static int forward_args_ok(const forward_args *a) {
  if (a->fmt != ORACLE_FMT_NVFP4 && a->fmt != ORACLE_FMT_MXFP4) return 0;
  const int B = fmt_block(a->fmt);
  return !(a->C < 0 || a->E <= 0 || a->k <= 0 || a->H <= 0 || a->I <= 0 || a->H % B || a->I % B ||
           !a->x || !a->ids || !a->w || !a->y);
}

/* The routed MoE output of C tokens given their selections:
 *   y[t] = sum_i w[t][i] * FFN_{ids[t][i]}(x[t])
 * Canonical weights are arrays over E experts:
 *   *_codes  [E][rows][K/2], *_scales [E][rows][K/16], *_g [E]
 * (gate/up: rows I, K H; down: rows H, K I).  The sum over i runs in the
 * order the ids are given.  An id outside [0, E) is an error.  The partial
 * sums over disjoint subsets of the selected experts add up to this result
 * ("SparkInfer-K3", "How the TP module works"). */
int oracle_moe_forward_fmt(int fmt, int C, int E, int k, int H, int I,
                           const uint8_t *gate_codes, const uint8_t *gate_scales, const float *gate_g,
                           const uint8_t *up_codes, const uint8_t *up_scales, const float *up_g,
                           const uint8_t *down_codes, const uint8_t *down_scales, const float *down_g,
                           const uint16_t *x, const int32_t *ids, const double *w,
                           double *y) {
  forward_args a = {fmt, C, E, k, H, I, gate_codes, gate_scales, gate_g, up_codes, up_scales, up_g,
                    down_codes, down_scales, down_g, x, ids, w, y, NULL, NULL, NULL, NULL};
  if (!forward_args_ok(&a)) return ORACLE_ERR_ARG;
  double *xt = (double *)malloc(sizeof(double) * (size_t)H);
  double *ye = (double *)malloc(sizeof(double) * (size_t)H);
  if (!xt || !ye) {
    free(xt);
    free(ye);
    return ORACLE_ERR_ARG;
  }
  int rc = ORACLE_OK;
  for (int t = 0; t < C && rc == ORACLE_OK; t++) rc = forward_token(&a, t, xt, ye);
  free(xt);
  free(ye);
  return rc;
}

int oracle_moe_forward(int C, int E, int k, int H, int I,
                       const uint8_t *gate_codes, const uint8_t *gate_scales, const float *gate_g,
                       const uint8_t *up_codes, const uint8_t *up_scales, const float *up_g,
                       const uint8_t *down_codes, const uint8_t *down_scales, const float *down_g,
                       const uint16_t *x, const int32_t *ids, const double *w,
                       double *y) {
  return oracle_moe_forward_fmt(ORACLE_FMT_NVFP4, C, E, k, H, I, gate_codes, gate_scales, gate_g, up_codes,
                                up_scales, up_g, down_codes, down_scales, down_g, x, ids, w, y);
}

/* The same result computed by `nthreads` POSIX threads.  The (token, slot)
 * pairs are dealt out to the threads (pair p = thread, thread + nthreads,
 * ...); each thread runs oracle_expert_ffn for its pairs into a buffer of
 * their outputs, and the calling thread then forms every y[t] exactly as
 * oracle_moe_forward does: from 0, adding w[t][i] * (expert output of slot i)
 * for i = 0, 1, ... .  Same values, same order: the output is bit-for-bit
 * the single-threaded one; the threads only change which core computes which
 * expert output. */
typedef struct {
  const forward_args *a;
  double *ye_all;                      /* [C * k][H] expert outputs of every pair */
  int first, step;
  int rc;
} forward_job;

static void *forward_worker(void *p) {
  forward_job *j = (forward_job *)p;
  const forward_args *a = j->a;
  const int H = a->H, k = a->k;
  double *xt = (double *)malloc(sizeof(double) * (size_t)H);
  j->rc = xt ? ORACLE_OK : ORACLE_ERR_ARG;
  for (int64_t pr = j->first; pr < (int64_t)a->C * k && j->rc == ORACLE_OK; pr += j->step) {
    const int64_t t = pr / k;
    const int e = a->ids[pr];
    if (e < 0 || e >= a->E) {
      j->rc = ORACLE_ERR_BAD_ID;
      break;
    }
    for (int q = 0; q < H; q++) xt[q] = oracle_bf16_value(a->x[t * H + q]);
    j->rc = run_expert(a, e, pr, xt, j->ye_all + pr * H);
  }
  free(xt);
  return NULL;
}

static int forward_mt(forward_args a, int nthreads);

int oracle_moe_forward_mt_fmt(int fmt, int nthreads, int C, int E, int k, int H, int I,
                              const uint8_t *gate_codes, const uint8_t *gate_scales, const float *gate_g,
                              const uint8_t *up_codes, const uint8_t *up_scales, const float *up_g,
                              const uint8_t *down_codes, const uint8_t *down_scales, const float *down_g,
                              const uint16_t *x, const int32_t *ids, const double *w,
                              double *y) {
  forward_args a = {fmt, C, E, k, H, I, gate_codes, gate_scales, gate_g, up_codes, up_scales, up_g,
                    down_codes, down_scales, down_g, x, ids, w, y, NULL, NULL, NULL, NULL};
  return forward_mt(a, nthreads);
}

/* The routed MoE output with W4A4 numerics (NVFP4 weights, activations
 * quantized to NVFP4 with each expert's static input scales, see
 * oracle_expert_ffn_w4a4), on `nthreads` threads as oracle_moe_forward_mt.
 * act, when not NULL, receives the float64 activation of every (token, slot)
 * pair [C * k][I] (rows of skipped slots are left as they were). */
int oracle_moe_forward_w4a4_mt(int nthreads, int C, int E, int k, int H, int I,
                               const uint8_t *gate_codes, const uint8_t *gate_scales, const float *gate_g,
                               const uint8_t *up_codes, const uint8_t *up_scales, const float *up_g,
                               const uint8_t *down_codes, const uint8_t *down_scales, const float *down_g,
                               const float *gate_a, const float *up_a, const float *down_a,
                               const uint16_t *x, const int32_t *ids, const double *w, double *y, double *act) {
  if (!gate_a || !up_a || !down_a) return ORACLE_ERR_ARG;
  forward_args a = {ORACLE_FMT_NVFP4, C, E, k, H, I, gate_codes, gate_scales, gate_g, up_codes, up_scales, up_g,
                    down_codes, down_scales, down_g, x, ids, w, y, gate_a, up_a, down_a, act};
  return forward_mt(a, nthreads);
}

static int forward_mt(forward_args a, int nthreads) {
  const int C = a.C, k = a.k, H = a.H;
  const double *w = a.w;
  double *y = a.y;
  if (!forward_args_ok(&a) || nthreads < 1) return ORACLE_ERR_ARG;
  init_tables();                       /* fill the shared tables before any thread reads them */
  const int64_t npairs = (int64_t)C * k;
  if (nthreads > npairs) nthreads = npairs > 0 ? (int)npairs : 1;
  double *ye_all = (double *)malloc(sizeof(double) * (size_t)(npairs > 0 ? npairs : 1) * (size_t)H);
  pthread_t *tids = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  forward_job *jobs = (forward_job *)malloc(sizeof(forward_job) * (size_t)nthreads);
  if (!ye_all || !tids || !jobs) {
    free(ye_all);
    free(tids);
    free(jobs);
    return ORACLE_ERR_ARG;
  }
  int started = 0;
  for (int i = 0; i < nthreads; i++) {
    jobs[i].a = &a;
    jobs[i].ye_all = ye_all;
    jobs[i].first = i;
    jobs[i].step = nthreads;
    jobs[i].rc = ORACLE_OK;
    if (pthread_create(&tids[i], NULL, forward_worker, &jobs[i]) != 0) break;
    started++;
  }
  for (int i = started; i < nthreads; i++) forward_worker(&jobs[i]);   /* no thread: run it here */
  int rc = ORACLE_OK;
  for (int i = 0; i < nthreads; i++) {
    if (i < started) pthread_join(tids[i], NULL);
    if (jobs[i].rc != ORACLE_OK && rc == ORACLE_OK) rc = jobs[i].rc;
  }
  for (int t = 0; t < C && rc == ORACLE_OK; t++) {
    for (int q = 0; q < H; q++) y[(int64_t)t * H + q] = 0.0;
    for (int i = 0; i < k; i++) {
      const double wi = w[(int64_t)t * k + i];
      const double *ye = ye_all + ((int64_t)t * k + i) * H;
      for (int q = 0; q < H; q++) y[(int64_t)t * H + q] += wi * ye[q];
    }
  }
  free(ye_all);
  free(tids);
  free(jobs);
  return rc;
}

int oracle_moe_forward_mt(int nthreads, int C, int E, int k, int H, int I,
                          const uint8_t *gate_codes, const uint8_t *gate_scales, const float *gate_g,
                          const uint8_t *up_codes, const uint8_t *up_scales, const float *up_g,
                          const uint8_t *down_codes, const uint8_t *down_scales, const float *down_g,
                          const uint16_t *x, const int32_t *ids, const double *w,
                          double *y) {
  return oracle_moe_forward_mt_fmt(ORACLE_FMT_NVFP4, nthreads, C, E, k, H, I, gate_codes, gate_scales, gate_g,
                                   up_codes, up_scales, up_g, down_codes, down_scales, down_g, x, ids, w, y);
}

/* ------------------------------------------------- around the routed sum */

/* Dense 4-bit GEMV of C vectors: y[t][m] = sum_k W[m][k] x[t][k] in float64,
 * W [M][K] in format `fmt` (codes [M][K/2], scales [M][K/B], tensor scale g).
 * The latent projections routed_down (7168 -> 3584) and routed_up
 * (3584 -> 7168) of "SparkInfer-K3", section "How the TP module works"
 * (FfnPartial: router -> routed_down -> experts; FfnFinish: routed_norm ->
 * routed_up -> shared experts), are of this form. */
int oracle_dense_gemv(int fmt, int M, int K, const uint8_t *codes, const uint8_t *scales, float g, int C,
                      const double *x, double *y) {
  if ((fmt != ORACLE_FMT_NVFP4 && fmt != ORACLE_FMT_MXFP4) || M <= 0 || K <= 0 || C < 0 ||
      K % fmt_block(fmt) || !codes || !scales || !x || !y)
    return ORACLE_ERR_ARG;
  init_tables();
  if (fmt_has_nan(fmt, scales, (int64_t)M * (K / fmt_block(fmt)))) return ORACLE_ERR_NAN_SCALE;
  for (int t = 0; t < C; t++)
    for (int m = 0; m < M; m++) {
      double s = 0.0;
      for (int k = 0; k < K; k++) s += fp4_weight(fmt, codes, scales, g, K, m, k) * x[(int64_t)t * K + k];
      y[(int64_t)t * M + m] = s;
    }
  return ORACLE_OK;
}

/* RMS norm of C vectors of length n (routed_norm, "SparkInfer-K3", "How the
 * TP module works": it follows the complete routed sum, because
 * rms_norm(sum of partials) != sum of rms_norm(partials)):
 *   out[t][i] = y[t][i] / sqrt(mean_j y[t][j]^2 + eps) * gamma[i]. */
int oracle_rms_norm(int C, int n, const double *y, const float *gamma, double eps, double *out) {
  if (C < 0 || n <= 0 || !y || !gamma || !out || !(eps >= 0.0)) return ORACLE_ERR_ARG;
  for (int t = 0; t < C; t++) {
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += y[(int64_t)t * n + i] * y[(int64_t)t * n + i];
    const double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int i = 0; i < n; i++) out[(int64_t)t * n + i] = y[(int64_t)t * n + i] * r * (double)gamma[i];
  }
  return ORACLE_OK;
}

/* float64 -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
uint16_t oracle_bf16_round(double v) {
  if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
  const int neg = v < 0.0;
  double a = fabs(v);
  int e;
  frexp(a, &e);                          /* a = m 2^e, m in [0.5, 1) */
  int eb = e - 1;                        /* a in [2^eb, 2^(eb+1)) */
  if (eb < -126) eb = -126;              /* subnormal range: fixed spacing 2^-133 */
  const double ulp = ldexp(1.0, eb - 7);
  double q = a / ulp;                    /* exact: a power-of-two division */
  double r = floor(q);
  const double frac = q - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  const double rv = r * ulp;             /* the rounded magnitude */
  float f = (float)rv;                   /* exact: 8 significant bits */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)((u >> 16) | (neg ? 0x8000u : 0u));
}

/* ------------------------------------------------------ W4A4 activations */

/* Round a non-negative float to e4m3 (nearest, ties to even mantissa, values
 * above the largest finite 448 saturate to 448): the byte. */
static uint8_t e4m3_rne_sat(float v) {
  if (!(v > 0.0f)) return 0;
  if (v >= 448.0f) return 0x7E;
  const double d = (double)v;                  /* exact */
  if (d < 0.015625) {                          /* subnormal: multiples of 2^-9 */
    double q = d * 512.0, r = floor(q), f = q - r;
    if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    return (uint8_t)(r >= 8.0 ? 0x08 : (int)r);  /* 8 * 2^-9 = 2^-6, the smallest normal */
  }
  int ex;
  const double m = frexp(d, &ex);              /* d = m 2^ex, m in [0.5, 1) */
  int e = ex - 1;
  double q = (2.0 * m - 1.0) * 8.0, r = floor(q), f = q - r;
  if (f > 0.5 || (f == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  if (r >= 8.0) { r = 0.0; e += 1; }
  if (e > 8 || (e == 8 && r > 6.0)) return 0x7E;
  return (uint8_t)(((e + 7) << 3) | (int)r);
}

/* Round a float to e2m1 (nearest, ties to even, |v| > 6 saturates to 6): the
 * 4-bit code, sign in bit 3 (a negative value that rounds to zero keeps its
 * sign bit). */
static uint8_t e2m1_rne_sat(float v) {
  const float a = fabsf(v);
  uint8_t mag;
  /* magnitudes 0 0.5 1 1.5 2 3 4 6; midpoints 0.25 0.75 1.25 1.75 2.5 3.5 5,
   * a tie goes to the even mantissa (codes 0, 2, 4, 6) */
  if (a <= 0.25f) mag = 0;
  else if (a < 0.75f) mag = 1;
  else if (a <= 1.25f) mag = 2;
  else if (a < 1.75f) mag = 3;
  else if (a <= 2.5f) mag = 4;
  else if (a < 3.5f) mag = 5;
  else if (a <= 5.0f) mag = 6;
  else mag = 7;
  return (uint8_t)(mag | (signbit(v) ? 8 : 0));
}

/* NVFP4 quantization of an activation vector v[n] (n a multiple of 16) with
 * the static per-tensor input scale a (the second fp32 of a matrix in the
 * NVFP4 checkpoint, "Kimi-K3 on the same pod, two engines", section "Same
 * hardware, same weights": 24 bytes of fp32 scalars per expert), in fp32
 * arithmetic step for step as the GPU does it:
 *   per block of 16: amax = max |v|;  s = e4m3(amax / (6 a))  (the byte);
 *   each element: code = e2m1(v / (e4m3value(s) a));  all-zero block: 0.
 * The dequantized element is e2m1(code) * e4m3value(s) * a.  Codes are
 * packed two per byte, low nibble = even element. */
int oracle_quantize_nvfp4(int n, const float *v, float a, uint8_t *codes, uint8_t *scales) {
  if (n <= 0 || n % 16 || !v || !codes || !scales || !(a > 0.0f)) return ORACLE_ERR_ARG;
  init_tables();
  for (int b = 0; b < n / 16; b++) {
    float amax = 0.0f;
    for (int i = 0; i < 16; i++) amax = fmaxf(amax, fabsf(v[16 * b + i]));
    const float denom = 6.0f * a;
    const float t = amax / denom;
    const uint8_t sb = e4m3_rne_sat(t);
    scales[b] = sb;
    const float sv = (float)e4m3_table[sb];     /* exact in float */
    const float m = sv * a;
    for (int i = 0; i < 16; i += 2) {
      uint8_t c0 = 0, c1 = 0;
      if (sv > 0.0f) {
        c0 = e2m1_rne_sat(v[16 * b + i] / m);
        c1 = e2m1_rne_sat(v[16 * b + i + 1] / m);
      }
      codes[(16 * b + i) / 2] = (uint8_t)(c0 | (c1 << 4));
    }
  }
  return ORACLE_OK;
}

/* The dequantized value of every element of a quantized activation vector:
 * e2m1(code) * e4m3(scale) * a (float64, exact). */
static void dequant_act(int n, const uint8_t *codes, const uint8_t *scales, float a, double *out) {
  for (int k = 0; k < n; k++) {
    const uint8_t byte = codes[k / 2];
    const uint8_t nib = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
    out[k] = e2m1_table[nib] * e4m3_table[scales[k / 16]] * (double)a;
  }
}

/* One expert's FFN with W4A4 numerics (NVFP4 weights and activations):
 *   xq  = Q(x, a_in)                  the input quantized with the gate
 *                                     matrix's input scale (gate and up see
 *                                     the same x)
 *   g = G xq, u = U xq;  act = silu(g) * u    (float64)
 *   aq  = Q((float) act, a_dn)        the down projection's input quantized
 *                                     with the down matrix's input scale
 *   y   = D aq
 * Q is oracle_quantize_nvfp4 followed by the exact dequantization.  The
 * float64 activation silu(g) * u before its rounding to float goes to
 * act_out[I] when act_out is not NULL. */
int oracle_expert_ffn_w4a4(int H, int I,
                           const uint8_t *gate_codes, const uint8_t *gate_scales, float gate_g,
                           const uint8_t *up_codes, const uint8_t *up_scales, float up_g,
                           const uint8_t *down_codes, const uint8_t *down_scales, float down_g,
                           float a_in, float a_dn, const double *x, double *y, double *act_out) {
  if (H <= 0 || I <= 0 || H % 16 || I % 16 || !x || !y || !(a_in > 0.0f) || !(a_dn > 0.0f)) return ORACLE_ERR_ARG;
  init_tables();
  if (fmt_has_nan(ORACLE_FMT_NVFP4, gate_scales, (int64_t)I * (H / 16)) ||
      fmt_has_nan(ORACLE_FMT_NVFP4, up_scales, (int64_t)I * (H / 16)) ||
      fmt_has_nan(ORACLE_FMT_NVFP4, down_scales, (int64_t)H * (I / 16)))
    return ORACLE_ERR_NAN_SCALE;
  float *xf = (float *)malloc(sizeof(float) * (size_t)H);
  double *xq = (double *)malloc(sizeof(double) * (size_t)H);
  float *af = (float *)malloc(sizeof(float) * (size_t)I);
  double *aq = (double *)malloc(sizeof(double) * (size_t)I);
  uint8_t *qc = (uint8_t *)malloc((size_t)(H > I ? H : I) / 2);
  uint8_t *qs = (uint8_t *)malloc((size_t)(H > I ? H : I) / 16);
  int rc = (xf && xq && af && aq && qc && qs) ? ORACLE_OK : ORACLE_ERR_ARG;
  if (rc == ORACLE_OK) {
    for (int k = 0; k < H; k++) xf[k] = (float)x[k];      /* x is bf16: exact */
    oracle_quantize_nvfp4(H, xf, a_in, qc, qs);
    dequant_act(H, qc, qs, a_in, xq);
    for (int r = 0; r < I; r++) {
      double g = 0.0, u = 0.0;
      for (int k = 0; k < H; k++) {
        g += fp4_weight(ORACLE_FMT_NVFP4, gate_codes, gate_scales, gate_g, H, r, k) * xq[k];
        u += fp4_weight(ORACLE_FMT_NVFP4, up_codes, up_scales, up_g, H, r, k) * xq[k];
      }
      const double h = silu(g) * u;
      if (act_out) act_out[r] = h;
      af[r] = (float)h;
    }
    oracle_quantize_nvfp4(I, af, a_dn, qc, qs);
    dequant_act(I, qc, qs, a_dn, aq);
    for (int r = 0; r < H; r++) {
      double s = 0.0;
      for (int k = 0; k < I; k++) s += fp4_weight(ORACLE_FMT_NVFP4, down_codes, down_scales, down_g, I, r, k) * aq[k];
      y[r] = s;
    }
  }
  free(xf); free(xq); free(af); free(aq); free(qc); free(qs);
  return rc;
}
