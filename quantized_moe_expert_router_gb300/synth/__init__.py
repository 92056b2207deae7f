"""Seeded synthetic inputs for the routed NVFP4 MoE layer (host side).

This module serves both the CUDA path and the float64 oracle with the same
inputs.  It holds a counter-based random generator and an NVFP4 *encoder* for
synthetic weights; it holds none of the method's arithmetic (no decode, no
router, no top-k, no FFN).  A device twin in ``synth.cu`` implements the same
generator for the 16.6 GB-per-layer expert weights; the two agree bit for bit
(a GPU test checks it), because every step is an integer operation or a single
correctly rounded IEEE float64 operation.

Generator
  draw(key, i) = splitmix64(key + i * 0x9E3779B97F4A7C15): the i-th output of a
  SplitMix64 stream started at ``key`` (Steele, Lea and Flood, "Fast
  splittable pseudorandom number generators", OOPSLA 2014).  Keys are derived
  from (seed, part, part, ...) by chaining splitmix64 over the parts.

Normal deviates
  z_i = (S_i - 262140) * c, S_i = sum of the eight 16-bit halves of draws 2i and
  2i+1, c = 1/sqrt(8 * (65536^2 - 1) / 12): an Irwin-Hall sum of 8 uniforms,
  standardised.  It is a textbook approximation of N(0,1) (|z| <= 4.899) that
  needs no transcendental function, which is what keeps host and device
  bit-identical.

NVFP4 encoder (weights N(0, 0.02) of one matrix [rows][K], global scale g):
  per 16-element block along K: amax = max|w|; scale byte = e4m3 round-to-
  nearest-even of amax / (6 g) (saturating at 448); s = its value; each code =
  the e2m1 value nearest to w / (s g) (ties to the even mantissa, saturating at
  6), found by comparing |w| with the midpoints times s*g, products that are
  exact in float64.  Low nibble = even element.
"""
from __future__ import annotations

import math

import numpy as np

MASK64 = (1 << 64) - 1
GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB

# 1/sqrt(variance of the sum of 8 uniform 16-bit integers) and the weight
# standard deviation 0.02 folded in.
IH8_CENTER = 8 * 65535 // 2 * 1.0          # 262140.0
IH8_INV_SD = 1.0 / math.sqrt(8 * (65536 ** 2 - 1) / 12)
WEIGHT_STD = 0.02
W_COEF = WEIGHT_STD * IH8_INV_SD          # multiplies (S - 262140) to give w
W_ABS_MAX = 262140.0 * W_COEF             # largest |w| the generator can emit
X_ABS_MAX = 262140.0 * IH8_INV_SD         # largest |z| of a standard deviate (4.899)

# Key kinds (first part after the seed).
KIND_WEIGHT = 1
KIND_ROUTER = 2
KIND_X = 3
KIND_BIAS_PERM = 4
KIND_GSCALE = 5
KIND_DRAFT = 6
KIND_FFN = 7            # the weights around the routed sum (latent projections, shared experts, norm)

FFN_ROUTED_DOWN, FFN_ROUTED_UP, FFN_SHARED, FFN_GAMMA = 0, 1, 2, 3

MAT_GATE, MAT_UP, MAT_DOWN = 0, 1, 2

# e2m1 rounding midpoints in units of s*g and the e4m3 encoder limits.
_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)
_E4M3_MAX = 448.0


def splitmix64_int(z: int) -> int:
    z = (z + GOLDEN) & MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def key(seed: int, *parts: int) -> int:
    """Stream key for (seed, parts...): splitmix64 chained over the parts."""
    h = splitmix64_int(seed & MASK64)
    for p in parts:
        h = splitmix64_int(h ^ (p & MASK64))
    return h


def draws(k: int, start: int, count: int) -> np.ndarray:
    """uint64 draws i = start .. start+count-1 of the stream with key k."""
    i = np.arange(start, start + count, dtype=np.uint64)
    z = np.uint64(k) + i * np.uint64(GOLDEN) + np.uint64(GOLDEN)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(M2)
    return z ^ (z >> np.uint64(31))


def _ih8_sum(k: int, count: int) -> np.ndarray:
    d = draws(k, 0, 2 * count).reshape(count, 2)
    s = np.zeros(count, np.int64)
    for j in range(2):
        a = d[:, j]
        for sh in (0, 16, 32, 48):
            s += ((a >> np.uint64(sh)) & np.uint64(0xFFFF)).astype(np.int64)
    return s


def normals(k: int, count: int) -> np.ndarray:
    """float64 standard-normal-like deviates z_0..z_{count-1} of stream k."""
    return (_ih8_sum(k, count).astype(np.float64) - IH8_CENTER) * IH8_INV_SD


def uniforms(k: int, count: int) -> np.ndarray:
    """float64 uniforms in [0, 1) with 53 random bits."""
    return (draws(k, 0, count) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


# ----------------------------------------------------------------- encoders

def e4m3_encode(v: np.ndarray):
    """Round non-negative float64 values to e4m3 (nearest, ties to even mantissa,
    saturating at 448).  Returns (codes uint8, exact values float64)."""
    v = np.asarray(v, np.float64)
    code = np.zeros(v.shape, np.int64)
    val = np.zeros(v.shape, np.float64)
    sat = v >= _E4M3_MAX
    sub = v < 2.0 ** -6
    nrm = ~sat & ~sub
    # subnormal range: multiples of 2^-9
    q = np.rint(v[sub] * 512.0).astype(np.int64)
    code[sub] = np.where(q >= 8, 0x08, q)
    val[sub] = np.where(q >= 8, 2.0 ** -6, q * 2.0 ** -9)
    # normal range
    m, ex = np.frexp(v[nrm])                  # v = m * 2^ex, m in [0.5, 1)
    e = ex.astype(np.int64) - 1               # v = (2m) * 2^e, 2m in [1, 2)
    q = np.rint((2.0 * m - 1.0) * 8.0).astype(np.int64)
    carry = q >= 8
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 0, q)
    over = e > 8
    code[nrm] = np.where(over, 0x7E, ((e + 7) << 3) | q)
    val[nrm] = np.where(over, _E4M3_MAX, np.ldexp(1.0 + q / 8.0, e))
    code[sat] = 0x7E
    val[sat] = _E4M3_MAX
    return code.astype(np.uint8), val


def e2m1_encode(w: np.ndarray, sg: np.ndarray) -> np.ndarray:
    """Nearest e2m1 code to w / sg (sg > 0), ties to even mantissa, saturating,
    decided by exact comparisons of |w| with midpoint * sg.  Returns uint8 codes
    0..15 (bit 3 = sign)."""
    a = np.abs(w)
    t = [m * sg for m in _E2M1_MIDPOINTS]
    mag = np.full(a.shape, 7, np.int64)
    mag = np.where(a <= t[6], 6, mag)
    mag = np.where(a < t[5], 5, mag)
    mag = np.where(a <= t[4], 4, mag)
    mag = np.where(a < t[3], 3, mag)
    mag = np.where(a <= t[2], 2, mag)
    mag = np.where(a < t[1], 1, mag)
    mag = np.where(a <= t[0], 0, mag)
    neg = (w < 0) & (mag != 0)
    return (mag | np.where(neg, 8, 0)).astype(np.uint8)


def quantize_nvfp4(w: np.ndarray, g: float):
    """Encode float64 weights [rows][K] with global scale g into canonical
    NVFP4: codes uint8 [rows][K/2] (low nibble = even k), scales uint8
    [rows][K/16]."""
    rows, K = w.shape
    blk = w.reshape(rows, K // 16, 16)
    amax = np.abs(blk).max(axis=2)
    g64 = float(np.float32(g))
    scode, sval = e4m3_encode(amax / (6.0 * g64))
    scode = np.where(amax == 0.0, 0, scode).astype(np.uint8)
    sval = np.where(amax == 0.0, 0.0, sval)
    sg = (sval * g64)[:, :, None]
    codes = np.where(sg > 0.0, e2m1_encode(blk, np.where(sg > 0.0, sg, 1.0)), 0).astype(np.uint8)
    codes = codes.reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, scode


def quantize_mxfp4(w: np.ndarray):
    """Encode float64 weights [rows][K] into canonical MXFP4 (OCP MX): per
    32-element block along K a shared e8m0 scale 2^e with e = floor(log2 amax)
    - 2 (the spec's rule: the exponent of amax minus e2m1's largest exponent,
    clamped to [-127, 127]; an all-zero block gets e = -127), and codes = the
    e2m1 value nearest to w / 2^e (ties to even, saturating at 6).  Returns
    codes uint8 [rows][K/2] (low nibble = even k) and scales uint8 [rows][K/32]
    (byte = e + 127)."""
    rows, K = w.shape
    blk = w.reshape(rows, K // 32, 32)
    amax = np.abs(blk).max(axis=2)
    _, ex = np.frexp(amax)                        # amax = m 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1
    e = np.where(amax > 0.0, ex.astype(np.int64) - 1 - 2, -127)
    e = np.clip(e, -127, 127)
    sc = np.ldexp(1.0, e)[:, :, None]
    codes = e2m1_encode(blk, sc).reshape(rows, K)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (e + 127).astype(np.uint8)


# ------------------------------------------------------------ layer inputs

def global_scales(seed: int, layer: int, E: int, H: int):
    """Per-(expert, matrix) fp32 weight scales g and input scales a.

    g = (W_ABS_MAX / (6 * 448)) * (1 + 0.5 u): the block scale never saturates
    and each matrix gets its own g.

    a is the static activation scale a calibration pass would store: the
    calibrated largest |input| over 6 * 448, so that an input block whose
    largest element reaches that bound gets the largest e4m3 block scale.
      gate, up: the input x is N(0, 1) with |x| <= X_ABS_MAX (the Irwin-Hall
                bound); a = X_ABS_MAX / (6 * 448) * (1 + 0.25 u), the same
                value for gate and up (they read the same input);
      down:     the input h = silu(g) u with g, u of standard deviation
                sigma = WEIGHT_STD sqrt(H) (H products of N(0, 0.02^2)
                weights with N(0, 1) inputs); a = 16 sigma^2 / (6 * 448) *
                (1 + 0.25 u), so |h| saturates only far in the tails.
    Only W4A4 layers use a.  Returns float32 arrays g[3][E], a[3][E]."""
    u = uniforms(key(seed, KIND_GSCALE, layer), 6 * E).reshape(6, E)
    base = W_ABS_MAX / (6.0 * _E4M3_MAX)
    g = (base * (1.0 + 0.5 * u[:3])).astype(np.float32)
    sigma2 = WEIGHT_STD * WEIGHT_STD * H
    a_x = (X_ABS_MAX / (6.0 * _E4M3_MAX)) * (1.0 + 0.25 * u[3])
    a_h = (16.0 * sigma2 / (6.0 * _E4M3_MAX)) * (1.0 + 0.25 * u[5])
    a = np.stack([a_x, a_x, a_h]).astype(np.float32)
    return g, a


def weight_key(seed: int, layer: int, expert: int, mat: int) -> int:
    return key(seed, KIND_WEIGHT, layer, expert, mat)


def expert_matrix(seed: int, layer: int, expert: int, mat: int, rows: int, K: int, g: float, fmt="nvfp4"):
    """Canonical (codes, scales) of one matrix of one expert: NVFP4 with
    global scale g, or MXFP4 (no global scale; the weights are the same draws)."""
    k = weight_key(seed, layer, expert, mat)
    w = (_ih8_sum(k, rows * K).astype(np.float64) - IH8_CENTER) * W_COEF
    if fmt == "mxfp4":
        return quantize_mxfp4(w.reshape(rows, K))
    return quantize_nvfp4(w.reshape(rows, K), g)


def canonical_layer(seed: int, layer: int, E: int, H: int, I: int, experts=None, fmt="nvfp4"):
    """Host-generated canonical layer, NVFP4 or MXFP4.

    Returns dict gate/up/down -> {'codes', 'scales', 'g', 'a'} with codes
    [n][rows][K/2], scales [n][rows][K/16] (NVFP4) or [n][rows][K/32] (MXFP4),
    g/a [n] for the experts listed (all E by default), in that order.  MXFP4
    matrices carry the tensor scale g = 1."""
    experts = list(range(E)) if experts is None else list(experts)
    g, a = global_scales(seed, layer, E, H)
    if fmt == "mxfp4":
        g = np.ones_like(g)
    blk = 32 if fmt == "mxfp4" else 16
    out = {}
    for mat, name, rows, K in ((MAT_GATE, "gate", I, H), (MAT_UP, "up", I, H), (MAT_DOWN, "down", H, I)):
        codes = np.empty((len(experts), rows, K // 2), np.uint8)
        scales = np.empty((len(experts), rows, K // blk), np.uint8)
        for j, e in enumerate(experts):
            codes[j], scales[j] = expert_matrix(seed, layer, e, mat, rows, K, float(g[mat][e]), fmt)
        out[name] = {"codes": codes, "scales": scales,
                     "g": g[mat][experts].copy(), "a": a[mat][experts].copy()}
    return out


def ffn_matrix(seed: int, layer: int, part: int, idx: int, rows: int, K: int, fmt="nvfp4"):
    """One N(0, 0.02) matrix [rows][K] of the FFN around the routed sum,
    quantized like the expert weights: (codes, scales, g).  NVFP4 gets a
    global scale g that keeps block scales unsaturated; MXFP4 g = 1."""
    k = key(seed, KIND_FFN, layer, part, idx)
    w = ((_ih8_sum(k, rows * K).astype(np.float64) - IH8_CENTER) * W_COEF).reshape(rows, K)
    if fmt == "mxfp4":
        c, sc = quantize_mxfp4(w)
        return c, sc, np.float32(1.0)
    g = np.float32(W_ABS_MAX / (6.0 * _E4M3_MAX) * (1.0 + 0.25 * (idx % 3)))
    c, sc = quantize_nvfp4(w, float(g))
    return c, sc, g


def ffn_weights(seed: int, layer: int, hidden: int, latent: int, shared: int, shared_inter: int,
                fmt="nvfp4", eps: float = 1e-6) -> dict:
    """Host-generated weights around the routed sum of one layer:
    routed_down [latent][hidden], routed_up [hidden][latent] (each
    {'codes','scales','g','a'}), 'shared' = gate/up [S][Is][hidden] and down
    [S][hidden][Is] in the routed experts' dict form, 'gamma' float32 [latent]
    = 1 + 0.1 z, and 'eps'."""
    def mat(part, idx, rows, K):
        c, sc, g = ffn_matrix(seed, layer, part, idx, rows, K, fmt)
        return {"codes": c, "scales": sc, "g": np.float32(g), "a": np.float32(1.0)}
    out = {"routed_down": mat(FFN_ROUTED_DOWN, 0, latent, hidden),
           "routed_up": mat(FFN_ROUTED_UP, 0, hidden, latent)}
    sh = {}
    for m, name, rows, K in ((0, "gate", shared_inter, hidden), (1, "up", shared_inter, hidden),
                             (2, "down", hidden, shared_inter)):
        ms = [mat(FFN_SHARED, 3 * s + m, rows, K) for s in range(shared)]
        blk = 32 if fmt == "mxfp4" else 16
        empty = {"codes": np.zeros((0, rows, K // 2), np.uint8), "scales": np.zeros((0, rows, K // blk), np.uint8),
                 "g": np.zeros(0, np.float32), "a": np.zeros(0, np.float32)}
        sh[name] = {f: np.stack([q[f] for q in ms]) if ms else empty[f] for f in ("codes", "scales", "g", "a")}
    out["shared"] = sh
    z = normals(key(seed, KIND_FFN, layer, FFN_GAMMA, 0), latent)
    out["gamma"] = (1.0 + 0.1 * z).astype(np.float32)
    out["eps"] = eps
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """float64 -> float32 (nearest) -> bfloat16 bits (nearest, ties to even)."""
    f = np.asarray(v, np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def tokens(seed: int, layer: int, C: int, H: int, attempts=None) -> np.ndarray:
    """x bf16 bits [C][H], N(0,1).  Token t uses stream (seed, X, layer, t,
    attempts[t]); a caller that needs a different draw for one token bumps its
    attempt number."""
    attempts = [0] * C if attempts is None else attempts
    x = np.empty((C, H), np.uint16)
    for t in range(C):
        x[t] = f64_to_bf16_bits(normals(key(seed, KIND_X, layer, t, attempts[t]), H))
    return x


def draft_rows(seed: int, layer: int, r: int, H: int, rho: float = 0.95, attempts=None) -> np.ndarray:
    """x bf16 bits [r][H] of r draft rows of one stream: row j is
    sqrt(rho) b + sqrt(1 - rho) z_j with b and z_j N(0,1) vectors (b shared by
    the rows, stream (seed, DRAFT, layer, 0); z_j from stream (seed, DRAFT,
    layer, 1 + j, attempts[j])), so the rows are N(0,1) with pairwise
    correlation rho and their top-k expert sets overlap."""
    attempts = [0] * r if attempts is None else attempts
    b = normals(key(seed, KIND_DRAFT, layer, 0), H)
    x = np.empty((r, H), np.uint16)
    for j in range(r):
        z = normals(key(seed, KIND_DRAFT, layer, 1 + j, attempts[j]), H)
        x[j] = f64_to_bf16_bits(math.sqrt(rho) * b + math.sqrt(1.0 - rho) * z)
    return x


def router_weights(seed: int, layer: int, E: int, H: int, std: float = 1.0) -> np.ndarray:
    """Wr float32 [E][H] with entries N(0, std^2 / H): logits of N(0,1) tokens
    then have standard deviation about ``std``."""
    z = normals(key(seed, KIND_ROUTER, layer), E * H).reshape(E, H)
    return (z * (std / math.sqrt(H))).astype(np.float32)


def zipf_bias(seed: int, layer: int, E: int, s: float = 1.1) -> np.ndarray:
    """Router bias b_e = ln p_{pi(e)}, p_r proportional to r^-s over ranks
    r = 1..E, pi a seeded permutation of the experts per layer."""
    r = np.arange(1, E + 1, dtype=np.float64)
    p = r ** -s
    p /= p.sum()
    order = np.argsort(draws(key(seed, KIND_BIAS_PERM, layer), 0, E), kind="stable")
    rank_of = np.empty(E, np.int64)
    rank_of[order] = np.arange(E)
    return np.log(p[rank_of]).astype(np.float32)


# The logit noise standard deviation that makes "bias + noise" behave like a
# Gumbel-perturbed Plackett-Luce draw: the Gumbel distribution's standard
# deviation is pi / sqrt(6).
ZIPF_ROUTER_STD = math.pi / math.sqrt(6.0)
