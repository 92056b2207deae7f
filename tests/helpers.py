"""Shared helpers of the test suite: tolerance checks, gap-enforced token
generation (via the oracle), and GPU layer set-up through the C ABI."""
from __future__ import annotations

import numpy as np

import oracle
from quantized_moe_expert_router_gb300 import synth

# Acceptance tolerance of the routed output against the float64 oracle:
# max |y - y_o| <= 2e-3 * max|y_o| and ||y - y_o||_2 <= 5e-4 ||y_o||_2;
# selected ids bit-exact given a logit gap >= 1e-3 at the k-th boundary.
MAX_ABS_REL = 2e-3
REL_L2 = 5e-4
MIN_GAP = 1e-3


def assert_close(y, y_ref, label=""):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    assert np.isfinite(y).all(), f"{label}: non-finite output"
    scale = np.abs(y_ref).max()
    err = np.abs(y - y_ref).max()
    l2 = np.linalg.norm(y - y_ref) / max(np.linalg.norm(y_ref), 1e-300)
    assert err <= MAX_ABS_REL * scale, f"{label}: max err {err:.3e} > {MAX_ABS_REL} * {scale:.3e}"
    assert l2 <= REL_L2, f"{label}: rel L2 {l2:.3e} > {REL_L2}"
    return err / max(scale, 1e-300), l2


def gapped_tokens(seed, layer, C, H, Wr, k, bias=None, min_gap=MIN_GAP, max_attempts=200, draft_rho=None):
    """x (bf16 bits [C][H]) whose oracle top-k boundary gap is >= min_gap for
    every token: a token that misses it is redrawn from its next attempt.
    With ``draft_rho`` the rows are draft rows of one stream
    (``synth.draft_rows``, pairwise correlation draft_rho)."""
    attempts = [0] * C

    def draw():
        if draft_rho is None:
            return synth.tokens(seed, layer, C, H, attempts)
        return synth.draft_rows(seed, layer, C, H, draft_rho, attempts)
    x = draw()
    for _ in range(max_attempts):
        _, _, gap = oracle.route(oracle.router_logits(Wr, x, bias), k)
        bad = [t for t in range(C) if gap[t] < min_gap]
        if not bad:
            return x
        for t in bad:
            attempts[t] += 1
        x = draw()
    raise RuntimeError("could not draw tokens with the required logit gap")


def golden_figures(name="k3_figures.txt"):
    """Parse a `name = value ; page ; section` fixture under tests/golden."""
    import os
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)
    out = {}
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split("=", 1)
            value = rest.split(";", 1)[0].strip()
            out[key.strip()] = float(value) if "." in value else int(value)
    return out


# W4A4 tolerance.  With activations quantized to NVFP4 the GPU and the oracle
# take the same fp32 decisions on the same inputs for x (bit-exact codes), but
# h = silu(g) u reaches the quantizer through different summation orders
# (fp32 tensor-core accumulation against float64), so an element of h that
# lies within that rounding noise of an e2m1 tie, or a block whose
# max|h| / (6 a) lies within it of an e4m3 tie, may be quantized to the
# neighbouring value on one side only.  W4A4_EPS bounds that noise relative
# to the block's max |h|: 2^-12, about 60 times the typical fp32 error of a
# 3584-term dot product (2^-24 * sqrt(3584) ~ 3.6e-6 of the terms' scale).
# For each element that close to a tie the allowance adds, to every output
# of its token, router weight * |D[:, j]| * (distance between the two
# candidate values); a block with an ambiguous scale counts every element
# with the bound (s_lo + s_hi) a <= 2 s_hi a on the change of its value.
W4A4_EPS = 2.0 ** -12
_E2M1_SIGNED = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])
_E2M1_TIES = ((0.25, 0.5), (0.75, 0.5), (1.25, 0.5), (1.75, 0.5), (2.5, 1.0), (3.5, 1.0), (5.0, 2.0))


def _e4m3_bytes(t):
    import torch
    t = np.minimum(np.asarray(t, np.float32), np.float32(448.0))
    return torch.from_numpy(np.ascontiguousarray(t)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def _e4m3_values(b):
    import torch
    return torch.from_numpy(np.asarray(b, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def w4a4_allowance(down, ids, w, act, eps=W4A4_EPS):
    """down: host weights of the experts `ids` indexes ('codes' [n][H][I/2],
    'scales' [n][H][I/16], 'g' [n], 'a' [n]); ids, w [C][k]; act [C][k][I] the
    oracle's float64 activations.  Returns (allowance [C][H], number of
    ambiguous elements)."""
    C, k, I = act.shape
    H = down["codes"].shape[1]
    allow = np.zeros((C, H))
    n_amb = 0
    for t in range(C):
        for i in range(k):
            e = int(ids[t, i])
            if e < 0:
                continue
            a = float(np.float32(down["a"][e]))
            h = act[t, i].reshape(-1, 16)
            amax = np.abs(h).max(1)
            tol = eps * amax
            tt = amax / (6.0 * a)
            b_lo, b_hi = _e4m3_bytes(tt * (1 - eps)), _e4m3_bytes(tt * (1 + eps))
            s_hi = _e4m3_values(b_hi)
            m = _e4m3_values(b_lo) * a
            dev = np.zeros_like(h)
            amb_scale = b_lo != b_hi
            dev[amb_scale] = (2.0 * s_hi * a)[amb_scale, None]
            ok = ~amb_scale & (m > 0)
            q = np.abs(h[ok]) / m[ok, None]
            r = tol[ok, None] / m[ok, None]
            d = np.zeros_like(q)
            for tie, step in _E2M1_TIES:
                d = np.where(np.abs(q - tie) <= r, step, d)
            dev[ok] = d * m[ok, None]
            cols = np.nonzero(dev.reshape(-1))[0]
            if cols.size == 0:
                continue
            n_amb += cols.size
            codes = down["codes"][e][:, cols // 2]
            nib = (codes >> (4 * (cols % 2))) & 15
            sc = _e4m3_values(down["scales"][e][:, cols // 16])
            Dcol = np.abs(_E2M1_SIGNED[nib] * sc) * float(np.float32(down["g"][e]))
            allow[t] += abs(float(w[t, i])) * (Dcol @ dev.reshape(-1)[cols])
    return allow, n_amb


def assert_close_w4a4(y, y_ref, allow, label=""):
    """The acceptance tolerance with the W4A4 allowance added element by
    element (max) and to the L2 excess."""
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    assert y.shape == y_ref.shape == allow.shape
    assert np.isfinite(y).all(), f"{label}: non-finite output"
    scale = np.abs(y_ref).max()
    d = np.abs(y - y_ref)
    worst = (d - allow).max()
    assert worst <= MAX_ABS_REL * scale, f"{label}: max err beyond allowance {worst:.3e} > {MAX_ABS_REL} * {scale:.3e}"
    excess = np.maximum(d - allow, 0.0)
    l2 = np.linalg.norm(excess) / max(np.linalg.norm(y_ref), 1e-300)
    assert l2 <= REL_L2, f"{label}: rel L2 beyond allowance {l2:.3e} > {REL_L2}"
    return d.max() / max(scale, 1e-300), l2
