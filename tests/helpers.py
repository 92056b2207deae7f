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
