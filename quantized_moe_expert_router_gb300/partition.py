"""Host-side helpers for the two ways the routed layer splits over G ranks.

Expert bands ("SparkInfer-K3", section "How the TP module works"): rank r
holds a contiguous band [lo, hi) of the experts, runs the same replicated
router as every other rank (so all agree on the top-k), evaluates only the
selected experts it holds and contributes zero for the rest; the sum of the
ranks' partial outputs (an all-reduce of C x H values) is the layer output.
A rank builds a layer of hi - lo experts from its band's weights and passes
its ids through ``band_ids``: in-band ids become band-local, the others -1,
which ``moe_forward`` skips as absent slots.

Intermediate-column slices ("Kimi-K3 on the same pod, two engines", section
"Reason 1 - slice every expert across all eight Sparks"): rank r holds the
gate/up rows and the down columns [i0, i1) of the intermediate dimension of
every expert.  Its layer has intermediate size i1 - i0 and computes, for every
selected expert, D[:, i0:i1] (silu(G[i0:i1] x) * (U[i0:i1] x)); the fixed-order
sum over the slices is the layer output, and every rank has the same work
whatever the router picks.

The helpers only slice the canonical NVFP4 arrays and remap ids (numpy, no
GPU); the partial outputs come from the library's own entry points.
"""
from __future__ import annotations

import numpy as np


def expert_bands(E: int, G: int):
    """[(lo, hi)] of G contiguous, near-equal bands covering 0..E-1."""
    if not 1 <= G <= E:
        raise ValueError(f"cannot split {E} experts into {G} bands")
    return [(E * r // G, E * (r + 1) // G) for r in range(G)]


def band_ids(ids, lo: int, hi: int):
    """ids int32 [C][k] -> band-local ids: e - lo inside [lo, hi), -1 elsewhere."""
    ids = np.asarray(ids, dtype=np.int32)
    inside = (ids >= lo) & (ids < hi)
    return np.where(inside, ids - lo, -1).astype(np.int32)


def band_weights(canon: dict, lo: int, hi: int) -> dict:
    """The canonical weights of experts [lo, hi) (arrays with a leading expert axis)."""
    return {n: {f: m[f][lo:hi] for f in m} for n, m in canon.items()}


def intermediate_slices(I: int, G: int, align: int = 64):
    """[(i0, i1)] of G contiguous slices of 0..I-1 with bounds on multiples of
    ``align`` (the library requires the intermediate size to be a multiple of
    64; the e4m3 scale blocks of the down rows are 16 wide)."""
    if I % align or (I // align) < G:
        raise ValueError(f"cannot cut I={I} into {G} slices on multiples of {align}")
    units = I // align
    return [(align * (units * r // G), align * (units * (r + 1) // G)) for r in range(G)]


def slice_weights(canon: dict, i0: int, i1: int) -> dict:
    """Canonical weights of intermediate columns [i0, i1): gate/up rows i0..i1-1
    (codes [E][I][H/2], scales [E][I][H/16]) and down columns i0..i1-1 (codes
    [E][H][I/2] bytes i0/2..i1/2-1, scales [E][H][I/16] blocks i0/16..i1/16-1).
    The per-matrix global and input scales are kept as they are."""
    if i0 % 16 or i1 % 16:
        raise ValueError("slice bounds must be multiples of 16 (one e4m3 scale block)")
    out = {}
    for n in ("gate", "up"):
        m = canon[n]
        out[n] = {"codes": m["codes"][:, i0:i1], "scales": m["scales"][:, i0:i1], "g": m["g"], "a": m["a"]}
    m = canon["down"]
    out["down"] = {"codes": m["codes"][:, :, i0 // 2:i1 // 2], "scales": m["scales"][:, :, i0 // 16:i1 // 16],
                   "g": m["g"], "a": m["a"]}
    return out
