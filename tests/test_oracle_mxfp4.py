"""Pins of the oracle's MXFP4 path (OCP Microscaling e2m1 codes with one e8m0
scale per 32 elements along K, the format of the ggml MUL_MAT_ID microbench in
"Kimi-K3 on 2x A40 - measured findings", section "Why the placement
experiments all looked the same").

The e8m0 decode is pinned on all 256 bytes against the closed form; the
dequant against a hand-built matrix; the FFN against the NVFP4 path, itself
pinned elsewhere: an MXFP4 matrix whose scales are powers of two that e4m3
holds exactly is the same matrix as the NVFP4 matrix with each 32-block scale
repeated over its two 16-blocks, so the two formats must give bit-identical
outputs; plus the closed-form one-hot expert and the byte count of one
MXFP4 tensor."""
import math

import numpy as np
import pytest

import oracle
from quantized_moe_expert_router_gb300 import synth

ONE = 0x2          # e2m1 code of +1.0


def test_e8m0_all_bytes():
    for b in range(255):
        assert oracle.e8m0_value(b) == math.ldexp(1.0, b - 127), b
    assert math.isnan(oracle.e8m0_value(255))
    assert oracle.e8m0_value(127) == 1.0 and oracle.e8m0_value(0) == 2.0 ** -127


def test_mxfp4_dequant_hand_built():
    # 2 rows x 64: block b of row r has scale byte 120 + 3r + b and codes
    # cycling through the 16 e2m1 codes
    rows, K = 2, 64
    codes4 = np.array([[(r * 5 + k) % 16 for k in range(K)] for r in range(rows)], np.uint8)
    packed = (codes4[:, 0::2] | (codes4[:, 1::2] << 4)).astype(np.uint8)
    scales = np.array([[120 + 3 * r + b for b in range(K // 32)] for r in range(rows)], np.uint8)
    g = 0.75
    out = oracle.dequant(packed, scales, g, rows, K, fmt="mxfp4")
    e2m1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    for r in range(rows):
        for k in range(K):
            c = int(codes4[r, k])
            v = (-1 if c & 8 else 1) * e2m1[c & 7] * math.ldexp(1.0, int(scales[r, k // 32]) - 127) * g
            assert out[r, k] == v, (r, k)


def test_mxfp4_nan_scale_is_an_error():
    packed = np.zeros((1, 16), np.uint8)
    with pytest.raises(ValueError):
        oracle.dequant(packed, np.array([[0xFF]], np.uint8), 1.0, 1, 32, fmt="mxfp4")


def _to_nvfp4(L):
    """The same matrices written as NVFP4: each e8m0 32-block scale 2^e becomes
    the e4m3 byte of 2^e on both 16-blocks (exact for -9 <= e <= 8)."""
    out = {}
    for n, m in L.items():
        e = m["scales"].astype(np.int64) - 127
        assert ((e >= -6) & (e <= 8)).all()
        e4 = ((e + 7) << 3).astype(np.uint8)          # normal e4m3 with zero mantissa = 2^e
        out[n] = {"codes": m["codes"], "scales": np.repeat(e4, 2, axis=-1), "g": m["g"], "a": m["a"]}
    return out


def test_mxfp4_ffn_equals_nvfp4_of_the_same_matrices():
    E, k, H, I, C = 6, 2, 64, 96, 3
    L = synth.canonical_layer(0, 0, E, H, I, fmt="mxfp4")
    for m in L.values():                       # power-of-two scales in e4m3's exact range
        m["scales"] = (127 + (m["scales"].astype(np.int64) - 127).clip(-6, 8)).astype(np.uint8)
    Wr = synth.router_weights(0, 0, E, H)
    x = synth.tokens(0, 0, C, H)
    ids, w, _ = oracle.route(oracle.router_logits(Wr, x), k)
    y_mx = oracle.moe_forward(L, x, ids, w, fmt="mxfp4")
    y_nv = oracle.moe_forward(_to_nvfp4(L), x, ids, w, fmt="nvfp4")
    assert (y_mx == y_nv).all()
    assert (oracle.moe_forward(L, x, ids, w, threads=4, fmt="mxfp4") == y_mx).all()


def test_mxfp4_closed_form_one_hot_expert():
    # G row j = one-hot(a_j), U row j = one-hot(b_j), D = partial identity,
    # every scale 2^0: y_m = silu(x_{a_m}) x_{b_m} for m < I
    H, I = 64, 32
    rng = np.random.default_rng(3)
    a, b = rng.integers(0, H, I), rng.integers(0, H, I)

    def one_hot(rows, K, cols):
        c = np.zeros((rows, K // 2), np.uint8)
        for r, col in enumerate(cols):
            if col is not None:
                c[r, col // 2] |= ONE << (4 * (col % 2))
        return c, np.full((rows, K // 32), 127, np.uint8), 1.0
    gate, up = one_hot(I, H, list(a)), one_hot(I, H, list(b))
    down = one_hot(H, I, [m if m < I else None for m in range(H)])
    x = rng.standard_normal(H)
    y = oracle.expert_ffn(H, I, gate, up, down, x, fmt="mxfp4")
    ref = np.zeros(H)
    for m in range(I):
        ga = x[a[m]]
        ref[m] = ga / (1.0 + math.exp(-ga)) * x[b[m]]
    np.testing.assert_allclose(y, ref, rtol=1e-15, atol=1e-300)


def test_mxfp4_tensor_bytes():
    # one 3584 -> 3072 MXFP4 tensor: 4-bit codes plus one scale byte per 32
    codes, scales = synth.quantize_mxfp4(np.zeros((3072, 3584)))
    assert codes.nbytes + scales.nbytes == 3072 * 3584 * 17 // 32 == 5_849_088


def test_mxfp4_encoder_scale_rule():
    # scale 2^(floor(log2 amax) - 2): the block maximum lands in [4, 8) units
    rng = np.random.default_rng(0)
    w = rng.standard_normal((4, 256)) * 0.02
    codes, scales = synth.quantize_mxfp4(w)
    amax = np.abs(w.reshape(4, 8, 32)).max(axis=2)
    e = scales.astype(np.int64) - 127
    assert ((amax / np.ldexp(1.0, e) >= 4.0) & (amax / np.ldexp(1.0, e) < 8.0)).all()
    dq = oracle.dequant(codes, scales, 1.0, 4, 256, fmt="mxfp4")
    assert np.abs(dq - w).max() <= 2.0 * np.ldexp(1.0, e).max()
