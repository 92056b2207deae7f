"""Pins of the oracle's steps around the routed sum ("SparkInfer-K3", "How
the TP module works": FfnPartial = router -> routed_down -> experts, then
FfnFinish = routed_norm -> routed_up -> shared experts): the dense 4-bit GEMV
against the pinned dequant and a library matmul and against one-hot rows,
the RMS norm against hand values (and the page's point that it is not
linear), the bf16 rounding against torch and hand ties, and the whole
composition against closed forms built from pinned pieces."""
import math

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_router_gb300 import synth


@pytest.mark.parametrize("fmt", ["nvfp4", "mxfp4"])
def test_dense_gemv_equals_dequant_matmul(fmt):
    c, sc, g = synth.ffn_matrix(1, 0, 0, 0, 48, 96, fmt)
    x = np.random.default_rng(2).standard_normal((3, 96))
    W = oracle.dequant(c, sc, g, 48, 96, fmt=fmt)
    np.testing.assert_allclose(oracle.dense_gemv(c, sc, g, x, fmt), x @ W.T, rtol=1e-13, atol=1e-13)


def test_dense_gemv_one_hot_rows():
    M, K = 16, 64
    cols = np.random.default_rng(4).integers(0, K, M)
    codes = np.zeros((M, K // 2), np.uint8)
    for m, col in enumerate(cols):
        codes[m, col // 2] |= 0x2 << (4 * (col % 2))          # e2m1 +1.0
    scales = np.full((M, K // 16), 0x38, np.uint8)           # e4m3 1.0
    x = np.random.default_rng(5).standard_normal((2, K))
    assert (oracle.dense_gemv(codes, scales, 1.0, x) == x[:, cols]).all()


def test_rms_norm_hand_values_and_nonlinearity():
    eps = 1e-6
    out = oracle.rms_norm(np.array([[3.0, 4.0]]), np.array([1.0, 2.0], np.float32), eps)
    r = 1.0 / math.sqrt(12.5 + eps)
    assert out[0, 0] == 3.0 * r * 1.0 and out[0, 1] == 4.0 * r * 2.0
    one = np.ones(2, np.float32)
    a, b = np.array([[3.0, 4.0]]), np.array([[1.0, -1.0]])
    # the reduce must come before the norm: norm(a + b) != norm(a) + norm(b)
    assert not np.allclose(oracle.rms_norm(a + b, one, eps), oracle.rms_norm(a, one, eps) + oracle.rms_norm(b, one, eps))
    # scale invariance (eps = 0)
    np.testing.assert_allclose(oracle.rms_norm(5.0 * a, one, 0.0), oracle.rms_norm(a, one, 0.0), rtol=1e-15)


def test_bf16_round_matches_torch_and_ties():
    rng = np.random.default_rng(0)
    v = rng.standard_normal(5000) * np.exp(rng.uniform(-20, 20, 5000))
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert (oracle.bf16_round(v.astype(np.float32).astype(np.float64)) == ref).all()
    # ties to even: 1 + 2^-8 sits halfway between 1 and 1 + 2^-7
    assert oracle.bf16_round(np.array([1 + 2 ** -8]))[0] == 0x3F80
    assert oracle.bf16_round(np.array([1 + 3 * 2 ** -8]))[0] == 0x3F82
    assert oracle.bf16_round(np.array([-0.0]))[0] == 0x8000


def _identity_rows(rows, K, col_of_row):
    codes = np.zeros((rows, K // 2), np.uint8)
    for r in range(rows):
        c = col_of_row(r)
        if c is not None:
            codes[r, c // 2] |= 0x2 << (4 * (c % 2))
    return {"codes": codes, "scales": np.full((rows, K // 16), 0x38, np.uint8), "g": np.float32(1.0),
            "a": np.float32(1.0)}


def test_ffn_layer_closed_form_with_identity_projections():
    # routed_down = [I | 0] and routed_up = [I ; 0], zero shared experts:
    # out[:, :L] = rms_norm(routed layer on u[:, :L]), out[:, L:] = 0
    Hd, L, E, k, I, S, Is, C = 128, 64, 12, 3, 96, 2, 32, 3
    ffn = synth.ffn_weights(0, 0, Hd, L, S, Is)
    ffn["routed_down"] = _identity_rows(L, Hd, lambda r: r)
    ffn["routed_up"] = _identity_rows(Hd, L, lambda r: r if r < L else None)
    for m in ffn["shared"].values():
        m["codes"][:] = 0
    routed = synth.canonical_layer(0, 0, E, L, I)
    Wr = synth.router_weights(0, 0, E, L)
    u = synth.tokens(0, 0, C, Hd)
    ids, w, _, x_bf16, y_r, out = oracle.ffn_layer(ffn, routed, Wr, u, k)
    assert (x_bf16 == u[:, :L]).all()                     # bf16 in, exact identity, bf16 out
    ids2, w2, _, y2 = oracle.full_layer(routed, Wr, u[:, :L], k)
    assert (ids == ids2).all() and (y_r == y2).all()
    assert (out[:, :L] == oracle.rms_norm(y2, ffn["gamma"], ffn["eps"])).all()
    assert (out[:, L:] == 0).all()


def test_ffn_layer_shared_experts_alone():
    # routed_up = 0: out = the sum of the shared experts' FFNs on u
    Hd, L, E, k, I, S, Is, C = 128, 64, 8, 2, 64, 2, 32, 2
    ffn = synth.ffn_weights(1, 0, Hd, L, S, Is)
    ffn["routed_up"]["codes"][:] = 0
    routed = synth.canonical_layer(1, 0, E, L, I)
    Wr = synth.router_weights(1, 0, E, L)
    u = synth.tokens(1, 0, C, Hd)
    _, _, _, _, _, out = oracle.ffn_layer(ffn, routed, Wr, u, k)
    uf = oracle.bf16_to_f64(u)
    sh = ffn["shared"]
    for t in range(C):
        ref = np.zeros(Hd)
        for s in range(S):
            ref += oracle.expert_ffn(Hd, Is, *[(sh[m]["codes"][s], sh[m]["scales"][s], float(sh[m]["g"][s]))
                                               for m in ("gate", "up", "down")], uf[t])
        assert (out[t] == ref).all()
