"""Pins of the oracle's expert FFN and combine: closed forms from hand-built
experts (one-hot gate/up rows, a partial-identity down matrix), exact
invariants (zero expert, k = 1, power-of-two scaling, expert permutation), and
an independent float64 torch composition (library float8 decode, softmax,
topk, silu, matmul) on the small synthetic layer."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from quantized_moe_expert_router_gb300 import synth

ONE = 0x2          # e2m1 code of +1.0
S_ONE = 0x38       # e4m3 byte of 1.0


def one_hot_matrix(rows, K, cols):
    """NVFP4 [rows][K] with row r = one-hot at column cols[r] (None = zero row)."""
    codes = np.zeros((rows, K // 2), np.uint8)
    scales = np.full((rows, K // 16), S_ONE, np.uint8)
    for r, c in enumerate(cols):
        if c is None:
            continue
        codes[r, c // 2] |= ONE << (4 * (c % 2))
    return codes, scales


def as_weights(mats):
    gate, up, down = mats
    return {n: {"codes": m[0][None], "scales": m[1][None], "g": np.array([m[2]], np.float32)}
            for n, m in zip(("gate", "up", "down"), (gate, up, down))}


def test_closed_form_one_hot_expert():
    H, I = 48, 32
    rng = np.random.default_rng(11)
    a = rng.integers(0, H, I)
    b = rng.integers(0, H, I)
    gate = one_hot_matrix(I, H, list(a)) + (1.0,)
    up = one_hot_matrix(I, H, list(b)) + (1.0,)
    down = one_hot_matrix(H, I, [r if r < I else None for r in range(H)]) + (1.0,)
    x = synth.f64_to_bf16_bits(rng.standard_normal((1, H)))
    xf = torch.from_numpy(synth.bf16_bits_to_f32(x)[0].astype(np.float64))
    want = torch.zeros(H, dtype=torch.float64)
    want[:I] = F.silu(xf[a]) * xf[b]
    y = oracle.expert_ffn(H, I, gate, up, down, xf.numpy())
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-15, atol=0)
    # through the routed forward with k = 1 and weight 1
    ym = oracle.moe_forward(as_weights((gate, up, down)), x, np.array([[0]]), np.array([[1.0]]))
    np.testing.assert_allclose(ym[0], want.numpy(), rtol=1e-15, atol=0)


def test_closed_form_scaled_codes():
    """Gate row r = 6.0 * 0.5 * 0.25 at column r: g_r = 0.75 x_r; up row r =
    -1.5 * 2 * 1 at column r+1: u_r = -3 x_{r+1}; down = identity * 4 (scale
    0x48) * 0.5 (g)."""
    H = I = 32
    gc = np.zeros((I, H // 2), np.uint8)
    uc = np.zeros((I, H // 2), np.uint8)
    dc = np.zeros((H, I // 2), np.uint8)
    for r in range(I):
        gc[r, r // 2] |= 0x7 << (4 * (r % 2))                  # +6
        c = (r + 1) % H
        uc[r, c // 2] |= 0xB << (4 * (c % 2))                  # -1.5
        dc[r, r // 2] |= ONE << (4 * (r % 2))
    gate = (gc, np.full((I, H // 16), 0x30, np.uint8), 0.25)  # scale 0.5
    up = (uc, np.full((I, H // 16), 0x40, np.uint8), 1.0)     # scale 2
    down = (dc, np.full((H, I // 16), 0x48, np.uint8), 0.5)   # scale 4
    rng = np.random.default_rng(5)
    x = synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(rng.standard_normal(H))).astype(np.float64)
    xt = torch.from_numpy(x)
    want = 2.0 * F.silu(0.75 * xt) * (-3.0 * torch.roll(xt, -1))
    y = oracle.expert_ffn(H, I, gate, up, down, x)
    np.testing.assert_allclose(y, want.numpy(), rtol=1e-15, atol=0)


def test_zero_expert_contributes_exactly_zero():
    L = synth.canonical_layer(0, 0, 4, 64, 32)
    for n in ("gate", "up", "down"):
        L[n]["codes"][2] = 0
    x = synth.tokens(0, 0, 2, 64)
    y = oracle.moe_forward(L, x, np.array([[2], [2]]), np.array([[1.0], [0.3]]))
    assert (y == 0.0).all()
    # and mixing it with a non-zero expert gives that expert's weighted output
    y1 = oracle.moe_forward(L, x, np.array([[1], [1]]), np.array([[0.7], [0.7]]))
    y2 = oracle.moe_forward(L, x, np.array([[1, 2], [2, 1]]), np.array([[0.7, 0.3], [0.3, 0.7]]))
    np.testing.assert_allclose(y2, y1, rtol=1e-15, atol=0)


def test_power_of_two_global_scale_doubles_contribution():
    L = synth.canonical_layer(0, 0, 3, 64, 32)
    x = synth.tokens(0, 0, 1, 64)
    ids, w = np.array([[0, 1]]), np.array([[0.25, 0.75]])
    y = oracle.moe_forward(L, x, ids, w)
    y_e0 = oracle.moe_forward(L, x, np.array([[0]]), np.array([[0.25]]))
    L["down"]["g"][0] *= 2
    y2 = oracle.moe_forward(L, x, ids, w)
    np.testing.assert_allclose(y2 - y, y_e0, rtol=1e-12, atol=1e-15)


def torch_reference_layer(L, Wr, x_bits, k, bias=None):
    """Independent float64 composition from torch library routines."""
    table = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                          -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=torch.float64)

    def deq(m, e):
        codes = torch.from_numpy(m["codes"][e]).long()
        rows = codes.shape[0]
        K = codes.shape[1] * 2
        el = torch.stack([table[codes & 15], table[codes >> 4]], -1).reshape(rows, K)
        sc = torch.from_numpy(m["scales"][e].copy()).view(torch.float8_e4m3fn).to(torch.float64)
        return (el.reshape(rows, K // 16, 16) * sc[..., None]).reshape(rows, K) * float(m["g"][e])

    x = torch.from_numpy(x_bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64)
    logits = x @ torch.from_numpy(Wr).to(torch.float64).T
    if bias is not None:
        logits = logits + torch.from_numpy(bias).to(torch.float64)
    p = torch.softmax(logits, dim=1)
    top = torch.topk(logits, k, dim=1).indices
    ids = torch.sort(top, dim=1).values
    w = torch.gather(p, 1, ids)
    w = w / w.sum(1, keepdim=True)
    y = torch.zeros_like(x)
    for t in range(x.shape[0]):
        for i in range(k):
            e = int(ids[t, i])
            G, U, D = deq(L["gate"], e), deq(L["up"], e), deq(L["down"], e)
            a = F.silu(G @ x[t]) * (U @ x[t])
            y[t] += w[t, i] * (D @ a)
    return ids.numpy(), w.numpy(), y.numpy()


@pytest.mark.parametrize("E,H,I,k,C", [(32, 256, 192, 4, 2), (12, 64, 96, 3, 3)])
def test_full_layer_matches_torch_composition(E, H, I, k, C):
    L = synth.canonical_layer(0, 0, E, H, I)
    Wr = synth.router_weights(0, 0, E, H)
    x = synth.tokens(0, 0, C, H)
    ids, w, gap, y = oracle.full_layer(L, Wr, x, k)
    rids, rw, ry = torch_reference_layer(L, Wr, x, k)
    assert (ids == rids).all()
    np.testing.assert_allclose(w, rw, rtol=1e-12)
    np.testing.assert_allclose(y, ry, rtol=1e-10, atol=1e-12 * np.abs(ry).max())


def test_permuting_experts_leaves_output_unchanged():
    E, H, I, k = 10, 64, 32, 3
    L = synth.canonical_layer(1, 0, E, H, I)
    Wr = synth.router_weights(1, 0, E, H)
    x = synth.tokens(1, 0, 2, H)
    _, _, _, y = oracle.full_layer(L, Wr, x, k)
    perm = np.random.default_rng(0).permutation(E)
    Lp = {n: {f: m[f][perm] for f in ("codes", "scales", "g")} for n, m in L.items()}
    _, _, _, yp = oracle.full_layer(Lp, Wr[perm], x, k)
    np.testing.assert_allclose(yp, y, rtol=1e-13, atol=1e-15)


def test_bad_expert_id_is_an_error():
    L = synth.canonical_layer(0, 0, 4, 64, 32)
    x = synth.tokens(0, 0, 1, 64)
    with pytest.raises(ValueError):
        oracle.moe_forward(L, x, np.array([[4]]), np.array([[1.0]]))


@pytest.mark.parametrize("C,threads", [(1, 3), (4, 2), (9, 7), (5, 64)])
def test_threaded_oracle_is_bitwise_the_single_threaded_one(C, threads):
    # the threaded forward only moves (token, slot) expert evaluations to other
    # cores and sums them in the same slot order
    E, k, H, I = 16, 3, 64, 96
    cw = synth.canonical_layer(2, 0, E, H, I)
    x = synth.tokens(2, 0, C, H)
    ids, w, _ = oracle.route(oracle.router_logits(synth.router_weights(2, 0, E, H), x), k)
    y1 = oracle.moe_forward(cw, x, ids, w)
    y2 = oracle.moe_forward(cw, x, ids, w, threads=threads)
    assert (y1 == y2).all()
    bad = ids.copy()
    bad[C - 1, 0] = E
    with pytest.raises(ValueError):
        oracle.moe_forward(cw, x, bad, w, threads=threads)
