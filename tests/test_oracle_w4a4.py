"""Pins of the oracle's W4A4 mode: activations quantized to NVFP4 with a
static per-tensor input scale ("Kimi-K3 on the same pod, two engines",
section "Same hardware, same weights": the NVFP4 checkpoint carries 24 bytes
of fp32 scalars per expert, a weight scale and an input scale per matrix).

The quantizer is checked against a brute-force restatement (nearest e2m1
magnitude by exhaustive search, e4m3 rounding by torch's float8 cast), hand
values with every rounding tie, saturation and scale underflow, exact round
trips of values on the grid and power-of-two invariance.  The expert and the
routed sum are checked against an independent numpy/torch composition, the
threaded forward against the one-thread composition, and the reading that
gate and up share one quantized x (scale max(a_gate, a_up))."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from quantized_moe_expert_router_gb300 import synth

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e4m3_byte(t):
    """Round-to-nearest-even e4m3 byte of t >= 0, saturating at 448 (torch's
    float8 cast rounds to nearest even; it does not saturate, so clamp first)."""
    t = np.minimum(np.asarray(t, np.float32), np.float32(448.0))
    return torch.from_numpy(np.ascontiguousarray(t)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def e4m3_val(b):
    return torch.from_numpy(np.asarray(b, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def e2m1_code(q):
    """Nearest e2m1 magnitude by exhaustive search, ties to the even code,
    saturating at 6; the sign bit is kept (so -0 is code 8)."""
    q = np.asarray(q, np.float64)
    mag = np.abs(q)
    d = np.abs(mag[..., None] - E2M1)
    best = d.min(-1, keepdims=True)
    cand = d == best                        # one or two nearest codes
    idx = np.arange(8)
    even_pick = np.where(cand & (idx % 2 == 0), idx, 99).min(-1)
    any_pick = np.where(cand, idx, 99).min(-1)
    code = np.where(cand.sum(-1) > 1, even_pick, any_pick)
    code = np.where(mag > 6.0, 7, code)
    return (code | np.where(np.signbit(q), 8, 0)).astype(np.uint8)


def brute_quant(v, a):
    """The NVFP4 activation quantizer restated with numpy float32 arithmetic:
    per block of 16, s = e4m3(max|v| / (6 a)); code = e2m1(v / (s a))."""
    v = np.asarray(v, np.float32).reshape(-1, 16)
    a32 = np.float32(a)
    amax = np.abs(v).max(1)
    t = amax / (np.float32(6.0) * a32)
    sb = e4m3_byte(t)
    sv = e4m3_val(sb).astype(np.float32)
    m = sv * a32
    with np.errstate(divide="ignore", invalid="ignore"):
        q = v / m[:, None]
    codes = np.where(sv[:, None] > 0, e2m1_code(q), 0).astype(np.uint8)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).reshape(-1)
    return packed, sb


def zero_sign_free(codes):
    """Codes with negative zero (nibble 8) mapped to zero."""
    lo, hi = codes & 0x0F, codes >> 4
    lo = np.where(lo == 8, 0, lo)
    hi = np.where(hi == 8, 0, hi)
    return (lo | (hi << 4)).astype(np.uint8)


def test_brute_force_helpers_on_hand_values():
    assert list(e2m1_code([0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.1, 9.0, -0.75])) == \
        [0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 8 | 2]
    assert list(e4m3_byte([1.0, 1.0625, 1.1875, 448.0, 460.0, 1e9, 2.0 ** -10])) == \
        [0x38, 0x38, 0x3A, 0x7E, 0x7E, 0x7E, 0x00]


def test_quantizer_hand_block():
    # a = 1/8: 6 a = 0.75 exactly; max|v| = 6 gives t = 8 (byte 0x50), so
    # s a = 1 and every code is the e2m1 rounding of v itself
    v = np.array([6, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5, -5, 5.5, 2.9, 3.1, 4.4, 0.5, -0.3, 0], np.float32)
    codes, scales = oracle.quantize_nvfp4_act(v, 0.125)
    want = [7, 0, 2, 2, 4, 4, 6, 6, 8 | 6, 7, 5, 5, 6, 1, 8 | 1, 0]
    got = [(codes[i // 2] >> (4 * (i % 2))) & 15 for i in range(16)]
    assert list(scales) == [0x50]
    assert got == want


def test_quantizer_scale_ties_saturation_underflow():
    a = np.float32(1.0) / np.float32(6.0)
    assert np.float32(6.0) * a == np.float32(1.0)          # t = max|v| exactly
    for amax, byte in [(1.0625, 0x38), (1.1875, 0x3A), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
                       (460.0, 0x7E), (1e6, 0x7E), (0.0, 0x00)]:
        v = np.zeros(16, np.float32)
        v[5] = -amax
        codes, scales = oracle.quantize_nvfp4_act(v, a)
        assert scales[0] == byte, (amax, scales[0])
        if byte == 0:
            assert not zero_sign_free(codes).any()          # scale 0: every code 0
    # saturation of the block scale clamps the codes at 6 too
    v = np.full(16, 1e6, np.float32)
    codes, scales = oracle.quantize_nvfp4_act(v, a)
    assert scales[0] == 0x7E and all(c == 0x77 for c in codes)


@pytest.mark.parametrize("a", [0.0019214, 0.125, 3e-5, 40.0, 1e-9])
def test_quantizer_matches_brute_force(a):
    rng = np.random.default_rng(int(a * 1e9) % 1000)
    n = 16 * 400
    # bf16 normals, wide-range blocks, exact ties and zero blocks
    v = synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(rng.standard_normal(n) * 3)).astype(np.float32)
    v[: 16 * 50] *= np.repeat(2.0 ** rng.integers(-20, 20, 50), 16).astype(np.float32)
    v[16 * 50: 16 * 60] = 0.0
    codes, scales = oracle.quantize_nvfp4_act(v, a)
    bc, bs = brute_quant(v, a)
    np.testing.assert_array_equal(scales, bs)
    np.testing.assert_array_equal(zero_sign_free(codes), zero_sign_free(bc))


def test_quantizer_round_trip_on_grid_and_power_of_two_invariance():
    rng = np.random.default_rng(3)
    a = np.float32(0.0123)
    for _ in range(50):
        s = e4m3_val(rng.integers(0x08, 0x7E))                # a normal block scale
        el = E2M1[rng.integers(0, 8, 16)] * rng.choice([-1, 1], 16)
        el[rng.integers(16)] = 6.0                             # the block max reaches 6 s
        v = (el * s * np.float64(a)).astype(np.float32)
        codes, scales = oracle.quantize_nvfp4_act(v, a)
        back = oracle.dequant_nvfp4_act(codes, scales, a)
        # v = e2m1 * s * a rounded to float32; the round trip gives the same
        # float32 value back whenever s a is itself exact (a power-of-two
        # ratio would be; here compare at float32 resolution)
        np.testing.assert_allclose(back, v.astype(np.float64), rtol=2 ** -23, atol=0)
    v = rng.standard_normal(16 * 64).astype(np.float32)
    c0, s0 = oracle.quantize_nvfp4_act(v, 0.01)
    for k in (-5, 3):
        c1, s1 = oracle.quantize_nvfp4_act(v * np.float32(2.0 ** k), np.float32(0.01) * np.float32(2.0 ** k))
        np.testing.assert_array_equal(c0, c1)
        np.testing.assert_array_equal(s0, s1)


# ---------------------------------------------------------------- the expert

TABLE = torch.tensor([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                      -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0], dtype=torch.float64)


def deq(m, e):
    """Library decode of one NVFP4 matrix: e2m1 table, torch float8 scales."""
    codes = torch.from_numpy(m["codes"][e]).long()
    rows, K = codes.shape[0], codes.shape[1] * 2
    el = torch.stack([TABLE[codes & 15], TABLE[codes >> 4]], -1).reshape(rows, K)
    sc = torch.from_numpy(m["scales"][e].copy()).view(torch.float8_e4m3fn).to(torch.float64)
    return ((el.reshape(rows, K // 16, 16) * sc[..., None]).reshape(rows, K) * float(m["g"][e])).numpy()


def brute_deq(v, a):
    codes, sb = brute_quant(v, a)
    nib = np.stack([codes & 15, codes >> 4], -1).reshape(-1)
    vals = TABLE.numpy()[nib]
    return vals * np.repeat(e4m3_val(sb), 16) * float(np.float32(a))


def composed_expert(L, e, x64, a_in, a_dn):
    """W4A4 expert restated with numpy matmuls and the brute-force quantizer."""
    G, U, D = deq(L["gate"], e), deq(L["up"], e), deq(L["down"], e)
    xq = brute_deq(x64.astype(np.float32), a_in)
    g, u = G @ xq, U @ xq
    h = (torch.from_numpy(g) * torch.sigmoid(torch.from_numpy(g))).numpy() * u
    return D @ brute_deq(h.astype(np.float32), a_dn), h


def mats(L, e):
    return [(L[n]["codes"][e], L[n]["scales"][e], L[n]["g"][e]) for n in ("gate", "up", "down")]


@pytest.mark.parametrize("H,I", [(64, 48), (256, 192)])
def test_expert_matches_independent_composition(H, I):
    L = synth.canonical_layer(5, 0, 3, H, I)
    x = synth.tokens(5, 0, 2, H)
    for e in range(3):
        for t in range(2):
            x64 = synth.bf16_bits_to_f32(x[t]).astype(np.float64)
            a_in, a_dn = L["gate"]["a"][e], L["down"]["a"][e]
            want, h_want = composed_expert(L, e, x64, a_in, a_dn)
            y, h = oracle.expert_ffn_w4a4(H, I, *mats(L, e), a_in, a_dn, x64, return_act=True)
            np.testing.assert_allclose(h, h_want, rtol=1e-12, atol=1e-15)
            np.testing.assert_allclose(y, want, rtol=1e-12, atol=1e-14 * np.abs(want).max())


def test_expert_one_hot_closed_form():
    """Gate/up rows one-hot: g_r = x[a_r], u_r = x[b_r]; down = partial
    identity: y[:I] = Q(silu(g) u), the quantized activation itself."""
    H, I = 64, 32
    rng = np.random.default_rng(2)
    a_idx, b_idx = rng.integers(0, H, I), rng.integers(0, H, I)

    def one_hot(rows, K, cols):
        codes = np.zeros((rows, K // 2), np.uint8)
        for r, c in enumerate(cols):
            if c is not None:
                codes[r, c // 2] |= 0x2 << (4 * (c % 2))       # +1.0
        return codes, np.full((rows, K // 16), 0x38, np.uint8)  # scale 1.0

    gate = one_hot(I, H, list(a_idx)) + (1.0,)
    up = one_hot(I, H, list(b_idx)) + (1.0,)
    down = one_hot(H, I, [r if r < I else None for r in range(H)]) + (1.0,)
    x64 = synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(rng.standard_normal(H))).astype(np.float64)
    a_in, a_dn = np.float32(4.9 / 2688), np.float32(0.004)
    xq = brute_deq(x64.astype(np.float32), a_in)
    h = F.silu(torch.from_numpy(xq[a_idx])).numpy() * xq[b_idx]
    want = np.zeros(H)
    want[:I] = brute_deq(h.astype(np.float32), a_dn)
    y = oracle.expert_ffn_w4a4(H, I, gate, up, down, a_in, a_dn, x64)
    np.testing.assert_allclose(y, want, rtol=1e-15, atol=0)
    # the quantized x really is coarser than x: the one-hot rows see xq, not x
    assert np.abs(xq - x64).max() > 1e-3


def test_expert_degenerate_inputs():
    H, I = 64, 48
    L = synth.canonical_layer(1, 0, 1, H, I)
    y = oracle.expert_ffn_w4a4(H, I, *mats(L, 0), L["gate"]["a"][0], L["down"]["a"][0], np.zeros(H))
    assert not y.any()
    # an input scale so large that every block scale underflows to zero
    x64 = synth.bf16_bits_to_f32(synth.tokens(1, 0, 1, H)[0]).astype(np.float64)
    y = oracle.expert_ffn_w4a4(H, I, *mats(L, 0), 1e30, L["down"]["a"][0], x64)
    assert not y.any()


# ---------------------------------------------------------------- the routed sum

def test_forward_composition_threads_and_shared_x_scale():
    E, H, I, k, C = 6, 128, 96, 3, 4
    L = synth.canonical_layer(7, 0, E, H, I)
    L["up"]["a"][1] = L["gate"]["a"][1] * np.float32(1.5)     # gate and up scales differ: x uses the larger
    x = synth.tokens(7, 0, C, H)
    rng = np.random.default_rng(0)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(C)]).astype(np.int32)
    w = rng.random((C, k))
    w /= w.sum(1, keepdims=True)
    y1, act = oracle.moe_forward_w4a4(L, x, ids, w, threads=1, return_act=True)
    y3 = oracle.moe_forward_w4a4(L, x, ids, w, threads=3)
    np.testing.assert_array_equal(y1, y3)
    for t in range(C):
        x64 = synth.bf16_bits_to_f32(x[t]).astype(np.float64)
        want = np.zeros(H)
        for i in range(k):
            e = int(ids[t, i])
            a_in = max(L["gate"]["a"][e], L["up"]["a"][e])
            ye, h = oracle.expert_ffn_w4a4(H, I, *mats(L, e), a_in, L["down"]["a"][e], x64, return_act=True)
            np.testing.assert_array_equal(act[t, i], h)
            want += w[t, i] * ye
        np.testing.assert_array_equal(y1[t], want)
    # expert 1 with the gate's own scale gives another x quantization
    t1, i1 = np.argwhere(ids == 1)[0]
    x64 = synth.bf16_bits_to_f32(x[t1]).astype(np.float64)
    y_gate_scale = oracle.expert_ffn_w4a4(H, I, *mats(L, 1), L["gate"]["a"][1], L["down"]["a"][1], x64)
    y_max_scale = oracle.expert_ffn_w4a4(H, I, *mats(L, 1), L["up"]["a"][1], L["down"]["a"][1], x64)
    assert np.abs(y_gate_scale - y_max_scale).max() > 0


def test_forward_is_w4a16_plus_activation_quantization_noise():
    """Relative to the weights-only result, quantizing x and h to 4 bits adds
    noise of the size NVFP4 rounding gives (a few per cent, not more)."""
    E, H, I, k, C = 8, 512, 384, 4, 3
    L = synth.canonical_layer(9, 0, E, H, I)
    x = synth.tokens(9, 0, C, H)
    ids = np.array([[0, 2, 5, 7], [1, 2, 3, 4], [6, 7, 0, 1]], np.int32)
    w = np.full((C, k), 0.25)
    y16 = oracle.moe_forward(L, x, ids, w)
    y4 = oracle.moe_forward_w4a4(L, x, ids, w)
    rel = np.linalg.norm(y4 - y16) / np.linalg.norm(y16)
    assert 0.02 < rel < 0.25, rel


# ---------------------------------------------------------------- the W4A4 tolerance

def simulated_outputs(L, ids, w, act, noise, rng, fold_weight=False, a_scale=1.0):
    """y from the oracle's activations perturbed by `noise` * (block max |h|)
    (what a different summation order can do), quantized by the brute-force
    quantizer; fold_weight quantizes w * h instead of h (a planted mistake);
    a_scale multiplies the down input scale (another)."""
    C, k, I = act.shape
    H = L["down"]["codes"].shape[1]
    y = np.zeros((C, H))
    for t in range(C):
        for i in range(k):
            e = int(ids[t, i])
            h = act[t, i].reshape(-1, 16)
            h = (h + noise * np.abs(h).max(1, keepdims=True) * rng.uniform(-1, 1, h.shape)).reshape(-1)
            if fold_weight:
                y[t] += deq(L["down"], e) @ brute_deq((w[t, i] * h).astype(np.float32), L["down"]["a"][e])
            else:
                aq = brute_deq(h.astype(np.float32), np.float32(L["down"]["a"][e] * a_scale))
                y[t] += w[t, i] * (deq(L["down"], e) @ aq)
    return y


def test_w4a4_tolerance_covers_tie_flips_and_catches_planted_mistakes():
    from helpers import W4A4_EPS, assert_close_w4a4, w4a4_allowance
    E, H, I, k, C = 6, 512, 384, 3, 3
    L = synth.canonical_layer(21, 0, E, H, I)
    x = synth.tokens(21, 0, C, H)
    ids = np.array([[0, 1, 2], [3, 4, 5], [5, 0, 2]], np.int32)
    w = np.array([[0.5, 0.3, 0.2], [0.4, 0.4, 0.2], [0.6, 0.3, 0.1]])
    oy, act = oracle.moe_forward_w4a4(L, x, ids, w, return_act=True)
    allow, n_amb = w4a4_allowance(L["down"], ids, w, act)
    assert n_amb > 0
    rng = np.random.default_rng(1)
    # noise at and below the bound: decisions near ties flip, the allowance covers them
    for noise in (1e-6, W4A4_EPS / 2, W4A4_EPS):
        assert_close_w4a4(simulated_outputs(L, ids, w, act, noise, rng), oy, allow, f"noise {noise}")
    # without the allowance the flips at noise = eps are visible
    y_flip = simulated_outputs(L, ids, w, act, W4A4_EPS, rng)
    assert np.abs(y_flip - oy).max() > 0
    # planted mistakes: router weight folded into h before quantization, wrong down scale
    for kw in ({"fold_weight": True}, {"a_scale": 1.5}):
        with pytest.raises(AssertionError):
            assert_close_w4a4(simulated_outputs(L, ids, w, act, 0.0, rng, **kw), oy, allow, str(kw))
