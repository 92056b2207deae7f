"""Pins of the oracle's router and top-k: numpy's float64 matmul for the logits,
brute-force sorting for the selection, scipy's softmax for k == E, and the
routing invariants (weights sum to 1, equal logits go to the lower index, a
one-hot router selects its expert, permuting experts permutes ids)."""
import numpy as np
import pytest
from scipy.special import softmax

import oracle
from quantized_moe_expert_router_gb300 import synth


def test_logits_match_numpy_matmul():
    rng = np.random.default_rng(2)
    E, H, C = 32, 256, 3
    Wr = rng.standard_normal((E, H)).astype(np.float32)
    x = synth.f64_to_bf16_bits(rng.standard_normal((C, H)))
    bias = rng.standard_normal(E).astype(np.float32)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ Wr.astype(np.float64).T + bias.astype(np.float64)
    got = oracle.router_logits(Wr, x, bias)
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-12)
    got_nb = oracle.router_logits(Wr, x, None)
    np.testing.assert_allclose(got_nb, xf @ Wr.astype(np.float64).T, rtol=1e-13, atol=1e-12)


@pytest.mark.parametrize("seed", range(5))
def test_route_brute_force(seed):
    rng = np.random.default_rng(seed)
    C, E, k = 4, 32, 4
    logits = rng.standard_normal((C, E))
    ids, w, gap = oracle.route(logits, k)
    for t in range(C):
        order = sorted(range(E), key=lambda e: (-logits[t, e], e))
        sel = sorted(order[:k])
        assert list(ids[t]) == sel
        p = softmax(logits[t])
        np.testing.assert_allclose(w[t], p[sel] / p[sel].sum(), rtol=1e-14)
        assert gap[t] == logits[t, order[k - 1]] - logits[t, order[k]]
        assert abs(w[t].sum() - 1.0) < 1e-14


def test_k_equals_e_is_plain_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((2, 16)) * 3
    ids, w, gap = oracle.route(logits, 16)
    assert (ids == np.arange(16)).all()
    np.testing.assert_allclose(w, softmax(logits, axis=1), rtol=1e-14)
    assert np.isinf(gap).all()


def test_ties_go_to_lower_index():
    logits = np.zeros((1, 8))
    logits[0, [1, 3, 5, 6]] = 2.0          # four-way tie for two slots
    ids, w, gap = oracle.route(logits, 2)
    assert list(ids[0]) == [1, 3]
    np.testing.assert_allclose(w[0], [0.5, 0.5], rtol=0, atol=0)
    assert gap[0] == 0.0


def test_one_hot_router_selects_expert():
    E, H = 16, 64
    rng = np.random.default_rng(3)
    x = synth.f64_to_bf16_bits(rng.standard_normal((1, H)))
    xf = synth.bf16_bits_to_f32(x)[0]
    for target in (0, 5, 15):
        Wr = np.zeros((E, H), np.float32)
        Wr[target] = xf                      # row e = x gives the largest score |x|^2
        ids, w, _ = oracle.route(oracle.router_logits(Wr, x), 1)
        assert ids[0, 0] == target and w[0, 0] == 1.0


def test_permuting_experts_permutes_ids():
    rng = np.random.default_rng(4)
    E, k = 24, 5
    logits = rng.standard_normal((3, E))
    perm = rng.permutation(E)                # new expert j is old expert perm[j]
    ids, w, _ = oracle.route(logits, k)
    ids2, w2, _ = oracle.route(logits[:, perm], k)
    for t in range(3):
        back = {int(perm[j]): wj for j, wj in zip(ids2[t], w2[t])}
        assert sorted(back) == list(ids[t])
        np.testing.assert_allclose([back[int(e)] for e in ids[t]], w[t], rtol=1e-14)


def test_softmax_is_shift_invariant_and_stable():
    logits = np.array([[1000.0, 999.0, 998.0, -1000.0]])
    ids, w, _ = oracle.route(logits, 3)
    p = softmax(logits[0, :3])
    assert list(ids[0]) == [0, 1, 2]
    np.testing.assert_allclose(w[0], p / p.sum(), rtol=1e-14)
