"""Host generator checks: determinism, shapes, the NVFP4 encoder against
torch's float8_e4m3fn rounding and against nearest-value search, and the
statistics of the synthetic weights."""
import numpy as np
import torch

import oracle
from quantized_moe_expert_router_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 started at state 0: the first outputs of the published
    # generator (Vigna's splitmix64.c) are these constants.
    assert synth.splitmix64_int(0) == 0xE220A8397B1DCDAF
    d = synth.draws(0, 0, 3)
    assert [int(v) for v in d] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_determinism_and_independence():
    a = synth.normals(synth.key(0, 1, 2), 1000)
    b = synth.normals(synth.key(0, 1, 2), 1000)
    c = synth.normals(synth.key(0, 1, 3), 1000)
    assert (a == b).all() and not (a == c).all()


def test_normal_statistics():
    z = synth.normals(synth.key(5, 9), 400_000)
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1.0) < 0.01
    assert np.abs(z).max() <= 4.899
    # Irwin-Hall(8) kurtosis is 3 - 6/(5*8) = 2.85
    k = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert abs(k - 2.85) < 0.05


def test_e4m3_encoder_matches_torch_rounding():
    rng = np.random.default_rng(0)
    v = np.concatenate([rng.uniform(0, 448, 20000), rng.uniform(0, 2 ** -5, 20000),
                        np.exp(rng.uniform(np.log(2 ** -10), np.log(448), 20000))])
    code, val = synth.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn)
    assert (code == ref.view(torch.uint8).numpy()).all()
    assert (val == ref.to(torch.float64).numpy()).all()
    assert synth.e4m3_encode(np.array([448.0, 500.0, 1e9]))[0].tolist() == [0x7E] * 3


def test_e2m1_encoder_is_nearest_with_ties_to_even():
    vals = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rng = np.random.default_rng(1)
    w = np.concatenate([rng.uniform(-7, 7, 5000), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -2.5]])
    codes = synth.e2m1_encode(w, np.ones_like(w))
    for wi, c in zip(w, codes):
        got = oracle.e2m1_value(int(c))
        d = np.abs(vals - min(abs(wi), 6.0))
        best = vals[d == d.min()]
        if len(best) == 2:      # tie: the value whose code has an even mantissa bit
            best = [b for b in best if (int(np.where(vals == b)[0][0]) & 1) == 0]
        assert abs(got) == best[0] and (got == 0 or np.sign(got) == np.sign(wi)), (wi, got)


def test_quantized_matrix_is_close_to_source():
    rows, K, g = 16, 256, 3.7e-5
    k = synth.weight_key(3, 0, 0, synth.MAT_GATE)
    w = ((synth._ih8_sum(k, rows * K) - synth.IH8_CENTER) * synth.W_COEF).reshape(rows, K)
    codes, scales = synth.quantize_nvfp4(w, g)
    deq = oracle.dequant(codes, scales, np.float32(g), rows, K)
    blk_amax = np.abs(w.reshape(rows, K // 16, 16)).max(2)
    err = np.abs(deq - w).reshape(rows, K // 16, 16).max(2)
    # half of the largest e2m1 step (2) in units of s*g, s <= 1.0625 * amax/(6g)
    assert (err <= blk_amax / 6 * 1.0625 + 1e-12).all()
    assert np.all(scales != 0x7F)


def test_canonical_layer_shapes_and_bytes():
    E, H, I = 4, 256, 192
    L = synth.canonical_layer(0, 0, E, H, I)
    total = sum(m["codes"].nbytes + m["scales"].nbytes + 8 * E for m in L.values())
    assert total == E * oracle.expert_bytes(H, I)
    assert L["gate"]["codes"].shape == (E, I, H // 2)
    assert L["down"]["scales"].shape == (E, H, I // 16)
    sub = synth.canonical_layer(0, 0, E, H, I, experts=[2])
    assert (sub["up"]["codes"][0] == L["up"]["codes"][2]).all()
    std = oracle.dequant(L["gate"]["codes"][0], L["gate"]["scales"][0], L["gate"]["g"][0], I, H).std()
    assert abs(std - 0.02) < 0.002


def test_zipf_bias_hot_set():
    E = 896
    b = synth.zipf_bias(0, 0, E)
    p = np.exp(b.astype(np.float64))
    assert abs(p.sum() - 1) < 1e-5
    top = np.sort(p)[::-1]
    assert abs(top[:104].sum() - 0.78) < 0.03
    assert not (np.argsort(b) == np.argsort(synth.zipf_bias(0, 1, E))).all()


def test_draft_rows_correlation_and_limits():
    # draft rows of one stream: N(0,1) rows with pairwise correlation rho;
    # rho = 1 gives identical rows, and a row's attempt number redraws that
    # row alone
    H = 4096
    x = synth.bf16_bits_to_f32(synth.draft_rows(3, 0, 4, H, 0.95)).astype(np.float64)
    assert np.abs(x.std(axis=1) - 1.0).max() < 0.05
    c = np.corrcoef(x)
    assert np.abs(c[np.triu_indices(4, 1)] - 0.95).max() < 0.02
    same = synth.draft_rows(3, 0, 3, H, 1.0)
    assert (same[0] == same[1]).all() and (same[1] == same[2]).all()
    a = synth.draft_rows(3, 0, 3, H, 0.9)
    b = synth.draft_rows(3, 0, 3, H, 0.9, attempts=[0, 1, 0])
    assert (a[0] == b[0]).all() and (a[2] == b[2]).all() and not (a[1] == b[1]).all()


def test_draft_rows_share_most_experts():
    # the verify pass's routing: with rho = 0.95 the 8 rows of a pass touch
    # far fewer distinct experts than 8 independent tokens would (16 each)
    E, H, k = 896, 3584, 16
    Wr = synth.router_weights(0, 0, E, H)
    for seed in range(3):
        ids, _, _ = oracle.route(oracle.router_logits(Wr, synth.draft_rows(seed, 0, 8, H, 0.95)), k)
        ind, _, _ = oracle.route(oracle.router_logits(Wr, synth.tokens(seed, 0, 8, H)), k)
        assert len(set(ids.ravel().tolist())) < 48 < len(set(ind.ravel().tolist()))
