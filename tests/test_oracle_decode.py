"""Pins of the oracle's number decoding and layout size against things other
than the oracle: the e2m1 value set of the OCP Microscaling format, torch's
float8_e4m3fn and bfloat16 conversions, and the sizes the pages print for the
K3 layer (tests/golden/k3_figures.txt: "Kimi-K3 on the same pod, two
engines", sections "Same hardware, same weights" and "Reason 1 -- slice every
expert across all eight Sparks"; "SparkInfer-K3", "The model")."""
import math

import numpy as np
import pytest
import torch

import oracle

from helpers import golden_figures

# The eight e2m1 magnitudes of the OCP MX v1.0 FP4 (E2M1) format, codes 0..7.
E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_all_sixteen_codes():
    for code in range(16):
        want = E2M1_MAGNITUDES[code & 7] * (-1.0 if code & 8 else 1.0)
        got = oracle.e2m1_value(code)
        assert got == want, (code, got, want)
        if code == 8:
            assert math.copysign(1.0, got) == -1.0  # negative zero keeps its sign


def test_e4m3_all_256_codes_match_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for code in range(256):
        got = oracle.e4m3_value(code)
        if code in (0x7F, 0xFF):
            assert math.isnan(got) and math.isnan(ref[code])
        else:
            assert got == ref[code], (code, got, ref[code])


def test_e4m3_landmarks():
    assert oracle.e4m3_value(0x7E) == 448.0          # largest finite
    assert oracle.e4m3_value(0x01) == 2.0 ** -9      # smallest subnormal
    assert oracle.e4m3_value(0x08) == 2.0 ** -6      # smallest normal
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert oracle.e2m1_value(7) == 6.0 and oracle.e2m1_value(1) == 0.5


def test_bf16_matches_torch():
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 16, size=4000, dtype=np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]             # skip inf/nan
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_value(int(b)) for b in bits])
    np.testing.assert_array_equal(got, ref)


def test_expert_bytes_match_the_k3_checkpoint():
    fig = golden_figures()
    H, I = fig["expert_latent_width"], fig["expert_ffn_width"]
    assert oracle.expert_bytes(H, I) == fig["expert_bytes_h3584_i3072"]
    # the small test layer (H 256, I 192)
    assert oracle.expert_bytes(256, 192) == 82_968
    # every layer but the leading dense one holds the routed experts
    assert (fig["layers"] - 1) * fig["routed_experts_per_layer"] == fig["routed_experts_per_checkpoint"]


def test_expert_slice_of_eight_matches_the_printed_size():
    # One eighth of the intermediate columns of an expert (gate/up rows and the
    # matching down columns, with their own scalars) is the printed ~2.32 MB.
    fig = golden_figures()
    H, I = fig["expert_latent_width"], fig["expert_ffn_width"]
    slice_bytes = oracle.expert_bytes(H, I // 8)
    assert round(slice_bytes / 1e6, 2) == fig["slice_megabytes_of_eight"]
    # the eight slices hold the whole expert except 7 extra copies of the 24 scalar bytes
    assert 8 * slice_bytes - oracle.expert_bytes(H, I) == 7 * 24


def test_expert_bands_of_eight_ranks():
    # 896 experts in 8 equal contiguous bands; the printed bands of ranks 3 and 7.
    fig = golden_figures()
    band = fig["routed_experts_per_layer"] // 8
    assert (3 * band, 4 * band) == (fig["expert_band_rank3_lo"], fig["expert_band_rank3_hi"])
    assert (7 * band, 8 * band) == (fig["expert_band_rank7_lo"], fig["expert_band_rank7_hi"])


def test_dequant_layout_nibbles_blocks_rows():
    """Hand-built 2x32 matrix: every element's code, block and row are
    distinguishable, so a swapped nibble, a transposed index or a wrong block
    stride changes the result."""
    rows, K = 2, 32
    codes = np.zeros((rows, K // 2), np.uint8)
    want_code = np.zeros((rows, K), np.int64)
    for r in range(rows):
        for k in range(K):
            want_code[r, k] = (3 * r + 5 * k + 1) % 16
    codes[:] = (want_code[:, 0::2] | (want_code[:, 1::2] << 4)).astype(np.uint8)
    scales = np.array([[0x38, 0x40], [0x30, 0x48]], np.uint8)   # 1, 2, 0.5, 4
    g = 0.75
    out = oracle.dequant(codes, scales, g, rows, K)
    sv = {0x38: 1.0, 0x40: 2.0, 0x30: 0.5, 0x48: 4.0}
    for r in range(rows):
        for k in range(K):
            c = want_code[r, k]
            v = E2M1_MAGNITUDES[c & 7] * (-1.0 if c & 8 else 1.0)
            assert out[r, k] == v * sv[int(scales[r, k // 16])] * g, (r, k)


def test_dequant_matches_torch_composition():
    """Random codes/scales: oracle dequant == a torch composition (float8
    decode of the scales, the literal e2m1 table for the codes)."""
    rng = np.random.default_rng(1)
    rows, K = 7, 64
    codes = rng.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7E, size=(rows, K // 16), dtype=np.uint8)
    g = np.float32(0.0123)
    lo = torch.from_numpy(codes & 0x0F).long()
    hi = torch.from_numpy(codes >> 4).long()
    table = torch.tensor([m for m in E2M1_MAGNITUDES] + [-m for m in E2M1_MAGNITUDES], dtype=torch.float64)
    elem = torch.stack([table[lo], table[hi]], dim=-1).reshape(rows, K)
    sc = torch.from_numpy(scales).view(torch.float8_e4m3fn).to(torch.float64)
    ref = (elem.reshape(rows, K // 16, 16) * sc[:, :, None]).reshape(rows, K) * float(g)
    got = oracle.dequant(codes, scales, g, rows, K)
    np.testing.assert_array_equal(got, ref.numpy())


def test_dequant_rejects_nan_scale():
    codes = np.zeros((1, 8), np.uint8)
    scales = np.array([[0x7F]], np.uint8)
    with pytest.raises(ValueError):
        oracle.dequant(codes, scales, 1.0, 1, 16)
