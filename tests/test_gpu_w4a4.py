"""GPU parity of the W4A4 numerics (MOE_CONFIG_W4A4): the activation
quantizer bit for bit against the oracle's, and the routed layer (the decode
kernels below 28 tokens, the grouped tcgen05 path from 28) against the
oracle's W4A4 mode within the acceptance tolerance plus the W4A4 allowance of
``helpers`` (rounding-tie decisions on h that fp32 accumulation noise can
move)."""
import numpy as np
import pytest
import torch

import oracle
from helpers import MIN_GAP, assert_close, assert_close_w4a4, gapped_tokens, w4a4_allowance
from quantized_moe_expert_router_gb300 import moe, synth
from quantized_moe_expert_router_gb300.synth import device as synth_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_moe_expert_router_gb300 import build
    build.build()
    moe.load_library()


def zero_sign_free(codes):
    lo, hi = codes & 0x0F, codes >> 4
    return (np.where(lo == 8, 0, lo) | (np.where(hi == 8, 0, hi) << 4)).astype(np.uint8)


def gpu_quantize(v, a, as_bf16):
    rows, n = v.shape
    if as_bf16:
        src = torch.from_numpy(synth.f64_to_bf16_bits(v.astype(np.float64)).view(np.int16)).to(DEV)
    else:
        src = torch.from_numpy(np.ascontiguousarray(v, np.float32)).to(DEV)
    codes = torch.empty((rows, n // 2), dtype=torch.uint8, device=DEV)
    scales = torch.empty((rows, n // 16), dtype=torch.uint8, device=DEV)
    moe.moe_quantize_nvfp4(src, a, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def tie_rich_inputs(rng, rows, n, a):
    """Normals, blocks scaled over a wide range, zero blocks, blocks whose
    elements sit on e2m1 rounding ties in units of s a (exactly for a = 1/8,
    where s = 8 gives s a = 1) and blocks whose max |v| / (6 a) sits on an
    e4m3 tie of the block scale."""
    a32 = np.float32(a)
    v = rng.standard_normal((rows, n)).astype(np.float32) * 3
    blk = v.reshape(-1, 16)
    nb = blk.shape[0]
    blk[: nb // 4] *= (2.0 ** rng.integers(-30, 30, nb // 4)).astype(np.float32)[:, None]
    blk[nb // 4: nb // 4 + 8] = 0.0
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    m = np.float32(8.0) * a32
    for b in range(nb // 2, nb // 2 + nb // 8):
        blk[b] = rng.choice(ties, 16) * rng.choice(np.array([-1, 1], np.float32), 16) * m
        blk[b, 0] = np.float32(6.0) * m                       # max |v| = 6 s a
    e4m3_ties = np.array([1.0625, 1.1875, 17.0, 34.0, 460.0, 2.0 ** -10], np.float32)
    for b in range(nb - 12, nb):
        tv = e4m3_ties[b % 6] * np.float32(6.0) * a32
        blk[b] = rng.standard_normal(16).astype(np.float32) * np.float32(0.1) * tv
        blk[b, 3] = tv
    return v


@pytest.mark.parametrize("as_bf16", [True, False])
@pytest.mark.parametrize("a", [0.125, 0.0019214, 7e-6])
def test_quantizer_bit_exact(as_bf16, a):
    rng = np.random.default_rng(11)
    v = tie_rich_inputs(rng, 48, 3584, a)
    if as_bf16:
        v = synth.bf16_bits_to_f32(synth.f64_to_bf16_bits(v.astype(np.float64)))
    codes, scales = gpu_quantize(v, a, as_bf16)
    oc, os_ = oracle.quantize_nvfp4_act(v.astype(np.float32), a)
    np.testing.assert_array_equal(scales, os_)
    np.testing.assert_array_equal(zero_sign_free(codes), zero_sign_free(oc))


def test_quantizer_rejects_bad_arguments():
    src = torch.zeros((2, 32), dtype=torch.float32, device=DEV)
    codes = torch.empty((2, 16), dtype=torch.uint8, device=DEV)
    scales = torch.empty((2, 2), dtype=torch.uint8, device=DEV)
    lib = moe.load_library()
    s = moe._stream(None)
    assert lib.moe_quantize_nvfp4(src.data_ptr(), 1, 2, 24, 1.0, codes.data_ptr(), scales.data_ptr(), s) != 0
    assert lib.moe_quantize_nvfp4(src.data_ptr(), 1, 2, 32, 0.0, codes.data_ptr(), scales.data_ptr(), s) != 0
    assert lib.moe_quantize_nvfp4(src.data_ptr(), 1, 2, 32, float("inf"), codes.data_ptr(), scales.data_ptr(), s) != 0
    assert lib.moe_quantize_nvfp4(src.data_ptr(), 7, 2, 32, 1.0, codes.data_ptr(), scales.data_ptr(), s) != 0
    assert lib.moe_quantize_nvfp4(src.data_ptr() + 4, 1, 1, 16, 1.0, codes.data_ptr(), scales.data_ptr(), s) != 0
    assert lib.moe_quantize_nvfp4(src.data_ptr(), 1, 2, 32, 1.0, codes.data_ptr(), scales.data_ptr(), s) == 0


# ------------------------------------------------------------------ the layer

class W4A4Layer:
    def __init__(self, E, k, H, I, max_tokens, seed=0, layer=0, zipf=False, device_gen=False):
        self.E, self.k, self.H, self.I = E, k, H, I
        self.h = moe.Layer(E, k, H, I, max_tokens, flags=moe.CONFIG_W4A4)
        if device_gen:
            self.canon_h = None
            self.canon = synth_dev.canonical_layer_device(seed, layer, E, H, I, DEV)
        else:
            self.canon_h = synth.canonical_layer(seed, layer, E, H, I)
            self.canon = {n: {f: torch.from_numpy(np.ascontiguousarray(m[f])).to(DEV)
                              for f in ("codes", "scales", "g", "a")} for n, m in self.canon_h.items()}
        self.packed = moe.alloc_packed(self.h)
        moe.moe_pack_weights(self.h, self.canon, self.packed)
        self.Wr = synth.router_weights(seed, layer, E, H)
        self.bias = synth.zipf_bias(seed, layer, E) if zipf else None
        self.Wr_d = torch.from_numpy(self.Wr).to(DEV)
        self.bias_d = None if self.bias is None else torch.from_numpy(self.bias).to(DEV)
        self.ws = moe.alloc_workspace(self.h, max_tokens)
        self.seed, self.layer = seed, layer

    def run(self, x_bits):
        C = x_bits.shape[0]
        x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
        ids = torch.empty((C, self.k), dtype=torch.int32, device=DEV)
        w = torch.empty((C, self.k), dtype=torch.float32, device=DEV)
        y = torch.empty((C, self.H), dtype=torch.float32, device=DEV)
        moe.moe_route_forward(self.h, x, C, self.Wr_d, self.bias_d, self.packed, ids, w, y, self.ws)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()

    def check(self, x_bits, label):
        ids, w, y = self.run(x_bits)
        logits = oracle.router_logits(self.Wr, x_bits, self.bias)
        oids, ow, gap = oracle.route(logits, self.k)
        assert (gap >= MIN_GAP).all()
        assert (ids == oids).all(), f"{label}: ids differ"
        assert moe.moe_get_device_status(self.h, self.ws) == 0
        sel = sorted(set(int(e) for e in oids.ravel()))
        remap = np.vectorize({e: i for i, e in enumerate(sel)}.get)(oids).astype(np.int32)
        if self.canon_h is None:
            Lw = synth_dev.gather_to_host(self.canon, sel)
        else:
            Lw = {n: {f: m[f][sel] for f in ("codes", "scales", "g", "a")} for n, m in self.canon_h.items()}
        oy, act = oracle.moe_forward_w4a4(Lw, x_bits, remap, ow, threads=oracle.default_threads(), return_act=True)
        allow, n_amb = w4a4_allowance(Lw["down"], remap, ow, act)
        err = assert_close_w4a4(y, oy, allow, label)
        # the layer really quantized: the weights-only result is far outside
        # the tolerance
        y16 = oracle.moe_forward(Lw, x_bits, remap, ow, threads=oracle.default_threads())
        with pytest.raises(AssertionError):
            assert_close(y, y16, label + " vs W4A16")
        return err, n_amb


@pytest.mark.parametrize("C", [1, 7, 12, 40])
def test_w4a4_parity_small(C):
    # C < 28: the decode kernels (12: two groups of at most 8); 40: the grouped path
    L = W4A4Layer(64, 8, 1024, 768, 64, seed=3)
    x = gapped_tokens(3, 0, C, 1024, L.Wr, 8)
    L.check(x, f"w4a4 E64 C={C}")


def test_w4a4_parity_odd_shape_zipf():
    L = W4A4Layer(40, 6, 576, 320, 64, seed=4, zipf=True)
    x = gapped_tokens(4, 0, 33, 576, L.Wr, 6, L.bias)
    L.check(x, "w4a4 odd shape zipf C=33")


@pytest.mark.parametrize("C", [1, 7])
def test_w4a4_parity_k3_shape(C):
    L = W4A4Layer(896, 16, 3584, 3072, 8, seed=5, device_gen=True)
    x = gapped_tokens(5, 0, C, 3584, L.Wr, 16)
    L.check(x, f"w4a4 K3 C={C}")


def test_w4a4_rejects_mxfp4_and_ffn():
    with pytest.raises(moe.MoEError):
        moe.Layer(64, 8, 512, 512, 8, flags=moe.CONFIG_W4A4 | moe.CONFIG_MXFP4)
    L = moe.Layer(64, 8, 512, 512, 8, flags=moe.CONFIG_W4A4)
    with pytest.raises(moe.MoEError):
        moe.Ffn(L, 1024, 0, 0, 1e-6)
