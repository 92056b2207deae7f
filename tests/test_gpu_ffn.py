"""GPU parity of the FFN around the routed sum (moe_ffn_* entry points):
routed_down, the routed layer, routed_norm, routed_up and the shared experts
("SparkInfer-K3", section "How the TP module works") against the float64
oracle on the same seeded inputs: the selected ids bit for bit, the routed sum
y_r and the layer output within the acceptance tolerance."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_close
from quantized_moe_expert_router_gb300 import moe, synth
from quantized_moe_expert_router_gb300.synth import device as synth_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_moe_expert_router_gb300 import build
    build.build()
    moe.load_library()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def ffn_to_device(fw):
    one = lambda m: {"codes": _dev(m["codes"]), "scales": _dev(m["scales"]),
                     "g": _dev(np.array([m["g"]], np.float32)), "a": _dev(np.array([m["a"]], np.float32))}
    sh = {n: {f: _dev(m[f]) for f in ("codes", "scales", "g", "a")} for n, m in fw["shared"].items()}
    return {"routed_down": one(fw["routed_down"]), "routed_up": one(fw["routed_up"]), "shared": sh,
            "gamma": _dev(fw["gamma"])}


class GpuFfn:
    def __init__(self, E, k, hidden, latent, I, S, Is, max_tokens=8, seed=0, fmt="nvfp4", device_gen=False):
        self.k, self.hidden, self.latent, self.fmt = k, hidden, latent, fmt
        flags = moe.CONFIG_MXFP4 if fmt == "mxfp4" else 0
        self.layer = moe.Layer(E, k, latent, I, max_tokens, flags=flags)
        if device_gen:
            self.canon = synth_dev.canonical_layer_device(seed, 0, E, latent, I, DEV, fmt=fmt)
            self.host_routed = lambda sel: synth_dev.gather_to_host(self.canon, sel)
        else:
            canon_h = synth.canonical_layer(seed, 0, E, latent, I, fmt=fmt)
            self.canon = {n: {f: _dev(m[f]) for f in ("codes", "scales", "g", "a")} for n, m in canon_h.items()}
            self.host_routed = lambda sel: {n: {f: m[f][list(sel)] for f in ("codes", "scales", "g", "a")}
                                            for n, m in canon_h.items()}
        self.packed = moe.alloc_packed(self.layer)
        moe.moe_pack_weights(self.layer, self.canon, self.packed)
        self.Wr = synth.router_weights(seed, 0, E, latent)
        self.Wr_d = _dev(self.Wr)
        self.fw = synth.ffn_weights(seed, 0, hidden, latent, S, Is, fmt=fmt)
        self.ffn = moe.Ffn(self.layer, hidden, S, Is, eps=self.fw["eps"])
        self.fpacked = moe.alloc_ffn_packed(self.ffn)
        moe.moe_ffn_pack_weights(self.ffn, ffn_to_device(self.fw), self.fpacked)
        self.ws = moe.alloc_ffn_workspace(self.ffn, max_tokens)

    def draw(self, C, seed=0):
        """Tokens whose routing gap (on the oracle's latent x) is >= 1e-3."""
        attempts = [0] * C
        for _ in range(200):
            u = synth.tokens(seed, 7, C, self.hidden, attempts)
            x = oracle.bf16_round(oracle.dense_gemv(self.fw["routed_down"]["codes"], self.fw["routed_down"]["scales"],
                                                    self.fw["routed_down"]["g"], oracle.bf16_to_f64(u), self.fmt))
            _, _, gap = oracle.route(oracle.router_logits(self.Wr, x), self.k)
            bad = [t for t in range(C) if gap[t] < 1e-3]
            if not bad:
                return u
            for t in bad:
                attempts[t] += 1
        raise RuntimeError("no tokens with the required gap")

    def run(self, u_bits, split=False):
        C = u_bits.shape[0]
        u = _dev(u_bits.view(np.int16))
        ids = torch.empty((C, self.k), dtype=torch.int32, device=DEV)
        w = torch.empty((C, self.k), dtype=torch.float32, device=DEV)
        out = torch.empty((C, self.hidden), dtype=torch.float32, device=DEV)
        y_r = torch.empty((C, self.latent), dtype=torch.float32, device=DEV)
        if split:
            moe.moe_ffn_partial(self.ffn, u, C, self.Wr_d, None, self.packed, self.fpacked, ids, w, y_r, self.ws)
            moe.moe_ffn_finish(self.ffn, u, C, y_r, self.fpacked, out, self.ws)
        else:
            moe.moe_ffn_forward(self.ffn, u, C, self.Wr_d, None, self.packed, self.fpacked, ids, w, out, self.ws)
            moe.moe_ffn_partial(self.ffn, u, C, self.Wr_d, None, self.packed, self.fpacked, ids, w, y_r, self.ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_status(self.layer, self.ws) == 0
        return ids.cpu().numpy(), w.cpu().numpy(), y_r.cpu().numpy(), out.cpu().numpy()

    def oracle(self, u_bits):
        return oracle.ffn_layer(self.fw, self.host_routed, self.Wr, u_bits, self.k, threads=oracle.default_threads(),
                                fmt=self.fmt)


def check(F, u, label):
    ids, w, y_r, out = F.run(u)
    oids, ow, _, _, oy_r, oout = F.oracle(u)
    assert (ids == oids).all(), f"{label}: ids differ"
    np.testing.assert_allclose(w, ow, rtol=2e-5, atol=1e-7)
    assert_close(y_r, oy_r, f"{label}: routed sum")
    assert_close(out, oout, f"{label}: layer output")
    return ids, y_r, out


@pytest.mark.parametrize("C", [1, 3, 8])
def test_tiny_ffn_parity(C):
    F = GpuFfn(32, 4, 512, 256, 192, 2, 128)
    check(F, F.draw(C), f"tiny ffn C={C}")


@pytest.mark.parametrize("hidden,latent,I,S,Is,C", [(192, 64, 128, 1, 64, 2), (1088, 320, 64, 0, 64, 5),
                                                    (8192, 256, 128, 1, 4096, 1)])
def test_ffn_odd_shapes_parity(hidden, latent, I, S, Is, C):
    F = GpuFfn(12, 3, hidden, latent, I, S, Is, seed=2)
    check(F, F.draw(C, seed=2), f"ffn H{hidden} L{latent} I{I} S{S} Is{Is} C{C}")


def test_tiny_ffn_mxfp4_parity():
    F = GpuFfn(32, 4, 512, 256, 192, 2, 128, fmt="mxfp4")
    check(F, F.draw(3, seed=1), "tiny ffn mxfp4 C=3")


def test_partial_finish_equal_forward_and_band_sum():
    # the two phases give the one-call output bit for bit; and two expert
    # bands' partial routed sums, added, then finished, give the layer
    # (the reduce at the latent width, before the norm)
    from quantized_moe_expert_router_gb300 import partition
    F = GpuFfn(32, 4, 512, 256, 192, 2, 128, seed=3)
    u = F.draw(4, seed=3)
    ids, w, y_r, out = F.run(u)
    ids2, w2, y_r2, out2 = F.run(u, split=True)
    assert (ids == ids2).all() and (y_r == y_r2).all() and (out == out2).all()
    # bands: each rank runs the routed experts it holds on the same x
    ud = _dev(u.view(np.int16))
    x_lat = oracle.bf16_round(oracle.dense_gemv(F.fw["routed_down"]["codes"], F.fw["routed_down"]["scales"],
                                                F.fw["routed_down"]["g"], oracle.bf16_to_f64(u)))
    xd = _dev(x_lat.view(np.int16))
    total = torch.zeros((4, 256), dtype=torch.float32, device=DEV)
    canon_h = synth.canonical_layer(3, 0, 32, 256, 192)
    for lo, hi in partition.expert_bands(32, 2):
        L = moe.Layer(hi - lo, 4, 256, 192, 8)
        pk = moe.alloc_packed(L)
        moe.moe_pack_weights(L, {n: {f: _dev(m[f]) for f in ("codes", "scales", "g", "a")}
                                 for n, m in partition.band_weights(canon_h, lo, hi).items()}, pk)
        yb = torch.empty((4, 256), dtype=torch.float32, device=DEV)
        moe.moe_forward(L, xd, 4, _dev(partition.band_ids(ids, lo, hi)), _dev(w), pk, yb, moe.alloc_workspace(L, 8))
        total += yb
    outb = torch.empty((4, 512), dtype=torch.float32, device=DEV)
    moe.moe_ffn_finish(F.ffn, ud, 4, total, F.fpacked, outb, F.ws)
    torch.cuda.synchronize()
    assert_close(total.cpu().numpy(), y_r, "band sum of the routed partials")
    assert_close(outb.cpu().numpy(), out, "finish of the band sum")


@pytest.mark.parametrize("C", [1, 7])
def test_k3_ffn_parity(C):
    # the K3 shape: hidden 7168, latent 3584, 896 experts top-16 with FFN
    # 3072, 2 shared experts of FFN 3072
    F = GpuFfn(896, 16, 7168, 3584, 3072, 2, 3072, seed=0, device_gen=True)
    check(F, F.draw(C, seed=C), f"k3 ffn C={C}")


def test_device_ffn_generator_matches_host():
    fd = synth_dev.ffn_weights_device(4, 0, 1024, 256, 2, 192, DEV)
    fh = synth.ffn_weights(4, 0, 1024, 256, 2, 192)
    for n in ("routed_down", "routed_up"):
        assert (fd[n]["codes"].cpu().numpy() == fh[n]["codes"]).all()
        assert (fd[n]["scales"].cpu().numpy() == fh[n]["scales"]).all()
        assert float(fd[n]["g"][0]) == float(fh[n]["g"])
    for n in ("gate", "up", "down"):
        for f in ("codes", "scales", "g"):
            assert (fd["shared"][n][f].cpu().numpy() == fh["shared"][n][f]).all(), (n, f)
    assert (fd["gamma"].cpu().numpy() == fh["gamma"]).all()
