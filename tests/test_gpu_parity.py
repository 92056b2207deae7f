"""GPU parity: the CUDA path through the C ABI against the float64 oracle on
the same seeded inputs.  Selected ids must match bit for bit (the generator
keeps a >= 1e-3 logit gap at the k-th boundary); outputs must meet the
acceptance tolerance in ``helpers``."""
import numpy as np
import pytest
import torch

import oracle
from helpers import MIN_GAP, assert_close, gapped_tokens
from quantized_moe_expert_router_gb300 import moe, synth
from quantized_moe_expert_router_gb300.synth import device as synth_dev

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    from quantized_moe_expert_router_gb300 import build
    build.build()
    moe.load_library()


def to_device(canon_h):
    return {n: {f: torch.from_numpy(np.ascontiguousarray(m[f])).to(DEV) for f in ("codes", "scales", "g", "a")}
            for n, m in canon_h.items()}


class GpuLayer:
    def __init__(self, E, k, H, I, max_tokens, seed=0, layer=0, device_gen=False, router_std=1.0,
                 zipf=False, fmt="nvfp4", grouped=False):
        self.E, self.k, self.H, self.I = E, k, H, I
        self.seed, self.layer_id, self.fmt = seed, layer, fmt
        flags = (moe.CONFIG_MXFP4 if fmt == "mxfp4" else 0) | (moe.CONFIG_GROUPED_ABOVE_8 if grouped else 0)
        self.h = moe.Layer(E, k, H, I, max_tokens, flags=flags)
        if device_gen:
            self.canon = synth_dev.canonical_layer_device(seed, layer, E, H, I, DEV, fmt=fmt)
        else:
            self.canon_h = synth.canonical_layer(seed, layer, E, H, I, fmt=fmt)
            self.canon = to_device(self.canon_h)
        self.packed = moe.alloc_packed(self.h)
        moe.moe_pack_weights(self.h, self.canon, self.packed)
        self.Wr = synth.router_weights(seed, layer, E, H, router_std)
        self.bias = synth.zipf_bias(seed, layer, E) if zipf else None
        self.Wr_d = torch.from_numpy(self.Wr).to(DEV)
        self.bias_d = None if self.bias is None else torch.from_numpy(self.bias).to(DEV)
        self.ws = moe.alloc_workspace(self.h, max_tokens)

    def host_weights(self, experts):
        if hasattr(self, "canon_h"):
            return {n: {f: m[f][list(experts)] for f in ("codes", "scales", "g", "a")}
                    for n, m in self.canon_h.items()}
        return synth_dev.gather_to_host(self.canon, experts)

    def run(self, x_bits):
        C = x_bits.shape[0]
        x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
        ids = torch.empty((C, self.k), dtype=torch.int32, device=DEV)
        w = torch.empty((C, self.k), dtype=torch.float32, device=DEV)
        y = torch.empty((C, self.H), dtype=torch.float32, device=DEV)
        moe.moe_route(self.h, x, C, self.Wr_d, self.bias_d, ids, w, self.ws)
        moe.moe_forward(self.h, x, C, ids, w, self.packed, y, self.ws)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()

    def run_fused(self, x_bits):
        """The whole layer in one call (moe_route_forward)."""
        C = x_bits.shape[0]
        x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
        ids = torch.empty((C, self.k), dtype=torch.int32, device=DEV)
        w = torch.empty((C, self.k), dtype=torch.float32, device=DEV)
        y = torch.empty((C, self.H), dtype=torch.float32, device=DEV)
        moe.moe_route_forward(self.h, x, C, self.Wr_d, self.bias_d, self.packed, ids, w, y, self.ws)
        torch.cuda.synchronize()
        return ids.cpu().numpy(), w.cpu().numpy(), y.cpu().numpy()

    def oracle(self, x_bits, threads=1):
        """Oracle routing + forward on the selected experts only."""
        logits = oracle.router_logits(self.Wr, x_bits, self.bias)
        ids, w, gap = oracle.route(logits, self.k)
        sel = sorted(set(int(e) for e in ids.ravel()))
        remap = {e: i for i, e in enumerate(sel)}
        y = oracle.moe_forward(self.host_weights(sel), x_bits, np.vectorize(remap.get)(ids).astype(np.int32), w,
                               threads=threads, fmt=getattr(self, "fmt", "nvfp4"))
        return ids, w, gap, y


def check_layer(L, x_bits, label, fused=False):
    ids, w, y = (L.run_fused if fused else L.run)(x_bits)
    oids, ow, gap, oy = L.oracle(x_bits)
    assert (gap >= MIN_GAP).all()
    assert (ids == oids).all(), f"{label}: ids differ\n{ids}\n{oids}"
    np.testing.assert_allclose(w, ow, rtol=2e-5, atol=1e-7)
    assert abs(w.sum(1) - 1).max() < 1e-5
    flags = moe.moe_get_device_status(L.h, L.ws)
    assert flags == 0, f"{label}: device flags {flags:#x}"
    return assert_close(y, oy, label)


# ------------------------------------------------------------------ generator

def test_device_generator_matches_host():
    E, H, I = 5, 256, 192
    d = synth_dev.canonical_layer_device(0, 3, E, H, I, DEV)
    h = synth.canonical_layer(0, 3, E, H, I)
    for n in ("gate", "up", "down"):
        for f in ("codes", "scales", "g", "a"):
            assert (d[n][f].cpu().numpy() == h[n][f]).all(), (n, f)


def test_device_generator_matches_host_k3_expert():
    E, H, I = 2, 3584, 3072
    d = synth_dev.canonical_layer_device(7, 1, E, H, I, DEV)
    h = synth.canonical_layer(7, 1, E, H, I, experts=[1])
    for n in ("gate", "up", "down"):
        assert (d[n]["codes"][1].cpu().numpy() == h[n]["codes"][0]).all(), n
        assert (d[n]["scales"][1].cpu().numpy() == h[n]["scales"][0]).all(), n


# ------------------------------------------------------------------ packer

def _unpack_tiles(buf, ntiles, W, K):
    """Tiles of 8 pair rows -> (rowA codes, rowB codes, rowA scales, rowB scales),
    each indexed [pair row][...] (the inverse of the packer's byte moves)."""
    tb = W * 4608
    t = buf[: ntiles * tb].reshape(ntiles, tb)
    codes = t[:, : W * 4096].reshape(ntiles, W, 8, 8, 4, 4, 4)     # tile w qg g q j byte
    codes = codes.transpose(0, 3, 1, 2, 5, 4, 6)                   # tile g w qg j q byte
    S = W * 32
    A = np.empty((ntiles, 8, S, 8), np.uint8)
    B = np.empty((ntiles, 8, S, 8), np.uint8)
    c = codes.reshape(ntiles, 8, S, 4, 4)                          # tile g S q byte
    A[..., :4], A[..., 4:] = c[..., 0], c[..., 2]
    B[..., :4], B[..., 4:] = c[..., 1], c[..., 3]
    sc = t[:, W * 4096:].reshape(ntiles, W, 4, 8, 8, 2)            # tile w q8 g i ab
    sc = sc.transpose(0, 3, 1, 2, 4, 5).reshape(ntiles, 8, S, 2)   # tile g S ab
    rows = ntiles * 8
    return (A.reshape(rows, S * 8)[:, : K // 2], B.reshape(rows, S * 8)[:, : K // 2],
            sc[..., 0].reshape(rows, S)[:, : K // 16], sc[..., 1].reshape(rows, S)[:, : K // 16])


def unpack_host(packed, E, H, I):
    """Reverse the packed tile layout on the host (byte moves only)."""
    Wg, Wd = -(-H // 512), -(-I // 512)
    gu_bytes = (I // 8) * Wg * 4608
    ebytes = gu_bytes + (H // 16) * Wd * 4608
    out = {n: {"codes": np.zeros((E, r, K // 2), np.uint8), "scales": np.zeros((E, r, K // 16), np.uint8)}
           for n, r, K in (("gate", I, H), ("up", I, H), ("down", H, I))}
    for e in range(E):
        base = e * ebytes
        ga, ub, gs, us = _unpack_tiles(packed[base: base + gu_bytes], I // 8, Wg, H)
        out["gate"]["codes"][e], out["up"]["codes"][e] = ga, ub
        out["gate"]["scales"][e], out["up"]["scales"][e] = gs, us
        da, db, das, dbs = _unpack_tiles(packed[base + gu_bytes: base + ebytes], H // 16, Wd, I)
        out["down"]["codes"][e][0::2], out["down"]["codes"][e][1::2] = da, db
        out["down"]["scales"][e][0::2], out["down"]["scales"][e][1::2] = das, dbs
    scal = packed[E * ebytes: E * ebytes + E * 24].view(np.float32).reshape(E, 6)
    return out, scal


@pytest.mark.parametrize("E,H,I", [(32, 256, 192), (3, 1024, 512)])
def test_pack_layout_roundtrip(E, H, I):
    L = GpuLayer(E, 2, H, I, 1)
    packed = L.packed.cpu().numpy()
    assert packed.size == moe.moe_packed_bytes(L.h)
    un, scal = unpack_host(packed, E, H, I)
    for n in ("gate", "up", "down"):
        assert (un[n]["codes"] == L.canon_h[n]["codes"]).all(), n
        assert (un[n]["scales"] == L.canon_h[n]["scales"]).all(), n
    for j, (n, f) in enumerate([("gate", "g"), ("gate", "a"), ("up", "g"), ("up", "a"), ("down", "g"), ("down", "a")]):
        assert (scal[:, j] == L.canon_h[n][f]).all()


def test_packed_bytes_equal_canonical_for_k3_shape():
    h = moe.Layer(896, 16, 3584, 3072, 1)
    assert moe.moe_packed_bytes(h) == 896 * oracle.expert_bytes(3584, 3072) + 16


def test_pack_rejects_nan_scale():
    L = GpuLayer(4, 2, 256, 192, 1)
    L.canon["down"]["scales"][2, 5, 3] = 0x7F
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_pack_weights(L.h, L.canon, L.packed)
    assert ei.value.status == 3


# ------------------------------------------------------------------ parity, small

@pytest.mark.parametrize("C", [1, 2, 3, 4, 7, 8, 11])
def test_tiny_layer_parity(C):
    L = GpuLayer(32, 4, 256, 192, 16)
    x = gapped_tokens(0, 0, C, 256, L.Wr, 4)
    check_layer(L, x, f"tiny C={C}")


@pytest.mark.parametrize("E,k,H,I,C", [(12, 3, 64, 128, 5), (40, 8, 576, 320, 2), (64, 32, 128, 64, 3),
                                       (7, 7, 192, 1088, 1)])
def test_odd_shapes_parity(E, k, H, I, C):
    L = GpuLayer(E, k, H, I, C, seed=3)
    x = gapped_tokens(3, 0, C, H, L.Wr, k)
    check_layer(L, x, f"E{E} k{k} H{H} I{I} C{C}")


@pytest.mark.parametrize("E,k,H,I,C", [(32, 4, 256, 192, 40), (12, 3, 64, 128, 20), (40, 8, 576, 320, 64),
                                       (7, 7, 192, 1088, 9), (8, 1, 4096, 4096, 9), (16, 2, 64, 4096, 12)])
def test_grouped_path_parity(E, k, H, I, C):
    # the grouped path for every C > 8 (the layer flag): expert-major, every
    # expert's weights once for all its tokens
    L = GpuLayer(E, k, H, I, C, seed=6, grouped=True)
    x = gapped_tokens(6, 0, C, H, L.Wr, k)
    check_layer(L, x, f"grouped E{E} k{k} H{H} I{I} C{C}")


@pytest.mark.parametrize("C", [520, 1100])
def test_grouped_path_multi_pass_parity(C):
    # more than 512 tokens: passes of 512 (and a ragged last one); ~65 pairs
    # per expert, so the grouped GEMMs split experts into several column
    # chunks (64 pairs for gate/up, 32 for down)
    L = GpuLayer(32, 4, 256, 192, C, seed=9, grouped=True)
    x = gapped_tokens(9, 0, C, 256, L.Wr, 4)
    check_layer(L, x, f"grouped multi-pass C={C}")


@pytest.mark.parametrize("C", [9, 16, 27, 28])
def test_default_path_switch_parity(C):
    # without the flag, 9 .. 27 tokens run the decode kernels in groups of 8
    # and 28 or more the grouped path: both sides of the switch against the
    # oracle
    L = GpuLayer(40, 8, 576, 320, C, seed=10)
    x = gapped_tokens(10, 0, C, 576, L.Wr, 8)
    check_layer(L, x, f"default path C={C}")


@pytest.mark.parametrize("C,grouped", [(1, False), (3, False), (8, False), (11, False), (11, True)])
def test_route_forward_equals_route_then_forward(C, grouped):
    # the one-call layer gives the separate calls' results bit for bit, call
    # after call
    L = GpuLayer(32, 4, 256, 192, 16, grouped=grouped)
    for rep in range(3):
        x = gapped_tokens(rep, 0, C, 256, L.Wr, 4)
        ids, w, y = L.run(x)
        ids2, w2, y2 = L.run_fused(x)
        assert (ids == ids2).all() and (w == w2).all() and (y == y2).all(), f"C={C} call {rep}"
        assert moe.moe_get_device_status(L.h, L.ws) == 0
    check_layer(L, x, f"fused tiny C={C}", fused=True)


@pytest.mark.parametrize("E,k,H,I,C", [(12, 3, 64, 128, 5), (7, 7, 192, 1088, 1), (200, 32, 4096, 64, 8)])
def test_route_forward_odd_shapes(E, k, H, I, C):
    L = GpuLayer(E, k, H, I, C, seed=5)
    x = gapped_tokens(5, 0, C, H, L.Wr, k)
    check_layer(L, x, f"fused E{E} k{k} H{H} I{I} C{C}", fused=True)


def _forward(h, x_bits, ids, w, canon_h, ws_tokens=8):
    """moe_forward of a layer built from host canonical weights."""
    packed = moe.alloc_packed(h)
    moe.moe_pack_weights(h, to_device(canon_h), packed)
    C, H = x_bits.shape
    y = torch.empty((C, H), dtype=torch.float32, device=DEV)
    ws = moe.alloc_workspace(h, ws_tokens)
    moe.moe_forward(h, torch.from_numpy(x_bits.view(np.int16)).to(DEV), C,
                    torch.from_numpy(np.ascontiguousarray(ids, np.int32)).to(DEV),
                    torch.from_numpy(np.ascontiguousarray(w, np.float32)).to(DEV), packed, y, ws)
    assert moe.moe_get_device_status(h, ws) == 0      # absent (negative) ids raise no flag
    return y.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("C", [3, 20])
def test_band_and_slice_partials_sum_to_the_layer(C):
    # the two splits of the layer over ranks (expert bands; intermediate
    # column slices), each partial computed by the CUDA path on its own
    # layer, summed in rank order (C = 20 runs the grouped path)
    from quantized_moe_expert_router_gb300 import partition
    E, k, H, I = 32, 4, 256, 192
    canon = synth.canonical_layer(0, 0, E, H, I)
    Wr = synth.router_weights(0, 0, E, H)
    x = gapped_tokens(0, 0, C, H, Wr, k)
    ids, w, _ = oracle.route(oracle.router_logits(Wr, x), k)
    y_o = oracle.moe_forward(canon, x, ids, w)
    total = np.zeros_like(y_o)
    gf = moe.CONFIG_GROUPED_ABOVE_8
    for lo, hi in partition.expert_bands(E, 2):
        total += _forward(moe.Layer(hi - lo, k, H, I, max(C, 8), flags=gf), x, partition.band_ids(ids, lo, hi), w,
                          partition.band_weights(canon, lo, hi), ws_tokens=max(C, 8))
    assert_close(total, y_o, "expert bands")
    total = np.zeros_like(y_o)
    for i0, i1 in partition.intermediate_slices(I, 2):
        total += _forward(moe.Layer(E, k, H, i1 - i0, max(C, 8), flags=gf), x, ids, w,
                          partition.slice_weights(canon, i0, i1), ws_tokens=max(C, 8))
    assert_close(total, y_o, "intermediate slices")


@pytest.mark.parametrize("C", [1, 2, 5])
def test_forward_reads_x_written_by_the_previous_kernel(C):
    # a caller's kernel writes x on the stream immediately before a standalone
    # moe_forward: the expert kernels must see the new x (the buffer held
    # other tokens before), whatever the launch overlap between kernels
    L = GpuLayer(32, 4, 256, 192, 8)
    x_bits = gapped_tokens(11, 0, C, 256, L.Wr, 4)
    x_src = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
    stale = gapped_tokens(12, 0, C, 256, L.Wr, 4)
    x = torch.from_numpy(stale.view(np.int16)).to(DEV)
    ids = torch.empty((C, 4), dtype=torch.int32, device=DEV)
    w = torch.empty((C, 4), dtype=torch.float32, device=DEV)
    y = torch.empty((C, 256), dtype=torch.float32, device=DEV)
    moe.moe_route(L.h, x_src, C, L.Wr_d, None, ids, w, L.ws)
    torch.cuda.synchronize()
    for _ in range(3):
        big = torch.ones(1 << 22, device=DEV).cumsum(0)          # a busy kernel first
        torch.bitwise_xor(x_src, torch.zeros_like(x_src), out=x)   # then x is written
        moe.moe_forward(L.h, x, C, ids, w, L.packed, y, L.ws)
        torch.cuda.synchronize()
        del big
        oids, ow, _, oy = L.oracle(x_bits)
        assert (ids.cpu().numpy() == oids).all()
        assert_close(y.cpu().numpy(), oy, f"x written right before moe_forward, C={C}")
        x.copy_(torch.from_numpy(stale.view(np.int16)).to(DEV))
        torch.cuda.synchronize()
    assert moe.moe_get_device_status(L.h, L.ws) == 0


@pytest.mark.parametrize("C", [1, 3])
def test_router_wait_timeout_is_reported_and_recovered(C):
    # the test hook makes every router block wait for bytes that never come:
    # the bounded wait runs out (20 ms), MOE_FLAG_TIMEOUT is raised, ids come
    # back as -1 with weights 0, moe_forward then treats every slot as absent
    # (y = 0), and the same workspace and the no-alloc router work normally on
    # the next call.  C = 1 takes the logits-only router, whose failed blocks
    # mark their logits NaN for the expert kernels' own selection.
    E, k, H, I = 32, 4, 256, 192
    good = GpuLayer(E, k, H, I, 8)
    stall = moe.Layer(E, k, H, I, 8, flags=moe.CONFIG_TEST_ROUTER_STALL)
    x_bits = gapped_tokens(0, 0, C, H, good.Wr, k)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
    ids = torch.zeros((C, k), dtype=torch.int32, device=DEV)
    w = torch.ones((C, k), dtype=torch.float32, device=DEV)
    y = torch.ones((C, H), dtype=torch.float32, device=DEV)
    moe.moe_route_forward(stall, x, C, good.Wr_d, None, good.packed, ids, w, y, good.ws)
    torch.cuda.synchronize()
    assert (ids.cpu().numpy() == -1).all() and (w.cpu().numpy() == 0).all()
    assert (y.cpu().numpy() == 0).all()
    flags = moe.moe_get_device_status(stall, good.ws)
    assert flags == moe.FLAG_TIMEOUT, f"{flags:#x}"
    oids, ow, _, oy = good.oracle(x_bits)
    for rep in range(2):                      # the workspace is as good as new
        ids2, w2, y2 = good.run(x_bits) if rep == 0 else good.run_fused(x_bits)
        assert (ids2 == oids).all()
        assert_close(y2, oy, f"after a router timeout, call {rep}")
        assert moe.moe_get_device_status(good.h, good.ws) == 0
    ids.fill_(0)
    moe.moe_route_noalloc(stall, x, C, good.Wr_d, None, ids, w)
    torch.cuda.synchronize()
    assert (ids.cpu().numpy() == -1).all()
    moe.moe_route_noalloc(good.h, x, C, good.Wr_d, None, ids, w)
    torch.cuda.synchronize()
    assert (ids.cpu().numpy() == oids).all()


@pytest.mark.parametrize("C,nan_token", [(3, 1), (12, 9)])
def test_nan_token_selects_nothing(C, nan_token):
    # a token whose router logits include a NaN (here from one NaN element of
    # its x) selects no expert: ids -1, weights 0, output 0, with no flag; the
    # other tokens of the call are unaffected (the fused router for C <= 8,
    # the tiled router and the per-token top-k above)
    L = GpuLayer(32, 4, 256, 192, 16)
    x_bits = gapped_tokens(7, 0, C, 256, L.Wr, 4)
    bad = x_bits.copy()
    bad[nan_token, 17] = 0x7FC0                  # a bf16 quiet NaN
    ids, w, y = L.run_fused(bad)
    assert moe.moe_get_device_status(L.h, L.ws) == 0
    assert (ids[nan_token] == -1).all() and (w[nan_token] == 0).all() and (y[nan_token] == 0).all()
    keep = [t for t in range(C) if t != nan_token]
    oids, ow, _, oy = L.oracle(x_bits[keep])
    assert (ids[keep] == oids).all()
    np.testing.assert_allclose(w[keep], ow, rtol=2e-5, atol=1e-7)
    assert_close(y[keep], oy, f"tokens beside a NaN token, C={C}")


def test_forward_is_deterministic():
    L = GpuLayer(32, 4, 256, 192, 8)
    x = gapped_tokens(0, 0, 8, 256, L.Wr, 4)
    _, _, y1 = L.run(x)
    _, _, y2 = L.run(x)
    assert (y1 == y2).all()


def test_bad_and_duplicate_ids_are_flagged_and_skipped():
    L = GpuLayer(32, 4, 256, 192, 2)
    x_bits = gapped_tokens(0, 0, 2, 256, L.Wr, 4)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
    ids = torch.tensor([[1, 5, 40, 9], [3, 3, 7, 8]], dtype=torch.int32, device=DEV)
    w = torch.tensor([[0.1, 0.2, 0.3, 0.4], [0.25, 0.25, 0.25, 0.25]], dtype=torch.float32, device=DEV)
    y = torch.empty((2, 256), dtype=torch.float32, device=DEV)
    moe.moe_forward(L.h, x, 2, ids, w, L.packed, y, L.ws)
    flags = moe.moe_get_device_status(L.h, L.ws)
    assert flags & moe.FLAG_BAD_EXPERT_ID and flags & moe.FLAG_DUPLICATE_ID
    # token 0 without its bad slot is exact; token 1 keeps one copy of expert 3
    y0 = oracle.moe_forward(L.host_weights(range(32)), x_bits[:1], np.array([[1, 5, 9]], np.int32),
                            np.array([[0.1, 0.2, 0.4]]))
    assert_close(y.cpu().numpy()[:1], y0, "bad id")
    y1 = oracle.moe_forward(L.host_weights(range(32)), x_bits[1:], np.array([[3, 7, 8]], np.int32),
                            np.array([[0.25, 0.25, 0.25]]))
    assert_close(y.cpu().numpy()[1:], y1, "duplicate id")
    assert moe.moe_get_device_status(L.h, L.ws) == 0    # cleared


def test_one_token_unsorted_bad_duplicate_and_absent_ids():
    # a single token takes its own dispatch path: slots in any order, an id
    # >= E and a repeated id are flagged and skipped (the repeat keeps its
    # lowest slot), negative ids are absent without a flag
    L = GpuLayer(32, 4, 256, 192, 2)
    x_bits = gapped_tokens(3, 0, 1, 256, L.Wr, 4)
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
    y = torch.empty((1, 256), dtype=torch.float32, device=DEV)
    cases = [([7, 40, 2, 7], [0.3, 0.1, 0.2, 0.4], [7, 2], [0.3, 0.2],
              moe.FLAG_BAD_EXPERT_ID | moe.FLAG_DUPLICATE_ID),
             ([-1, 5, -1, 1], [0.5, 0.25, 0.5, 0.75], [5, 1], [0.25, 0.75], 0),
             ([31, 0, 16, 8], [0.25, 0.125, 0.5, 0.125], [31, 0, 16, 8], [0.25, 0.125, 0.5, 0.125], 0)]
    for ids_l, w_l, oids, ow, want in cases:
        ids = torch.tensor([ids_l], dtype=torch.int32, device=DEV)
        w = torch.tensor([w_l], dtype=torch.float32, device=DEV)
        moe.moe_forward(L.h, x, 1, ids, w, L.packed, y, L.ws)
        assert moe.moe_get_device_status(L.h, L.ws) == want, ids_l
        yo = oracle.moe_forward(L.host_weights(range(32)), x_bits, np.array([oids], np.int32), np.array([ow]))
        assert_close(y.cpu().numpy(), yo, f"one token, ids {ids_l}")


def test_grouped_bad_duplicate_and_absent_ids():
    # C > 8 (expert-major dispatch): a bad id and a repeated id are flagged
    # and skipped, negative ids are absent slots, a token with no slot left
    # gets a zero output
    C, k = 12, 4
    L = GpuLayer(32, k, 256, 192, C, seed=4, grouped=True)
    x_bits = gapped_tokens(4, 0, C, 256, L.Wr, k)
    ids_h, w_h, _ = oracle.route(oracle.router_logits(L.Wr, x_bits), k)
    ids_h = ids_h.astype(np.int32).copy()
    w_h = w_h.astype(np.float32).copy()
    ids_h[0, 2] = 40                       # bad
    ids_h[1, 3] = ids_h[1, 0]              # repeat of slot 0
    ids_h[2, 1] = -1                       # absent
    ids_h[3, :] = -1                       # nothing left
    x = torch.from_numpy(x_bits.view(np.int16)).to(DEV)
    y = torch.empty((C, 256), dtype=torch.float32, device=DEV)
    moe.moe_forward(L.h, x, C, torch.from_numpy(ids_h).to(DEV), torch.from_numpy(w_h).to(DEV), L.packed, y, L.ws)
    flags = moe.moe_get_device_status(L.h, L.ws)
    assert flags & moe.FLAG_BAD_EXPERT_ID and flags & moe.FLAG_DUPLICATE_ID
    keep = (ids_h >= 0) & (ids_h < 32)
    keep[1, 3] = False
    y_o = oracle.moe_forward(L.host_weights(range(32)), x_bits, np.where(keep, ids_h, 0).astype(np.int32),
                             np.where(keep, w_h, 0.0))
    yg = y.cpu().numpy()
    assert (yg[3] == 0).all()
    assert_close(yg, y_o, "grouped bad / repeated / absent ids")
    assert moe.moe_get_device_status(L.h, L.ws) == 0    # cleared


def test_argument_errors_return_status_without_launch():
    L = GpuLayer(32, 4, 256, 192, 2)
    x = torch.zeros((2, 256), dtype=torch.int16, device=DEV)
    ids = torch.zeros((2, 4), dtype=torch.int32, device=DEV)
    w = torch.zeros((2, 4), dtype=torch.float32, device=DEV)
    y = torch.empty((2, 256), dtype=torch.float32, device=DEV)
    small = torch.zeros(64, dtype=torch.uint8, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_forward(L.h, x, 2, ids, w, L.packed, y, small)
    assert ei.value.status == 4
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_forward(L.h, x, 3, ids, w, L.packed, y, L.ws)       # C > max_tokens
    assert ei.value.status == 1
    ybuf = torch.empty(2 * 256 + 1, dtype=torch.float32, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_forward(L.h, x, 2, ids, w, L.packed, ybuf[1:], L.ws)  # misaligned y
    assert ei.value.status == 1
    for bad in [(0, 4, 256, 192), (32, 0, 256, 192), (32, 33, 256, 192), (32, 4, 100, 192), (32, 4, 256, 8192),
                (2000, 4, 256, 192)]:
        with pytest.raises(moe.MoEError):
            moe.Layer(*bad, 1)


@pytest.mark.parametrize("C,k", [(1, 8), (3, 12), (11, 8)])
def test_router_ties_take_lower_ids(C, k):
    # Zero router weights: every logit is its bias exactly.  Ten experts share
    # each bias value (with +0 and -0 in one group), so the k-th boundary
    # falls inside a tie and the lower expert ids must be kept.
    E, H = 40, 64
    h = moe.Layer(E, k, H, 64, 16)
    ws = moe.alloc_workspace(h, 16)
    rng = np.random.default_rng(7)
    bias = rng.permutation(np.repeat(np.array([2.0, 1.0, 0.0, -1.0], np.float32), 10))
    zero_idx = np.nonzero(bias == 0.0)[0]
    bias[zero_idx[::2]] = -0.0
    xb = synth.tokens(7, 0, C, H)
    x = torch.from_numpy(xb.view(np.int16)).to(DEV)
    ids = torch.empty((C, k), dtype=torch.int32, device=DEV)
    w = torch.empty((C, k), dtype=torch.float32, device=DEV)
    Wr = torch.zeros((E, H), dtype=torch.float32, device=DEV)
    moe.moe_route(h, x, C, Wr, torch.from_numpy(bias).to(DEV), ids, w, ws)
    oids, ow, _ = oracle.route(np.tile(bias.astype(np.float64), (C, 1)), k)
    assert (ids.cpu().numpy() == oids).all(), (ids.cpu().numpy(), oids)
    np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-6, atol=1e-8)


# ------------------------------------------------------------------ K3 shape

@pytest.fixture(scope="module")
def k3_layer():
    L = GpuLayer(896, 16, 3584, 3072, 8, seed=0, device_gen=True)
    yield L
    del L.canon


def test_k3_router_parity(k3_layer):
    L = k3_layer
    x = gapped_tokens(0, 0, 8, 3584, L.Wr, 16)
    for C in (1, 8):
        xd = torch.from_numpy(x[:C].view(np.int16)).to(DEV)
        ids = torch.empty((C, 16), dtype=torch.int32, device=DEV)
        w = torch.empty((C, 16), dtype=torch.float32, device=DEV)
        moe.moe_route(L.h, xd, C, L.Wr_d, None, ids, w, L.ws)
        oids, ow, _ = oracle.route(oracle.router_logits(L.Wr, x[:C]), 16)
        assert (ids.cpu().numpy() == oids).all()
        np.testing.assert_allclose(w.cpu().numpy(), ow, rtol=2e-5, atol=1e-7)


def test_k3_decode_batch1_parity(k3_layer):
    L = k3_layer
    x = gapped_tokens(0, 0, 1, 3584, L.Wr, 16)
    check_layer(L, x, "k3 C=1 top-16")
    check_layer(L, x, "k3 C=1 top-16 fused", fused=True)


@pytest.mark.parametrize("k", [8, 16])
def test_k3_decode_batch7_parity(k3_layer, k):
    L = k3_layer
    if k != 16:
        h = moe.Layer(896, k, 3584, 3072, 8)
        L = _retarget(k3_layer, h, k)
    x = gapped_tokens(1, 0, 7, 3584, L.Wr, k)
    check_layer(L, x, f"k3 C=7 top-{k}")
    check_layer(L, x, f"k3 C=7 top-{k} fused", fused=True)


def test_k3_grouped_zipf_parity(k3_layer):
    # 48 tokens of a Zipf-routed batch on the expert-major path (hot experts
    # chosen by most of the tokens); every token's output against the oracle
    L = k3_layer
    v = _retarget(L, moe.Layer(896, 16, 3584, 3072, 48), 16)
    v.ws = moe.alloc_workspace(v.h, 48)
    v.Wr = synth.router_weights(0, 0, 896, 3584, synth.ZIPF_ROUTER_STD)
    v.bias = synth.zipf_bias(0, 0, 896)
    v.Wr_d = torch.from_numpy(v.Wr).to(DEV)
    v.bias_d = torch.from_numpy(v.bias).to(DEV)
    x = gapped_tokens(3, 0, 48, 3584, v.Wr, 16, bias=v.bias)
    ids, w, y = v.run(x)
    assert moe.moe_get_device_status(v.h, v.ws) == 0
    oids, ow, gap, oy = v.oracle(x, threads=oracle.default_threads())
    assert (ids == oids).all()
    np.testing.assert_allclose(w, ow, rtol=2e-5, atol=1e-7)
    for t in range(48):
        assert_close(y[t:t + 1], oy[t:t + 1], f"k3 grouped zipf token {t}")
    assert_close(y, oy, "k3 grouped zipf, all 48 tokens")


def test_k3_prefill512_parity(k3_layer):
    # the prefill workload as the bench runs it: 512 Zipf-routed tokens in one
    # call (one grouped pass; hot experts split into several column chunks);
    # every token's ids, weights and output against the oracle (its tokens
    # spread over the host cores)
    L = k3_layer
    C = 512
    v = _retarget(L, moe.Layer(896, 16, 3584, 3072, C), 16)
    v.ws = moe.alloc_workspace(v.h, C)
    v.Wr = synth.router_weights(0, 0, 896, 3584, synth.ZIPF_ROUTER_STD)
    v.bias = synth.zipf_bias(0, 0, 896)
    v.Wr_d = torch.from_numpy(v.Wr).to(DEV)
    v.bias_d = torch.from_numpy(v.bias).to(DEV)
    x = gapped_tokens(5, 0, C, 3584, v.Wr, 16, bias=v.bias)
    ids, w, y = v.run_fused(x)
    assert moe.moe_get_device_status(v.h, v.ws) == 0
    oids, ow, gap = oracle.route(oracle.router_logits(v.Wr, x, v.bias), 16)
    assert (ids == oids).all()
    np.testing.assert_allclose(w, ow, rtol=2e-5, atol=1e-7)
    counts = np.bincount(ids.ravel(), minlength=896)
    assert counts.max() > 64                      # a gate/up unit holds 64 pairs: several chunks
    _, _, _, oy = v.oracle(x, threads=oracle.default_threads())
    for t in range(C):
        assert_close(y[t:t + 1], oy[t:t + 1], f"k3 prefill512 token {t}")
    assert_close(y, oy, "k3 prefill512, all 512 tokens")


@pytest.mark.parametrize("C", [1, 7])
def test_k3_zipf_routing_parity(k3_layer, C):
    # the 8-layer workload's routing: a Zipf router bias (per-layer permutation
    # of ranks, s = 1.1) and logit noise of std pi / sqrt(6); hot experts are
    # shared by several tokens of a group
    L = k3_layer
    v = _retarget(L, L.h, 16)
    v.Wr = synth.router_weights(0, 0, 896, 3584, synth.ZIPF_ROUTER_STD)
    v.bias = synth.zipf_bias(0, 0, 896)
    v.Wr_d = torch.from_numpy(v.Wr).to(DEV)
    v.bias_d = torch.from_numpy(v.bias).to(DEV)
    x = gapped_tokens(2, 0, C, 3584, v.Wr, 16, bias=v.bias)
    check_layer(v, x, f"k3 zipf C={C}")
    check_layer(v, x, f"k3 zipf C={C} one call", fused=True)


@pytest.mark.parametrize("r", [2, 4, 8])
def test_k3_verify_pass_parity(k3_layer, r):
    # the multi-row verify pass: r draft rows of one stream (pairwise
    # correlation 0.95) in one call; the rows share most of their experts, so
    # many experts carry several rows (the down kernel's second pass of four
    # token slots runs for experts that more than four rows chose)
    L = k3_layer
    x = gapped_tokens(4, 0, r, 3584, L.Wr, 16, draft_rho=0.95)
    ids, _, _ = L.run(x)
    assert len(set(ids.ravel().tolist())) < 16 * r
    counts = np.bincount(ids.ravel(), minlength=896)
    if r == 8:
        assert counts.max() > 4                  # an expert chosen by more than four rows
    check_layer(L, x, f"k3 verify pass r={r}")
    check_layer(L, x, f"k3 verify pass r={r} one call", fused=True)


def test_tiny_verify_pass_parity():
    L = GpuLayer(32, 4, 256, 192, 8, seed=8)
    x = gapped_tokens(8, 0, 8, 256, L.Wr, 4, draft_rho=0.95)
    check_layer(L, x, "tiny verify pass r=8")


def test_tiny_zipf_routing_parity():
    L = GpuLayer(32, 4, 256, 192, 8, seed=4, router_std=synth.ZIPF_ROUTER_STD, zipf=True)
    x = gapped_tokens(4, 0, 8, 256, L.Wr, 4, bias=L.bias)
    check_layer(L, x, "tiny zipf C=8")


def _retarget(L, h, k):
    """Same weights, another top-k: a new handle over the same packed buffer."""
    class View:
        pass
    v = View()
    v.__dict__.update(L.__dict__)
    v.h, v.k = h, k
    v.ws = moe.alloc_workspace(h, 8)
    v.run = GpuLayer.run.__get__(v)
    v.run_fused = GpuLayer.run_fused.__get__(v)
    v.oracle = GpuLayer.oracle.__get__(v)
    v.host_weights = GpuLayer.host_weights.__get__(v)
    return v


# ------------------------------------------------------------------ MXFP4 weights

def test_device_generator_matches_host_mxfp4():
    E, H, I = 3, 256, 192
    d = synth_dev.canonical_layer_device(0, 5, E, H, I, DEV, fmt="mxfp4")
    h = synth.canonical_layer(0, 5, E, H, I, fmt="mxfp4")
    for n in ("gate", "up", "down"):
        for f in ("codes", "scales", "g"):
            assert (d[n][f].cpu().numpy() == h[n][f]).all(), (n, f)


def _unpack_tiles_mx(buf, ntiles, W, K):
    """MXFP4 tiles -> (rowA codes, rowB codes, rowA scales, rowB scales)."""
    tb = W * 4352
    t = buf[: ntiles * tb].reshape(ntiles, tb)
    codes = t[:, : W * 4096].reshape(ntiles, W, 8, 8, 4, 4, 4).transpose(0, 3, 1, 2, 5, 4, 6)
    S = W * 32
    c = codes.reshape(ntiles, 8, S, 4, 4)
    A = np.empty((ntiles, 8, S, 8), np.uint8)
    B = np.empty((ntiles, 8, S, 8), np.uint8)
    A[..., :4], A[..., 4:] = c[..., 0], c[..., 2]
    B[..., :4], B[..., 4:] = c[..., 1], c[..., 3]
    sc = t[:, W * 4096:].reshape(ntiles, W, 2, 8, 8, 2).transpose(0, 3, 1, 2, 4, 5).reshape(ntiles, 8, W * 16, 2)
    rows = ntiles * 8
    return (A.reshape(rows, S * 8)[:, : K // 2], B.reshape(rows, S * 8)[:, : K // 2],
            sc[..., 0].reshape(rows, W * 16)[:, : K // 32], sc[..., 1].reshape(rows, W * 16)[:, : K // 32])


@pytest.mark.parametrize("E,H,I", [(5, 256, 192), (2, 1024, 576)])
def test_pack_layout_roundtrip_mxfp4(E, H, I):
    L = GpuLayer(E, 2, H, I, 1, fmt="mxfp4")
    packed = L.packed.cpu().numpy()
    assert packed.size == moe.moe_packed_bytes(L.h)
    Wg, Wd = -(-H // 512), -(-I // 512)
    gu_bytes = (I // 8) * Wg * 4352
    ebytes = gu_bytes + (H // 16) * Wd * 4352
    for e in range(E):
        base = e * ebytes
        ga, ub, gs, us = _unpack_tiles_mx(packed[base: base + gu_bytes], I // 8, Wg, H)
        assert (ga == L.canon_h["gate"]["codes"][e]).all() and (ub == L.canon_h["up"]["codes"][e]).all()
        assert (gs == L.canon_h["gate"]["scales"][e]).all() and (us == L.canon_h["up"]["scales"][e]).all()
        da, db, das, dbs = _unpack_tiles_mx(packed[base + gu_bytes: base + ebytes], H // 16, Wd, I)
        assert (da == L.canon_h["down"]["codes"][e][0::2]).all() and (db == L.canon_h["down"]["codes"][e][1::2]).all()
        assert (das == L.canon_h["down"]["scales"][e][0::2]).all()
        assert (dbs == L.canon_h["down"]["scales"][e][1::2]).all()


def test_packed_bytes_mxfp4_k3_shape():
    h = moe.Layer(896, 16, 3584, 3072, 1, flags=moe.CONFIG_MXFP4)
    assert moe.moe_packed_bytes(h) == 896 * (3 * 3072 * 3584 * 17 // 32 + 24) + 16


def test_pack_rejects_nan_scale_mxfp4():
    L = GpuLayer(4, 2, 256, 192, 1, fmt="mxfp4")
    L.canon["up"]["scales"][1, 7, 3] = 0xFF
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_pack_weights(L.h, L.canon, L.packed)
    assert ei.value.status == 3


@pytest.mark.parametrize("C", [1, 2, 3, 8, 11, 20])
def test_mxfp4_tiny_parity(C):
    # C > 8 runs in groups of 8 tokens on the decode kernels
    L = GpuLayer(32, 4, 256, 192, 24, fmt="mxfp4")
    x = gapped_tokens(0, 0, C, 256, L.Wr, 4)
    check_layer(L, x, f"mxfp4 tiny C={C}")


@pytest.mark.parametrize("E,k,H,I,C", [(12, 3, 64, 128, 5), (40, 8, 576, 320, 2), (7, 7, 192, 1088, 1),
                                       (9, 2, 4096, 4096, 3)])
def test_mxfp4_odd_shapes_parity(E, k, H, I, C):
    L = GpuLayer(E, k, H, I, C, seed=3, fmt="mxfp4")
    x = gapped_tokens(3, 0, C, H, L.Wr, k)
    check_layer(L, x, f"mxfp4 E{E} k{k} H{H} I{I} C{C}")


@pytest.fixture(scope="module")
def k3_layer_mx():
    L = GpuLayer(896, 16, 3584, 3072, 8, seed=0, device_gen=True, fmt="mxfp4")
    yield L
    del L.canon


@pytest.mark.parametrize("C,k", [(1, 16), (1, 8), (7, 16), (7, 8)])
def test_k3_mxfp4_parity(k3_layer_mx, C, k):
    # the ggml microbench's shapes: 8 or 16 of the K3-shape experts at C = 1
    # and C = 7, MXFP4
    L = k3_layer_mx if k == 16 else _retarget(k3_layer_mx, moe.Layer(896, k, 3584, 3072, 8, flags=moe.CONFIG_MXFP4), k)
    x = gapped_tokens(6, 0, C, 3584, L.Wr, k)
    check_layer(L, x, f"k3 mxfp4 C={C} top-{k}")
    check_layer(L, x, f"k3 mxfp4 C={C} top-{k} one call", fused=True)
