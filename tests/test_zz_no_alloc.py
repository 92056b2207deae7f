"""moe_route_noalloc: the router for callers that cannot allocate device
memory (stream capture that forbids cudaMalloc, host frameworks that own all
device buffers, loops that must not pay cudaMalloc's synchronisation).  It
must give what moe_route gives with a caller-allocated workspace, on two
calls in a row (the library's fixed scratch array keeps the previous call's
contents, which must not leak into the next).

This file sorts last so that a run stopping at the first failure has run
every other test before it."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_route_noalloc_matches_route_twice():
    from quantized_moe_expert_router_gb300 import build, moe, synth
    build.build()
    E, k, H = 896, 16, 3584
    layer = moe.Layer(E, k, H, 3072, 8)
    Wr = torch.from_numpy(synth.router_weights(5, 0, E, H)).to(DEV)
    ws = moe.alloc_workspace(layer, 8)
    for call, C in enumerate((8, 3)):            # two calls in a row, different sizes
        x = torch.from_numpy(synth.tokens(5, call, C, H).view(np.int16)).to(DEV)
        ids_ref = torch.empty((C, k), dtype=torch.int32, device=DEV)
        w_ref = torch.empty((C, k), dtype=torch.float32, device=DEV)
        moe.moe_route(layer, x, C, Wr, None, ids_ref, w_ref, ws)
        ids = torch.full((C, k), -1, dtype=torch.int32, device=DEV)
        w = torch.zeros((C, k), dtype=torch.float32, device=DEV)
        moe.moe_route_noalloc(layer, x, C, Wr, None, ids, w)
        torch.cuda.synchronize()
        assert (ids.cpu() == ids_ref.cpu()).all(), f"call {call}: ids differ"
        np.testing.assert_allclose(w.cpu().numpy(), w_ref.cpu().numpy(), rtol=2e-5, atol=1e-7)


def test_route_noalloc_rejects_sizes_beyond_its_scratch():
    from quantized_moe_expert_router_gb300 import build, moe
    build.build()
    layer = moe.Layer(896, 16, 3584, 3072, 16)
    x = torch.zeros((9, 3584), dtype=torch.int16, device=DEV)
    Wr = torch.zeros((896, 3584), dtype=torch.float32, device=DEV)
    ids = torch.empty((9, 16), dtype=torch.int32, device=DEV)
    w = torch.empty((9, 16), dtype=torch.float32, device=DEV)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_route_noalloc(layer, x, 9, Wr, None, ids, w)
    assert ei.value.status == 4     # MOE_ERR_WORKSPACE_TOO_SMALL
