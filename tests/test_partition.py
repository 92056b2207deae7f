"""The layer's two splits over ranks, on CPU ranks (gloo, world size 2): each
rank evaluates its partial with the float64 oracle, an all-reduce sums the
partials, and the sum must equal the unsplit oracle output.

  expert bands      ("SparkInfer-K3", "How the TP module works")
  intermediate cuts ("Kimi-K3 on the same pod, two engines", "Reason 1 --
                     slice every expert across all eight Sparks")

The partition helpers (band ids, weight slicing) are the library's own
(quantized_moe_expert_router_gb300.partition); the GPU path's partials are
checked in test_gpu_parity.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from quantized_moe_expert_router_gb300 import partition, synth

E, K, H, I, C = 32, 4, 256, 192, 3


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer():
    canon = synth.canonical_layer(0, 0, E, H, I)
    Wr = synth.router_weights(0, 0, E, H)
    x = synth.tokens(0, 0, C, H)
    ids, w, _ = oracle.route(oracle.router_logits(Wr, x), K)
    return canon, x, ids, w


def _band_partial(canon, x, ids, w, lo, hi):
    local = partition.band_ids(ids, lo, hi)
    keep = local >= 0
    # absent slots: any valid index with weight 0 contributes exactly 0
    return oracle.moe_forward(partition.band_weights(canon, lo, hi), x, np.where(keep, local, 0).astype(np.int32),
                              np.where(keep, w, 0.0))


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        canon, x, ids, w = _layer()           # every rank: same weights, same replicated router
        lo, hi = partition.expert_bands(E, world)[rank]
        part = torch.from_numpy(_band_partial(canon, x, ids, w, lo, hi))
        dist.all_reduce(part)
        i0, i1 = partition.intermediate_slices(I, world)[rank]
        sl = torch.from_numpy(oracle.moe_forward(partition.slice_weights(canon, i0, i1), x, ids, w))
        dist.all_reduce(sl)
        if rank == 0:
            np.save(os.path.join(out_dir, "band.npy"), part.numpy())
            np.save(os.path.join(out_dir, "slice.npy"), sl.numpy())
    finally:
        dist.destroy_process_group()


def test_band_and_slice_partials_sum_to_the_layer(tmp_path):
    oracle.build()
    mp.spawn(_rank_main, args=(2, _free_port(), str(tmp_path)), nprocs=2, join=True)
    canon, x, ids, w = _layer()
    y = oracle.moe_forward(canon, x, ids, w)
    band = np.load(tmp_path / "band.npy")
    sl = np.load(tmp_path / "slice.npy")
    np.testing.assert_allclose(band, y, rtol=1e-12, atol=1e-15 * np.abs(y).max())
    np.testing.assert_allclose(sl, y, rtol=1e-11, atol=1e-14 * np.abs(y).max())


def test_band_helpers():
    assert partition.expert_bands(896, 8)[3] == (336, 448)     # the band printed for rank 3
    assert partition.expert_bands(896, 8)[7] == (784, 896)
    ids = np.array([[1, 5, 17, 30]], np.int32)
    assert partition.band_ids(ids, 16, 32).tolist() == [[-1, -1, 1, 14]]
    assert partition.intermediate_slices(3072, 8)[0] == (0, 384)
    with pytest.raises(ValueError):
        partition.intermediate_slices(3072, 100)


def test_slice_weights_shapes():
    canon = synth.canonical_layer(0, 0, 2, 64, 128)
    s = partition.slice_weights(canon, 64, 128)
    assert s["gate"]["codes"].shape == (2, 64, 32) and s["gate"]["scales"].shape == (2, 64, 4)
    assert s["down"]["codes"].shape == (2, 64, 32) and s["down"]["scales"].shape == (2, 64, 4)
    # the two slices' down bytes concatenate back to the full rows
    a = partition.slice_weights(canon, 0, 64)["down"]["codes"]
    assert (np.concatenate([a, s["down"]["codes"]], axis=2) == canon["down"]["codes"]).all()
