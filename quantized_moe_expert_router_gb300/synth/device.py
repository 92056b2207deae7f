"""Device-side synthetic NVFP4 layers (the CUDA twin of the host generator).

Full K3-shape layers (16.6 GB of canonical NVFP4 each) are generated on the
GPU by ``synth.cu``; they are bit-identical to ``canonical_layer`` in this
package's ``__init__`` (a GPU test checks a sample).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

from . import (FFN_GAMMA, FFN_ROUTED_DOWN, FFN_ROUTED_UP, FFN_SHARED, KIND_FFN, MAT_DOWN, MAT_GATE, MAT_UP, W_ABS_MAX,
               W_COEF, _E4M3_MAX, global_scales, key, normals, weight_key)

_LIB_PATH = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                         "_lib", "libmoe_synth.so")
_lock = threading.Lock()
_lib = None


def _load():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(f"{_LIB_PATH} is missing: run the package build first")
            lib = ctypes.CDLL(_LIB_PATH)
            lib.synth_generate_matrices.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_generate_matrices.restype = ctypes.c_int
            lib.synth_generate_matrices_mx.argtypes = [
                ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_double, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
            lib.synth_generate_matrices_mx.restype = ctypes.c_int
            _lib = lib
    return _lib


def canonical_layer_device(seed: int, layer: int, E: int, H: int, I: int, device="cuda:0",
                           stream=None, fmt="nvfp4"):
    """Canonical NVFP4 (or MXFP4) layer on the device: dict gate/up/down ->
    {'codes', 'scales', 'g', 'a'} torch tensors ([E][rows][K/2] uint8,
    [E][rows][K/16] (NVFP4) or [E][rows][K/32] (MXFP4) uint8, [E] float32,
    [E] float32; MXFP4 matrices have g = 1)."""
    lib = _load()
    g, a = global_scales(seed, layer, E, H)
    if fmt == "mxfp4":
        g = np.ones_like(g)
    stream = stream or torch.cuda.current_stream(device)
    out = {}
    for mat, name, rows, K in ((MAT_GATE, "gate", I, H), (MAT_UP, "up", I, H), (MAT_DOWN, "down", H, I)):
        keys = np.array([weight_key(seed, layer, e, mat) for e in range(E)], dtype=np.uint64)
        keys_d = torch.from_numpy(keys.view(np.int64)).to(device)
        g_d = torch.from_numpy(g[mat].copy()).to(device)
        a_d = torch.from_numpy(a[mat].copy()).to(device)
        codes = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=device)
        if fmt == "mxfp4":
            scales = torch.empty((E, rows, K // 32), dtype=torch.uint8, device=device)
            rc = lib.synth_generate_matrices_mx(keys_d.data_ptr(), E, rows, K, W_COEF, codes.data_ptr(),
                                                scales.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        else:
            scales = torch.empty((E, rows, K // 16), dtype=torch.uint8, device=device)
            rc = lib.synth_generate_matrices(keys_d.data_ptr(), g_d.data_ptr(), E, rows, K, W_COEF,
                                             codes.data_ptr(), scales.data_ptr(),
                                             ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"synth_generate_matrices failed with cudaError {rc}")
        out[name] = {"codes": codes, "scales": scales, "g": g_d, "a": a_d, "_keys": keys_d}
    return out


def gather_to_host(canon_dev: dict, experts) -> dict:
    """Copy the listed experts' canonical NVFP4 matrices to host numpy arrays
    (the oracle's input for full-size layers)."""
    idx = torch.as_tensor(list(experts), dtype=torch.long, device=canon_dev["gate"]["codes"].device)
    out = {}
    for name, m in canon_dev.items():
        out[name] = {f: m[f].index_select(0, idx).cpu().numpy() for f in ("codes", "scales", "g", "a")}
    return out


def free(canon_dev: dict) -> None:
    for m in canon_dev.values():
        m.clear()


def ffn_weights_device(seed: int, layer: int, hidden: int, latent: int, shared: int, shared_inter: int,
                       device="cuda:0", stream=None, eps: float = 1e-6) -> dict:
    """The NVFP4 weights around the routed sum on the device, bit-identical to
    ``ffn_weights`` of the host generator (same keys, same global scales,
    same encoder): routed_down / routed_up {'codes','scales','g','a'} (g, a
    one-element tensors), 'shared' in the routed experts' dict form,
    'gamma', 'eps'."""
    lib = _load()
    stream = stream or torch.cuda.current_stream(device)

    def mat(part, idx, rows, K):
        k = torch.tensor([np.uint64(key(seed, KIND_FFN, layer, part, idx)).view(np.int64)], device=device)
        g = np.float32(W_ABS_MAX / (6.0 * _E4M3_MAX) * (1.0 + 0.25 * (idx % 3)))
        g_d = torch.tensor([g], dtype=torch.float32, device=device)
        codes = torch.empty((1, rows, K // 2), dtype=torch.uint8, device=device)
        scales = torch.empty((1, rows, K // 16), dtype=torch.uint8, device=device)
        rc = lib.synth_generate_matrices(k.data_ptr(), g_d.data_ptr(), 1, rows, K, W_COEF, codes.data_ptr(),
                                         scales.data_ptr(), ctypes.c_void_p(stream.cuda_stream))
        if rc != 0:
            raise RuntimeError(f"synth_generate_matrices failed with cudaError {rc}")
        return {"codes": codes[0], "scales": scales[0], "g": g_d,
                "a": torch.ones(1, dtype=torch.float32, device=device)}
    out = {"routed_down": mat(FFN_ROUTED_DOWN, 0, latent, hidden), "routed_up": mat(FFN_ROUTED_UP, 0, hidden, latent)}
    sh = {}
    for m, name, rows, K in ((0, "gate", shared_inter, hidden), (1, "up", shared_inter, hidden),
                             (2, "down", hidden, shared_inter)):
        ms = [mat(FFN_SHARED, 3 * s + m, rows, K) for s in range(shared)]
        sh[name] = {"codes": torch.stack([q["codes"] for q in ms]), "scales": torch.stack([q["scales"] for q in ms]),
                    "g": torch.cat([q["g"] for q in ms]), "a": torch.cat([q["a"] for q in ms])}
    out["shared"] = sh
    z = normals(key(seed, KIND_FFN, layer, FFN_GAMMA, 0), latent)
    out["gamma"] = torch.from_numpy((1.0 + 0.1 * z).astype(np.float32)).to(device)
    out["eps"] = eps
    return out
