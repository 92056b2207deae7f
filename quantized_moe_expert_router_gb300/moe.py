"""Thin ctypes binding of the C ABI in include/moe.h (argument marshalling only).

Every function here has the name of the C entry point it calls.  Tensors are
torch tensors on the layer's CUDA device (PyTorch is used for device memory
and streams only); the computation runs in the library's kernels.  The module
raises if ``_lib/libmoe.so`` is missing: there is no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED_SHAPE",
    3: "MOE_ERR_INVALID_VALUE", 4: "MOE_ERR_WORKSPACE_TOO_SMALL",
    5: "MOE_ERR_OUT_OF_MEMORY", 6: "MOE_ERR_CUDA", 7: "MOE_ERR_DEVICE_TIMEOUT",
    8: "MOE_ERR_BAD_EXPERT_ID",
}
FLAG_BAD_EXPERT_ID = 0x1
FLAG_DUPLICATE_ID = 0x2
FLAG_TIMEOUT = 0x4
CONFIG_TEST_ROUTER_STALL = 0x80000000   # test hook: the router's bounded wait runs out
CONFIG_MXFP4 = 0x1                      # MXFP4 weights (e8m0 scale per 32 elements)
CONFIG_GROUPED_ABOVE_8 = 0x2            # the grouped tcgen05 path for every call of more than 8 tokens
CONFIG_W4A4 = 0x4                       # activations quantized to NVFP4 with each matrix's input scale
ACT_BF16, ACT_F32 = 0, 1                # source types of moe_quantize_nvfp4

EXPORTED = (
    "moe_layer_create", "moe_layer_destroy", "moe_packed_bytes", "moe_workspace_bytes",
    "moe_pack_weights", "moe_route", "moe_forward", "moe_get_device_status",
    "moe_set_stage_events", "moe_route_noalloc", "moe_route_forward",
    "moe_ffn_create", "moe_ffn_destroy", "moe_ffn_packed_bytes", "moe_ffn_workspace_bytes",
    "moe_ffn_pack_weights", "moe_ffn_partial", "moe_ffn_finish", "moe_ffn_forward", "moe_quantize_nvfp4",
    "moe_status_string",
)


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS_NAMES.get(status, status)}")


class moe_config(ctypes.Structure):
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("max_tokens", ctypes.c_int32), ("flags", ctypes.c_uint32)]


class moe_fp4_tensor(ctypes.Structure):
    _fields_ = [("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("global_scale", ctypes.c_void_p), ("input_scale", ctypes.c_void_p)]


class moe_canonical_weights(ctypes.Structure):
    _fields_ = [("gate", moe_fp4_tensor), ("up", moe_fp4_tensor), ("down", moe_fp4_tensor)]


class moe_ffn_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("shared_experts", ctypes.c_int32),
                ("shared_intermediate", ctypes.c_int32), ("eps", ctypes.c_float), ("flags", ctypes.c_uint32)]


class moe_ffn_weights(ctypes.Structure):
    _fields_ = [("routed_down", moe_fp4_tensor), ("routed_up", moe_fp4_tensor),
                ("shared", moe_canonical_weights), ("norm_gamma", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None


def load_library(path: str = LIB_PATH):
    """Load libmoe.so (built by ``build.build()``); raise if it is absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: run quantized_moe_expert_router_gb300.build.build() "
                                   "(there is no CPU fallback)")
            lib = ctypes.CDLL(path)
            P, I32, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            lib.moe_layer_create.argtypes = [ctypes.POINTER(moe_config), I32, ctypes.POINTER(P)]
            lib.moe_layer_destroy.argtypes = [P]
            lib.moe_packed_bytes.argtypes = [P, ctypes.POINTER(SZ)]
            lib.moe_workspace_bytes.argtypes = [P, I32, ctypes.POINTER(SZ)]
            lib.moe_pack_weights.argtypes = [P, ctypes.POINTER(moe_canonical_weights), P, P]
            lib.moe_route.argtypes = [P, P, I32, P, P, P, P, P, SZ, P]
            lib.moe_forward.argtypes = [P, P, I32, P, P, P, P, P, SZ, P]
            lib.moe_get_device_status.argtypes = [P, P, P, ctypes.POINTER(ctypes.c_int32)]
            lib.moe_set_stage_events.argtypes = [P, P, I32]
            lib.moe_route_noalloc.argtypes = [P, P, I32, P, P, P, P, P]
            lib.moe_route_forward.argtypes = [P, P, I32, P, P, P, P, P, P, P, SZ, P]
            lib.moe_ffn_create.argtypes = [ctypes.POINTER(moe_ffn_config), P, ctypes.POINTER(P)]
            lib.moe_ffn_destroy.argtypes = [P]
            lib.moe_ffn_packed_bytes.argtypes = [P, ctypes.POINTER(SZ)]
            lib.moe_ffn_workspace_bytes.argtypes = [P, I32, ctypes.POINTER(SZ)]
            lib.moe_ffn_pack_weights.argtypes = [P, ctypes.POINTER(moe_ffn_weights), P, P]
            lib.moe_ffn_partial.argtypes = [P, P, I32, P, P, P, P, P, P, P, P, SZ, P]
            lib.moe_ffn_finish.argtypes = [P, P, I32, P, P, P, P, SZ, P]
            lib.moe_ffn_forward.argtypes = [P, P, I32, P, P, P, P, P, P, P, P, SZ, P]
            lib.moe_quantize_nvfp4.argtypes = [P, I32, ctypes.c_int64, I32, ctypes.c_float, P, P, P]
            lib.moe_status_string.argtypes = [I32]
            lib.moe_status_string.restype = ctypes.c_char_p
            for name in EXPORTED[:-1]:
                getattr(lib, name).restype = I32
            _lib = lib
    return _lib


def _check(fn, status):
    if status != MOE_OK:
        raise MoEError(fn, status)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


class Layer:
    """Owns one ``moe_layer_t`` handle (host memory only)."""

    def __init__(self, num_experts, top_k, hidden, intermediate, max_tokens, device=0, flags=0):
        lib = load_library()
        self.cfg = moe_config(num_experts, top_k, hidden, intermediate, max_tokens, flags)
        self.device = device
        h = ctypes.c_void_p()
        _check("moe_layer_create", lib.moe_layer_create(ctypes.byref(self.cfg), device, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.moe_layer_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


def moe_layer_create(num_experts, top_k, hidden, intermediate, max_tokens, device=0) -> Layer:
    return Layer(num_experts, top_k, hidden, intermediate, max_tokens, device)


def moe_layer_destroy(layer: Layer) -> None:
    layer.close()


def moe_packed_bytes(layer: Layer) -> int:
    n = ctypes.c_size_t()
    _check("moe_packed_bytes", load_library().moe_packed_bytes(layer.handle, ctypes.byref(n)))
    return n.value


def moe_workspace_bytes(layer: Layer, num_tokens: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_workspace_bytes", load_library().moe_workspace_bytes(layer.handle, num_tokens, ctypes.byref(n)))
    return n.value


def _fp4(m):
    return moe_fp4_tensor(_ptr(m["codes"]), _ptr(m["scales"]), _ptr(m["g"]), _ptr(m["a"]))


def moe_pack_weights(layer: Layer, canon: dict, packed: torch.Tensor, stream=None) -> None:
    """canon: {'gate'|'up'|'down': {'codes','scales','g','a'}} device tensors."""
    cw = moe_canonical_weights(_fp4(canon["gate"]), _fp4(canon["up"]), _fp4(canon["down"]))
    _check("moe_pack_weights", load_library().moe_pack_weights(
        layer.handle, ctypes.byref(cw), _ptr(packed), _stream(stream)))


def moe_route(layer, x, num_tokens, w_router, bias, ids, weights, ws, stream=None) -> None:
    _check("moe_route", load_library().moe_route(
        layer.handle, _ptr(x), num_tokens, _ptr(w_router), _ptr(bias), _ptr(ids), _ptr(weights),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_forward(layer, x, num_tokens, ids, weights, packed, y, ws, stream=None) -> None:
    _check("moe_forward", load_library().moe_forward(
        layer.handle, _ptr(x), num_tokens, _ptr(ids), _ptr(weights), _ptr(packed), _ptr(y),
        _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_forward(layer, x, num_tokens, w_router, bias, packed, ids, weights, y, ws, stream=None) -> None:
    """The whole layer: routing then the routed experts (ids/weights written)."""
    _check("moe_route_forward", load_library().moe_route_forward(
        layer.handle, _ptr(x), num_tokens, _ptr(w_router), _ptr(bias), _ptr(packed), _ptr(ids),
        _ptr(weights), _ptr(y), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_route_noalloc(layer, x, num_tokens, w_router, bias, ids, weights, stream=None) -> None:
    """moe_route for callers that cannot allocate a workspace: the router's
    scratch lives in a fixed array inside the library (C <= 8 tokens).  Calls
    that overlap on the GPU share that array and race; the first call on a
    device must happen outside stream capture."""
    _check("moe_route_noalloc", load_library().moe_route_noalloc(
        layer.handle, _ptr(x), num_tokens, _ptr(w_router), _ptr(bias), _ptr(ids), _ptr(weights),
        _stream(stream)))


def moe_get_device_status(layer, ws, stream=None) -> int:
    f = ctypes.c_int32()
    _check("moe_get_device_status", load_library().moe_get_device_status(
        layer.handle, _ptr(ws), _stream(stream), ctypes.byref(f)))
    return f.value


def moe_set_stage_events(layer, events) -> None:
    lib = load_library()
    if events is None:
        _check("moe_set_stage_events", lib.moe_set_stage_events(layer.handle, None, 0))
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    layer._stage_events = (events, arr)      # keep alive
    _check("moe_set_stage_events", lib.moe_set_stage_events(layer.handle, arr, len(events)))


def moe_quantize_nvfp4(src: torch.Tensor, a: float, codes: torch.Tensor, scales: torch.Tensor, stream=None) -> None:
    """NVFP4 quantization of src [rows][n] (torch.bfloat16, or uint16 bf16
    bits, or torch.float32) with input scale a into codes uint8 [rows][n/2]
    and scales uint8 [rows][n/16] (device tensors)."""
    dtype = ACT_F32 if src.dtype == torch.float32 else ACT_BF16
    if src.dtype not in (torch.float32, torch.bfloat16, torch.uint16, torch.int16):
        raise TypeError(f"moe_quantize_nvfp4: unsupported source dtype {src.dtype}")
    n = src.shape[-1]
    rows = src.numel() // n if n else 0
    _check("moe_quantize_nvfp4", load_library().moe_quantize_nvfp4(
        _ptr(src), dtype, rows, n, float(a), _ptr(codes), _ptr(scales), _stream(stream)))


def moe_status_string(status: int) -> str:
    return load_library().moe_status_string(status).decode()


# ------------------------------------------------------------ conveniences

def alloc_workspace(layer: Layer, num_tokens: int, device=None) -> torch.Tensor:
    """Zero-filled workspace (uint8) of moe_workspace_bytes(num_tokens)."""
    n = moe_workspace_bytes(layer, num_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device or f"cuda:{layer.device}")


def alloc_packed(layer: Layer, device=None) -> torch.Tensor:
    return torch.empty(moe_packed_bytes(layer), dtype=torch.uint8, device=device or f"cuda:{layer.device}")


# ------------------------------------------------ the FFN around the routed sum

class Ffn:
    """Owns one ``moe_ffn_t`` handle tied to a routed ``Layer`` (host memory only)."""

    def __init__(self, routed: Layer, hidden, shared_experts, shared_intermediate, eps=1e-6):
        lib = load_library()
        self.routed = routed
        self.cfg = moe_ffn_config(hidden, shared_experts, shared_intermediate, eps, 0)
        h = ctypes.c_void_p()
        _check("moe_ffn_create", lib.moe_ffn_create(ctypes.byref(self.cfg), routed.handle, ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and _lib is not None:
            _lib.moe_ffn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        self.close()


def moe_ffn_packed_bytes(ffn: Ffn) -> int:
    n = ctypes.c_size_t()
    _check("moe_ffn_packed_bytes", load_library().moe_ffn_packed_bytes(ffn.handle, ctypes.byref(n)))
    return n.value


def moe_ffn_workspace_bytes(ffn: Ffn, num_tokens: int) -> int:
    n = ctypes.c_size_t()
    _check("moe_ffn_workspace_bytes", load_library().moe_ffn_workspace_bytes(ffn.handle, num_tokens, ctypes.byref(n)))
    return n.value


def _fp4_1(m):
    return moe_fp4_tensor(_ptr(m["codes"]), _ptr(m["scales"]), _ptr(m["g"]), _ptr(m["a"]))


def moe_ffn_pack_weights(ffn: Ffn, w: dict, packed: torch.Tensor, stream=None) -> None:
    """w: {'routed_down', 'routed_up': {'codes','scales','g','a'} (g, a: one-element tensors),
    'shared': {'gate'|'up'|'down': ...}, 'gamma'} device tensors."""
    sh = w["shared"]
    cw = moe_ffn_weights(_fp4_1(w["routed_down"]), _fp4_1(w["routed_up"]),
                         moe_canonical_weights(_fp4(sh["gate"]), _fp4(sh["up"]), _fp4(sh["down"])),
                         _ptr(w["gamma"]))
    _check("moe_ffn_pack_weights", load_library().moe_ffn_pack_weights(
        ffn.handle, ctypes.byref(cw), _ptr(packed), _stream(stream)))


def moe_ffn_partial(ffn, u, num_tokens, w_router, bias, routed_packed, ffn_packed, ids, weights, y_routed, ws,
                    stream=None) -> None:
    _check("moe_ffn_partial", load_library().moe_ffn_partial(
        ffn.handle, _ptr(u), num_tokens, _ptr(w_router), _ptr(bias), _ptr(routed_packed), _ptr(ffn_packed),
        _ptr(ids), _ptr(weights), _ptr(y_routed), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def moe_ffn_finish(ffn, u, num_tokens, y_routed, ffn_packed, out, ws, stream=None) -> None:
    _check("moe_ffn_finish", load_library().moe_ffn_finish(
        ffn.handle, _ptr(u), num_tokens, _ptr(y_routed), _ptr(ffn_packed), _ptr(out), _ptr(ws),
        ws.numel() * ws.element_size(), _stream(stream)))


def moe_ffn_forward(ffn, u, num_tokens, w_router, bias, routed_packed, ffn_packed, ids, weights, out, ws,
                    stream=None) -> None:
    _check("moe_ffn_forward", load_library().moe_ffn_forward(
        ffn.handle, _ptr(u), num_tokens, _ptr(w_router), _ptr(bias), _ptr(routed_packed), _ptr(ffn_packed),
        _ptr(ids), _ptr(weights), _ptr(out), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream)))


def alloc_ffn_workspace(ffn: Ffn, num_tokens: int, device=None) -> torch.Tensor:
    n = moe_ffn_workspace_bytes(ffn, num_tokens)
    return torch.zeros(n, dtype=torch.uint8, device=device or f"cuda:{ffn.routed.device}")


def alloc_ffn_packed(ffn: Ffn, device=None) -> torch.Tensor:
    return torch.empty(moe_ffn_packed_bytes(ffn), dtype=torch.uint8, device=device or f"cuda:{ffn.routed.device}")
