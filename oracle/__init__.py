"""Float64 CPU oracle for the routed NVFP4 MoE FFN -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The product
package never imports it and has no CPU fallback.  The arithmetic lives in
``moe_oracle.c`` (plain C, float64; one thread, or the (token, slot) expert
evaluations spread over POSIX threads with bit-identical results); this module only compiles it
with gcc and marshals numpy arrays through ctypes.

Each function names the passage it follows in ``moe_oracle.c``.  Parity pins
(tests under ``tests/test_oracle_*.py``) tie it to things other than itself:
the pages' byte count per expert, library decodes of e4m3/bf16, the e2m1 value
set, brute-force routing, closed-form experts, invariants and an independent
float64 torch composition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_NAN_SCALE, ERR_BAD_ID = 0, 1, 2, 3
FMT_NVFP4, FMT_MXFP4 = 0, 1
_FMT = {"nvfp4": FMT_NVFP4, "mxfp4": FMT_MXFP4}


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, -O2, no FMA contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-pthread",
                           "-shared", "-o", tmp, _SRC, "-lm"])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64 = ctypes.c_int, ctypes.c_int64
            lib.oracle_e2m1_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e2m1_value.restype = ctypes.c_double
            lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e4m3_value.restype = ctypes.c_double
            lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
            lib.oracle_e8m0_value.restype = ctypes.c_double
            lib.oracle_dequant_fmt.argtypes = [i32, P, P, ctypes.c_float, i64, i64, P]
            lib.oracle_dequant_fmt.restype = i32
            lib.oracle_expert_ffn_fmt.argtypes = [i32, i32, i32] + [P, P, ctypes.c_float] * 3 + [P, P]
            lib.oracle_expert_ffn_fmt.restype = i32
            lib.oracle_moe_forward_fmt.argtypes = [i32] * 6 + [P, P, P] * 3 + [P, P, P, P]
            lib.oracle_moe_forward_fmt.restype = i32
            lib.oracle_moe_forward_mt_fmt.argtypes = [i32] * 7 + [P, P, P] * 3 + [P, P, P, P]
            lib.oracle_moe_forward_mt_fmt.restype = i32
            lib.oracle_dense_gemv.argtypes = [i32, i32, i32, P, P, ctypes.c_float, i32, P, P]
            lib.oracle_dense_gemv.restype = i32
            lib.oracle_rms_norm.argtypes = [i32, i32, P, P, ctypes.c_double, P]
            lib.oracle_rms_norm.restype = i32
            lib.oracle_bf16_round.argtypes = [ctypes.c_double]
            lib.oracle_bf16_round.restype = ctypes.c_uint16
            lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_value.restype = ctypes.c_double
            lib.oracle_expert_bytes.argtypes = [i64, i64]
            lib.oracle_expert_bytes.restype = ctypes.c_uint64
            lib.oracle_dequant.argtypes = [P, P, ctypes.c_float, i64, i64, P]
            lib.oracle_dequant.restype = i32
            lib.oracle_router_logits.argtypes = [i32, i32, i32, P, P, P, P]
            lib.oracle_router_logits.restype = i32
            lib.oracle_route.argtypes = [i32, i32, i32, P, P, P, P]
            lib.oracle_route.restype = i32
            lib.oracle_expert_ffn.argtypes = [i32, i32] + [P, P, ctypes.c_float] * 3 + [P, P]
            lib.oracle_expert_ffn.restype = i32
            lib.oracle_moe_forward.argtypes = [i32] * 5 + [P, P, P] * 3 + [P, P, P, P]
            lib.oracle_moe_forward.restype = i32
            lib.oracle_moe_forward_mt.argtypes = [i32] * 6 + [P, P, P] * 3 + [P, P, P, P]
            lib.oracle_moe_forward_mt.restype = i32
            lib.oracle_quantize_nvfp4.argtypes = [i32, P, ctypes.c_float, P, P]
            lib.oracle_quantize_nvfp4.restype = i32
            lib.oracle_expert_ffn_w4a4.argtypes = ([i32, i32] + [P, P, ctypes.c_float] * 3 +
                                                   [ctypes.c_float, ctypes.c_float, P, P, P])
            lib.oracle_expert_ffn_w4a4.restype = i32
            lib.oracle_moe_forward_w4a4_mt.argtypes = [i32] * 6 + [P, P, P] * 4 + [P, P, P, P, P]
            lib.oracle_moe_forward_w4a4_mt.restype = i32
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def e2m1_value(nibble: int) -> float:
    return _load().oracle_e2m1_value(nibble)


def e4m3_value(byte: int) -> float:
    return _load().oracle_e4m3_value(byte)


def e8m0_value(byte: int) -> float:
    return _load().oracle_e8m0_value(byte)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def expert_bytes(hidden: int, inter: int) -> int:
    return int(_load().oracle_expert_bytes(hidden, inter))


def dequant(codes, scales, g, rows, K, fmt="nvfp4"):
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    out = np.empty((rows, K), np.float64)
    rc = _load().oracle_dequant_fmt(_FMT[fmt], _ptr(codes), _ptr(scales), float(g), rows, K, _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_dequant failed ({rc})")
    return out


def router_logits(Wr, x_bf16, bias=None):
    """Wr float32 [E][H], x_bf16 uint16 [C][H] -> float64 logits [C][E]."""
    Wr = _c(Wr, np.float32)
    x = _c(x_bf16, np.uint16)
    E, H = Wr.shape
    C = x.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    out = np.empty((C, E), np.float64)
    rc = _load().oracle_router_logits(C, E, H, _ptr(Wr), _ptr(x), _ptr(b), _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_router_logits failed ({rc})")
    return out


def route(logits, k):
    """float64 logits [C][E] -> (ids int32 [C][k] ascending, weights float64 [C][k], gap [C])."""
    logits = _c(logits, np.float64)
    C, E = logits.shape
    ids = np.empty((C, k), np.int32)
    w = np.empty((C, k), np.float64)
    gap = np.empty((C,), np.float64)
    rc = _load().oracle_route(C, E, k, _ptr(logits), _ptr(ids), _ptr(w), _ptr(gap))
    if rc != OK:
        raise ValueError(f"oracle_route failed ({rc})")
    return ids, w, gap


def expert_ffn(H, I, gate, up, down, x, fmt="nvfp4"):
    """gate/up/down = (codes, scales, g) of one expert; x float64 [H] -> y float64 [H]."""
    x = _c(x, np.float64)
    y = np.empty((H,), np.float64)
    mats = []
    args = []
    for m in (gate, up, down):
        c, s = _c(m[0], np.uint8), _c(m[1], np.uint8)
        mats.append((c, s))
        args += [_ptr(c), _ptr(s), float(m[2])]
    rc = _load().oracle_expert_ffn_fmt(_FMT[fmt], H, I, *args, _ptr(x), _ptr(y))
    if rc != OK:
        raise ValueError(f"oracle_expert_ffn failed ({rc})")
    return y


def default_threads() -> int:
    """Host cores this process may use (the threaded oracle's default)."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def moe_forward(weights, x_bf16, ids, w, threads=1, fmt=None):
    """Routed MoE output.

    weights: dict with 'gate', 'up', 'down', each a dict of 'codes' [E][rows][K/2],
    'scales' [E][rows][K/16], 'g' [E] (canonical NVFP4).  x_bf16 uint16 [C][H],
    ids int32 [C][k], w float64 [C][k] -> y float64 [C][H].  ``threads`` > 1
    spreads the (token, slot) expert evaluations over that many POSIX threads
    (oracle_moe_forward_mt) and sums them in slot order as the one-thread
    code does, so the result is bit-for-bit the same.  ``fmt`` names the
    weight format, "nvfp4" (default) or "mxfp4".
    """
    fmt = _FMT[fmt or "nvfp4"]
    gate, up, down = weights["gate"], weights["up"], weights["down"]
    E, I, Hh = gate["codes"].shape
    H = Hh * 2
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    C, k = ids.shape
    keep = []
    args = []
    for m in (gate, up, down):
        c, s, g = _c(m["codes"], np.uint8), _c(m["scales"], np.uint8), _c(m["g"], np.float32)
        keep.append((c, s, g))
        args += [_ptr(c), _ptr(s), _ptr(g)]
    y = np.empty((C, H), np.float64)
    if threads > 1:
        rc = _load().oracle_moe_forward_mt_fmt(fmt, int(threads), C, E, k, H, I, *args, _ptr(x), _ptr(ids), _ptr(w),
                                               _ptr(y))
    else:
        rc = _load().oracle_moe_forward_fmt(fmt, C, E, k, H, I, *args, _ptr(x), _ptr(ids), _ptr(w), _ptr(y))
    if rc != OK:
        raise ValueError(f"oracle_moe_forward failed ({rc})")
    return y


def quantize_nvfp4_act(v, a):
    """NVFP4 quantization of activations with the static input scale a, in
    fp32 as the GPU does it (oracle_quantize_nvfp4): v float32 [..., n] (n a
    multiple of 16) -> (codes uint8 [..., n/2], scales uint8 [..., n/16])."""
    v = _c(v, np.float32)
    n = v.shape[-1]
    rows = v.reshape(-1, n)
    codes = np.empty((rows.shape[0], n // 2), np.uint8)
    scales = np.empty((rows.shape[0], n // 16), np.uint8)
    for i in range(rows.shape[0]):
        r = np.ascontiguousarray(rows[i])
        c, s = codes[i], scales[i]
        rc = _load().oracle_quantize_nvfp4(n, _ptr(r), float(a), _ptr(c), _ptr(s))
        if rc != OK:
            raise ValueError(f"oracle_quantize_nvfp4 failed ({rc})")
    return codes.reshape(v.shape[:-1] + (n // 2,)), scales.reshape(v.shape[:-1] + (n // 16,))


def dequant_nvfp4_act(codes, scales, a):
    """Values of quantized activations: e2m1(code) * e4m3(scale) * a (float64)."""
    codes = np.asarray(codes, np.uint8)
    scales = np.asarray(scales, np.uint8)
    n = codes.shape[-1] * 2
    nib = np.stack([codes & 0x0F, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (n,))
    e2 = np.array([e2m1_value(i) for i in range(16)])[nib]
    e4 = np.array([e4m3_value(i) for i in range(256)])[scales]
    return e2 * np.repeat(e4, 16, axis=-1) * float(np.float32(a))


def expert_ffn_w4a4(H, I, gate, up, down, a_in, a_dn, x, return_act=False):
    """One expert with W4A4 numerics (oracle_expert_ffn_w4a4): gate/up/down =
    (codes, scales, g); x float64 [H] (bf16 values) -> y float64 [H] (and the
    float64 activation [I] when return_act)."""
    x = _c(x, np.float64)
    y = np.empty((H,), np.float64)
    act = np.empty((I,), np.float64)
    keep, args = [], []
    for m in (gate, up, down):
        c, s = _c(m[0], np.uint8), _c(m[1], np.uint8)
        keep.append((c, s))
        args += [_ptr(c), _ptr(s), float(m[2])]
    rc = _load().oracle_expert_ffn_w4a4(H, I, *args, float(a_in), float(a_dn), _ptr(x), _ptr(y), _ptr(act))
    if rc != OK:
        raise ValueError(f"oracle_expert_ffn_w4a4 failed ({rc})")
    return (y, act) if return_act else y


def moe_forward_w4a4(weights, x_bf16, ids, w, threads=1, return_act=False):
    """Routed MoE output with W4A4 numerics (oracle_moe_forward_w4a4_mt):
    weights as for moe_forward (NVFP4) plus each matrix's input scales 'a'
    [E]; x is quantized per (token, expert) with max(gate a, up a), the
    activation h with the down matrix's a.  Returns y float64 [C][H] (and the
    float64 activations [C][k][I] when return_act)."""
    gate, up, down = weights["gate"], weights["up"], weights["down"]
    E, I, Hh = gate["codes"].shape
    H = Hh * 2
    x = _c(x_bf16, np.uint16)
    ids = _c(ids, np.int32)
    w = _c(w, np.float64)
    C, k = ids.shape
    keep, args, scl = [], [], []
    for m in (gate, up, down):
        c, s, g = _c(m["codes"], np.uint8), _c(m["scales"], np.uint8), _c(m["g"], np.float32)
        a = _c(m["a"], np.float32)
        keep.append((c, s, g, a))
        args += [_ptr(c), _ptr(s), _ptr(g)]
        scl.append(_ptr(a))
    y = np.empty((C, H), np.float64)
    act = np.zeros((C, k, I), np.float64)
    rc = _load().oracle_moe_forward_w4a4_mt(int(max(1, threads)), C, E, k, H, I, *args, *scl, _ptr(x), _ptr(ids),
                                            _ptr(w), _ptr(y), _ptr(act))
    if rc != OK:
        raise ValueError(f"oracle_moe_forward_w4a4 failed ({rc})")
    return (y, act) if return_act else y


def full_layer(weights, Wr, x_bf16, k, bias=None, fmt="nvfp4"):
    """Router + top-k + routed FFN for C tokens: returns (ids, w, gap, y)."""
    logits = router_logits(Wr, x_bf16, bias)
    ids, w, gap = route(logits, k)
    y = moe_forward(weights, x_bf16, ids, w, fmt=fmt)
    return ids, w, gap, y


# ------------------------------------------------- around the routed sum

def dense_gemv(codes, scales, g, x, fmt="nvfp4"):
    """y [C][M] = W x for W [M][K] 4-bit (codes [M][K/2], scales, tensor
    scale g) and x float64 [C][K] (oracle_dense_gemv)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8)
    x = _c(np.atleast_2d(x), np.float64)
    M, K = codes.shape[0], codes.shape[1] * 2
    C = x.shape[0]
    y = np.empty((C, M), np.float64)
    rc = _load().oracle_dense_gemv(_FMT[fmt], M, K, _ptr(codes), _ptr(scales), float(g), C, _ptr(x), _ptr(y))
    if rc != OK:
        raise ValueError(f"oracle_dense_gemv failed ({rc})")
    return y


def rms_norm(y, gamma, eps):
    """RMS norm of the rows of y (oracle_rms_norm)."""
    y = _c(np.atleast_2d(y), np.float64)
    gamma = _c(gamma, np.float32)
    out = np.empty_like(y)
    rc = _load().oracle_rms_norm(y.shape[0], y.shape[1], _ptr(y), _ptr(gamma), float(eps), _ptr(out))
    if rc != OK:
        raise ValueError(f"oracle_rms_norm failed ({rc})")
    return out


def bf16_round(v):
    """float64 array -> bfloat16 bits (nearest, ties to even)."""
    v = np.asarray(v, np.float64)
    f = _load().oracle_bf16_round
    return np.array([f(float(a)) for a in v.ravel()], np.uint16).reshape(v.shape)


def bf16_to_f64(bits):
    return np.array([bf16_value(int(b)) for b in np.asarray(bits).ravel()], np.float64).reshape(np.shape(bits))


def ffn_layer(ffn, routed, Wr, u_bf16, k, bias=None, threads=1, fmt="nvfp4", ids_w=None):
    """The MoE FFN of a Kimi-K3-class layer around the routed sum
    ("SparkInfer-K3", "How the TP module works" and "The model"):

      x   = routed_down u           (u: bf16 hidden [C][Hd]; x rounded to bf16)
      ids, w = top-k of the router on x;  y_r = routed sum of the experts on x
      n   = routed_norm(y_r)         (RMS norm with gamma, eps)
      out = routed_up n + sum over the shared experts s of FFN_s(u)

    routed: the experts' canonical dict, or a function mapping a sorted list
    of expert ids to the dict of those experts.
    ffn: dict with 'routed_down' and 'routed_up' ({'codes','scales','g'}),
    'shared' (gate/up/down dicts over the shared experts, as the routed
    weights), 'gamma' float32 [latent], 'eps'.  Returns (ids, w, gap, x_bf16,
    y_r, out).  ``ids_w``: use these (ids, w) instead of the router's."""
    u = np.asarray(u_bf16, np.uint16)
    C = u.shape[0]
    uf = bf16_to_f64(u)
    rd = ffn["routed_down"]
    x_f = dense_gemv(rd["codes"], rd["scales"], rd["g"], uf, fmt)
    x_bf16 = bf16_round(x_f)
    if ids_w is None:
        ids, w, gap = route(router_logits(Wr, x_bf16, bias), k)
    else:
        (ids, w), gap = ids_w, None
    if callable(routed):                       # the experts' weights are fetched for the selected ones
        sel = sorted(set(int(e) for e in np.asarray(ids).ravel()))
        remap = {e: i for i, e in enumerate(sel)}
        y_r = moe_forward(routed(sel), x_bf16, np.vectorize(remap.get)(ids).astype(np.int32), w, threads=threads,
                          fmt=fmt)
    else:
        y_r = moe_forward(routed, x_bf16, ids, w, threads=threads, fmt=fmt)
    n = rms_norm(y_r, ffn["gamma"], ffn["eps"])
    ru = ffn["routed_up"]
    out = dense_gemv(ru["codes"], ru["scales"], ru["g"], n, fmt)
    sh = ffn["shared"]
    Hd = u.shape[1]
    Is = sh["gate"]["codes"].shape[1]
    for s in range(sh["gate"]["codes"].shape[0]):
        mats = [(sh[m]["codes"][s], sh[m]["scales"][s], float(sh[m]["g"][s])) for m in ("gate", "up", "down")]
        for t in range(C):
            out[t] += expert_ffn(Hd, Is, *mats, uf[t], fmt=fmt)
    return ids, w, gap, x_bf16, y_r, out
