"""ctypes wrapper around the plain C oracle (oracle/k3moe_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
CPU-baseline leg of bench.py, never by the product path.  The C file is
compiled on first use if the shared object is missing (gcc, -O2, OpenMP,
no fast-math, no FMA contraction).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k3moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libk3oracle.so")
_lock = threading.Lock()
_lib = None

GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11"]


def compile_oracle(out: str = _SO) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.check_call(["gcc", *GCC_FLAGS, _SRC, "-o", out, "-lm"])
    return out


class OraDims(C.Structure):
    _fields_ = [
        ("hidden", C.c_int), ("latent", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
        ("inter", C.c_int), ("group", C.c_int),
        ("beta", C.c_double), ("beta_lin", C.c_double), ("rms_eps", C.c_double),
        ("routed_scaling", C.c_double), ("norm_topk", C.c_int),
        ("n_shared", C.c_int), ("shared_inter", C.c_int), ("bank2_begin", C.c_int),
    ]


class OraWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in (
        "router_w", "router_bias", "down_proj", "w1_packed", "w1_scale", "w3_packed", "w3_scale",
        "w2_packed", "w2_scale", "norm_w", "up_proj", "shared_w1", "shared_w3", "shared_w2",
        "b2_w1q", "b2_w1s", "b2_w1b", "b2_w3q", "b2_w3s", "b2_w3b", "b2_w2q", "b2_w2s", "b2_w2b")]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
                compile_oracle()
            L = C.CDLL(_SO)
            vp, i32 = C.c_void_p, C.c_int
            L.ora_bf16_to_double.restype = C.c_double
            L.ora_bf16_to_double.argtypes = [C.c_uint16]
            L.ora_bf16_from_double.restype = C.c_uint16
            L.ora_bf16_from_double.argtypes = [C.c_double]
            L.ora_e2m1_value.restype = C.c_double
            L.ora_e2m1_value.argtypes = [C.c_uint]
            L.ora_e8m0_value.restype = C.c_double
            L.ora_e8m0_value.argtypes = [C.c_uint]
            L.ora_situ_glu.restype = C.c_double
            L.ora_situ_glu.argtypes = [C.c_double] * 4
            L.ora_sigmoid.restype = C.c_double
            L.ora_sigmoid.argtypes = [C.c_double]
            L.ora_mxfp4_dequant_bf16.restype = None
            L.ora_mxfp4_dequant_bf16.argtypes = [vp, vp, i32, i32, vp]
            L.ora_forward.restype = None
            L.ora_forward.argtypes = [C.POINTER(OraDims), C.POINTER(OraWeights), vp, i32, vp, vp, vp,
                                      vp, vp, vp, vp, vp, vp, vp, vp]
            L.ora_route.restype = None
            L.ora_route.argtypes = [C.POINTER(OraDims), vp, i32, vp, vp, vp, vp, vp, vp]
            L.ora_route_from_logits.restype = None
            L.ora_route_from_logits.argtypes = [C.POINTER(OraDims), vp, vp, vp, vp, vp]
            L.ora_forward_dense_masked.restype = None
            L.ora_forward_dense_masked.argtypes = [C.POINTER(OraDims), C.POINTER(OraWeights), vp, i32, vp]
            L.ora_reap_saliency.restype = None
            L.ora_reap_saliency.argtypes = [C.POINTER(OraDims), C.POINTER(OraWeights), vp, i32, vp, vp]
            L.ora_forward_partial.restype = None
            L.ora_forward_partial.argtypes = [C.POINTER(OraDims), C.POINTER(OraWeights), vp, i32, i32, i32, vp]
            L.ora_finish.restype = None
            L.ora_finish.argtypes = [C.POINTER(OraDims), C.POINTER(OraWeights), vp, vp, i32, vp]
            L.ora_affine2_element.restype = C.c_double
            L.ora_affine2_element.argtypes = [vp, vp, vp, i32]
            L.ora_num_threads.restype = C.c_int
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data


def dims_struct(d) -> OraDims:
    """`d` is any object with the LayerDims attribute names."""
    return OraDims(d.hidden, d.latent, d.n_experts, d.top_k, d.inter, d.group, float(d.beta),
                   float(d.beta_lin), float(d.rms_eps), float(d.routed_scaling), int(d.norm_topk),
                   int(getattr(d, "n_shared", 0)), int(getattr(d, "shared_inter", 0)),
                   int(getattr(d, "bank2_begin", 0)))


_WEIGHT_DTYPES = {
    "router_w": np.uint16, "router_bias": np.float32, "down_proj": np.uint16,
    "w1_packed": np.uint8, "w1_scale": np.uint8, "w3_packed": np.uint8, "w3_scale": np.uint8,
    "w2_packed": np.uint8, "w2_scale": np.uint8, "norm_w": np.uint16, "up_proj": np.uint16,
    "shared_w1": np.uint16, "shared_w3": np.uint16, "shared_w2": np.uint16,
    "b2_w1q": np.uint8, "b2_w1s": np.uint16, "b2_w1b": np.uint16, "b2_w3q": np.uint8, "b2_w3s": np.uint16,
    "b2_w3b": np.uint16, "b2_w2q": np.uint8, "b2_w2s": np.uint16, "b2_w2b": np.uint16,
}
_OPTIONAL = ("shared_w1", "shared_w3", "shared_w2", "b2_w1q", "b2_w1s", "b2_w1b", "b2_w3q", "b2_w3s", "b2_w3b",
             "b2_w2q", "b2_w2s", "b2_w2b")


def weights_struct(w: dict) -> OraWeights:
    s = OraWeights()
    for name, dt in _WEIGHT_DTYPES.items():
        if name in _OPTIONAL and name not in w:
            setattr(s, name, None)
            continue
        a = w[name]
        assert a.dtype == dt and a.flags.c_contiguous, name
        setattr(s, name, a.ctypes.data)
    return s


# ---------------------------------------------------------------- scalars
def bf16_to_float(bits):
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_from_double(v: float) -> int:
    return int(lib().ora_bf16_from_double(float(v)))


def e2m1_value(code: int) -> float:
    return float(lib().ora_e2m1_value(int(code)))


def e8m0_value(s: int) -> float:
    return float(lib().ora_e8m0_value(int(s)))


def situ_glu(g: float, u: float, beta: float = 4.0, beta_lin: float = 25.0) -> float:
    return float(lib().ora_situ_glu(float(g), float(u), float(beta), float(beta_lin)))


def sigmoid(z: float) -> float:
    return float(lib().ora_sigmoid(float(z)))


# ---------------------------------------------------------------- arrays
def mxfp4_dequant_bf16(packed: np.ndarray, scale: np.ndarray) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    scale = np.ascontiguousarray(scale, dtype=np.uint8)
    rows, half = packed.shape
    cols = half * 2
    assert scale.shape == (rows, cols // 32)
    out = np.empty((rows, cols), dtype=np.uint16)
    lib().ora_mxfp4_dequant_bf16(_p(packed), _p(scale), rows, cols, _p(out))
    return out


def route(dims, x: np.ndarray, router_w: np.ndarray, bias: np.ndarray, want_keys: bool = False):
    """Router only.  Returns (idx [T,K] i32, w [T,K] f32, logits [T,E] f32[, keys [T,K+1]])."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    K, E = dims.top_k, dims.n_experts
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    logits = np.empty((T, E), np.float32)
    keys = np.empty((T, K + 1), np.float32) if want_keys else None
    ds = dims_struct(dims)
    lib().ora_route(C.byref(ds), _p(x), T, _p(np.ascontiguousarray(router_w)),
                    _p(np.ascontiguousarray(bias, dtype=np.float32)), _p(idx), _p(w), _p(logits), _p(keys))
    return (idx, w, logits, keys) if want_keys else (idx, w, logits)


def route_from_logits(dims, logits: np.ndarray, bias: np.ndarray):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T = logits.shape[0]
    K = dims.top_k
    idx = np.empty((T, K), np.int32)
    w = np.empty((T, K), np.float32)
    ds = dims_struct(dims)
    b = np.ascontiguousarray(bias, dtype=np.float32)
    for t in range(T):
        lib().ora_route_from_logits(C.byref(ds), _p(logits[t]), _p(b), _p(idx[t]), _p(w[t]), None)
    return idx, w


def forward(dims, weights: dict, x: np.ndarray, probes: bool = False) -> dict:
    """The whole layer for every row of x.  Returns y, idx, w and, with
    probes=True, the intermediates logits, lat, h [T,K,I], o [T,K,L], c, n
    and, for dims with shared experts, hs [T,Is] and z [T,H]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    H, L, E, K, I = dims.hidden, dims.latent, dims.n_experts, dims.top_k, dims.inter
    out = {
        "y": np.empty((T, H), np.uint16),
        "idx": np.empty((T, K), np.int32),
        "w": np.empty((T, K), np.float32),
    }
    if probes:
        out.update(logits=np.empty((T, E), np.float32), lat=np.empty((T, L), np.uint16),
                   h=np.empty((T, K, I), np.uint16), o=np.empty((T, K, L), np.float64),
                   c=np.empty((T, L), np.float64), n=np.empty((T, L), np.uint16))
        Is = getattr(dims, "n_shared", 0) * getattr(dims, "shared_inter", 0)
        if Is:
            out.update(hs=np.empty((T, Is), np.uint16), z=np.empty((T, H), np.uint16))
    if getattr(dims, "n_shared", 0):
        assert all(n in weights for n in _OPTIONAL[:3]), "dims with shared experts need shared_w1/w3/w2"
    if getattr(dims, "bank2_begin", 0):
        assert all(n in weights for n in _OPTIONAL[3:]), "two-bank dims need the b2_* tensors"
    ds, ws = dims_struct(dims), weights_struct(weights)
    g = out.get
    lib().ora_forward(C.byref(ds), C.byref(ws), _p(x), T, _p(out["y"]), _p(out["idx"]), _p(out["w"]),
                      _p(g("logits")), _p(g("lat")), _p(g("h")), _p(g("o")), _p(g("c")), _p(g("n")),
                      _p(g("hs")), _p(g("z")))
    return out


def forward_dense_masked_c(dims, weights: dict, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.uint16)
    T = x.shape[0]
    c = np.empty((T, dims.latent), np.float64)
    ds, ws = dims_struct(dims), weights_struct(weights)
    lib().ora_forward_dense_masked(C.byref(ds), C.byref(ws), _p(x), T, _p(c))
    return c


def reap_saliency(dims, weights: dict, x: np.ndarray):
    """REAP saliency S [E] of the calibration tokens x and the undivided sums."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    S = np.empty(dims.n_experts, np.float64)
    S_sum = np.empty(dims.n_experts, np.float64)
    ds, ws = dims_struct(dims), weights_struct(weights)
    lib().ora_reap_saliency(C.byref(ds), C.byref(ws), _p(x), x.shape[0], _p(S), _p(S_sum))
    return S, S_sum


def forward_partial(dims, weights: dict, x: np.ndarray, e_begin: int, e_count: int) -> np.ndarray:
    """Partial combine c_r [T, L] (fp64) of the experts [e_begin, e_begin + e_count)."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    c = np.empty((x.shape[0], dims.latent), np.float64)
    ds, ws = dims_struct(dims), weights_struct(weights)
    lib().ora_forward_partial(C.byref(ds), C.byref(ws), _p(x), x.shape[0], int(e_begin), int(e_count), _p(c))
    return c


def finish(dims, weights: dict, x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """y [T, H] bf16 bits from a combine c [T, L]: RMSNorm, up_proj, shared experts."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    c = np.ascontiguousarray(c, dtype=np.float64)
    y = np.empty((x.shape[0], dims.hidden), np.uint16)
    ds, ws = dims_struct(dims), weights_struct(weights)
    lib().ora_finish(C.byref(ds), C.byref(ws), _p(x), _p(c), x.shape[0], _p(y))
    return y


def affine2_element(q_row: np.ndarray, s_row: np.ndarray, b_row: np.ndarray, j: int) -> float:
    q_row = np.ascontiguousarray(q_row, np.uint8)
    s_row = np.ascontiguousarray(s_row, np.uint16)
    b_row = np.ascontiguousarray(b_row, np.uint16)
    return float(lib().ora_affine2_element(_p(q_row), _p(s_row), _p(b_row), int(j)))


def num_threads() -> int:
    return int(lib().ora_num_threads())
