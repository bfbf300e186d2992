"""Python binding of libk3moe (include/k3moe.h): argument marshalling only.

Every step of the layer runs in the library's CUDA kernels; this module
passes pointers and sizes.  torch tensors are accepted for device buffers
(their data_ptr() is passed) and numpy arrays for host buffers.  If the
shared library has not been built the import fails: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from .dims import LayerDims
from .native import LIB

OK, EINVAL, ENOMEM, ECUDA, ETIMEOUT, EBADSCALE, ESTATE = 0, -1, -2, -3, -4, -5, -6
BUF = dict(logits=0, lat=1, counts=2, offsets=3, perm=4, slot=5, h=6, o=7, n=8, active=9, shared_h=10,
           shared_z=11)
Q = dict(workspace_bytes=0, weight_bytes=1, launches_last=2, path_last=3, device=4)
EXPORTS = ["k3moe_create", "k3moe_load_weights", "k3moe_forward", "k3moe_forward_host", "k3moe_status",
           "k3moe_last_error", "k3moe_destroy", "k3moe_mxfp4_dequant", "k3moe_route", "k3moe_fetch",
           "k3moe_query", "k3moe_profile", "k3moe_profile_read", "k3moe_profile_name", "k3moe_route_noalloc",
           "k3moe_saliency", "k3moe_saliency_read", "k3moe_saliency_reset", "k3moe_forward_partial",
           "k3moe_finish", "k3moe_check_guards", "k3moe_test_withhold_copies"]


class K3Error(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"k3moe error {code}: {msg}")
        self.code = code


class Config(C.Structure):
    _fields_ = [("hidden", C.c_int), ("latent", C.c_int), ("n_experts", C.c_int), ("top_k", C.c_int),
                ("inter", C.c_int), ("group", C.c_int), ("beta", C.c_float), ("beta_lin", C.c_float),
                ("rms_eps", C.c_float), ("routed_scaling", C.c_float), ("norm_topk", C.c_int),
                ("max_tokens", C.c_int), ("spin_timeout_ms", C.c_int), ("force_path", C.c_int),
                ("n_shared", C.c_int), ("shared_inter", C.c_int), ("expert_begin", C.c_int),
                ("expert_count", C.c_int), ("bank2_begin", C.c_int)]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("router_w", "router_bias", "down_proj", "w1_packed", "w1_scale",
                                          "w3_packed", "w3_scale", "w2_packed", "w2_scale", "norm_w", "up_proj",
                                          "shared_w1", "shared_w3", "shared_w2", "b2_w1q", "b2_w1s", "b2_w1b",
                                          "b2_w3q", "b2_w3s", "b2_w3b", "b2_w2q", "b2_w2s", "b2_w2b")]


OPTIONAL_WEIGHTS = ("shared_w1", "shared_w3", "shared_w2", "b2_w1q", "b2_w1s", "b2_w1b", "b2_w3q", "b2_w3s",
                    "b2_w3b", "b2_w2q", "b2_w2s", "b2_w2b")


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise ImportError(f"{LIB} is missing: build it with __graft_entry__.build() "
                              "(the layer has no CPU fallback)")
        L = C.CDLL(LIB)
        vp, i32 = C.c_void_p, C.c_int
        L.k3moe_create.argtypes = [C.POINTER(Config), i32, C.POINTER(vp)]
        L.k3moe_load_weights.argtypes = [vp, C.POINTER(Weights)]
        L.k3moe_forward.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.k3moe_forward_host.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.k3moe_status.argtypes = [vp]
        L.k3moe_last_error.argtypes = [vp]
        L.k3moe_last_error.restype = C.c_char_p
        L.k3moe_destroy.argtypes = [vp]
        L.k3moe_destroy.restype = None
        L.k3moe_mxfp4_dequant.argtypes = [vp, vp, i32, i32, vp, i32, vp]
        L.k3moe_route.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, C.c_float, vp, vp, vp, vp]
        L.k3moe_route_noalloc.argtypes = [vp, i32, vp, vp, i32, i32, i32, i32, C.c_float, vp, vp, vp]
        L.k3moe_fetch.argtypes = [vp, i32, vp, C.c_size_t]
        L.k3moe_query.argtypes = [vp, i32, C.POINTER(C.c_longlong)]
        L.k3moe_profile.argtypes = [vp, i32]
        L.k3moe_profile_read.argtypes = [vp, C.POINTER(C.c_float), i32, C.POINTER(C.c_int)]
        L.k3moe_profile_name.argtypes = [vp, i32]
        L.k3moe_profile_name.restype = C.c_char_p
        L.k3moe_saliency.argtypes = [vp, i32]
        L.k3moe_forward_partial.argtypes = [vp, vp, i32, vp, vp, vp, vp]
        L.k3moe_check_guards.argtypes = [vp]
        L.k3moe_test_withhold_copies.argtypes = [vp]
        L.k3moe_finish.argtypes = [vp, vp, vp, i32, vp, vp]
        L.k3moe_saliency_read.argtypes = [vp, vp, i32, C.POINTER(C.c_ulonglong)]
        L.k3moe_saliency_reset.argtypes = [vp]
        for f in ("k3moe_create", "k3moe_load_weights", "k3moe_forward", "k3moe_forward_host", "k3moe_status",
                  "k3moe_mxfp4_dequant", "k3moe_route", "k3moe_route_noalloc", "k3moe_fetch", "k3moe_query",
                  "k3moe_profile", "k3moe_profile_read", "k3moe_saliency", "k3moe_saliency_read",
                  "k3moe_saliency_reset", "k3moe_forward_partial", "k3moe_finish", "k3moe_check_guards",
                  "k3moe_test_withhold_copies"):
            getattr(L, f).restype = C.c_int
        _lib = L
    return _lib


def _ptr(a):
    if a is None:
        return None
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if isinstance(a, np.ndarray):
        return a.ctypes.data
    return int(a)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def last_error(ctx=None) -> str:
    return lib().k3moe_last_error(ctx).decode()


def _check(rc: int, ctx=None):
    if rc != OK:
        raise K3Error(rc, last_error(ctx))


PATH_AUTO, PATH_CUDA_CORE, PATH_BLOCK_SCALED = 0, 1, 4


def make_config(d: LayerDims, max_tokens: int, spin_timeout_ms: int = 0, force_path: int = 0,
                expert_begin: int = 0, expert_count: int = 0) -> Config:
    return Config(d.hidden, d.latent, d.n_experts, d.top_k, d.inter, d.group, d.beta, d.beta_lin, d.rms_eps,
                  d.routed_scaling, int(d.norm_topk), int(max_tokens), int(spin_timeout_ms), int(force_path),
                  int(d.n_shared), int(d.shared_inter), int(expert_begin), int(expert_count),
                  int(d.bank2_begin))


# ------------------------------------------------------------------ raw calls
def create(cfg: Config, device: int = 0):
    h = C.c_void_p()
    _check(lib().k3moe_create(C.byref(cfg), int(device), C.byref(h)))
    return h


def load_weights(ctx, w: dict):
    s = Weights()
    keep = {}
    for name, _ in Weights._fields_:
        if name in OPTIONAL_WEIGHTS and name not in w:
            setattr(s, name, None)
            continue
        a = np.ascontiguousarray(w[name])
        keep[name] = a
        setattr(s, name, a.ctypes.data)
    _check(lib().k3moe_load_weights(ctx, C.byref(s)), ctx)


def forward(ctx, x, T: int, y, topk_idx, topk_w, stream=None):
    _check(lib().k3moe_forward(ctx, _ptr(x), int(T), _ptr(y), _ptr(topk_idx), _ptr(topk_w), _stream(stream)), ctx)


def forward_host(ctx, x_host, T: int, y_host, idx_host=None, w_host=None, stream=None):
    _check(lib().k3moe_forward_host(ctx, _ptr(x_host), int(T), _ptr(y_host), _ptr(idx_host), _ptr(w_host),
                                    _stream(stream)), ctx)


def forward_partial(ctx, x, T: int, c_partial, topk_idx, topk_w, stream=None):
    _check(lib().k3moe_forward_partial(ctx, _ptr(x), int(T), _ptr(c_partial), _ptr(topk_idx), _ptr(topk_w),
                                       _stream(stream)), ctx)


def finish(ctx, x, c_sum, T: int, y, stream=None):
    _check(lib().k3moe_finish(ctx, _ptr(x), _ptr(c_sum), int(T), _ptr(y), _stream(stream)), ctx)


def status(ctx) -> int:
    return int(lib().k3moe_status(ctx))


def destroy(ctx):
    lib().k3moe_destroy(ctx)


def mxfp4_dequant(packed, scale, rows: int, cols: int, out, kind: int = 0, stream=None):
    _check(lib().k3moe_mxfp4_dequant(_ptr(packed), _ptr(scale), int(rows), int(cols), _ptr(out), int(kind),
                                     _stream(stream)))


def route(x, T, router_w, bias, E, H, K, norm_topk, routed_scaling, logits, topk_idx, topk_w, stream=None):
    _check(lib().k3moe_route(_ptr(x), int(T), _ptr(router_w), _ptr(bias), int(E), int(H), int(K), int(norm_topk),
                             float(routed_scaling), _ptr(logits), _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def fetch(ctx, which: str, dst: np.ndarray):
    _check(lib().k3moe_fetch(ctx, BUF[which], dst.ctypes.data, dst.nbytes), ctx)
    return dst


def query(ctx, what: str) -> int:
    v = C.c_longlong()
    _check(lib().k3moe_query(ctx, Q[what], C.byref(v)), ctx)
    return int(v.value)


def profile(ctx, enable: bool = True):
    _check(lib().k3moe_profile(ctx, int(enable)), ctx)


def profile_read(ctx) -> list:
    """[(group name, milliseconds)] of the last forward."""
    buf = (C.c_float * 16)()
    n = C.c_int()
    _check(lib().k3moe_profile_read(ctx, buf, 16, C.byref(n)), ctx)
    return [(lib().k3moe_profile_name(ctx, i).decode(), float(buf[i])) for i in range(min(n.value, 16))]


def saliency(ctx, enable: bool = True):
    _check(lib().k3moe_saliency(ctx, int(enable)), ctx)


def saliency_read(ctx, n_experts: int):
    """(sums [E] float64, tokens): REAP saliency S = sums / tokens."""
    sums = np.empty(n_experts, np.float64)
    tok = C.c_ulonglong()
    _check(lib().k3moe_saliency_read(ctx, sums.ctypes.data, int(n_experts), C.byref(tok)), ctx)
    return sums, int(tok.value)


def saliency_reset(ctx):
    _check(lib().k3moe_saliency_reset(ctx), ctx)


# ------------------------------------------------------------------ convenience
class Layer:
    """One context: create + load_weights on construction, destroy on close."""

    def __init__(self, d: LayerDims, weights: dict, max_tokens: int, device: int = 0, spin_timeout_ms: int = 0,
                 force_path: int = PATH_AUTO, expert_begin: int = 0, expert_count: int = 0):
        """`weights` holds the expert tensors of experts [expert_begin,
        expert_begin + expert_count) only when expert_count > 0 (a shard)."""
        self.d = d
        self.max_tokens = max_tokens
        self.force_path = force_path
        self.ctx = create(make_config(d, max_tokens, spin_timeout_ms, force_path, expert_begin, expert_count),
                          device)
        try:
            load_weights(self.ctx, weights)
        except Exception:
            destroy(self.ctx)
            self.ctx = None
            raise

    def forward(self, x, y, topk_idx, topk_w, stream=None, T=None):
        T = x.shape[0] if T is None else T
        forward(self.ctx, x, T, y, topk_idx, topk_w, stream)

    def forward_torch(self, x, stream=None):
        import torch
        T = x.shape[0]
        y = torch.empty((T, self.d.hidden), dtype=torch.uint16 if hasattr(torch, "uint16") else torch.int16,
                        device=x.device)
        idx = torch.empty((T, self.d.top_k), dtype=torch.int32, device=x.device)
        w = torch.empty((T, self.d.top_k), dtype=torch.float32, device=x.device)
        forward(self.ctx, x, T, y, idx, w, stream if stream is not None else torch.cuda.current_stream())
        return y, idx, w

    def fetch(self, which: str, shape, dtype):
        return fetch(self.ctx, which, np.empty(shape, dtype))

    def query(self, what: str) -> int:
        return query(self.ctx, what)

    def status(self) -> int:
        return status(self.ctx)

    def check_guards(self) -> int:
        return int(lib().k3moe_check_guards(self.ctx))

    def close(self):
        if self.ctx is not None:
            destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
