"""Seeded synthetic inputs (binding of csrc/synth/k3synth.c).

Holds no arithmetic of the layer: it only draws numbers.  Recipe (per layer
seed; every tensor has its own counter stream):
  x            ~ N(0, 1) bf16                       (row t of attempt a: stream 1000 + a)
  router_w     ~ N(0, 1/H) bf16                     [E, H]
  router_bias  ~ U(-0.1, 0.1) f32                   [E]   (+2.0 on `hot` experts, if given)
  down_proj    ~ N(0, 1/H) bf16                     [L, H]
  up_proj      ~ N(0, 1/L) bf16                     [H, L]
  norm_w       ~ 1 + N(0, 0.02) bf16                [L]
  w1/w3/w2 packed bytes uniform over 0..255; e8m0 scale bytes uniform in 118..124.
  second bank (dims with bank2_begin > 0): the MXFP4 tensors hold experts
  [0, bank2_begin); experts from there are 2-bit affine: code bytes uniform
  over 0..255, per 64-element group scale s = bf16(0.14 * U(0.7, 1.3)) and
  bias b = bf16(-1.5 s * U(0.9, 1.1)) (weights of RMS ~0.16, like the MXFP4 ones).
  shared experts (when the dims have them; Is = n_shared * shared_inter):
  shared_w1, shared_w3 ~ N(0, 1/H) bf16 [Is, H]; shared_w2 ~ N(0, 1/Is) bf16 [H, Is].
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

from .dims import LayerDims

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth", "k3synth.c")
_SO = os.path.join(_HERE, "_lib", "libk3synth.so")
_lock = threading.Lock()
_lib = None

SYNTH_GCC_FLAGS = ["-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-std=c11"]

S_ROUTER_W, S_BIAS, S_DOWN, S_UP, S_GAMMA = 1, 2, 3, 4, 5
S_W1P, S_W1S, S_W3P, S_W3S, S_W2P, S_W2S = 6, 7, 8, 9, 10, 11
S_HOT = 12
S_SW1, S_SW3, S_SW2 = 13, 14, 15
S_B2 = 16  # second-bank streams: 16 + 3 * matrix + {0 codes, 1 scale, 2 bias}
S_X = 1000
SCALE_LO, SCALE_HI = 118, 124


def compile_synth(out: str = _SO) -> str:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    subprocess.check_call(["gcc", *SYNTH_GCC_FLAGS, _SRC, "-o", out, "-lm"])
    return out


def lib():
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
                compile_synth()
            L = C.CDLL(_SO)
            u64, vp, sz = C.c_uint64, C.c_void_p, C.c_size_t
            L.k3s_counter_u64.restype = u64
            L.k3s_counter_u64.argtypes = [u64, u64, u64]
            L.k3s_normal.restype = C.c_double
            L.k3s_normal.argtypes = [u64, u64, u64]
            L.k3s_fill_bf16_normal.argtypes = [u64, u64, u64, C.c_double, C.c_double, vp, sz]
            L.k3s_fill_f32_uniform.argtypes = [u64, u64, u64, C.c_double, C.c_double, vp, sz]
            L.k3s_fill_u8_full.argtypes = [u64, u64, vp, sz]
            L.k3s_fill_u8_range.argtypes = [u64, u64, C.c_uint8, C.c_uint8, vp, sz]
            L.k3s_permutation.argtypes = [u64, u64, vp, C.c_int]
            L.k3s_num_threads.restype = C.c_int
            _lib = L
    return _lib


def bf16_normal(seed: int, stream: int, shape, mean=0.0, std=1.0, index0: int = 0) -> np.ndarray:
    out = np.empty(shape, np.uint16)
    lib().k3s_fill_bf16_normal(seed, stream, index0, mean, std, out.ctypes.data, out.size)
    return out


def f32_uniform(seed: int, stream: int, shape, lo: float, hi: float) -> np.ndarray:
    out = np.empty(shape, np.float32)
    lib().k3s_fill_f32_uniform(seed, stream, 0, lo, hi, out.ctypes.data, out.size)
    return out


def u8_full(seed: int, stream: int, shape, out: np.ndarray | None = None) -> np.ndarray:
    out = np.empty(shape, np.uint8) if out is None else out
    lib().k3s_fill_u8_full(seed, stream, out.ctypes.data, out.size)
    return out


def u8_range(seed: int, stream: int, shape, lo: int, hi: int) -> np.ndarray:
    out = np.empty(shape, np.uint8)
    lib().k3s_fill_u8_range(seed, stream, lo, hi, out.ctypes.data, out.size)
    return out


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.int32)
    lib().k3s_permutation(seed, stream, out.ctypes.data, n)
    return out


def hot_experts(d: LayerDims, seed: int, n_hot: int) -> np.ndarray:
    """The first n_hot entries of a seeded permutation of the expert ids."""
    return np.sort(permutation(seed, S_HOT, d.n_experts)[:n_hot])


def layer_weights(d: LayerDims, seed: int, n_hot: int = 0, hot_bias: float = 2.0) -> dict:
    H, L, I = d.hidden, d.latent, d.inter
    E = d.n_bank1  # MXFP4 experts (all of them with one bank)
    w = {
        "router_w": bf16_normal(seed, S_ROUTER_W, (d.n_experts, H), 0.0, 1.0 / np.sqrt(H)),
        "down_proj": bf16_normal(seed, S_DOWN, (L, H), 0.0, 1.0 / np.sqrt(H)),
        "w1_packed": u8_full(seed, S_W1P, (E, I, L // 2)),
        "w1_scale": u8_range(seed, S_W1S, (E, I, L // 32), SCALE_LO, SCALE_HI),
        "w3_packed": u8_full(seed, S_W3P, (E, I, L // 2)),
        "w3_scale": u8_range(seed, S_W3S, (E, I, L // 32), SCALE_LO, SCALE_HI),
        "w2_packed": u8_full(seed, S_W2P, (E, L, I // 2)),
        "w2_scale": u8_range(seed, S_W2S, (E, L, I // 32), SCALE_LO, SCALE_HI),
        "norm_w": bf16_normal(seed, S_GAMMA, (L,), 1.0, 0.02),
        "up_proj": bf16_normal(seed, S_UP, (H, L), 0.0, 1.0 / np.sqrt(L)),
    }
    w["router_bias"] = f32_uniform(seed, S_BIAS, (d.n_experts,), -0.1, 0.1)
    if n_hot:
        w["router_bias"][hot_experts(d, seed, n_hot)] = np.float32(hot_bias)
    if d.bank2_begin:
        w.update(bank2_weights(d, seed))
    if d.n_shared:
        w.update(shared_weights(d, seed))
    return w


def bank2_weights(d: LayerDims, seed: int) -> dict:
    """The second bank's 2-bit affine tensors (experts bank2_begin..E-1)."""
    E2, L, I = d.n_experts - d.bank2_begin, d.latent, d.inter
    out = {}
    for m, (name, rows, cols) in enumerate((("w1", I, L), ("w3", I, L), ("w2", L, I))):
        st = S_B2 + 3 * m
        out[f"b2_{name}q"] = u8_full(seed, st, (E2, rows, cols // 4))
        sc = f32_uniform(seed, st + 1, (E2, rows, cols // 64), 0.7, 1.3).astype(np.float64) * 0.14
        bi = -1.5 * sc * f32_uniform(seed, st + 2, (E2, rows, cols // 64), 0.9, 1.1).astype(np.float64)
        out[f"b2_{name}s"] = f32_to_bf16_bits(sc)
        out[f"b2_{name}b"] = f32_to_bf16_bits(bi)
    return out


def f32_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round to bf16 (nearest, ties to even) through float32; inputs here are
    ordinary finite numbers."""
    u = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def shared_weights(d: LayerDims, seed: int) -> dict:
    """The shared experts' bf16 weights alone (the same values layer_weights
    gives dims with shared experts)."""
    H, Is = d.hidden, d.shared_total
    return {"shared_w1": bf16_normal(seed, S_SW1, (Is, H), 0.0, 1.0 / np.sqrt(H)),
            "shared_w3": bf16_normal(seed, S_SW3, (Is, H), 0.0, 1.0 / np.sqrt(H)),
            "shared_w2": bf16_normal(seed, S_SW2, (H, Is), 0.0, 1.0 / np.sqrt(Is))}


def token_rows(d: LayerDims, seed: int, T: int, attempts: np.ndarray | None = None) -> np.ndarray:
    """x [T, H] bf16 ~ N(0,1).  Row t comes from stream S_X + attempts[t]
    (all attempts 0 by default), element index t*H + h, so redrawing one row
    leaves every other row unchanged."""
    H = d.hidden
    x = np.empty((T, H), np.uint16)
    if attempts is None or not np.any(attempts):
        lib().k3s_fill_bf16_normal(seed, S_X, 0, 0.0, 1.0, x.ctypes.data, x.size)
        return x
    for t in range(T):
        a = int(attempts[t])
        lib().k3s_fill_bf16_normal(seed, S_X + a, t * H, 0.0, 1.0, x[t].ctypes.data, H)
    return x


def token_row_into(d: LayerDims, seed: int, t: int, attempt: int, out: np.ndarray) -> None:
    """Row t of attempt `attempt` (the same values token_rows would give it)."""
    assert out.dtype == np.uint16 and out.size == d.hidden and out.flags.c_contiguous
    lib().k3s_fill_bf16_normal(seed, S_X + attempt, t * d.hidden, 0.0, 1.0, out.ctypes.data, d.hidden)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def num_threads() -> int:
    return int(lib().k3s_num_threads())
