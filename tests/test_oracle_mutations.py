"""The oracle's pins catch plausible mistakes.

Each case copies oracle/k3moe_oracle.c, plants one mistake in the copy (on
the CPU, in a temporary directory), compiles it, and checks that the pin
written for that part of the oracle rejects the mutant while the original
passes.  The mistakes are the ones a reader could make from the pages:
the wrong nibble first, the wrong exponent bias, swapped SiTU temperatures,
the bias leaking into the weights, ties to the higher id, a dropped RMSNorm
epsilon, a transposed down projection, and two slips in the K+1 routing
keys that guard the parity inputs' routing gap (only K keys written,
ranking by the unbiased score), and two in the shared experts (fed the
latent instead of the residual, gate and up weights swapped), and two in the
second bank's 2-bit decode (high bits first, bias dropped).
"""
import ctypes as C
import math
import os
import subprocess

import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import synth
from mxfp4_routed_expert_k3_gb300.dims import LayerDims
from oracle import oracle as ora

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "k3moe_oracle.c")
E2M1_INT = [0, 1, 2, 3, 4, 6, 8, 12]

MUTATIONS = {
    "high_nibble_first": ("unsigned code = (j % 2 == 0) ? (byte & 0x0Fu) : (byte >> 4);",
                          "unsigned code = (j % 2 == 0) ? (byte >> 4) : (byte & 0x0Fu);"),
    "e2m1_bias_0": ("ldexp(1.0 + 0.5 * (double)m, (int)e - 1)", "ldexp(1.0 + 0.5 * (double)m, (int)e)"),
    "e8m0_bias_128": ("return ldexp(1.0, (int)S - 127);", "return ldexp(1.0, (int)S - 128);"),
    "situ_betas_swapped": ("return beta * tanh(g / beta) * ora_sigmoid(g) * beta_lin * tanh(u / beta_lin);",
                           "return beta_lin * tanh(g / beta_lin) * ora_sigmoid(g) * beta * tanh(u / beta);"),
    "bias_in_weights": ("for (int k = 0; k < K; ++k) sum += (double)s[idx[k]];",
                        "for (int k = 0; k < K; ++k) sum += (double)key[idx[k]];"),
    "ties_to_higher_id": ("if (best < 0 || key[e] > key[best]) best = e;",
                          "if (best < 0 || key[e] >= key[best]) best = e;"),
    "rmsnorm_no_eps": ("double inv = 1.0 / sqrt(ms + d->rms_eps);", "double inv = 1.0 / sqrt(ms);"),
    "keys_top_only_k": ("for (int k = 0; k <= K; ++k) {\n        if (k >= E) {",
                        "for (int k = 0; k < K; ++k) {\n        if (k >= E) {"),
    "keys_top_by_score": ("float ke = s[e] + bias[e], kb = best < 0 ? 0.f : s[best] + bias[best];",
                          "float ke = s[e], kb = best < 0 ? 0.f : s[best];"),
    "shared_on_latent": ("        double a = ora_bf16_to_double(x[i]);\n        gs +=",
                         "        double a = ora_bf16_to_double(lat[i % L]);\n        gs +="),
    "shared_gate_up_swapped": ("        gs += ora_bf16_to_double(W->shared_w1[",
                               "        gs += ora_bf16_to_double(W->shared_w3["),
    "bank2_high_bits_first": ("unsigned q = (q_row[j / 4] >> (2 * (j % 4))) & 3u;",
                              "unsigned q = (q_row[j / 4] >> (6 - 2 * (j % 4))) & 3u;"),
    "bank2_bias_dropped": ("return ora_bf16_to_double(s_row[j / 64]) * (double)q + ora_bf16_to_double(b_row[j / 64]);",
                           "return ora_bf16_to_double(s_row[j / 64]) * (double)q;"),
    "down_proj_transposed": ("acc += ora_bf16_to_double(W->down_proj[(size_t)l * H + j]) * ora_bf16_to_double(x[j]);",
                             "acc += ora_bf16_to_double(W->down_proj[(size_t)j * L + l]) * ora_bf16_to_double(x[j]);"),
}


def build_variant(tmp, name):
    src = open(SRC).read()
    if name is not None:
        old, new = MUTATIONS[name]
        assert src.count(old) >= 1, name
        src = src.replace(old, new, 1)
    path = os.path.join(tmp, f"v_{name}.c")
    open(path, "w").write(src)
    so = path[:-2] + ".so"
    subprocess.check_call(["gcc", *ora.GCC_FLAGS, path, "-o", so, "-lm"])
    L = C.CDLL(so)
    L.ora_bf16_to_double.restype = C.c_double
    L.ora_bf16_to_double.argtypes = [C.c_uint16]
    L.ora_situ_glu.restype = C.c_double
    L.ora_situ_glu.argtypes = [C.c_double] * 4
    L.ora_mxfp4_dequant_bf16.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p]
    L.ora_route_from_logits.argtypes = [C.POINTER(ora.OraDims)] + [C.c_void_p] * 5
    L.ora_route.argtypes = [C.POINTER(ora.OraDims), C.c_void_p, C.c_int] + [C.c_void_p] * 6
    L.ora_forward.argtypes = [C.POINTER(ora.OraDims), C.POINTER(ora.OraWeights)] + [C.c_void_p, C.c_int] + \
        [C.c_void_p] * 11
    return L


# ---- the pins, as functions of a compiled variant (True = pin passes)
def pin_dequant(L):
    packed = np.tile(np.arange(256, dtype=np.uint8), (256, 1))
    scale = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 16, axis=1)
    out = np.empty((256, 512), np.uint16)
    L.ora_mxfp4_dequant_bf16(packed.ctypes.data, scale.ctypes.data, 256, 512, out.ctypes.data)
    f = ora.bf16_to_float(out)
    for S in range(0, 253, 7):
        for b in range(256):
            for hi in (0, 1):
                code = (b >> 4) if hi else (b & 0xF)
                v = E2M1_INT[code & 7] * 2.0 ** (S - 128) * (-1 if code >> 3 else 1)
                if f[S, 2 * b + hi] != v:
                    return False
    return True


def pin_situ(L):
    for u in (-3.0, 0.5, 7.0):
        if abs(L.ora_situ_glu(60.0, u, 4.0, 25.0) - 100 * math.tanh(u / 25)) > 1e-9:
            return False
    return True


def pin_router(L):
    d = LayerDims(hidden=64, latent=64, n_experts=8, top_k=3, inter=64)
    ds = ora.dims_struct(d)
    logits = np.zeros(8, np.float32)
    bias = np.array([0, 0.5, 0.5, 0, 0.5, 0, 0.5, 0], np.float32)
    idx = np.empty(3, np.int32)
    w = np.empty(3, np.float32)
    L.ora_route_from_logits(C.byref(ds), logits.ctypes.data, bias.ctypes.data, idx.ctypes.data, w.ctypes.data, None)
    if idx.tolist() != [1, 2, 4]:
        return False
    # the weights use the unbiased score: all selected scores are sigmoid(0)
    return bool(np.allclose(w, 1 / 3, rtol=1e-6))


def pin_keys(L):
    """The K+1 routing keys (the parity tests' gap guard) against a numpy
    sort of s + bias; the output is pre-filled with NaN so that a slot the
    oracle leaves unwritten fails."""
    d = LayerDims(hidden=128, latent=128, n_experts=16, top_k=4, inter=128)
    w = synth.layer_weights(d, seed=23)
    # a bias wide enough to reorder the sigmoid scores
    w["router_bias"] = np.random.default_rng(5).uniform(-0.3, 0.3, d.n_experts).astype(np.float32)
    x = synth.token_rows(d, 24, 64)
    T, E, K = 64, d.n_experts, d.top_k
    idx = np.empty((T, K), np.int32)
    wt = np.empty((T, K), np.float32)
    logits = np.empty((T, E), np.float32)
    keys = np.full((T, K + 1), np.nan, np.float32)
    ds = ora.dims_struct(d)
    L.ora_route(C.byref(ds), x.ctypes.data, T, w["router_w"].ctypes.data, w["router_bias"].ctypes.data,
                idx.ctypes.data, wt.ctypes.data, logits.ctypes.data, keys.ctypes.data)
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    key = (s + w["router_bias"]).astype(np.float32)
    return bool(np.array_equal(keys, -np.sort(-key, axis=1)[:, : K + 1]))


def pin_shared(L):
    """The shared experts against the numpy per-expert formulation."""
    from test_oracle_pins import np_shared
    d = LayerDims(hidden=128, latent=128, n_experts=8, top_k=2, inter=128, n_shared=2, shared_inter=64)
    w = synth.layer_weights(d, seed=14)
    x = synth.token_rows(d, 15, 3)
    T = 3
    y = np.empty((T, d.hidden), np.uint16)
    idx = np.empty((T, d.top_k), np.int32)
    wt = np.empty((T, d.top_k), np.float32)
    z = np.empty((T, d.hidden), np.uint16)
    ds, ws = ora.dims_struct(d), ora.weights_struct(w)
    L.ora_forward(C.byref(ds), C.byref(ws), x.ctypes.data, T, y.ctypes.data, idx.ctypes.data, wt.ctypes.data,
                  None, None, None, None, None, None, None, z.ctypes.data)
    _, zr = np_shared(d, w, x)
    zo = ora.bf16_to_float(z)
    return bool(np.max(np.abs(zo - zr)) <= 2 ** -7 * np.abs(zr).max())


def pin_bank2(L):
    """Second-bank decode against the integer formula on every code byte."""
    L.ora_affine2_element.restype = C.c_double
    L.ora_affine2_element.argtypes = [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int]
    sc = np.array([0x3E00], np.uint16)  # 0.125
    bi = np.array([0xBE40], np.uint16)  # -0.1875
    for byte in range(256):
        row = np.full(16, byte, np.uint8)
        for j in range(4):
            v = L.ora_affine2_element(row.ctypes.data, sc.ctypes.data, bi.ctypes.data, j)
            if v != 0.125 * ((byte >> (2 * j)) & 3) - 0.1875:
                return False
    return True


def pin_layer(L):
    """Against the independent numpy formulation in test_oracle_pins."""
    from test_oracle_pins import np_layer
    # eps of the order of mean(c^2), so that dropping it changes n visibly
    d = LayerDims(hidden=128, latent=128, n_experts=8, top_k=2, inter=128, rms_eps=4.0)
    w = synth.layer_weights(d, seed=12)
    x = synth.token_rows(d, 13, 3)
    ref = np_layer(d, w, x)
    T = 3
    y = np.empty((T, d.hidden), np.uint16)
    idx = np.empty((T, d.top_k), np.int32)
    wt = np.empty((T, d.top_k), np.float32)
    c = np.empty((T, d.latent), np.float64)
    n = np.empty((T, d.latent), np.uint16)
    ds, ws = ora.dims_struct(d), ora.weights_struct(w)
    L.ora_forward(C.byref(ds), C.byref(ws), x.ctypes.data, T, y.ctypes.data, idx.ctypes.data, wt.ctypes.data,
                  None, None, None, None, c.ctypes.data, n.ctypes.data, None, None)
    assert 0.1 < d.rms_eps / np.mean(ref["c"] ** 2) < 10
    yf, nf = ora.bf16_to_float(y), ora.bf16_to_float(n)
    return bool(np.abs(c - ref["c"]).max() < 1e-9 * np.abs(ref["c"]).max()
                and np.abs(nf - ref["n"]).max() <= 2 ** -7 * np.abs(ref["n"]).max()
                and np.abs(yf - ref["y"]).max() <= 2 ** -6 * np.abs(ref["y"]).max())


PIN_OF = {
    "high_nibble_first": pin_dequant, "e2m1_bias_0": pin_dequant, "e8m0_bias_128": pin_dequant,
    "situ_betas_swapped": pin_situ, "bias_in_weights": pin_router, "ties_to_higher_id": pin_router,
    "rmsnorm_no_eps": pin_layer, "down_proj_transposed": pin_layer,
    "keys_top_only_k": pin_keys, "keys_top_by_score": pin_keys,
    "shared_on_latent": pin_shared, "shared_gate_up_swapped": pin_shared,
    "bank2_high_bits_first": pin_bank2, "bank2_bias_dropped": pin_bank2,
}


@pytest.fixture(scope="module")
def tmpdir_mod(tmp_path_factory):
    return str(tmp_path_factory.mktemp("mutants"))


def test_original_passes_every_pin(tmpdir_mod):
    L = build_variant(tmpdir_mod, None)
    for pin in set(PIN_OF.values()):
        assert pin(L), pin.__name__


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pin_rejects_mutant(tmpdir_mod, name):
    L = build_variant(tmpdir_mod, name)
    assert not PIN_OF[name](L), f"mutation {name} was not caught by {PIN_OF[name].__name__}"
