"""Pins of the CPU oracle against facts that do not come from the oracle.

Each check is chosen so that a plausible slip in the oracle (a swapped
nibble, a wrong exponent bias, a dropped term, a transposed operand, a
bias used in the weights, a tie broken the wrong way) fails at least one:

  * MXFP4 dequant: all 256 packed bytes x 256 e8m0 bytes against the
    integer form v = (-1)^s * M[m] * 2^(S-128), M = {0,1,2,3,4,6,8,12}
    (the OCP e2m1 table written as integers), and the low-nibble-first
    order the pages state.
  * bf16 rounding: against torch's float32->bfloat16 conversion and
    hand-made ties.
  * SiTU-GLU: closed-form limits, oddness in u, the SwiGLU limit.
  * Router: sort-based top-k (numpy stable argsort), the pruning invariant
    (-inf bias == expert removed), bias-shift invariance, the hot-expert
    set, the sum of the weights.
  * Whole layer: an independent numpy formulation that evaluates every
    expert for every token with zero weight for unselected ones, and a
    pure-Python brute force on a tiny layer.
  * Work counts: the byte, parameter and PFLOP figures the pages print.
"""
import math

import numpy as np
import pytest
import torch

from mxfp4_routed_expert_k3_gb300 import synth
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY, LayerDims
from oracle import oracle as ora

E2M1_INT = [0, 1, 2, 3, 4, 6, 8, 12]  # e2m1 magnitudes times 2 (OCP MX FP4 table)


# ----------------------------------------------------------------------------- helpers
def exact_mxfp4(byte: int, hi: bool, S: int) -> float:
    code = (byte >> 4) if hi else (byte & 0xF)
    s, m = code >> 3, code & 7
    if S == 255:
        return math.nan
    v = E2M1_INT[m] * 2.0 ** (S - 128)
    return -v if s else v


def bf16_rne_py(v: float) -> float:
    """Round a float to bf16 (8 significant bits, exponent >= -126 normal,
    subnormal spacing 2^-133, overflow to inf), written from the format."""
    if math.isnan(v) or math.isinf(v) or v == 0.0:
        return v
    a = abs(v)
    m, e = math.frexp(a)  # a = m 2^e, m in [0.5, 1)
    E = max(e - 1, -126)
    ulp = 2.0 ** (E - 7)
    r = round(a / ulp) * ulp  # Python round: ties to even
    if r >= 2.0 ** 128:
        r = math.inf
    return math.copysign(r, v)


def bits_to_f64(bits):
    return ora.bf16_to_float(bits)


def f64_to_bits_torch(v: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(v, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ----------------------------------------------------------------------------- dequant
def test_e2m1_table_is_ocp():
    vals = [ora.e2m1_value(c) for c in range(16)]
    expect = [0, .5, 1, 1.5, 2, 3, 4, 6, -0.0, -.5, -1, -1.5, -2, -3, -4, -6]
    assert vals == expect
    assert math.copysign(1.0, vals[8]) == -1.0  # code 0x8 is -0.0


def test_e8m0_scale_values():
    assert ora.e8m0_value(127) == 1.0
    assert ora.e8m0_value(0) == 2.0 ** -127
    assert ora.e8m0_value(254) == 2.0 ** 127
    assert math.isnan(ora.e8m0_value(255))


def test_low_nibble_first():
    # byte 0x21 with scale 1.0: element 0 is the low nibble (code 1 = 0.5),
    # element 1 the high nibble (code 2 = 1.0).
    packed = np.zeros((1, 16), np.uint8)
    packed[0, 0] = 0x21
    scale = np.full((1, 1), 127, np.uint8)
    out = bits_to_f64(ora.mxfp4_dequant_bf16(packed, scale))
    assert out[0, 0] == 0.5 and out[0, 1] == 1.0 and np.all(out[0, 2:] == 0)


def test_dequant_bruteforce_all_bytes_all_scales():
    packed = np.tile(np.arange(256, dtype=np.uint8), (256, 1))  # row S, byte i
    scale = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 512 // 32, axis=1)
    got = ora.mxfp4_dequant_bf16(packed, scale)
    gotf = bits_to_f64(got)
    for S in range(256):
        for b in range(256):
            for hi in (0, 1):
                g = gotf[S, 2 * b + hi]
                x = exact_mxfp4(b, bool(hi), S)
                if math.isnan(x):
                    assert math.isnan(g)
                    continue
                want = bf16_rne_py(x)
                assert g == want or (math.isinf(want) and g == want), (S, b, hi, g, want)
                if S <= 252:
                    assert g == x  # exact: every product is a bf16 value
                if x == 0.0:  # keep the sign of zero
                    assert math.copysign(1.0, g) == math.copysign(1.0, x)


def test_dequant_overflow_only_above_252():
    packed = np.tile(np.arange(256, dtype=np.uint8), (256, 1))
    scale = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 16, axis=1)
    f = bits_to_f64(ora.mxfp4_dequant_bf16(packed, scale))
    assert np.all(np.isfinite(f[:253]))
    assert np.any(np.isinf(f[253])) and np.any(np.isinf(f[254]))
    assert np.all(np.isnan(f[255]))


# ----------------------------------------------------------------------------- bf16
def test_bf16_rounding_matches_torch_on_floats():
    rng = np.random.default_rng(1)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),  # subnormal range
        np.clip(rng.standard_normal(2000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),
        np.array([1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 - 2 ** -9, 3.3895314e38, 2 ** -133, 2 ** -134], np.float32),
    ])
    ours = np.array([ora.bf16_from_double(float(v)) for v in vals], np.uint16)
    ref = f64_to_bits_torch(vals)
    assert np.array_equal(ours, ref)


def test_bf16_rounding_ties_to_even_direct_from_double():
    # 1 + 2^-8 is exactly halfway between 1 and 1 + 2^-7 -> even (1.0)
    assert ora.bf16_from_double(1 + 2 ** -8) == 0x3F80
    # a hair above the tie rounds up; a float detour would have lost the hair
    assert ora.bf16_from_double(1 + 2 ** -8 + 2 ** -40) == 0x3F81
    assert ora.bf16_from_double(1 + 3 * 2 ** -8) == 0x3F82
    assert ora.bf16_from_double(-2.0) == 0xC000
    assert ora.bf16_from_double(1e39) == 0x7F80


# ----------------------------------------------------------------------------- SiTU-GLU
def test_situ_limits():
    for u in (-30.0, -3.0, -0.1, 0.0, 0.5, 7.0, 80.0):
        # g -> +inf: sigmoid -> 1, tanh(g/4) -> 1
        assert ora.situ_glu(60.0, u) == pytest.approx(4 * 25 * math.tanh(u / 25), rel=1e-12, abs=1e-12)
        # g -> -inf: the gate closes
        assert abs(ora.situ_glu(-60.0, u)) < 1e-20
    # |h| < 4 * 25 everywhere
    grid = np.linspace(-200, 200, 81)
    assert max(abs(ora.situ_glu(g, u)) for g in grid for u in grid) < 100.0


def test_situ_odd_in_u_and_swiglu_limit():
    rng = np.random.default_rng(2)
    for g, u in rng.standard_normal((50, 2)) * 5:
        assert ora.situ_glu(g, -u) == -ora.situ_glu(g, u)
    for g, u in rng.standard_normal((50, 2)) * 1e-3:
        silu = g / (1 + math.exp(-g))
        assert ora.situ_glu(g, u) == pytest.approx(silu * u, rel=1e-5)


def test_situ_is_not_symmetric_in_g_and_u():
    # beta = 4 on the gate, beta_lin = 25 on the linear branch: swapping fails
    assert abs(ora.situ_glu(8.0, 2.0) - ora.situ_glu(2.0, 8.0)) > 1.0


# ----------------------------------------------------------------------------- router
def _keys_from_logits(logits, bias):
    s = (1.0 / (1.0 + np.exp(-logits.astype(np.float64)))).astype(np.float32)
    return s, (s + bias.astype(np.float32)).astype(np.float32)


def test_router_topk_matches_sort():
    d = TINY
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((200, d.n_experts)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, d.n_experts).astype(np.float32)
    idx, w = ora.route_from_logits(d, logits, bias)
    s, key = _keys_from_logits(logits, bias)
    for t in range(200):
        order = np.argsort(-key[t], kind="stable")[: d.top_k]
        assert np.array_equal(idx[t], order)
        sel = s[t, order].astype(np.float64)
        assert np.allclose(w[t], sel / sel.sum(), rtol=1e-6)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6
        # the weights use the unbiased score, not the key
        assert not np.allclose(w[t], key[t, order] / key[t, order].sum(), rtol=1e-6)


def test_router_ties_go_to_lower_id():
    d = LayerDims(hidden=64, latent=64, n_experts=8, top_k=3, inter=64)
    logits = np.zeros((1, 8), np.float32)
    bias = np.array([0, 0.5, 0.5, 0, 0.5, 0, 0.5, 0], np.float32)
    idx, _ = ora.route_from_logits(d, logits, bias)
    assert idx[0].tolist() == [1, 2, 4]


def test_router_pruning_invariant_and_bias_shift():
    d = TINY
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((64, d.n_experts)).astype(np.float32)
    bias = rng.uniform(-0.1, 0.1, d.n_experts).astype(np.float32)
    pruned = bias.copy()
    drop = [3, 17, 40]
    pruned[drop] = -np.inf
    idx_p, w_p = ora.route_from_logits(d, logits, pruned)
    keep = np.array([e for e in range(d.n_experts) if e not in drop])
    d_small = d.with_(n_experts=len(keep))
    idx_s, w_s = ora.route_from_logits(d_small, np.ascontiguousarray(logits[:, keep]), bias[keep])
    assert np.array_equal(idx_p, keep[idx_s])
    assert np.array_equal(w_p, w_s)
    # a constant shift of the bias (exact in fp32 here) never changes the selection
    idx0, _ = ora.route_from_logits(d, logits, bias)
    idx1, _ = ora.route_from_logits(d, logits, (bias + np.float32(0.25)).astype(np.float32))
    assert np.array_equal(idx0, idx1)


def test_router_hot_set_and_scaling_options():
    d = TINY
    w = synth.layer_weights(d, seed=7, n_hot=2 * d.top_k)
    hot = synth.hot_experts(d, 7, 2 * d.top_k)
    x = synth.token_rows(d, 70, 16)
    idx, wts, logits = ora.route(d, x, w["router_w"], w["router_bias"])
    assert np.isin(idx, hot).all()
    d0 = d.with_(norm_topk=0, routed_scaling=2.5)
    idx0, w0, _ = ora.route(d0, x, w["router_w"], w["router_bias"])
    assert np.array_equal(idx, idx0)
    s = (1.0 / (1.0 + np.exp(-np.take_along_axis(logits, idx, 1).astype(np.float64)))).astype(np.float32)
    assert np.allclose(w0, s.astype(np.float64) * 2.5, rtol=1e-6)


def _keys_top_by_sort(d, logits, bias):
    """The K+1 largest keys per token by a numpy sort of s + bias (fp32),
    -inf padded when the layer has only K experts."""
    _, key = _keys_from_logits(logits, bias)
    top = -np.sort(-key, axis=1)[:, : d.top_k + 1]
    if top.shape[1] < d.top_k + 1:
        top = np.concatenate([top, np.full((top.shape[0], d.top_k + 1 - top.shape[1]), -np.inf, np.float32)], 1)
    return top


@pytest.mark.parametrize("dims", [TINY, LayerDims(hidden=128, latent=128, n_experts=8, top_k=8, inter=128),
                                  LayerDims(hidden=128, latent=128, n_experts=9, top_k=8, inter=128)],
                         ids=["tiny", "k_equals_e", "k_plus_one_equals_e"])
def test_route_keys_top_match_sort(dims):
    """The K+1 keys the parity tests use as the routing-gap guard are the
    K+1 largest of s + bias, descending, exactly (selection uses the biased
    key, the (K+1)-th slot is filled, and -inf stands in when K == E)."""
    d = dims
    w = synth.layer_weights(d, seed=21)
    x = synth.token_rows(d, 22, 300)
    idx, _, logits, keys = ora.route(d, x, w["router_w"], w["router_bias"], want_keys=True)
    ref = _keys_top_by_sort(d, logits, w["router_bias"])
    assert np.array_equal(keys, ref)
    # the first K keys are those of the selected experts, in the selection order
    _, key = _keys_from_logits(logits, w["router_bias"])
    assert np.array_equal(keys[:, : d.top_k], np.take_along_axis(key, idx, 1))
    gap = keys[:, d.top_k - 1].astype(np.float64) - keys[:, d.top_k].astype(np.float64)
    assert np.all(gap >= 0)
    if d.top_k == d.n_experts:
        assert np.all(np.isinf(gap))


def test_router_logits_match_library_matmul():
    d = TINY
    w = synth.layer_weights(d, seed=1)
    x = synth.token_rows(d, 11, 8)
    _, _, logits = ora.route(d, x, w["router_w"], w["router_bias"])
    ref = (bits_to_f64(x) @ bits_to_f64(w["router_w"]).T).astype(np.float32)
    assert np.max(np.abs(logits.astype(np.float64) - ref) / np.maximum(np.abs(ref), 1e-30)) < 2e-7


# ----------------------------------------------------------------------------- whole layer
def np_dequant(packed, scale):
    """Independent numpy dequant (integer table x 2^(S-128)) -> float64."""
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    mag = np.array(E2M1_INT, np.float64)[codes & 7] * np.where(codes >> 3, -1.0, 1.0)
    sc = np.ldexp(1.0, scale.astype(np.int64) - 128)
    return mag * np.repeat(sc, 32, axis=-1)


def np_bf16(v):
    return np.vectorize(bf16_rne_py, otypes=[np.float64])(v)


def np_layer(d, w, x):
    """Dense all-expert masked formulation of the layer in numpy fp64."""
    xf = bits_to_f64(x)
    logits = (xf @ bits_to_f64(w["router_w"]).T).astype(np.float32)
    s, key = _keys_from_logits(logits, w["router_bias"])
    T = x.shape[0]
    gate = np.zeros((T, d.n_experts))
    for t in range(T):
        sel = np.argsort(-key[t], kind="stable")[: d.top_k]
        wk = (s[t, sel].astype(np.float64) / s[t, sel].astype(np.float64).sum()).astype(np.float32)
        gate[t, sel] = wk.astype(np.float64) * d.routed_scaling
    lat = np_bf16(xf @ bits_to_f64(w["down_proj"]).T)
    c = np.zeros((T, d.latent))
    for e in range(d.n_experts):
        W1 = np_dequant(w["w1_packed"][e], w["w1_scale"][e])
        W3 = np_dequant(w["w3_packed"][e], w["w3_scale"][e])
        W2 = np_dequant(w["w2_packed"][e], w["w2_scale"][e])
        g, u = lat @ W1.T, lat @ W3.T
        h = np_bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
        c += gate[:, e:e + 1] * (h @ W2.T)
    inv = 1.0 / np.sqrt((c * c).mean(axis=1, keepdims=True) + d.rms_eps)
    n = np_bf16(c * inv * bits_to_f64(w["norm_w"]))
    y = np_bf16(n @ bits_to_f64(w["up_proj"]).T)
    return {"c": c, "lat": lat, "n": n, "y": y, "gate": gate}


@pytest.fixture(scope="module")
def tiny_case():
    d = TINY
    w = synth.layer_weights(d, seed=0)
    x = synth.token_rows(d, 100, 12)
    return d, w, x, ora.forward(d, w, x, probes=True)


def test_layer_matches_dense_masked_numpy(tiny_case):
    d, w, x, out = tiny_case
    ref = np_layer(d, w, x)
    assert np.array_equal(bits_to_f64(out["lat"]), ref["lat"])
    rel = np.abs(out["c"] - ref["c"]).max() / np.sqrt((ref["c"] ** 2).mean())
    assert rel < 1e-9
    # n and y are bf16: identical except where fp64 reordering lands on a tie
    assert np.mean(bits_to_f64(out["n"]) == ref["n"]) > 0.999
    yo, yr = bits_to_f64(out["y"]), ref["y"]
    assert np.mean(yo == yr) > 0.999
    assert np.max(np.abs(yo - yr)) / np.sqrt((yr ** 2).mean()) < 1e-2
    # selection and weights agree with the masked formulation
    for t in range(x.shape[0]):
        assert np.array_equal(np.sort(out["idx"][t]), np.flatnonzero(ref["gate"][t]))


def test_layer_sparse_equals_c_dense_masked(tiny_case):
    d, w, x, out = tiny_case
    c_dense = ora.forward_dense_masked_c(d, w, x[:4])
    assert np.allclose(out["c"][:4], c_dense, rtol=1e-12, atol=1e-12)


def test_rmsnorm_removes_routing_weight_scale(tiny_case):
    d, w, x, out = tiny_case
    for dd in (d.with_(norm_topk=0), d.with_(routed_scaling=2.0)):
        o2 = ora.forward(dd, w, x)
        a, b = bits_to_f64(out["y"]), bits_to_f64(o2["y"])
        assert np.array_equal(out["idx"], o2["idx"])
        assert np.abs(a - b).mean() / np.abs(a).mean() < 2e-3


def test_layer_tokens_independent(tiny_case):
    d, w, x, out = tiny_case
    part = ora.forward(d, w, x[5:7])
    assert np.array_equal(part["y"], out["y"][5:7])


def test_brute_force_tiny_layer_pure_python():
    d = LayerDims(hidden=64, latent=64, n_experts=4, top_k=2, inter=64)
    w = synth.layer_weights(d, seed=5)
    x = synth.token_rows(d, 55, 2)
    out = ora.forward(d, w, x, probes=True)
    f = lambda b: float(bits_to_f64(np.uint16(b)))
    for t in range(2):
        xs = [f(v) for v in x[t]]
        logits = []
        for e in range(4):
            acc = math.fsum(xs[j] * f(w["router_w"][e, j]) for j in range(64))
            logits.append(float(np.float32(acc)))
        s = [float(np.float32(1 / (1 + math.exp(-z)))) for z in logits]
        key = [float(np.float32(np.float32(s[e]) + w["router_bias"][e])) for e in range(4)]
        sel = sorted(range(4), key=lambda e: (-key[e], e))[:2]
        assert list(out["idx"][t]) == sel
        wk = [float(np.float32(s[e] / (s[sel[0]] + s[sel[1]]))) for e in sel]
        lat = [bf16_rne_py(math.fsum(f(w["down_proj"][l, j]) * xs[j] for j in range(64))) for l in range(64)]
        c = [0.0] * 64
        for k, e in enumerate(sel):
            def wv(P, Sc, r, j):
                return exact_mxfp4(int(P[e, r, j // 2]), j % 2 == 1, int(Sc[e, r, j // 32]))
            h = []
            for j in range(64):
                g = math.fsum(wv(w["w1_packed"], w["w1_scale"], j, l) * lat[l] for l in range(64))
                u = math.fsum(wv(w["w3_packed"], w["w3_scale"], j, l) * lat[l] for l in range(64))
                h.append(bf16_rne_py(4 * math.tanh(g / 4) / (1 + math.exp(-g)) * 25 * math.tanh(u / 25)))
            assert [bits_to_f64(v) for v in out["h"][t, k]] == h
            for l in range(64):
                o = math.fsum(wv(w["w2_packed"], w["w2_scale"], l, j) * h[j] for j in range(64))
                c[l] += wk[k] * o
        assert np.allclose(out["c"][t], c, rtol=1e-12, atol=1e-14)
        inv = 1 / math.sqrt(math.fsum(v * v for v in c) / 64 + 1e-6)
        n = [bf16_rne_py(c[l] * inv * f(w["norm_w"][l])) for l in range(64)]
        y = [bf16_rne_py(math.fsum(f(w["up_proj"][j, l]) * n[l] for l in range(64))) for j in range(64)]
        assert np.mean(np.array(y) == bits_to_f64(out["y"][t])) > 0.98
        assert np.allclose(bits_to_f64(out["y"][t]), y, rtol=1e-2, atol=1e-2)


# ----------------------------------------------------------------------------- shared experts
def np_shared(d, w, x):
    """The shared experts in numpy fp64, one expert at a time, their outputs
    summed before the single bf16 rounding of the block's shared branch."""
    xf = bits_to_f64(x)
    Ie = d.shared_inter
    zsum = np.zeros((x.shape[0], d.hidden))
    hs = []
    for e in range(d.n_shared):
        rows = slice(e * Ie, (e + 1) * Ie)
        g = xf @ bits_to_f64(w["shared_w1"][rows]).T
        u = xf @ bits_to_f64(w["shared_w3"][rows]).T
        h = np_bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
        hs.append(h)
        zsum += h @ bits_to_f64(w["shared_w2"][:, rows]).T
    return np.concatenate(hs, axis=1), np_bf16(zsum)


@pytest.fixture(scope="module")
def shared_case():
    from mxfp4_routed_expert_k3_gb300.dims import TINY_SHARED
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=3)
    x = synth.token_rows(d, 30, 6)
    return d, w, x, ora.forward(d, w, x, probes=True)


def test_shared_experts_match_numpy_per_expert_sum(shared_case):
    """Shared experts act on the residual x (not the latent), each a SiTU-GLU
    MLP; z = bf16(sum of the experts' outputs) and y = bf16(y_routed + z)."""
    d, w, x, out = shared_case
    hs, z = np_shared(d, w, x)
    assert np.mean(bits_to_f64(out["hs"]) == hs) > 0.999
    zo = bits_to_f64(out["z"])
    assert np.mean(zo == z) > 0.999
    assert np.max(np.abs(zo - z)) <= 2 ** -7 * np.abs(z).max()
    routed = ora.forward(d.with_(n_shared=0, shared_inter=0), w, x)
    y = np_bf16(bits_to_f64(routed["y"]) + zo)
    assert np.array_equal(bits_to_f64(out["y"]), y)
    # the shared branch is a sizeable part of the output on these inputs
    assert np.sqrt(np.mean(zo ** 2)) > 0.1 * np.sqrt(np.mean(bits_to_f64(routed["y"]) ** 2))


def test_shared_experts_zero_weights_leave_routed_output(shared_case):
    d, w, x, _ = shared_case
    w0 = dict(w)
    for n in ("shared_w1", "shared_w3", "shared_w2"):
        w0[n] = np.zeros_like(w[n])
    a = ora.forward(d, w0, x)
    b = ora.forward(d.with_(n_shared=0, shared_inter=0), w, x)
    assert np.array_equal(a["y"], b["y"])
    assert np.array_equal(a["idx"], b["idx"])


def test_shared_experts_brute_force_pure_python():
    d = LayerDims(hidden=64, latent=64, n_experts=4, top_k=2, inter=64, n_shared=2, shared_inter=32)
    w = synth.layer_weights(d, seed=6)
    x = synth.token_rows(d, 66, 1)
    out = ora.forward(d, w, x, probes=True)
    f = lambda b: float(bits_to_f64(np.uint16(b)))
    xs = [f(v) for v in x[0]]
    hs = []
    for j in range(64):
        g = math.fsum(f(w["shared_w1"][j, i]) * xs[i] for i in range(64))
        u = math.fsum(f(w["shared_w3"][j, i]) * xs[i] for i in range(64))
        hs.append(bf16_rne_py(4 * math.tanh(g / 4) / (1 + math.exp(-g)) * 25 * math.tanh(u / 25)))
    assert [bits_to_f64(v) for v in out["hs"][0]] == hs
    z = [bf16_rne_py(math.fsum(f(w["shared_w2"][i, j]) * hs[j] for j in range(64))) for i in range(64)]
    assert [bits_to_f64(v) for v in out["z"][0]] == z


# ----------------------------------------------------------------------------- REAP saliency
def test_reap_saliency_matches_dense_numpy(tiny_case):
    """S_j = mean over tokens of g_j(x) ||e_j(x)||_2 with g_j = 0 for
    unselected experts, from the dense all-expert numpy formulation."""
    d, w, x, _ = tiny_case
    ref = np_layer(d, w, x)
    xf = bits_to_f64(x)
    lat = ref["lat"]
    S_ref = np.zeros(d.n_experts)
    for e in range(d.n_experts):
        W1 = np_dequant(w["w1_packed"][e], w["w1_scale"][e])
        W3 = np_dequant(w["w3_packed"][e], w["w3_scale"][e])
        W2 = np_dequant(w["w2_packed"][e], w["w2_scale"][e])
        g, u = lat @ W1.T, lat @ W3.T
        h = np_bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
        o = h @ W2.T
        S_ref[e] = np.mean(ref["gate"][:, e] * np.linalg.norm(o, axis=1))
    S, S_sum = ora.reap_saliency(d, w, x)
    assert np.allclose(S, S_ref, rtol=1e-9, atol=0)
    assert np.allclose(S_sum, S * x.shape[0], rtol=1e-15)
    assert xf.shape[0] == x.shape[0]
    # experts no token selected score exactly zero
    assert np.array_equal(S == 0, np.all(ref["gate"] == 0, axis=0))


def test_reap_saliency_streams_over_the_calibration_set(tiny_case):
    """The score of a set is the token-weighted mean of its parts' scores
    (the calibration streams batches through the layer) and does not depend
    on the token order."""
    d, w, x, _ = tiny_case
    S, _ = ora.reap_saliency(d, w, x)
    S1, _ = ora.reap_saliency(d, w, x[:5])
    S2, _ = ora.reap_saliency(d, w, x[5:])
    assert np.allclose(S, (5 * S1 + (x.shape[0] - 5) * S2) / x.shape[0], rtol=1e-12, atol=1e-300)
    perm = np.random.default_rng(0).permutation(x.shape[0])
    Sp, _ = ora.reap_saliency(d, w, np.ascontiguousarray(x[perm]))
    assert np.allclose(Sp, S, rtol=1e-12, atol=1e-300)


def test_reap_saliency_of_a_pruned_expert_is_zero(tiny_case):
    """An expert removed by a -inf correction bias (the pruning identity)
    is never selected, so it scores zero."""
    d, w, x, _ = tiny_case
    S, _ = ora.reap_saliency(d, w, x)
    top = int(np.argmax(S))
    w2 = dict(w)
    w2["router_bias"] = w["router_bias"].copy()
    w2["router_bias"][top] = -np.inf
    S2, _ = ora.reap_saliency(d, w2, x)
    assert S[top] > 0 and S2[top] == 0.0


# ----------------------------------------------------------------------------- expert parallelism
def test_expert_shards_sum_to_the_combine(shared_case):
    """The two ranks' partial combines add up to the whole combine, and the
    finish step on that sum gives the block's output exactly."""
    d, w, x, out = shared_case
    h = d.n_experts // 2
    c0 = ora.forward_partial(d, w, x, 0, h)
    c1 = ora.forward_partial(d, w, x, h, d.n_experts - h)
    assert np.allclose(c0 + c1, out["c"], rtol=1e-12, atol=1e-12 * np.abs(out["c"]).max())
    assert np.array_equal(ora.finish(d, w, x, out["c"]), out["y"])
    # a rank whose experts no token selected contributes zero
    sel = np.unique(out["idx"])
    unused = [e for e in range(d.n_experts) if e not in sel]
    if unused:
        assert not np.any(ora.forward_partial(d, w, x, unused[0], 1))
    # uneven shards and one shard of everything
    c_all = ora.forward_partial(d, w, x, 0, d.n_experts)
    assert np.array_equal(c_all, out["c"])
    parts = sum(ora.forward_partial(d, w, x, b, n) for b, n in ((0, 5), (5, 40), (45, d.n_experts - 45)))
    assert np.allclose(parts, out["c"], rtol=1e-12, atol=1e-12 * np.abs(out["c"]).max())


# ----------------------------------------------------------------------------- two-bank experts
def np_affine2(q, sc, bi):
    """Independent numpy dequant of 2-bit affine rows: codes low bits first,
    scale and bias per 64."""
    codes = np.stack([(q >> (2 * i)) & 3 for i in range(4)], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 4)
    return codes * np.repeat(bits_to_f64(sc), 64, axis=-1) + np.repeat(bits_to_f64(bi), 64, axis=-1)


def test_affine2_decode_every_byte():
    q = np.arange(256, dtype=np.uint8)
    rng = np.random.default_rng(9)
    for _ in range(6):
        sc = f64_to_bits_torch(rng.uniform(-2, 2, 1) * 2.0 ** rng.integers(-20, 10))
        bi = f64_to_bits_torch(rng.uniform(-2, 2, 1) * 2.0 ** rng.integers(-20, 10))
        s, b = float(bits_to_f64(sc[0])), float(bits_to_f64(bi[0]))
        for byte in range(256):
            row = np.full(16, byte, np.uint8)
            for j in range(4):
                code = (byte >> (2 * j)) & 3
                assert ora.affine2_element(row, sc, bi, j) == s * code + b
        ref = np_affine2(q[None, :16], sc[None, :], bi[None, :])
        got = [ora.affine2_element(q[:16], sc, bi, j) for j in range(64)]
        assert np.array_equal(ref[0], got)


def mxfp4_twin_of_bank2(d, w, seed):
    """Second-bank tensors holding exactly the values of MXFP4 experts:
    scales 2^k and biases -2^k make every weight one of {-1, 0, 1, 2} 2^k,
    which e2m1 codes {0xA, 0x0, 0x2, 0x4} with e8m0 byte 127 + k store
    exactly.  Returns (two-bank weights, the equivalent one-bank weights)."""
    rng = np.random.default_rng(seed)
    E2 = d.n_experts - d.bank2_begin
    two = dict(w)
    one = dict(w)
    e2m1_of = np.array([0xA, 0x0, 0x2, 0x4], np.uint8)
    for name, rows, cols in (("w1", d.inter, d.latent), ("w3", d.inter, d.latent), ("w2", d.latent, d.inter)):
        q = rng.integers(0, 256, (E2, rows, cols // 4), dtype=np.uint8)
        k = rng.integers(-9, -3, (E2, rows, cols // 64))
        two[f"b2_{name}q"] = q
        two[f"b2_{name}s"] = f64_to_bits_torch(np.ldexp(1.0, k)).reshape(k.shape)
        two[f"b2_{name}b"] = f64_to_bits_torch(-np.ldexp(1.0, k)).reshape(k.shape)
        codes = np.stack([(q >> (2 * i)) & 3 for i in range(4)], -1).reshape(E2, rows, cols)
        nib = e2m1_of[codes]
        packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
        scale = np.repeat((127 + k).astype(np.uint8), 2, axis=-1)
        one[f"{name}_packed"] = np.ascontiguousarray(np.concatenate([w[f"{name}_packed"], packed]))
        one[f"{name}_scale"] = np.ascontiguousarray(np.concatenate([w[f"{name}_scale"], scale]))
    return two, one


def test_two_banks_of_identical_values_match_one_bank():
    """The graded two-bank layer with the second bank holding exactly the
    values of MXFP4 experts equals the one-bank layer, bit for bit (the
    page's own correctness test for the two-bank design)."""
    d2 = TINY.with_(bank2_begin=40)
    w = synth.layer_weights(d2, seed=7)
    two, one = mxfp4_twin_of_bank2(d2, w, 8)
    x = synth.token_rows(TINY, 77, 10)
    a = ora.forward(d2, two, x, probes=True)
    b = ora.forward(TINY, one, x, probes=True)
    assert np.any(a["idx"] >= 40)  # the second bank is used
    for k in ("y", "idx", "w", "h", "n"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(a["o"], b["o"])


def test_two_bank_layer_matches_dense_numpy():
    d = TINY.with_(bank2_begin=40)
    w = synth.layer_weights(d, seed=12)
    x = synth.token_rows(d, 78, 6)
    out = ora.forward(d, w, x, probes=True)
    xf = bits_to_f64(x)
    lat = np_bf16(xf @ bits_to_f64(w["down_proj"]).T)
    assert np.array_equal(bits_to_f64(out["lat"]), lat)
    for t in range(x.shape[0]):
        for k, e in enumerate(out["idx"][t]):
            if e < 40:
                W1 = np_dequant(w["w1_packed"][e], w["w1_scale"][e])
                W3 = np_dequant(w["w3_packed"][e], w["w3_scale"][e])
                W2 = np_dequant(w["w2_packed"][e], w["w2_scale"][e])
            else:
                e2 = e - 40
                W1 = np_affine2(w["b2_w1q"][e2], w["b2_w1s"][e2], w["b2_w1b"][e2])
                W3 = np_affine2(w["b2_w3q"][e2], w["b2_w3s"][e2], w["b2_w3b"][e2])
                W2 = np_affine2(w["b2_w2q"][e2], w["b2_w2s"][e2], w["b2_w2b"][e2])
            g, u = W1 @ lat[t], W3 @ lat[t]
            h = np_bf16(4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25))
            assert np.mean(bits_to_f64(out["h"][t, k]) == h) > 0.99
            o = bits_to_f64(out["h"][t, k]) @ W2.T
            assert np.allclose(out["o"][t, k], o, rtol=1e-12, atol=1e-12 * np.abs(o).max())


# ----------------------------------------------------------------------------- work counts
def test_page_byte_figures(golden):
    g = golden["expert_tensors"]
    assert K3.expert_bytes() == g["bytes_per_expert"] == 17547264
    assert K3.inter * K3.latent // 2 == g["w1_packed"]["bytes"]
    assert K3.inter * (K3.latent // K3.group) == g["w1_scale"]["bytes"]
    assert [K3.latent, K3.inter // 2] == g["w2_packed"]["shape"]
    assert [K3.inter, K3.latent // 32] == g["w1_scale"]["shape"]
    assert golden["tiers"]["mxfp4_expert_bpw"] == 4 + 8 / K3.group
    assert round(K3.n_experts * K3.hidden * 2 / 1e6, 2) == golden["router"]["weight_mb"]


def test_page_parameter_and_flop_figures(golden):
    a = golden["architecture"]
    layers = a["moe_layers"]
    routed = layers * K3.n_experts * 3 * K3.inter * K3.latent
    assert round(routed / 1e9, 1) == a["routed_expert_params_billion"]
    assert round(layers * 2 * K3.hidden * K3.latent / 1e9, 1) == a["latent_up_down_params_billion"]
    for row in golden["reap_compute"]["rows"]:
        tokens = row["seqs"] * row["seqlen"]
        pflop = K3.expert_flop_per_token() * tokens * layers / 1e15
        assert round(pflop, 1) == row["pflop"]
    # per-token routed expert traffic ~= 87 GB - 61 GB from the published builds
    routed_gb = layers * K3.top_k * K3.expert_bytes() / 1e9
    dt = golden["decode_traffic"]
    assert abs(routed_gb - (dt["gb_read_per_token"] - dt["gb_non_expert_per_token"])) < 1.0
