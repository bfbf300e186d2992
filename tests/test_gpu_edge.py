"""Layer-level edge cases of the block-scaled expert path (decode tiles:
kind::mxf4 with six e2m1 activation terms, T = 8; prefill tiles:
kind::mxf8f6f4 with two e4m3 terms, T = 200), against the CPU oracle
through the C ABI:

  * e8m0 scale extremes through the tensor cores: scale bytes 0..2
    (products below the fp32 normal range) and 228..240 (products near the
    top of it) in some groups of the gate, up and down weights, chosen so
    that no exact fp32 partial sum overflows;
  * an all-zero token (c = 0: RMSNorm divides by sqrt(eps) alone);
  * latent groups holding one bf16 outlier 2^20 above the rest of its 32
    (decode tiles: the six-term split adapts its scale per term and keeps
    them; prefill tiles: the two-term e4m3 split is exact within 2^13 of a
    group's maximum, so there the outliers are 2^12 above the rest, and the
    2^20 case is held to the bound that follows from the split's absolute
    error, below 2^-20 of the group maximum, in a test of its own);
  * latent groups found by a search to be the hardest for the six-term
    e2m1 split (largest residual after six terms).

The latent is steered through a one-hot down_proj (lat[l] = x[2l], exact);
the router ignores those positions (zero columns), so the routing gap of
the inputs stays forced."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import TINY
from oracle import oracle as ora

from _cases import GAP, assert_routing_equal, assert_y_close, bf16_f64, bf16_round, gapped_tokens

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D = TINY
BF16_ONE = np.uint16(0x3F80)


def run(layer, x_np):
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y = torch.empty((T, D.hidden), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, D.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, D.top_k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, w, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert layer.status() == 0
    return y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()


def check_h(layer, ref, T):
    """h per slot against the oracle's h: identical on >= 99.5 % of the
    elements and within one bf16 ulp on >= 99.9 % (fp32 against fp64
    accumulation of g and u moves a few roundings, more where g or u
    cancels)."""
    K = D.top_k
    slot = layer.fetch("slot", (T * K,), np.int32)
    h = layer.fetch("h", (T * K, D.inter), np.uint16)
    hg = bf16_f64(h[slot]).reshape(T, K, D.inter)
    hr = bf16_f64(ref["h"])
    assert np.all(np.isfinite(hg))
    assert np.mean(hg == hr) > 0.995
    ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(np.abs(hr), 2.0 ** -126))) - 7).astype(np.int64))
    assert np.mean(np.abs(hg - hr) <= ulp) > 0.999


# ------------------------------------------------------------------ scale extremes
def extreme_scales(w, seed):
    """One group in ~6% of the rows of every expert matrix gets a tiny scale
    byte (0..2) and one in another ~6% a large one (gate/up 228..240, down
    228..236): at most one large group per row, so |partial sums| stay
    below 2^127 for these inputs (|lat| < 8, |h| < 100)."""
    rng = np.random.default_rng(seed)
    w = dict(w)
    for name, hi in (("w1_scale", 240), ("w3_scale", 240), ("w2_scale", 236)):
        sc = w[name].copy()
        E, R, G = sc.shape
        for e in range(E):
            rows = rng.permutation(R)
            n = max(1, R // 16)
            tiny_rows, big_rows = rows[:n], rows[n:2 * n]
            sc[e, tiny_rows, rng.integers(0, G, n)] = rng.integers(0, 3, n)
            sc[e, big_rows, rng.integers(0, G, n)] = rng.integers(228, hi + 1, n)
        w[name] = sc
    return w


@pytest.fixture(scope="module")
def scale_layer():
    w = extreme_scales(synth.layer_weights(D, seed=20), seed=21)
    layer = k3moe.Layer(D, w, max_tokens=256)
    yield w, layer
    layer.close()


@pytest.mark.parametrize("T", [8, 200])
def test_scale_extremes_through_the_tensor_cores(scale_layer, T):
    w, layer = scale_layer
    x = gapped_tokens(D, w, seed=2000 + T, T=T)
    ref = ora.forward(D, w, x, probes=True)
    assert np.abs(ref["c"]).max() > 1e30  # the large scales reach the output
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    check_h(layer, ref, T)
    assert_y_close(y, ref["y"], f"scale extremes T={T}")


# ------------------------------------------------------------------ activation edge cases
def steered_weights(seed):
    """One-hot down_proj (lat[l] = x[2l]) and a router blind to those inputs;
    the bias keeps a gap above GAP at the K-th key of an all-zero token."""
    w = synth.layer_weights(D, seed=seed)
    wd = np.zeros((D.latent, D.hidden), np.uint16)
    wd[np.arange(D.latent), 2 * np.arange(D.latent)] = BF16_ONE
    w["down_proj"] = wd
    rw = w["router_w"].copy()
    rw[:, 0::2] = 0
    w["router_w"] = rw
    b = w["router_bias"].copy()
    order = np.argsort(-b, kind="stable")
    b[order[: D.top_k]] += np.float32(3 * GAP)
    w["router_bias"] = b
    return w


def worst_case_group():
    """A bf16 group whose six-term e2m1 split leaves about the largest
    residual found by a random search refined by hill climbing (1.4e-6 of
    the group maximum; the proved bound is 3^-6)."""
    v = np.array([-5.546875e-01, -1.72615051e-04, 1.34765625e-01, -6.3671875e-01, -4.43359375e-01,
                  -2.23632812e-01, -3.02734375e-01, -6.796875e-01, 2.109375e-01, -3.8671875e-01,
                  -3.34472656e-02, -6.6796875e-01, -6.2109375e-01, 8.69140625e-02, -9.96093750e-02,
                  5.5078125e-01, -2.59765625e-01, 4.8046875e-01, 5.859375e-01, 6.40625e-01, 6.6796875e-01,
                  4.00390625e-01, 6.2109375e-01, -6.5625e-01, 1.93359375e-01, -3.515625e-02, 4.6484375e-01,
                  -8.74023438e-02, 6.71875e-01, -6.796875e-01, -2.71484375e-01, -4.921875e-01])
    return bf16_round(v)


def steered_tokens(w, T, seed, outlier_log2=20):
    x = gapped_tokens(D, w, seed=seed, T=T)
    xf = bf16_f64(x)
    rng = np.random.default_rng(seed)
    G = D.latent // 32
    wc = worst_case_group()
    for t in range(T):
        lat = xf[t, 0::2].reshape(G, 32)
        kind = t % 4
        if kind == 1:  # one outlier 2^20 above the rest of each group
            j = rng.integers(0, 32, G)
            lat[np.arange(G), j] = (np.sign(lat[np.arange(G), j] + 1e-3) * np.ldexp(1.0, outlier_log2)
                                    * np.abs(lat).max())
        elif kind == 2:  # the hard group, scaled and sign-flipped per group
            lat[:] = wc[None, :] * rng.choice([-1.0, 1.0], (G, 1)) * np.ldexp(1.0, rng.integers(-4, 5, (G, 1)))
        elif kind == 3 and t == 3:  # an all-zero token
            xf[t, :] = 0.0
            continue
        xf[t, 0::2] = bf16_round(lat.reshape(-1))
    bits = np.array([ora.bf16_from_double(float(v)) for v in xf.reshape(-1)], np.uint16).reshape(T, D.hidden)
    return bits


@pytest.fixture(scope="module")
def steered_layer():
    w = steered_weights(30)
    layer = k3moe.Layer(D, w, max_tokens=256)
    yield w, layer
    layer.close()


@pytest.mark.parametrize("T,outlier_log2", [(8, 20), (200, 12)], ids=["decode-2^20", "prefill-2^12"])
def test_outliers_worst_case_groups_and_zero_token(steered_layer, T, outlier_log2):
    w, layer = steered_layer
    x = steered_tokens(w, T, seed=3000 + T, outlier_log2=outlier_log2)
    ref = ora.forward(D, w, x, probes=True)
    keys = ora.route(D, x, w["router_w"], w["router_bias"], want_keys=True)[3]
    assert np.all(keys[:, D.top_k - 1].astype(np.float64) - keys[:, D.top_k] > GAP)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    lat = layer.fetch("lat", (T, D.latent), np.uint16)
    assert np.array_equal(lat, ref["lat"])  # the one-hot down_proj is exact
    check_h(layer, ref, T)
    # the all-zero token: c = 0, so n = 0 and y = 0 on both sides
    assert not np.any(bf16_f64(ref["y"][3])) and not np.any(bf16_f64(y[3]))
    assert_y_close(y, ref["y"], f"steered T={T}")


def test_prefill_tiles_with_2e20_outliers_stay_within_the_split_bound(steered_layer):
    """Prefill tiles carry the latent as two e4m3 terms: exact within 2^13
    of a group's maximum, an absolute error below 2^-20 of it for smaller
    elements.  With an outlier 2^20 above the rest of every group, those
    elements are all but dropped, which moves a few SiTU-GLU gates near zero
    (measured: y rel-RMS 1.06e-2 and mean relative error 8.7e-3 on the
    outlier tokens, 3e-4 and 3e-5 on the others).  Held here: routing and
    the zero token exact, every other token within the usual tolerance, the
    outlier tokens within 2e-2 rel-RMS and 1.5e-2 mean relative error."""
    w, layer = steered_layer
    T = 200
    x = steered_tokens(w, T, seed=3200, outlier_log2=20)
    ref = ora.forward(D, w, x, probes=True)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], "prefill 2^20")
    assert not np.any(bf16_f64(y[3]))
    out_tok = np.arange(1, T, 4)
    rest = np.setdiff1d(np.arange(T), out_tok)
    assert_y_close(y[rest], ref["y"][rest], "prefill 2^20, tokens without outliers")
    yg, yr = bf16_f64(y[out_tok]), bf16_f64(ref["y"][out_tok])
    assert np.all(np.isfinite(yg))
    assert np.sqrt(np.mean((yg - yr) ** 2) / np.mean(yr ** 2)) <= 2e-2
    assert np.mean(np.abs(yg - yr)) / np.mean(np.abs(yr)) <= 1.5e-2
