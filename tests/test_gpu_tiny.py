"""GPU parity on the tiny layer (H=1024, L=512, E=64, top-8, I=384): every
step of the CUDA path against the CPU oracle, element by element, through
the C ABI."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import TINY, LayerDims
from oracle import oracle as ora

from _cases import (assert_routing_equal, assert_y_close, bf16_f64, bf16_round, bf16_ulp, expert_matrix,
                    gapped_tokens, stable_permutation, y_metrics)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAXT = 320


@pytest.fixture(scope="module",
                params=[k3moe.PATH_AUTO, k3moe.PATH_CUDA_CORE], ids=["auto", "cudacore"])
def tiny(request):
    d = TINY
    w = synth.layer_weights(d, seed=0)
    layer = k3moe.Layer(d, w, max_tokens=MAXT, force_path=request.param)
    yield d, w, layer
    layer.close()


def run(layer, x_np):
    d = layer.d
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y = torch.empty((T, d.hidden), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    layer.forward(x, y, idx, w, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert layer.status() == 0
    return y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()


@pytest.mark.parametrize("T", [1, 3, 32, 77, 128, 200, MAXT])
def test_tiny_layer_matches_oracle(tiny, T):
    d, w, layer = tiny
    x = gapped_tokens(d, w, seed=100 + T, T=T)
    ref = ora.forward(d, w, x, probes=True)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    # intermediates, step by step
    logits = layer.fetch("logits", (T, d.n_experts), np.float32)
    assert np.allclose(logits, ref["logits"], rtol=1e-5, atol=1e-5)
    lat = layer.fetch("lat", (T, d.latent), np.uint16)
    lg, lr = bf16_f64(lat), bf16_f64(ref["lat"])
    assert np.mean(lg == lr) > 0.995
    assert np.max(np.abs(lg - lr) / np.maximum(np.abs(lr), 1e-3)) <= 2 ** -7
    counts, offsets, perm, slot = stable_permutation(idx, d.n_experts)
    assert np.array_equal(layer.fetch("counts", (d.n_experts,), np.int32), counts)
    assert np.array_equal(layer.fetch("offsets", (d.n_experts + 1,), np.int32), offsets)
    assert np.array_equal(layer.fetch("perm", (T * d.top_k,), np.int32), perm)
    assert np.array_equal(layer.fetch("slot", (T * d.top_k,), np.int32), slot)
    active = layer.fetch("active", (d.n_experts + 1,), np.int32)
    assert active[0] == np.count_nonzero(counts)
    assert np.array_equal(active[1:1 + active[0]], np.flatnonzero(counts))
    # h and o per slot, each against the oracle's arithmetic applied to the
    # GPU's own input of that step (so a one-ulp bf16 flip upstream does not
    # hide or fake an error here)
    h = layer.fetch("h", (T * d.top_k, d.inter), np.uint16)
    o = layer.fetch("o", (T * d.top_k, d.latent), np.float32)
    situ = np.vectorize(lambda g, u: ora.situ_glu(g, u, d.beta, d.beta_lin), otypes=[np.float64])
    for e in np.unique(idx):
        sl = np.flatnonzero(idx.reshape(-1) == e)  # assignments t*K+k of expert e
        s_of = slot[sl]
        W1, W3, W2 = (expert_matrix(w, n, e) for n in ("w1", "w3", "w2"))
        xl = lg[sl // d.top_k]
        h_ref = bf16_round(situ(xl @ W1.T, xl @ W3.T))
        hg = bf16_f64(h[s_of])
        assert np.mean(hg == h_ref) > 0.995, e
        # one bf16 ulp, plus an fp32-accumulation floor: where g or u cancel to
        # near zero, h is small and fp32 vs fp64 sums differ by several of its ulps
        floor = 1e-4 * np.sqrt(np.mean(h_ref ** 2))
        assert np.all(np.abs(hg - h_ref) <= bf16_ulp(h_ref) + floor), e
        o_ref = hg @ W2.T
        assert np.max(np.abs(o[s_of] - o_ref)) <= 2e-5 * np.sqrt(np.mean(o_ref ** 2)) + 1e-6, e
    n = layer.fetch("n", (T, d.latent), np.uint16)
    # n is bf16 after two bf16 roundings upstream (lat, h): one-ulp flips there
    # move c by ~1e-4 relative and flip a few percent of n's roundings
    nn, nr = bf16_f64(n), bf16_f64(ref["n"])
    assert np.mean(nn == nr) > 0.95
    assert np.sqrt(np.mean((nn - nr) ** 2) / np.mean(nr ** 2)) < 2e-3
    m = assert_y_close(y, ref["y"], f"T={T}")
    print(f"T={T}", m)


def test_tiny_zero_and_too_many_tokens(tiny):
    d, w, layer = tiny
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    k3moe.forward(layer.ctx, dummy, 0, dummy, dummy, dummy)  # T = 0: no-op
    assert layer.query("launches_last") == 0
    with pytest.raises(k3moe.K3Error) as e:
        k3moe.forward(layer.ctx, dummy, MAXT + 1, dummy, dummy, dummy)
    assert e.value.code == k3moe.EINVAL


def test_tiny_forward_host_matches_device(tiny):
    d, w, layer = tiny
    x = gapped_tokens(d, w, seed=7, T=20)
    y_dev, idx_dev, w_dev = run(layer, x)
    y_h = np.empty((20, d.hidden), np.uint16)
    i_h = np.empty((20, d.top_k), np.int32)
    w_h = np.empty((20, d.top_k), np.float32)
    k3moe.forward_host(layer.ctx, x, 20, y_h, i_h, w_h)
    assert np.array_equal(y_h, y_dev) and np.array_equal(i_h, idx_dev) and np.array_equal(w_h, w_dev)


def test_tiny_deterministic(tiny):
    d, w, layer = tiny
    x = gapped_tokens(d, w, seed=8, T=50)
    a = run(layer, x)
    b = run(layer, x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_tiny_slot_order_does_not_change_y(tiny):
    """Permutation neutrality: the same tokens in another order give the
    same per-token outputs (the expert slot order changes)."""
    d, w, layer = tiny
    x = gapped_tokens(d, w, seed=9, T=40)
    y0, i0, w0 = run(layer, x)
    p = np.random.default_rng(0).permutation(40)
    y1, i1, w1 = run(layer, np.ascontiguousarray(x[p]))
    assert np.array_equal(y1, y0[p]) and np.array_equal(i1, i0[p]) and np.array_equal(w1, w0[p])


@pytest.mark.parametrize("opt", [dict(norm_topk=0), dict(routed_scaling=2.5), dict(n_hot=16)])
def test_tiny_routing_options(opt):
    n_hot = opt.pop("n_hot", 0)
    d = TINY.with_(**opt)
    w = synth.layer_weights(d, seed=3, n_hot=n_hot)
    layer = k3moe.Layer(d, w, max_tokens=32)
    try:
        x = gapped_tokens(d, w, seed=33, T=32)
        ref = ora.forward(d, w, x)
        y, idx, wts = run(layer, x)
        assert_routing_equal(idx, wts, ref["idx"], ref["w"], str(opt))
        assert_y_close(y, ref["y"], str(opt))
        if n_hot:
            assert np.isin(idx, synth.hot_experts(d, 3, n_hot)).all()
    finally:
        layer.close()


def test_pruned_expert_never_selected():
    d = TINY
    w = synth.layer_weights(d, seed=4)
    w["router_bias"][[1, 5, 9]] = -np.inf
    layer = k3moe.Layer(d, w, max_tokens=32)
    try:
        x = gapped_tokens(d, w, seed=44, T=32)
        ref = ora.forward(d, w, x)
        y, idx, wts = run(layer, x)
        assert not np.isin(idx, [1, 5, 9]).any()
        assert_routing_equal(idx, wts, ref["idx"], ref["w"])
        assert_y_close(y, ref["y"])
    finally:
        layer.close()


def test_bad_scale_rejected_on_load():
    d = TINY
    w = synth.layer_weights(d, seed=1)
    w["w2_scale"][3, 7, 2] = 255
    with pytest.raises(k3moe.K3Error) as e:
        k3moe.Layer(d, w, max_tokens=8)
    assert e.value.code == k3moe.EBADSCALE


def test_route_entry_point_matches_oracle():
    d = TINY
    w = synth.layer_weights(d, seed=2)
    T = 64
    x = gapped_tokens(d, w, seed=22, T=T)
    idx_r, w_r, logits_r = ora.route(d, x, w["router_w"], w["router_bias"])
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    rw = torch.from_numpy(w["router_w"].view(np.int16)).cuda()
    b = torch.from_numpy(w["router_bias"]).cuda()
    logits = torch.empty((T, d.n_experts), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    k3moe.route(xd, T, rw, b, d.n_experts, d.hidden, d.top_k, 1, 1.0, logits, idx, wt,
                torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert np.allclose(logits.cpu().numpy(), logits_r, rtol=1e-5, atol=1e-5)
    assert_routing_equal(idx.cpu().numpy(), wt.cpu().numpy(), idx_r, w_r)


@pytest.mark.parametrize("n_experts", [64, 896])
def test_route_exact_ties_go_to_lower_ids(n_experts):
    """Duplicated router rows with equal bias give bit-identical keys: the
    selection must take the lower expert ids, in the oracle's order
    (kimi-k3-mlx README, "Architecture": top-k by score + bias; ties are
    this implementation's reading, lower id first)."""
    d = TINY.with_(n_experts=n_experts)
    w = synth.layer_weights(d, seed=5)
    rw = w["router_w"].copy()
    bias = w["router_bias"].copy()
    # experts 3, 17, 40, 41, 60 (and more when E is large) copy expert 9
    dups = [3, 17, 40, 41, 60] + ([100, 333, 700, 701, 895] if n_experts > 64 else [])
    for e in dups:
        rw[e] = rw[9]
        bias[e] = bias[9]
    bias[9] += np.float32(0.5)  # push the tied group into the top-K
    for e in dups:
        bias[e] = bias[9]
    T = 16
    x = synth.token_rows(d, 77, T)
    idx_r, w_r, logits_r = ora.route(d, x, rw, bias)
    xd = torch.from_numpy(x.view(np.int16)).cuda()
    rwd = torch.from_numpy(rw.view(np.int16)).cuda()
    b = torch.from_numpy(bias).cuda()
    logits = torch.empty((T, d.n_experts), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    wt = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    k3moe.route(xd, T, rwd, b, d.n_experts, d.hidden, d.top_k, 1, 1.0, logits, idx, wt,
                torch.cuda.current_stream())
    torch.cuda.synchronize()
    lg = logits.cpu().numpy()
    # the duplicated rows produce identical logits on the device, so the keys tie exactly there
    for e in dups:
        assert np.array_equal(lg[:, e], lg[:, 9])
    # selection from the device's own logits by the oracle's rule
    idx_dev_rule, w_dev_rule = ora.route_from_logits(d, lg, bias)
    assert np.array_equal(idx.cpu().numpy(), idx_dev_rule)
    assert np.allclose(wt.cpu().numpy(), w_dev_rule, rtol=1e-6, atol=0)
    # at least one token has a tie crossing the K-th position or inside the top-K
    sel = idx.cpu().numpy()
    tied = [e for e in [9] + dups]
    assert any(len(set(sel[t]) & set(tied)) >= 2 for t in range(T))
