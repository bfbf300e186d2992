"""GPU parity at K3 dims (H=7168, L=3584, 896 experts, top-16, I=3072) in
the launch configuration the benchmark times: decode T = 1, 8, 64 against
the oracle on every token; prefill T = 8192 and the skewed T = 4096 case
with the routing of every token checked bit for bit and the outputs on a
seeded sample of tokens."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3
from oracle import oracle as ora

from _cases import assert_routing_equal, assert_y_close, bf16_f64, gapped_tokens, y_metrics

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

MAXT = 8192


@pytest.fixture(scope="module")
def k3weights():
    return synth.layer_weights(K3, seed=1)


@pytest.fixture(scope="module", params=[k3moe.PATH_BLOCK_SCALED], ids=["blockscaled"])
def k3layer(request, k3weights):
    layer = k3moe.Layer(K3, k3weights, max_tokens=MAXT, force_path=request.param)
    yield k3weights, layer
    layer.close()


@pytest.fixture(scope="module", params=[k3moe.PATH_CUDA_CORE, k3moe.PATH_BLOCK_SCALED],
                ids=["cudacore", "blockscaled"])
def k3decode(request, k3weights):
    layer = k3moe.Layer(K3, k3weights, max_tokens=64, force_path=request.param)
    yield k3weights, layer
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


@pytest.mark.parametrize("T", [1, 8, 64])
def test_k3_decode_all_tokens(k3decode, T):
    w, layer = k3decode
    x = gapped_tokens(K3, w, seed=200 + T, T=T)
    ref = ora.forward(K3, w, x)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"decode T={T}")
    m = assert_y_close(y, ref["y"], f"decode T={T}")
    print(f"decode T={T} path={layer.query('path_last')}", m)


def test_k3_decode_tiles_unfused_route_t96(k3weights):
    """T = 96: decode tiles (T <= 128) with T*K = 1536 > 1024 slots, so the
    routing runs the multi-kernel top-k / permute / tile-list chain instead
    of the fused small-batch kernel; every token against the oracle."""
    layer = k3moe.Layer(K3, k3weights, max_tokens=128)
    try:
        x = gapped_tokens(K3, k3weights, seed=296, T=96)
        ref = ora.forward(K3, k3weights, x)
        y, idx, wts = run(layer, x)
        assert layer.query("path_last") == k3moe.PATH_BLOCK_SCALED
        assert_routing_equal(idx, wts, ref["idx"], ref["w"], "decode tiles T=96")
        m = assert_y_close(y, ref["y"], "decode tiles T=96")
        print("decode tiles T=96", m)
    finally:
        layer.close()


def _sampled(layer, w, x, n_sample, seed, label):
    T = x.shape[0]
    idx_ref, w_ref, _ = ora.route(K3, x, w["router_w"], w["router_bias"])
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, idx_ref, w_ref, label)
    sample = np.sort(np.random.default_rng(seed).choice(T, n_sample, replace=False))
    sample[-1] = T - 1  # always include the ragged tail
    ref = ora.forward(K3, w, np.ascontiguousarray(x[sample]), probes=True)
    # per-step diagnostics on the sampled tokens
    logits = layer.fetch("logits", (T, K3.n_experts), np.float32)[sample].astype(np.float64)
    lat = bf16_f64(layer.fetch("lat", (T, K3.latent), np.uint16)[sample])
    n = bf16_f64(layer.fetch("n", (T, K3.latent), np.uint16)[sample])
    dl = np.abs(logits - ref["logits"])
    diag = {"logits_max_abs": float(dl.max()), "logits_rms": float(np.sqrt(np.mean(ref["logits"] ** 2))),
            "lat_identical": float(np.mean(lat == bf16_f64(ref["lat"]))),
            "lat_max_rel": float(np.max(np.abs(lat - bf16_f64(ref["lat"])) / np.maximum(np.abs(bf16_f64(ref["lat"])), 1e-3))),
            "n_identical": float(np.mean(n == bf16_f64(ref["n"]))),
            "n_rel_rms": float(np.sqrt(np.mean((n - bf16_f64(ref["n"])) ** 2) / np.mean(bf16_f64(ref["n"]) ** 2)))}
    print(label, "steps", diag)
    m = assert_y_close(y[sample], ref["y"], label)
    # properties that hold for every token
    yf = (y.astype(np.uint32) << 16).view(np.float32)
    assert np.all(np.isfinite(yf))
    assert np.allclose(wts.sum(1), K3.routed_scaling, rtol=1e-5)
    print(label, f"path={layer.query('path_last')}", m)
    return idx


def test_k3_prefill_8192(k3layer):
    w, layer = k3layer
    x = gapped_tokens(K3, w, seed=300, T=8192)
    _sampled(layer, w, x, 128, 1, "prefill T=8192")


@pytest.mark.parametrize("path", [k3moe.PATH_BLOCK_SCALED], ids=["blockscaled"])
def test_k3_skewed_4096(path):
    w = synth.layer_weights(K3, seed=3, n_hot=32)
    hot = synth.hot_experts(K3, 3, 32)
    layer = k3moe.Layer(K3, w, max_tokens=4096, force_path=path)
    try:
        x = gapped_tokens(K3, w, seed=301, T=4096)
        idx = _sampled(layer, w, x, 128, 2, "skew T=4096")
        assert np.isin(idx, hot).all()
        counts = layer.fetch("counts", (K3.n_experts,), np.int32)
        assert np.count_nonzero(counts) == 32 and counts.sum() == 4096 * 16
    finally:
        layer.close()
