"""GPU parity of the K3 MoE block with its shared experts (two bf16 SiTU-GLU
MLPs on the residual, summed and added to the routed branch's output):
the CUDA path against the CPU oracle through the C ABI, on the tiny layer
at decode and prefill sizes and on K3 dims at decode sizes, eagerly and as
a CUDA-graph replay (the shared experts run on a forked side stream)."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3_SHARED, TINY_SHARED
from oracle import oracle as ora

from _cases import assert_routing_equal, assert_y_close, bf16_f64, gapped_tokens

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def run(layer, x_np, graph=False):
    d = layer.d
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y = torch.empty((T, d.hidden), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        layer.forward(x, y, idx, w, stream=s)
        if graph:
            g = torch.cuda.CUDAGraph()
            y.zero_()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                layer.forward(x, y, idx, w, stream=s)
            g.replay()
    s.synchronize()
    assert layer.status() == 0, k3moe.last_error(layer.ctx)
    return y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()


def check_shared_step(layer, d, ref, T):
    hs = layer.fetch("shared_h", (T, d.shared_total), np.uint16)
    z = layer.fetch("shared_z", (T, d.hidden), np.uint16)
    hg, hr = bf16_f64(hs), bf16_f64(ref["hs"])
    assert np.mean(hg == hr) > 0.995
    assert np.max(np.abs(hg - hr)) <= 2 ** -7 * np.abs(hr).max() + 1e-30
    # z sums thousands of bf16 h terms: one-ulp differences in h move some of
    # its bf16 roundings (more the longer the sum), so z is held to an error
    # bound, not to identical bits
    zg, zr = bf16_f64(z), bf16_f64(ref["z"])
    zrms = np.sqrt(np.mean(zr ** 2))
    assert np.sqrt(np.mean((zg - zr) ** 2)) <= 2e-3 * zrms
    assert np.max(np.abs(zg - zr)) <= 2 ** -5 * zrms


def branch_terms(ref):
    """The two bf16 terms of y = bf16(y_routed + z): z, and y_routed ~ y - z."""
    z = bf16_f64(ref["z"])
    return (z, bf16_f64(ref["y"]) - z)


@pytest.fixture(scope="module", params=[k3moe.PATH_AUTO], ids=["auto"])
def tiny_shared(request):
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=8)
    layer = k3moe.Layer(d, w, max_tokens=256, force_path=request.param)
    yield d, w, layer
    layer.close()


@pytest.mark.parametrize("T", [1, 5, 64, 65, 200])
def test_tiny_block_with_shared_experts(tiny_shared, T):
    d, w, layer = tiny_shared
    x = gapped_tokens(d, w, seed=800 + T, T=T)
    ref = ora.forward(d, w, x, probes=True)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    check_shared_step(layer, d, ref, T)
    m = assert_y_close(y, ref["y"], f"T={T}", rounded_terms=branch_terms(ref))
    assert m["identical_frac"] > 0.9


@pytest.mark.parametrize("T", [8, 150])
def test_tiny_block_with_shared_experts_graph_replay(tiny_shared, T):
    """The side stream is forked and joined inside the captured graph."""
    d, w, layer = tiny_shared
    x = gapped_tokens(d, w, seed=850 + T, T=T)
    ref = ora.forward(d, w, x, probes=True)
    y_eager, _, _ = run(layer, x)
    y_graph, idx, wts = run(layer, x, graph=True)
    assert np.array_equal(y_graph, y_eager)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    assert_y_close(y_graph, ref["y"], f"graph T={T}", rounded_terms=branch_terms(ref))


@pytest.fixture(scope="module")
def k3_shared():
    d = K3_SHARED
    w = synth.layer_weights(d, seed=9)
    layer = k3moe.Layer(d, w, max_tokens=64)
    yield d, w, layer
    layer.close()


@pytest.mark.parametrize("T", [1, 8])
def test_k3_block_with_shared_experts(k3_shared, T):
    d, w, layer = k3_shared
    x = gapped_tokens(d, w, seed=900 + T, T=T)
    ref = ora.forward(d, w, x, probes=True)
    y, idx, wts = run(layer, x, graph=True)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"K3 T={T}")
    check_shared_step(layer, d, ref, T)
    assert_y_close(y, ref["y"], f"K3 T={T}", rounded_terms=branch_terms(ref))
