"""GPU parity of the REAP saliency accumulation (kimi-k3-mlx README, "REAP
expert pruning": S_j = 1/|C| sum over calibration tokens of g_j(x)
||e_j(x)||_2) against the CPU oracle through the C ABI: two batches
streamed through the layer (eager and graph replay, decode and prefill tile
kinds), determinism of the fp64 running sums, zero for unselected experts,
and reset."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY
from oracle import oracle as ora

from _cases import gapped_tokens

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

# the GPU's expert outputs o carry fp32 accumulation (and, on decode tiles,
# the six-term activation split): ~1e-5 relative per element; a norm of
# thousands of them and the mean over tokens keep S within this
S_RTOL = 1e-3


def forward(layer, x_np, graph=False):
    d = layer.d
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y = torch.empty((T, d.hidden), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, d.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, d.top_k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        if graph:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
                layer.forward(x, y, idx, w, stream=s)
            g.replay()
        else:
            layer.forward(x, y, idx, w, stream=s)
    s.synchronize()
    assert layer.status() == 0
    return idx.cpu().numpy()


def check(S_gpu, S_ref, label):
    assert np.array_equal(S_gpu == 0, S_ref == 0), f"{label}: zero pattern differs"
    assert np.allclose(S_gpu, S_ref, rtol=S_RTOL, atol=1e-12 * S_ref.max()), \
        f"{label}: max rel {np.max(np.abs(S_gpu - S_ref) / np.maximum(S_ref, 1e-30)):.3e}"


@pytest.mark.parametrize("path", [k3moe.PATH_AUTO, k3moe.PATH_CUDA_CORE], ids=["auto", "cudacore"])
def test_tiny_saliency_over_two_batches(path):
    d = TINY
    w = synth.layer_weights(d, seed=10)
    xa = gapped_tokens(d, w, seed=1001, T=40)
    xb = gapped_tokens(d, w, seed=1002, T=150)  # prefill tile kind on path 4
    layer = k3moe.Layer(d, w, max_tokens=256, force_path=path)
    try:
        k3moe.saliency(layer.ctx, True)
        forward(layer, xa)
        forward(layer, xb, graph=True)  # the replay accumulates too (capture itself launches nothing)
        sums, tokens = k3moe.saliency_read(layer.ctx, d.n_experts)
        assert tokens == 190
        S_ref, _ = ora.reap_saliency(d, w, np.concatenate([xa, xb]))
        check(sums / tokens, S_ref, f"path {path}")
        # the sums are deterministic: the same stream again doubles them exactly
        forward(layer, xa)
        forward(layer, xb)
        sums2, tokens2 = k3moe.saliency_read(layer.ctx, d.n_experts)
        assert tokens2 == 380 and np.array_equal(sums2, 2 * sums)
        k3moe.saliency_reset(layer.ctx)
        sums3, tokens3 = k3moe.saliency_read(layer.ctx, d.n_experts)
        assert tokens3 == 0 and not np.any(sums3)
        # disabled: forwards leave the totals alone
        k3moe.saliency(layer.ctx, False)
        forward(layer, xa)
        assert k3moe.saliency_read(layer.ctx, d.n_experts)[1] == 0
    finally:
        layer.close()


def test_k3_saliency_decode_batch():
    d = K3
    w = synth.layer_weights(d, seed=11)
    x = gapped_tokens(d, w, seed=1003, T=24)
    layer = k3moe.Layer(d, w, max_tokens=64)
    try:
        k3moe.saliency(layer.ctx, True)
        forward(layer, x[:8], graph=True)
        forward(layer, x[8:])
        sums, tokens = k3moe.saliency_read(layer.ctx, d.n_experts)
        assert tokens == 24
        S_ref, _ = ora.reap_saliency(d, w, x)
        check(sums / tokens, S_ref, "K3 T=8+16")
    finally:
        layer.close()
