"""Expert parallelism on one GPU: two shard contexts (experts [0, E/2) and
[E/2, E), dense weights whole) run k3moe_forward_partial, their partial
combines are summed (c_0 + c_1, what the all-reduce computes), and
k3moe_finish completes the block; checked against the oracle's partial
combines and whole block, and against the unsharded context, through the
C ABI.  (The ranks run one after the other here: every call of this run
uses a single GPU.)"""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import expert_parallel as ep
from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY_SHARED
from oracle import oracle as ora

from _cases import assert_routing_equal, assert_y_close, bf16_f64, gapped_tokens


def branch_terms(ref):
    """The two bf16 terms of y = bf16(y_routed + z) (shared experts)."""
    z = bf16_f64(ref["z"])
    return (z, bf16_f64(ref["y"]) - z)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def c_close(c_gpu, c_ref, label):
    rms = np.sqrt(np.mean(c_ref ** 2))
    err = np.abs(c_gpu.astype(np.float64) - c_ref)
    assert np.sqrt(np.mean(err ** 2)) <= 1e-3 * rms, (label, np.sqrt(np.mean(err ** 2)) / rms)


@pytest.fixture(scope="module")
def tiny_ep():
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=40)
    full = k3moe.Layer(d, w, max_tokens=256)
    ranks = [ep.ExpertShardLayer(d, w, r, 2, max_tokens=256) for r in range(2)]
    yield d, w, full, ranks
    full.close()
    for r in ranks:
        r.close()


@pytest.mark.parametrize("T", [5, 64, 150])
def test_tiny_two_shards_match_the_block(tiny_ep, T):
    d, w, full, ranks = tiny_ep
    x_np = gapped_tokens(d, w, seed=4000 + T, T=T)
    ref = ora.forward(d, w, x_np, probes=True)
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    # the unsharded context: finish(partial) is the forward, bit for bit
    y_full, idx_full, w_full = full.forward_torch(x)
    c_all = torch.empty((T, d.latent), dtype=torch.float32, device="cuda")
    idx = torch.empty_like(idx_full)
    wt = torch.empty_like(w_full)
    k3moe.forward_partial(full.ctx, x, T, c_all, idx, wt, torch.cuda.current_stream())
    y2 = torch.empty_like(y_full)
    k3moe.finish(full.ctx, x, c_all, T, y2, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert torch.equal(y2, y_full) and torch.equal(idx, idx_full)
    c_close(c_all.cpu().numpy(), ref["c"], "whole combine")
    # two shards
    parts = [r.partial(x) for r in ranks]
    torch.cuda.synchronize()
    for r, (b, n), c in zip(ranks, [ep.shard_range(i, 2, d.n_experts) for i in range(2)], parts):
        assert torch.equal(r.idx, idx_full) and torch.equal(r.w, w_full)  # the router is replicated
        c_close(c.cpu().numpy(), ora.forward_partial(d, w, x_np, b, n), f"shard {b}+{n}")
    c = parts[0] + parts[1]
    ys = [r.finish(x, c) for r in ranks]
    torch.cuda.synchronize()
    assert torch.equal(ys[0], ys[1])
    y_ep = ys[0].cpu().numpy().view(np.uint16)
    assert_routing_equal(idx_full.cpu().numpy(), w_full.cpu().numpy(), ref["idx"], ref["w"], f"T={T}")
    assert_y_close(y_ep, ref["y"], f"expert parallel T={T}", rounded_terms=branch_terms(ref))
    assert np.mean(y_ep == y_full.cpu().numpy().view(np.uint16)) > 0.97


def test_shard_rejects_the_whole_forward(tiny_ep):
    d, w, full, ranks = tiny_ep
    x = torch.zeros((2, d.hidden), dtype=torch.int16, device="cuda")
    with pytest.raises(k3moe.K3Error) as ei:
        ranks[0].layer.forward_torch(x)
    assert ei.value.code == k3moe.ESTATE


def test_k3_two_shards_decode():
    d = K3
    w = synth.layer_weights(d, seed=41)
    ranks = [ep.ExpertShardLayer(d, w, r, 2, max_tokens=64) for r in range(2)]
    try:
        for T in (1, 8):
            x_np = gapped_tokens(d, w, seed=4100 + T, T=T)
            ref = ora.forward(d, w, x_np)
            x = torch.from_numpy(x_np.view(np.int16)).cuda()
            c = ranks[0].partial(x) + ranks[1].partial(x)
            y = ranks[0].finish(x, c)
            torch.cuda.synchronize()
            assert ranks[0].layer.status() == 0 and ranks[1].layer.status() == 0
            assert_routing_equal(ranks[0].idx.cpu().numpy(), ranks[0].w.cpu().numpy(), ref["idx"], ref["w"],
                                 f"K3 T={T}")
            assert_y_close(y.cpu().numpy().view(np.uint16), ref["y"], f"K3 expert parallel T={T}")
    finally:
        for r in ranks:
            r.close()
