"""GPU parity of two-bank graded experts (kimi-k3-mlx README, "REAP expert
pruning": graded mode and the two-bank SwitchGLU): experts [0, bank2_begin)
MXFP4 on the block-scaled tensor cores, the rest 2-bit affine (group 64,
bf16 scale and bias) decoded exactly and fed to the tensor cores as bf16
hi + lo terms; the split of the sorted selections between the banks is
found on the device.  Against the CPU oracle through the C ABI, at decode
and prefill tile sizes, plus the pages' own correctness test: a second bank
holding exactly the values of MXFP4 experts gives the one-bank layer's
output."""
import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY
from oracle import oracle as ora

from _cases import assert_routing_equal, assert_y_close, bf16_f64, gapped_tokens
from test_oracle_pins import mxfp4_twin_of_bank2, np_affine2

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

D2 = TINY.with_(bank2_begin=40)


def run(layer, x_np):
    d = layer.d
    T = x_np.shape[0]
    x = torch.from_numpy(x_np.view(np.int16)).cuda()
    y, idx, w = layer.forward_torch(x)
    torch.cuda.synchronize()
    assert layer.status() == 0, k3moe.last_error(layer.ctx)
    return y.cpu().numpy().view(np.uint16), idx.cpu().numpy(), w.cpu().numpy()


def check_h(layer, d, w, ref, T):
    """h of every slot against the oracle's arithmetic applied to the GPU's
    own latent (a one-ulp bf16 difference in the latent of a token shifts
    every h of that token, which would hide or fake an error here): weights
    dequantised by the numpy formulas of the oracle pins, SiTU-GLU in
    float64, bf16 rounding through the oracle."""
    from _cases import bf16_round, expert_matrix
    K = d.top_k
    slot = layer.fetch("slot", (T * K,), np.int32)
    h = layer.fetch("h", (T * K, d.inter), np.uint16)
    lat = bf16_f64(layer.fetch("lat", (T, d.latent), np.uint16))
    hg = bf16_f64(h[slot]).reshape(T, K, d.inter)
    idx = ref["idx"]
    bank2 = idx >= d.bank2_begin
    assert np.any(bank2) and np.any(~bank2)
    situ = lambda g, u: 4 * np.tanh(g / 4) / (1 + np.exp(-g)) * 25 * np.tanh(u / 25)
    same = {True: [], False: []}
    for e in np.unique(idx):
        tk = np.argwhere(idx == e)
        if e >= d.bank2_begin:
            e2 = e - d.bank2_begin
            W1 = np_affine2(w["b2_w1q"][e2], w["b2_w1s"][e2], w["b2_w1b"][e2])
            W3 = np_affine2(w["b2_w3q"][e2], w["b2_w3s"][e2], w["b2_w3b"][e2])
        else:
            W1, W3 = expert_matrix(w, "w1", e), expert_matrix(w, "w3", e)
        xl = lat[tk[:, 0]]
        h_ref = bf16_round(situ(xl @ W1.T, xl @ W3.T))
        same[bool(e >= d.bank2_begin)].append(hg[tk[:, 0], tk[:, 1]] == h_ref)
    for b2, name in ((True, "second bank"), (False, "first bank")):
        assert np.mean(np.concatenate(same[b2])) > 0.995, name


@pytest.fixture(scope="module")
def two_bank():
    w = synth.layer_weights(D2, seed=50)
    layer = k3moe.Layer(D2, w, max_tokens=256)
    yield w, layer
    layer.close()


@pytest.mark.parametrize("T", [1, 8, 64, 200])
def test_tiny_two_bank_layer(two_bank, T):
    w, layer = two_bank
    x = gapped_tokens(D2, w, seed=5000 + T, T=T)
    ref = ora.forward(D2, w, x, probes=True)
    y, idx, wts = run(layer, x)
    assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"T={T}")
    check_h(layer, D2, w, ref, T)
    assert_y_close(y, ref["y"], f"two banks T={T}")


@pytest.mark.parametrize("T", [8, 150])
def test_second_bank_of_mxfp4_values_matches_one_bank(T):
    """The page's test: both banks holding the same values must give the
    one-bank result.  The oracle gives identical outputs for the two
    layouts; on the GPU the second bank runs other kernels, so both GPU
    outputs are held to the oracle and to each other."""
    w = synth.layer_weights(D2, seed=51)
    two, one = mxfp4_twin_of_bank2(D2, w, 52)
    x = gapped_tokens(TINY, one, seed=5100 + T, T=T)
    ref = ora.forward(TINY, one, x)
    assert np.array_equal(ora.forward(D2, two, x)["y"], ref["y"])
    l2 = k3moe.Layer(D2, two, max_tokens=256)
    l1 = k3moe.Layer(TINY, one, max_tokens=256)
    try:
        y2, idx2, w2 = run(l2, x)
        y1, idx1, w1 = run(l1, x)
    finally:
        l2.close()
        l1.close()
    assert np.array_equal(idx2, idx1) and np.array_equal(w2, w1)
    assert_routing_equal(idx2, w2, ref["idx"], ref["w"], f"T={T}")
    assert_y_close(y2, ref["y"], f"two banks T={T}")
    assert_y_close(y1, ref["y"], f"one bank T={T}")
    assert np.mean(y1 == y2) > 0.95


def test_k3_two_bank_decode():
    d = K3.with_(bank2_begin=448)
    w = synth.layer_weights(d, seed=53)
    layer = k3moe.Layer(d, w, max_tokens=64)
    try:
        for T in (1, 8):
            x = gapped_tokens(d, w, seed=5200 + T, T=T)
            ref = ora.forward(d, w, x, probes=True)
            y, idx, wts = run(layer, x)
            assert_routing_equal(idx, wts, ref["idx"], ref["w"], f"K3 T={T}")
            check_h(layer, d, w, ref, T)
            assert_y_close(y, ref["y"], f"K3 two banks T={T}")
    finally:
        layer.close()
