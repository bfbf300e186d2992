"""k3moe_route_noalloc: the router step for callers that cannot allocate
device memory where they route (inside a CUDA-graph capture, inside another
framework's memory pool or fixed budget, in services that allow no
allocation after start-up).  Its scratch is a static device array; this
checks, through the C ABI, that two calls in a row give the same routing
as k3moe_route (which uses caller-provided scratch), that the call works
inside a CUDA-graph capture without allocating, and that oversized
requests are refused.  Kept in a file of its own that pytest collects last.
"""
import ctypes as C

import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import k3moe, synth
from mxfp4_routed_expert_k3_gb300.dims import K3

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _router(seed):
    E, H = K3.n_experts, K3.hidden
    rw = synth.bf16_normal(seed, synth.S_ROUTER_W, (E, H), 0.0, 1.0 / np.sqrt(H))
    bias = synth.f32_uniform(seed, synth.S_BIAS, (E,), -0.1, 0.1)
    return torch.from_numpy(rw.view(np.int16)).cuda(), torch.from_numpy(bias).cuda()


def _route(fn, x, T, rw, b, with_scratch):
    E, H, K = K3.n_experts, K3.hidden, K3.top_k
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    if with_scratch:
        logits = torch.empty((T, E), dtype=torch.float32, device="cuda")
        rc = fn(x.data_ptr(), T, rw.data_ptr(), b.data_ptr(), E, H, K, 1, C.c_float(1.0), logits.data_ptr(),
                idx.data_ptr(), w.data_ptr(), s)
    else:
        rc = fn(x.data_ptr(), T, rw.data_ptr(), b.data_ptr(), E, H, K, 1, C.c_float(1.0), idx.data_ptr(),
                w.data_ptr(), s)
    assert rc == k3moe.OK, k3moe.last_error()
    torch.cuda.synchronize()
    return idx.cpu().numpy(), w.cpu().numpy()


def test_noalloc_route_matches_route_on_two_calls_in_a_row():
    L = k3moe.lib()
    rw, b = _router(21)
    for call, (T, seed) in enumerate([(64, 301), (37, 302)]):
        x = torch.from_numpy(synth.token_rows(K3, seed, T).view(np.int16)).cuda()
        idx_ref, w_ref = _route(L.k3moe_route, x, T, rw, b, with_scratch=True)
        idx, w = _route(L.k3moe_route_noalloc, x, T, rw, b, with_scratch=False)
        assert np.array_equal(idx, idx_ref), f"call {call}: expert ids differ"
        assert np.array_equal(w, w_ref), f"call {call}: routing weights differ"
        assert np.all((idx >= 0) & (idx < K3.n_experts))
        assert np.allclose(w.sum(1), 1.0, rtol=1e-5)


def test_noalloc_route_rejects_more_than_its_scratch():
    L = k3moe.lib()
    rw, b = _router(21)
    T = 147  # 147 * 896 > 131072 logits
    x = torch.zeros((T, K3.hidden), dtype=torch.int16, device="cuda")
    idx = torch.empty((T, K3.top_k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, K3.top_k), dtype=torch.float32, device="cuda")
    rc = L.k3moe_route_noalloc(x.data_ptr(), T, rw.data_ptr(), b.data_ptr(), K3.n_experts, K3.hidden, K3.top_k, 1,
                               C.c_float(1.0), idx.data_ptr(), w.data_ptr(), None)
    assert rc == k3moe.EINVAL
    assert "scratch" in k3moe.last_error()


def test_noalloc_route_inside_a_graph_capture():
    """The use the entry point exists for: the call captured into a CUDA
    graph after one eager call, the graph replayed on new tokens copied
    into the captured input; idx and w bit-equal to k3moe_route's, and
    neither the torch allocator nor the device's free memory moves across
    the replays (nor the torch allocator across the captured call)."""
    L = k3moe.lib()
    rw, b = _router(21)
    T, E, H, K = 16, K3.n_experts, K3.hidden, K3.top_k
    x = torch.from_numpy(synth.token_rows(K3, 401, T).view(np.int16)).cuda()
    idx = torch.full((T, K), -1, dtype=torch.int32, device="cuda")
    w = torch.full((T, K), -1.0, dtype=torch.float32, device="cuda")
    side = torch.cuda.Stream()

    def call():
        rc = L.k3moe_route_noalloc(x.data_ptr(), T, rw.data_ptr(), b.data_ptr(), E, H, K, 1, C.c_float(1.0),
                                   idx.data_ptr(), w.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert rc == k3moe.OK, k3moe.last_error()

    with torch.cuda.stream(side):
        call()  # the eager call before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        # (entering the capture context allocates a little itself; a device
        # allocation by the call would end the capture with an error)
        alloc0 = torch.cuda.memory_allocated()
        call()
        alloc_in = torch.cuda.memory_allocated()
    assert alloc_in == alloc0, "the captured call allocated"
    saved = [torch.empty_like(x) for _ in range(2)]  # allocated before the measurements
    alloc1 = torch.cuda.memory_allocated()
    got, free = [], []
    for i, seed in enumerate((402, 403)):
        x.copy_(torch.from_numpy(synth.token_rows(K3, seed, T).view(np.int16)))
        g.replay()
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        saved[i].copy_(x)
        got.append((idx.cpu().numpy().copy(), w.cpu().numpy().copy(), saved[i]))
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == alloc1, "a replay allocated"
    assert free[0] == free[1], "device memory changed between replays"
    for i, (gi, gw, xi) in enumerate(got):
        idx_ref, w_ref = _route(L.k3moe_route, xi, T, rw, b, with_scratch=True)
        assert np.array_equal(gi, idx_ref), f"replay {i}: expert ids differ"
        assert np.array_equal(gw, w_ref), f"replay {i}: routing weights differ"
