"""Expert parallelism, host side, on CPU: the rank ranges, the weights a
rank loads, and the all-reduce between the partial combine and the rest of
the block, run as two gloo ranks with the oracle standing in for each
rank's GPU (partial combine of its experts; RMSNorm, up_proj and shared
experts on the sum).  Every rank must end with the whole block's output."""
import json
import os
import socket

import numpy as np
import pytest

from mxfp4_routed_expert_k3_gb300 import expert_parallel as ep
from mxfp4_routed_expert_k3_gb300 import synth
from mxfp4_routed_expert_k3_gb300.dims import K3, TINY_SHARED


def test_shard_ranges_cover_every_expert_once():
    for E, world in [(896, 2), (64, 2), (64, 3), (9, 4), (896, 8)]:
        ranges = [ep.shard_range(r, world, E) for r in range(world)]
        ids = np.concatenate([np.arange(b, b + n) for b, n in ranges])
        assert np.array_equal(ids, np.arange(E))
        assert max(n for _, n in ranges) - min(n for _, n in ranges) <= 1
    assert ep.shard_range(1, 2, K3.n_experts) == (448, 448)  # the 50/50 split
    with pytest.raises(ValueError):
        ep.shard_range(2, 2, 64)


def test_shard_weights_slice_experts_only():
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=4)
    s = ep.shard_weights(w, 10, 20)
    for name in ep.EXPERT_TENSORS:
        assert s[name].shape[0] == 20 and np.array_equal(s[name], w[name][10:30])
    for name in ("router_w", "router_bias", "down_proj", "up_proj", "norm_w", "shared_w1", "shared_w2"):
        assert s[name] is w[name]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _rank(rank, world, port, out):
    import torch
    import torch.distributed as dist
    from oracle import oracle as ora
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=5)
    x = synth.token_rows(d, 55, 6)
    b, n = ep.shard_range(rank, world, d.n_experts)

    def partial(xv):  # this rank's "device": the partial combine of its experts
        return torch.from_numpy(ora.forward_partial(d, w, xv, b, n))

    def finish(xv, c):
        return ora.finish(d, w, xv, c.numpy())

    y = ep.ep_forward(partial, finish, x)
    np.save(f"{out}.{rank}.npy", y)
    dist.destroy_process_group()


def test_two_rank_expert_parallel_block_gloo(tmp_path):
    import torch.multiprocessing as mp
    from oracle import oracle as ora
    out = str(tmp_path / "y")
    mp.spawn(_rank, args=(2, _free_port(), out), nprocs=2, join=True)
    d = TINY_SHARED
    w = synth.layer_weights(d, seed=5)
    x = synth.token_rows(d, 55, 6)
    ref = ora.forward(d, w, x)["y"]
    y0, y1 = np.load(f"{out}.0.npy"), np.load(f"{out}.1.npy")
    assert np.array_equal(y0, y1)  # both ranks hold the same output
    # c_0 + c_1 regroups the fp64 combine: bf16 outputs agree but for ties
    same = np.mean(y0 == ref)
    assert same > 0.999, same
    a, r = ora.bf16_to_float(y0), ora.bf16_to_float(ref)
    assert np.max(np.abs(a - r)) <= 2 ** -7 * np.abs(r).max()
