"""Expert parallelism over ranks: the host side of the block split at the
combine (Kimi-K3-Alis-MLX-Dynamic model card, "Performance" and "Usage":
dense weights replicated, the routed experts split between the machines).

Every rank holds the whole router, down_proj, RMSNorm weight, up_proj and
shared experts, and a contiguous range of the routed experts.  One block
forward is

    c_r = k3moe_forward_partial(x)        on every rank (its experts only)
    c   = sum over ranks of c_r           one all-reduce of [T, L] fp32
    y   = k3moe_finish(x, c)              on every rank (identical results)

RMSNorm needs the whole combine, so the all-reduce sits before it; that is
the block's only exchange.  The reduction uses torch.distributed (NCCL on
GPUs); for two ranks every element is c_0 + c_1, the same on both ranks.
"""
from __future__ import annotations

from typing import Callable

import numpy as np

from .dims import LayerDims

EXPERT_TENSORS = ("w1_packed", "w1_scale", "w3_packed", "w3_scale", "w2_packed", "w2_scale")


def shard_range(rank: int, world: int, n_experts: int) -> tuple[int, int]:
    """(begin, count) of rank's contiguous expert range; the first
    n_experts % world ranks take one more (an even 50/50 split for two)."""
    if not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside [0, {world})")
    base, extra = divmod(n_experts, world)
    begin = rank * base + min(rank, extra)
    return begin, base + (1 if rank < extra else 0)


def shard_weights(w: dict, begin: int, count: int) -> dict:
    """The weights a rank loads: every dense tensor, and the expert tensors
    of experts [begin, begin + count) only."""
    out = dict(w)
    for name in EXPERT_TENSORS:
        out[name] = np.ascontiguousarray(w[name][begin:begin + count])
    return out


def all_reduce_sum(c, group=None):
    """Sum of the ranks' partial combines, in place (identity on one rank)."""
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(c, op=dist.ReduceOp.SUM, group=group)
    return c


def ep_forward(partial_fn: Callable, finish_fn: Callable, x, group=None):
    """One block forward under expert parallelism: partial combine of this
    rank's experts, one all-reduce, the rest of the block on the sum."""
    c = partial_fn(x)
    all_reduce_sum(c, group)
    return finish_fn(x, c)


class ExpertShardLayer:
    """A rank's context: the routed experts [begin, begin + count) of a
    layer, dense weights whole (binding of k3moe_forward_partial /
    k3moe_finish; device buffers are torch tensors)."""

    def __init__(self, d: LayerDims, weights: dict, rank: int, world: int, max_tokens: int, device: int = 0):
        from . import k3moe
        self.d = d
        self.begin, self.count = shard_range(rank, world, d.n_experts)
        whole = self.count == d.n_experts
        self.layer = k3moe.Layer(d, weights if whole else shard_weights(weights, self.begin, self.count),
                                 max_tokens=max_tokens, device=device, expert_begin=0 if whole else self.begin,
                                 expert_count=0 if whole else self.count)

    def partial(self, x, stream=None):
        import torch
        from . import k3moe
        T = x.shape[0]
        c = torch.empty((T, self.d.latent), dtype=torch.float32, device=x.device)
        self.idx = torch.empty((T, self.d.top_k), dtype=torch.int32, device=x.device)
        self.w = torch.empty((T, self.d.top_k), dtype=torch.float32, device=x.device)
        k3moe.forward_partial(self.layer.ctx, x, T, c, self.idx, self.w,
                              stream if stream is not None else torch.cuda.current_stream())
        return c

    def finish(self, x, c, stream=None):
        import torch
        from . import k3moe
        T = x.shape[0]
        y = torch.empty((T, self.d.hidden), dtype=torch.int16, device=x.device)
        k3moe.finish(self.layer.ctx, x, c, T, y, stream if stream is not None else torch.cuda.current_stream())
        return y

    def forward(self, x, group=None, stream=None):
        return ep_forward(lambda v: self.partial(v, stream), lambda v, c: self.finish(v, c, stream), x, group)

    def close(self):
        self.layer.close()
