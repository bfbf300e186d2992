"""Layer dimensions and the standard shapes.

K3 figures: 7168-d residual, 3584-d latent, 896 routed experts, top-16,
moe_intermediate_size 3072, MXFP4 group 32, SiTU-GLU beta 4 / beta_lin 25
(kimi-k3-mlx README, "Architecture" table; K3_ARTIFACT_AUDIT section 4.3
for the expert tensor shapes).
"""
from __future__ import annotations

from dataclasses import dataclass, replace


@dataclass(frozen=True)
class LayerDims:
    hidden: int
    latent: int
    n_experts: int
    top_k: int
    inter: int
    group: int = 32
    beta: float = 4.0
    beta_lin: float = 25.0
    rms_eps: float = 1e-6
    routed_scaling: float = 1.0
    norm_topk: int = 1
    # shared experts on the residual (0 = the routed path alone); K3 has 2,
    # each with intermediate 3072 (kimi-k3-mlx README, "Architecture" table
    # and "Parameter budget": 12.2 B shared-expert parameters over 92 MoE
    # layers = 3 x 7168 x 6144 per layer)
    n_shared: int = 0
    shared_inter: int = 0
    # two-bank graded experts (kimi-k3-mlx README, "REAP expert pruning"):
    # 0 = one MXFP4 bank; else experts >= bank2_begin are stored as 2-bit
    # affine weights (group 64, bf16 scale and bias: 2.5 bits per weight)
    bank2_begin: int = 0

    def with_(self, **kw) -> "LayerDims":
        return replace(self, **kw)

    # --- storage figures (bytes) -------------------------------------------------
    def expert_bytes(self) -> int:
        """Packed nibbles + e8m0 scales of one expert's w1, w3 and w2."""
        gate_up = 2 * (self.inter * self.latent // 2 + self.inter * self.latent // self.group)
        down = self.latent * self.inter // 2 + self.latent * self.inter // self.group
        return gate_up + down

    def expert_gate_up_bytes(self) -> int:
        return 2 * (self.inter * self.latent // 2 + self.inter * self.latent // self.group)

    def expert_down_bytes(self) -> int:
        return self.latent * self.inter // 2 + self.latent * self.inter // self.group

    @property
    def shared_total(self) -> int:
        """Concatenated intermediate of the shared experts."""
        return self.n_shared * self.shared_inter

    def shared_bytes(self) -> int:
        """bf16 gate, up and down weights of the shared experts."""
        return 3 * self.hidden * self.shared_total * 2

    @property
    def n_bank1(self) -> int:
        """Experts in the MXFP4 bank."""
        return self.bank2_begin if self.bank2_begin else self.n_experts

    def expert_bytes_bank2(self) -> int:
        """2-bit codes + bf16 scale and bias of one second-bank expert."""
        per = lambda rows, cols: rows * cols // 4 + 2 * 2 * rows * (cols // 64)
        return 2 * per(self.inter, self.latent) + per(self.latent, self.inter)

    def dense_bytes(self) -> int:
        """Router weight + bias, down_proj, up_proj and the RMSNorm weight."""
        return (self.n_experts * self.hidden * 2 + self.n_experts * 4 + self.latent * self.hidden * 2
                + self.hidden * self.latent * 2 + self.latent * 2)

    # --- work figures (multiply-adds counted as 2 FLOP) -------------------------
    def expert_flop_per_token(self) -> int:
        return self.top_k * (2 * self.latent * 2 * self.inter + 2 * self.inter * self.latent)

    def shared_flop_per_token(self) -> int:
        return 3 * 2 * self.hidden * self.shared_total

    def flop_per_token(self) -> int:
        router = 2 * self.n_experts * self.hidden
        proj = 2 * 2 * self.latent * self.hidden
        return router + proj + self.expert_flop_per_token() + self.shared_flop_per_token()


TINY = LayerDims(hidden=1024, latent=512, n_experts=64, top_k=8, inter=384)
K3 = LayerDims(hidden=7168, latent=3584, n_experts=896, top_k=16, inter=3072)
# the K3 MoE block: the routed layer plus its two shared experts
K3_SHARED = K3.with_(n_shared=2, shared_inter=3072)
TINY_SHARED = TINY.with_(n_shared=2, shared_inter=384)
