"""The layer-level call a user makes: prepacked weights resident on the GPU,
then gate_up -> silu_and_mul -> down per batch of routed tokens.

Every step is a call into the C-ABI library (``ops``); this module only
allocates buffers (torch device memory) and sequences the calls on one
stream.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import ops


@dataclass
class PackedExperts:
    """Prepacked expert weights of one projection: [num_experts, n, k]."""
    packed: torch.Tensor
    num_experts: int
    n: int
    k: int

    layout: int = ops.W4A16_LAYOUT_KTILE64

    @classmethod
    def from_checkpoint(cls, q: torch.Tensor, scales: torch.Tensor, group: int = 32,
                        layout: int = ops.W4A16_LAYOUT_KTILE64):
        """layout W4A16_LAYOUT_KTILE64_GLU16 (gate_up weights only) enables the
        fused gate_up + activation call."""
        e, n, kh = q.shape
        return cls(ops.w4a16_prepack(q, scales, group, layout), e, n, kh * 2, layout)


def single_launch_default(gate_up_layout: int, deterministic: bool, inter: int,
                          block_m: int = 32) -> bool:
    """Whether a layer runs gate_up, the activation and down as one launch
    (w4a16_moe_layer) by default: GLU16 gate_up weights, no deterministic
    pass, a long down reduction (inter >= 1024) and routing blocks of at most
    32 rows. Measured: 303.8 vs 314.6 us at the EP8 decode shard (I = 2048,
    block_m 32); slower at the TP8 shard, I = 256, whose down items are two
    pipeline stages long (516.4 vs 418.5 us at T = 256), and at the EP8
    prefill shard, whose 64-row blocks need the early-release epilogue the
    single launch does not have (703.8 vs 634.3 us)."""
    return (gate_up_layout == ops.W4A16_LAYOUT_KTILE64_GLU16 and not deterministic
            and inter >= 1024 and block_m <= 32)


class W4A16MoE:
    """One MoE layer's expert pair on one GPU (gate_up [E, 2I, H], down [E, H, I])."""

    def __init__(self, gate_up: PackedExperts, down: PackedExperts, topk: int,
                 max_tokens: int, tok_e_hint: float = 0.0, device=None,
                 deterministic: bool = False, single_launch: Optional[bool] = None):
        """With gate_up packed as W4A16_LAYOUT_KTILE64_GLU16 the activation is
        fused into the gate_up call (forward skips the separate pass). With
        deterministic=True the down pass adds each token's top-k rows in a
        fixed order (W4A16_FLAG_DETERMINISTIC): the output bits do not depend
        on the schedule. single_launch=True (GLU16 gate_up weights) runs
        gate_up, the activation and down in one launch (w4a16_moe_layer);
        None applies single_launch_default."""
        assert gate_up.num_experts == down.num_experts
        assert gate_up.n == 2 * down.k and gate_up.k == down.n
        self.gate_up, self.down = gate_up, down
        self.num_experts = gate_up.num_experts
        self.hidden, self.inter = gate_up.k, down.k
        self.topk = topk
        self.device = device or gate_up.packed.device
        self.max_tokens = max_tokens
        self.tok_e_hint = tok_e_hint
        self.deterministic = deterministic
        glu = gate_up.layout == ops.W4A16_LAYOUT_KTILE64_GLU16
        if single_launch is None:
            block_m = ops.w4a16_plan(max_tokens, topk, gate_up.num_experts, gate_up.n, gate_up.k,
                                     tok_e_hint).block_m
            single_launch = single_launch_default(gate_up.layout, deterministic, down.k, block_m)
        self.single_launch = single_launch
        if single_launch and (not glu or deterministic):
            raise ValueError("single_launch needs GLU16 gate_up weights and no deterministic pass")
        self._plan_for(max_tokens)

    def _plan_for(self, tokens: int):
        hint = self.tok_e_hint
        self.plan_gu = ops.w4a16_plan(tokens, self.topk, self.num_experts, self.gate_up.n,
                                      self.gate_up.k, hint)
        self.plan_dn = ops.w4a16_plan(tokens, self.topk, self.num_experts, self.down.n,
                                      self.down.k, hint)
        self.fused_act = self.gate_up.layout == ops.W4A16_LAYOUT_KTILE64_GLU16
        self.plan_gu.layout = self.gate_up.layout
        if self.single_launch:
            # one launch over one set of routing blocks
            if self.plan_gu.block_m > 128:
                raise ValueError("single_launch needs routing blocks of at most 128 rows")
            self.plan_dn.block_m = self.plan_gu.block_m
        self.block_m = self.plan_gu.block_m
        numel = self.max_tokens * self.topk
        self.capacity = ops.w4a16_align_capacity(numel, self.num_experts, self.block_m)
        dev = self.device
        self.sorted_ids = torch.empty(self.capacity, dtype=torch.int32, device=dev)
        self.expert_ids = torch.empty(self.capacity // self.block_m, dtype=torch.int32, device=dev)
        self.ntp = torch.empty(1, dtype=torch.int32, device=dev)
        # The down GEMM may take other blocks than gate_up (when the plans
        # differ, e.g. a 256-row gate_up plan): gate_up writes its rows in
        # token order, so each GEMM reads its own routing.
        self.block_m_dn = self.plan_dn.block_m
        if self.block_m_dn != self.block_m:
            self.capacity_dn = ops.w4a16_align_capacity(numel, self.num_experts, self.block_m_dn)
            self.sorted_ids_dn = torch.empty(self.capacity_dn, dtype=torch.int32, device=dev)
            self.expert_ids_dn = torch.empty(self.capacity_dn // self.block_m_dn,
                                             dtype=torch.int32, device=dev)
            self.ntp_dn = torch.empty(1, dtype=torch.int32, device=dev)
        else:
            self.capacity_dn = self.capacity
            self.sorted_ids_dn, self.expert_ids_dn, self.ntp_dn = (
                self.sorted_ids, self.expert_ids, self.ntp)
        self.inter_buf = torch.empty((numel, 2 * self.inter), dtype=torch.bfloat16, device=dev)
        self.act_buf = torch.empty((numel, self.inter), dtype=torch.bfloat16, device=dev)
        # one workspace for both GEMMs (ordered on one stream): status words
        # and the routed rows of the wider activation (x, k = hidden)
        self.workspace = ops.new_workspace(
            self.plan_gu, dev, max(self.capacity, self.capacity_dn), max(self.hidden, self.inter),
            det_n=self.hidden if self.deterministic else 0, det_numel=numel)
        if self.single_launch:
            self.layer_workspace = torch.zeros(
                ops.w4a16_layer_workspace_size(self.plan_gu, self.capacity, self.hidden,
                                               self.inter), dtype=torch.uint8, device=dev)

    def align(self, topk_ids: torch.Tensor, stream=None):
        """Routing blocks of both GEMMs (one align, two when their block sizes
        differ)."""
        self._align_down(topk_ids, stream)
        return ops.w4a16_moe_align_block_size(
            topk_ids, self.num_experts, self.block_m, self.capacity,
            out=(self.sorted_ids, self.expert_ids, self.ntp), stream=stream)

    def _align_down(self, topk_ids: torch.Tensor, stream=None):
        if self.block_m_dn != self.block_m:
            ops.w4a16_moe_align_block_size(
                topk_ids, self.num_experts, self.block_m_dn, self.capacity_dn,
                out=(self.sorted_ids_dn, self.expert_ids_dn, self.ntp_dn), stream=stream)

    def gate_up_gemm(self, x: torch.Tensor, tokens: int, stream=None):
        numel = tokens * self.topk
        return ops.w4a16_moe_indexed_gemm(
            ops.W4A16_GATE_UP, self.gate_up.packed, self.num_experts, self.gate_up.n,
            self.gate_up.k, x, tokens, self.topk, self.sorted_ids, self.expert_ids, self.ntp,
            self.plan_gu, self.workspace, out=self.inter_buf[:numel], stream=stream)

    def gate_up_act(self, x: torch.Tensor, tokens: int, stream=None):
        """gate_up with the activation fused: writes act_buf directly."""
        numel = tokens * self.topk
        return ops.w4a16_moe_indexed_gemm(
            ops.W4A16_GATE_UP_SILU, self.gate_up.packed, self.num_experts, self.gate_up.n,
            self.gate_up.k, x, tokens, self.topk, self.sorted_ids, self.expert_ids, self.ntp,
            self.plan_gu, self.workspace, out=self.act_buf[:numel], stream=stream)

    def layer_single_launch(self, x: torch.Tensor, tokens: int, topk_weights: torch.Tensor,
                            out: torch.Tensor, stream=None):
        """gate_up, activation and down in one launch (w4a16_moe_layer)."""
        return ops.w4a16_moe_layer(
            self.gate_up.packed, self.down.packed, self.num_experts, self.hidden, self.inter, x,
            tokens, self.topk, self.sorted_ids, self.expert_ids, self.ntp, self.plan_gu,
            self.layer_workspace, topk_weights, out=out, stream=stream)

    def activation(self, tokens: int, stream=None):
        numel = tokens * self.topk
        return ops.w4a16_silu_and_mul(self.inter_buf[:numel], out=self.act_buf[:numel],
                                      stream=stream)

    def down_gemm(self, tokens: int, topk_weights: torch.Tensor, out: torch.Tensor, stream=None):
        numel = tokens * self.topk
        return ops.w4a16_moe_indexed_gemm(
            ops.W4A16_DOWN, self.down.packed, self.num_experts, self.down.n, self.down.k,
            self.act_buf[:numel], tokens, self.topk, self.sorted_ids_dn, self.expert_ids_dn,
            self.ntp_dn, self.plan_dn, self.workspace, topk_weights=topk_weights, out=out,
            flags=ops.W4A16_FLAG_DETERMINISTIC if self.deterministic else 0, stream=stream)

    def route(self, router_logits: torch.Tensor, expert_offset: int = 0,
              renormalize: bool = True, stream=None):
        """Router logits [T, E_global] (fp32 or BF16) -> (topk_ids, topk_weights)
        for this GPU's experts [expert_offset, expert_offset + num_experts),
        on the device (w4a16_topk_softmax)."""
        tokens = router_logits.shape[0]
        if not hasattr(self, "_route_ids") or self._route_ids.shape[0] < tokens:
            self._route_ids = torch.empty((self.max_tokens, self.topk), dtype=torch.int32,
                                          device=self.device)
            self._route_w = torch.empty((self.max_tokens, self.topk), dtype=torch.float32,
                                        device=self.device)
        out = (self._route_ids[:tokens], self._route_w[:tokens])
        return ops.w4a16_topk_softmax(router_logits, self.topk, renormalize, expert_offset,
                                      self.num_experts, out=out, stream=stream)

    def route_align(self, router_logits: torch.Tensor, expert_offset: int = 0,
                    renormalize: bool = True, stream=None):
        """route() and align() in one launch (w4a16_moe_route_align): returns
        (topk_ids, topk_weights) and fills the layer's routing tensors."""
        tokens = router_logits.shape[0]
        if tokens > self.max_tokens:
            raise ValueError("more tokens than the layer was planned for")
        if not hasattr(self, "_route_ids"):
            self._route_ids = torch.empty((self.max_tokens, self.topk), dtype=torch.int32,
                                          device=self.device)
            self._route_w = torch.empty((self.max_tokens, self.topk), dtype=torch.float32,
                                        device=self.device)
        if not hasattr(self, "_arrivals"):
            self._arrivals = torch.zeros(1, dtype=torch.int32, device=self.device)
        ids, w = self._route_ids[:tokens], self._route_w[:tokens]
        ops.w4a16_moe_route_align(
            router_logits, self.topk, self.block_m, self._arrivals, renormalize, expert_offset,
            self.num_experts, self.capacity,
            out=(ids, w, self.sorted_ids, self.expert_ids, self.ntp), stream=stream)
        # the down GEMM's own blocks over the same local ids
        self._align_down(ids, stream)
        return ids, w

    def forward_from_logits(self, x: torch.Tensor, router_logits: torch.Tensor,
                            expert_offset: int = 0, renormalize: bool = True,
                            out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """The whole layer from router logits: route + align (one launch),
        gate_up(+act), down."""
        _, w = self.route_align(router_logits, expert_offset, renormalize, stream)
        return self.experts(x, w, out=out, stream=stream)

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_weights: torch.Tensor,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """x BF16 [T, H], topk_ids int32 [T, topk], topk_weights fp32 [T, topk]
        -> fp32 [T, H] (this GPU's experts' share of the top-k weighted sum)."""
        tokens = x.shape[0]
        if tokens > self.max_tokens:
            raise ValueError("more tokens than the layer was planned for")
        if out is None:
            out = torch.empty((tokens, self.hidden), dtype=torch.float32, device=x.device)
        self.align(topk_ids, stream)
        return self.experts(x, topk_weights, out=out, stream=stream)

    def experts(self, x: torch.Tensor, topk_weights: torch.Tensor,
                out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
        """gate_up(+act) and down over the routing tensors already aligned."""
        tokens = x.shape[0]
        if out is None:
            out = torch.empty((tokens, self.hidden), dtype=torch.float32, device=x.device)
        if self.single_launch:
            return self.layer_single_launch(x, tokens, topk_weights, out, stream)
        if self.fused_act:
            self.gate_up_act(x, tokens, stream)
        else:
            self.gate_up_gemm(x, tokens, stream)
            self.activation(tokens, stream)
        self.down_gemm(tokens, topk_weights, out, stream)
        return out
