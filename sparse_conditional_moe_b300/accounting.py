"""Algorithmic work of one MoE layer forward pass: FLOPs, bytes, roofline time.

Counts only what the method itself must touch (no intermediates):
  FLOPs = 6 d F per kept assignment (gate, up, down: 3 GEMV-sized products of
          2 d F each) + 6 d F_s per token per shared expert + 2 d E per token
          for the router;
  bytes = 3 d F per touched expert (an expert with >= 1 kept row) and per shared
          expert, times the activation element size, + the fp32 router weight
          (4 d E) + x read and out written (N d each, activation size).
Parameter counting follows the page "混合专家 MoE", section "总参数与激活参数"
(total minus the (E - k) unused experts per MoE layer) and its exercise 1.
"""
from __future__ import annotations

import dataclasses


def expert_params(d: int, d_ff: int) -> int:
    """gate [d_ff,d] + up [d_ff,d] + down [d,d_ff]."""
    return 3 * d * d_ff


def moe_param_counts(n_experts: int, top_k: int, d: int, d_ff: int, moe_layers: int):
    """(total, active) expert parameters over all MoE layers."""
    per = expert_params(d, d_ff)
    return n_experts * per * moe_layers, top_k * per * moe_layers


@dataclasses.dataclass
class Work:
    flops: float
    bytes: float

    def roofline_s(self, peak_flops: float, peak_bytes: float) -> float:
        return max(self.flops / peak_flops, self.bytes / peak_bytes)

    def bound(self, peak_flops: float, peak_bytes: float) -> str:
        return "tensor" if self.flops / peak_flops >= self.bytes / peak_bytes else "hbm"


# W4A16 expert weights: half a byte per code + one fp32 scale per 128 weights.
W4_BYTES_PER_WEIGHT = 0.5 + 4.0 / 128


def layer_work(N: int, d: int, d_ff: int, E: int, k: int, n_shared: int, d_ff_shared: int,
               act_bytes: int, kept_assignments: int, touched_experts: int,
               weight_bytes: float = 0.0) -> Work:
    """weight_bytes: bytes per expert weight (default: the activation size)."""
    wb = weight_bytes or act_bytes
    flops = (6.0 * d * d_ff * kept_assignments + 6.0 * d * d_ff_shared * n_shared * N
             + 2.0 * d * E * N)
    byts = (3.0 * d * d_ff * wb * touched_experts
            + 3.0 * d * d_ff_shared * wb * n_shared
            + 4.0 * d * E + 2.0 * N * d * act_bytes)
    return Work(flops, byts)


def gateup_flops(d: int, d_ff: int, rows: int) -> float:
    """gate + up projections over `rows` token rows (2 products of 2 d F each)."""
    return 4.0 * d * d_ff * rows


def down_flops(d: int, d_ff: int, rows: int) -> float:
    return 2.0 * d * d_ff * rows


def gateup_bytes(d: int, d_ff: int, rows: int, groups_touched: int, act_bytes: int = 2) -> float:
    """weights of the touched groups + the A rows read + the H rows written."""
    return act_bytes * (2.0 * d * d_ff * groups_touched + rows * d + rows * d_ff)


def down_bytes(d: int, d_ff: int, rows: int, groups_touched: int, act_bytes: int = 2) -> float:
    return act_bytes * (1.0 * d * d_ff * groups_touched + rows * d_ff + rows * d)
