"""Seeded synthetic inputs for the top-k routed MoE FFN layer.

This module is the only code shared by the CUDA path's tests/bench and the CPU
oracle's tests.  It draws random tensors and describes layer shapes; it holds
none of the layer's arithmetic (no routing, no FFN, no grouping).

Recipe (all layers): one seeded ``torch.Generator``; draw order x, W_r, W_gate,
W_up, W_down, then the shared experts' Ws_gate, Ws_up, Ws_down.
  x ~ N(0, 1); W_r, W_gate, W_up, Ws_gate, Ws_up ~ N(0, 1/d);
  W_down ~ N(0, 1/d_ff); Ws_down ~ N(0, 1/d_ff_shared).
Values are drawn in fp32; bf16 layers round x and the expert weights to
nearest-even bf16, the router weight stays fp32.  Layouts follow nn.Linear
(out x in, input dim contiguous): W_r [E, d], W_gate/W_up [E, F, d],
W_down [E, d, F], shared [S, F_s, d] / [S, d, F_s].

The skewed layer adds a router bias b_e = ln((e+1)^-s / H_E(s)) with s = 1.2,
a Zipf law over expert rank, so low-index experts are overloaded.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import torch

F32 = "f32"
BF16 = "bf16"


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    name: str
    N: int            # tokens in the batch
    d: int            # model dim
    d_ff: int         # routed expert hidden dim
    E: int            # routed experts
    k: int            # experts per token
    n_shared: int = 0
    d_ff_shared: int = 0
    capacity_factor: float = 0.0   # <= 0: no capacity limit
    dtype: str = BF16
    zipf_bias: float = 0.0         # > 0: router bias ln Zipf(s) over expert rank
    renorm: int = 1
    bias_mode: int = 1             # how a router bias enters: 1 logits, 2 top-k choice only
    w4a16: bool = False            # expert weights run as 4-bit codes + per-128 scales

    def with_(self, **kw) -> "LayerSpec":
        return dataclasses.replace(self, **kw)


# The five layers of the workload set, plus the page's own self-test shape.
TINY = LayerSpec("tiny_fp32", N=64, d=128, d_ff=256, E=8, k=2, n_shared=1,
                 d_ff_shared=256, dtype=F32)
MIXTRAL = LayerSpec("mixtral_8x_bf16", N=4096, d=4096, d_ff=14336, E=8, k=2)
DSV3_PREFILL = LayerSpec("deepseek_v3_prefill_bf16", N=8192, d=7168, d_ff=2048,
                         E=256, k=8, n_shared=1, d_ff_shared=2048)
DSV3_DECODE = DSV3_PREFILL.with_(name="deepseek_v3_decode_bf16", N=64)
DSV3_DECODE_W4 = DSV3_DECODE.with_(name="deepseek_v3_decode_w4a16", w4a16=True)
QWEN3_SKEWED = LayerSpec("qwen3_30b_a3b_skewed_bf16", N=16384, d=2048, d_ff=768,
                         E=128, k=8, capacity_factor=1.25, zipf_bias=1.2)
PAGE_SELFTEST = LayerSpec("page_selftest_fp32", N=50, d=64, d_ff=128, E=16, k=4,
                          n_shared=1, d_ff_shared=128, dtype=F32)

WORKLOADS = {s.name: s for s in (TINY, MIXTRAL, DSV3_PREFILL, DSV3_DECODE, QWEN3_SKEWED,
                                  DSV3_DECODE_W4)}


def zipf_bias(E: int, s: float) -> torch.Tensor:
    """b_e = ln((e+1)^-s / H) with H = sum_{r=1..E} r^-s (expert e has rank e+1)."""
    ranks = torch.arange(1, E + 1, dtype=torch.float64)
    h = torch.sum(ranks ** (-s))
    return (torch.log(ranks ** (-s) / h)).to(torch.float32)


def _randn(gen: torch.Generator, shape, std: float, device) -> torch.Tensor:
    t = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        t.mul_(std)
    return t


def make_layer(spec: LayerSpec, seed: int = 0, device: str | torch.device = "cpu",
               x_only: bool = False) -> Dict[str, Optional[torch.Tensor]]:
    """Draw one layer's inputs.  Returns a dict of tensors on ``device``.

    Expert weights are drawn one expert at a time so that the fp32 staging
    buffer stays one expert large even for 256-expert layers.
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    act = torch.bfloat16 if spec.dtype == BF16 else torch.float32
    d, F, E, S, Fs = spec.d, spec.d_ff, spec.E, spec.n_shared, spec.d_ff_shared

    out: Dict[str, Optional[torch.Tensor]] = {}
    out["x"] = _randn(gen, (spec.N, d), 1.0, device).to(act)
    out["W_r"] = _randn(gen, (E, d), d ** -0.5, device)
    out["b_r"] = zipf_bias(E, spec.zipf_bias).to(device) if spec.zipf_bias > 0 else None
    if x_only:
        return out

    def bank(n_exp: int, rows: int, cols: int, std: float) -> torch.Tensor:
        t = torch.empty((n_exp, rows, cols), dtype=act, device=device)
        for e in range(n_exp):
            t[e].copy_(_randn(gen, (rows, cols), std, device))
        return t

    out["W_gate"] = bank(E, F, d, d ** -0.5)
    out["W_up"] = bank(E, F, d, d ** -0.5)
    out["W_down"] = bank(E, d, F, F ** -0.5)
    if S > 0:
        out["Ws_gate"] = bank(S, Fs, d, d ** -0.5)
        out["Ws_up"] = bank(S, Fs, d, d ** -0.5)
        out["Ws_down"] = bank(S, d, Fs, Fs ** -0.5)
    else:
        out["Ws_gate"] = out["Ws_up"] = out["Ws_down"] = None
    return out


def make_x(spec: LayerSpec, seed: int, device="cpu") -> torch.Tensor:
    """A fresh activation batch (used for per-step inputs in the end-to-end timing)."""
    gen = torch.Generator(device=torch.device(device))
    gen.manual_seed(seed)
    act = torch.bfloat16 if spec.dtype == BF16 else torch.float32
    return _randn(gen, (spec.N, spec.d), 1.0, device).to(act)


def capacity_note(spec: LayerSpec) -> str:
    if spec.capacity_factor <= 0:
        return "none"
    return f"CF={spec.capacity_factor}"


def sample_tokens(N: int, n: int, seed: int) -> torch.Tensor:
    """A seeded, sorted sample of n distinct token indices out of N (for sampled checks)."""
    n = min(n, N)
    gen = torch.Generator()
    gen.manual_seed(seed)
    return torch.sort(torch.randperm(N, generator=gen)[:n]).values


def numel_bytes(spec: LayerSpec) -> int:
    """Bytes of all layer inputs (x + router + routed + shared weights)."""
    a = 2 if spec.dtype == BF16 else 4
    w = 3 * spec.E * spec.d * spec.d_ff + 3 * spec.n_shared * spec.d * spec.d_ff_shared
    return spec.N * spec.d * a + spec.E * spec.d * 4 + w * a


__all__ = ["LayerSpec", "make_layer", "make_x", "zipf_bias", "sample_tokens", "WORKLOADS",
           "TINY", "MIXTRAL", "DSV3_PREFILL", "DSV3_DECODE", "QWEN3_SKEWED", "PAGE_SELFTEST",
           "F32", "BF16"]
