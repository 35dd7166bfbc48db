"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run the oracle on
the same seeded inputs, and compare what is unique.

Tolerances (the layer's stated bar):
  routing indices, counts, offsets, permutation, positions: bit-exact, except tokens whose
  k-th and (k+1)-th oracle probabilities differ by less than 1e-6 (their expert set is not
  numerically unique), which are reported and excluded;
  routing weights and the near-tie gap: |w - w_oracle| <= 2e-6.  Derivation: the GPU logit is
  an fp32 FMA chain over each 32-wide slice of d, slices combined with compensated summation,
  so its error is about u*sqrt(32) ~ 3.4e-7 rms (u = 2^-24) whatever d is, against the
  oracle's correctly rounded logit; w_j = softmax over the selected logits moves by at most
  half the spread of the logit errors, so 6 sigma stays under 2e-6;
  fp32 layers: max-abs error of the output <= 1e-4;
  bf16 layers: per-token relative L2 error ||y - y*|| / ||y*|| <= 2e-2, and a token whose
  every assignment was dropped (y* = 0 without shared experts) must be exactly 0.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

TIE = 1e-6
W_TOL = 2e-6
F32_TOL = 1e-4
BF16_REL = 2e-2


def dtype_code(spec) -> int:
    return oracle.BF16 if spec.dtype == "bf16" else oracle.F32


def to_dev(layer: dict) -> dict:
    return {k: (None if v is None else v.cuda()) for k, v in layer.items()}


def out_f64(out, spec) -> np.ndarray:
    if isinstance(out, torch.Tensor):
        return out.detach().float().cpu().double().numpy()
    if spec.dtype == "bf16":
        return oracle.bf16_bits_to_f32(out).astype(np.float64)
    return out.astype(np.float64)


def internal_tie(probs: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Tokens whose selected probabilities contain two within TIE (slot order not unique)."""
    sel = np.take_along_axis(probs.astype(np.float64), idx.astype(np.int64), axis=1)
    if sel.shape[1] < 2:
        return np.zeros(sel.shape[0], bool)
    return np.any(np.abs(np.diff(sel, axis=1)) < TIE, axis=1)


def check_routing(idx_g, w_g, gap_g, idx_o, w_o, probs_o, gap_o, scores_o=None):
    """Bit-exact routing on every token whose expert set is unique; returns (excluded mask,
    tokens whose GPU routing differs from the oracle's).  scores_o: the selection scores when
    they are not the probabilities (selection-only bias)."""
    idx_g = np.asarray(idx_g)
    w_g = np.asarray(w_g)
    excl = gap_o < TIE
    order_tie = internal_tie(probs_o if scores_o is None else scores_o, idx_o)
    strict = ~excl & ~order_tie
    bad = np.nonzero(strict & np.any(idx_g != idx_o, axis=1))[0]
    assert bad.size == 0, f"routing differs on tokens {bad[:10]} ({bad.size})"
    np.testing.assert_array_less(np.abs(w_g[strict] - w_o[strict]), W_TOL)
    loose = ~excl & order_tie
    for t in np.nonzero(loose)[0]:
        assert sorted(idx_g[t]) == sorted(idx_o[t])
    if gap_g is not None:
        g = np.asarray(gap_g, np.float64)
        fin = np.isfinite(gap_o)
        np.testing.assert_allclose(g[fin], gap_o[fin].astype(np.float64), atol=W_TOL, rtol=0)
    differs = np.nonzero(np.any(np.sort(idx_g, 1) != np.sort(idx_o, 1), axis=1))[0]
    assert np.all(excl[differs])
    return excl, differs


def compare_rows(got: np.ndarray, ref: np.ndarray, spec, rows=None, what="output"):
    """got/ref float64 [n, d]."""
    if rows is not None:
        got, ref = got[rows], ref[rows]
    if got.size == 0:
        return
    if spec.dtype == "f32":
        err = np.abs(got - ref).max()
        assert err <= F32_TOL, f"{what}: max-abs error {err:.3e} > {F32_TOL}"
        return
    nref = np.linalg.norm(ref, axis=1)
    nerr = np.linalg.norm(got - ref, axis=1)
    zero = nref == 0
    assert np.all(nerr[zero] == 0), f"{what}: rows that must be exactly 0 are not"
    rel = nerr[~zero] / nref[~zero]
    if rel.size:
        worst = int(np.argmax(rel))
        assert rel.max() <= BF16_REL, f"{what}: relative L2 error {rel.max():.3e} (row {worst})"


class ExpertCache:
    """Host copies of individual experts' matrices (for sampled oracle checks)."""

    def __init__(self, layer_dev: dict):
        self.L = layer_dev
        self.cache = {}

    def routed(self, e: int):
        key = ("r", e)
        if key not in self.cache:
            self.cache[key] = tuple(self.L[n][e].cpu() for n in ("W_gate", "W_up", "W_down"))
        return self.cache[key]

    def shared(self):
        if self.L.get("Ws_gate") is None:
            return []
        out = []
        for s in range(self.L["Ws_gate"].shape[0]):
            key = ("s", s)
            if key not in self.cache:
                self.cache[key] = tuple(self.L[n][s].cpu() for n in ("Ws_gate", "Ws_up", "Ws_down"))
            out.append(self.cache[key])
        return out


def oracle_tokens(spec, x_host, tokens, idx_o, w_o, keep_o, cache: ExpertCache) -> np.ndarray:
    """Oracle layer output for the given tokens (threads: the C calls release the GIL)."""
    code = dtype_code(spec)
    shared = cache.shared()
    for t in tokens:                       # fill the cache in this thread
        for e in idx_o[t]:
            cache.routed(int(e))

    def one(t):
        experts = [cache.routed(int(e)) for e in idx_o[t]]
        o = oracle.moe_token(x_host[t], w_o[t], keep_o[t], experts, shared, code,
                             1 if code == oracle.BF16 else 0)
        return out_f64(o, spec)

    workers = max(1, min(32, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(workers) as ex:
        rows = list(ex.map(one, tokens))
    return np.stack(rows) if rows else np.zeros((0, spec.d))


def run_layer(spec, layer_dev: dict):
    cfg = moe.cfg_from_spec(spec)
    lay = moe.MoELayer(cfg, layer_dev)
    out = lay.forward(layer_dev["x"]).clone()
    torch.cuda.synchronize()
    return lay, out
