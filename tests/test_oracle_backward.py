"""Pins of the oracle's backward pass: central finite differences of the (separately pinned)
oracle forward, on small fp32 layers whose routing margins keep the top-k choice and the
capacity drops fixed under the perturbation.

Loss: L = sum_t <dout_t, out_t> + a * L_aux + b * L_z with out from oracle.forward_naive,
L_aux from oracle.stats (E sum f P, f counted, i.e. constant while routing is fixed) and L_z
from oracle.router_stats.  Readings under test: no gradient through the top-k choice or the
capacity drop; the selection-only bias has no gradient; a dropped assignment passes nothing.
Step sizes: 1e-2 on expert weights and x (the loss is smooth there; the fp32 output rounding,
~6e-8 relative, then costs < 1e-4), 1e-3 on the router (probabilities move less than the
margins).  Tolerance |fd - g| <= 2e-3 (1 + |g|).
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle

TOL = 2e-3


def loss(layer, spec, dout, a, b):
    bm = spec.bias_mode if spec.zipf_bias > 0 else None
    out, ex = oracle.forward_naive(layer, spec.k, oracle.F32, cf=spec.capacity_factor,
                                   renorm=spec.renorm, round_h=0, bias_mode=bm)
    st = oracle.stats(ex["idx"], ex["probs"], ex["keep"], ex["gap"])
    _, _, _, _, lse = oracle.route(layer["x"], layer["W_r"], layer["b_r"], spec.k, oracle.F32,
                                   renorm=spec.renorm, bias_mode=bm, with_lse=True)
    z = oracle.router_stats(ex["idx"], ex["w"], lse, spec.E)["z_loss"]
    return float(np.sum(dout * out.astype(np.float64)) + a * st["aux"] + b * z), ex


def check_fd(spec, seed, a=0.3, b=0.05, n_pick=12, tensors=None):
    L = moe_synth.make_layer(spec, seed=seed)
    L = {k: (None if v is None else v.clone()) for k, v in L.items()}
    rng = np.random.default_rng(seed)
    dout = rng.standard_normal((spec.N, spec.d))
    bm = spec.bias_mode if spec.zipf_bias > 0 else None
    g = oracle.backward(L, spec.k, oracle.F32, dout, cf=spec.capacity_factor, renorm=spec.renorm,
                        round_h=0, bias_mode=bm, aux_coef=a, z_coef=b)
    base, ex0 = loss(L, spec, dout, a, b)
    names = tensors or [("x", "dx"), ("W_r", "dW_r"), ("W_gate", "dW_gate"), ("W_up", "dW_up"),
                        ("W_down", "dW_down"), ("Ws_gate", "dWs_gate"), ("Ws_up", "dWs_up"),
                        ("Ws_down", "dWs_down"), ("b_r", "db")]
    checked = 0
    for pname, gname in names:
        if L.get(pname) is None:
            continue
        t = L[pname]
        flat = t.view(-1)
        h = 1e-3 if pname in ("W_r", "b_r") else 1e-2
        for i in rng.choice(flat.numel(), size=min(n_pick, flat.numel()), replace=False):
            old = float(flat[i])
            flat[i] = old + h
            lp, exp_ = loss(L, spec, dout, a, b)
            flat[i] = old - h
            lm, exm = loss(L, spec, dout, a, b)
            flat[i] = old
            assert np.array_equal(exp_["idx"], ex0["idx"]) and np.array_equal(exm["idx"], ex0["idx"])
            assert np.array_equal(exp_["keep"], ex0["keep"]) and np.array_equal(exm["keep"], ex0["keep"])
            fd = (lp - lm) / (2 * h)
            gv = float(g[gname].reshape(-1)[i])
            assert abs(fd - gv) <= TOL * (1 + abs(gv)), (pname, int(i), fd, gv)
            checked += 1
    return g, checked


BASE = moe_synth.LayerSpec("bwd", N=6, d=8, d_ff=12, E=4, k=2, n_shared=1, d_ff_shared=10,
                           dtype="f32")


def test_fd_all_parameters_shared_aux_z():
    g, n = check_fd(BASE, seed=3)
    assert n > 80


def test_fd_logit_bias():
    spec = BASE.with_(zipf_bias=1.2, bias_mode=1, N=5)
    g, n = check_fd(spec, seed=4)
    assert np.any(g["db"] != 0)


def test_fd_selection_only_bias_has_no_bias_gradient():
    spec = BASE.with_(zipf_bias=1.2, bias_mode=2, N=5, n_shared=0)
    g, n = check_fd(spec, seed=5)
    assert np.all(g["db"] == 0)


def test_fd_capacity_drops():
    spec = BASE.with_(N=10, E=4, k=2, capacity_factor=0.6, n_shared=0)
    seed = 16                                      # routing margin 0.058 (selection gap)
    L = moe_synth.make_layer(spec, seed=seed)
    _, ex = oracle.forward_naive(L, spec.k, oracle.F32, cf=spec.capacity_factor, round_h=0)
    assert ex["keep"].min() == 0                   # some assignments really are dropped
    assert ex["gap"].min() > 0.05
    check_fd(spec, seed=seed)


def test_fd_without_renormalisation():
    check_fd(BASE.with_(renorm=0, n_shared=0), seed=7)


def test_single_expert_router_gets_no_gradient_from_the_output():
    """E = k = 1: w = 1 whatever the logits, so only the aux and z terms move W_r."""
    spec = moe_synth.LayerSpec("one", N=4, d=6, d_ff=8, E=1, k=1, dtype="f32")
    L = moe_synth.make_layer(spec, seed=1)
    dout = np.random.default_rng(1).standard_normal((4, 6))
    g = oracle.backward(L, 1, oracle.F32, dout, round_h=0)
    assert np.all(g["dW_r"] == 0)
    assert np.any(g["dW_down"] != 0)


def test_zero_upstream_gradient_leaves_only_the_losses():
    L = moe_synth.make_layer(BASE, seed=2)
    z = np.zeros((BASE.N, BASE.d))
    g = oracle.backward(L, BASE.k, oracle.F32, z, round_h=0)
    for n in ("dx", "dW_r", "dW_gate", "dW_up", "dW_down", "dWs_gate"):
        assert np.all(g[n] == 0), n
    g2 = oracle.backward(L, BASE.k, oracle.F32, z, round_h=0, aux_coef=1.0)
    assert np.any(g2["dW_r"] != 0) and np.all(g2["dW_down"] == 0)
