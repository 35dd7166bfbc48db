"""Pins for the oracle's expert FFNs, shared experts and the whole layer.

Page: "混合专家 MoE", sections "结构" (y = sum over the top-k of w_i Expert_i(x),
shared expert on every token) and "实现：逐 token 与按专家分组" (Expert =
down(silu(gate x) * up x) without biases; forward_naive == forward_grouped,
checked there with allclose(atol=1e-5) on d=64, d_ff=128, 16 experts, top-4,
50 tokens, one shared expert).
"""
import numpy as np
import pytest
import torch

import moe_synth


def _np64(t):
    return t.to(torch.float64).numpy()


def _swiglu_np(x, Wg, Wu, Wd):
    """Textbook SwiGLU with numpy matmuls (fp64)."""
    g = x @ Wg.T
    u = x @ Wu.T
    return (g / (1.0 + np.exp(-g)) * u) @ Wd.T


def _bf16_round_torch(a):
    return torch.from_numpy(a).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def test_bf16_rounding_matches_torch(orc):
    g = torch.Generator().manual_seed(0)
    vals = torch.cat([torch.randn(4000, generator=g) * 10.0 ** torch.randint(-30, 30, (4000,), generator=g),
                      torch.tensor([1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 3e38, -3.4e38,
                                    1e-40, -1e-41, 0.0, -0.0])])
    ref = vals.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.round_bf16(float(v)) for v in vals], np.uint16)
    np.testing.assert_array_equal(got, ref)


def test_single_expert_is_dense_swiglu(orc):
    """E = k = 1, no shared expert: the layer is one SwiGLU FFN (numpy matmul)."""
    spec = moe_synth.LayerSpec("dense", N=12, d=24, d_ff=40, E=1, k=1, dtype="f32")
    L = moe_synth.make_layer(spec, seed=4)
    out, ex = orc.forward_naive(L, 1, orc.F32)
    ref = _swiglu_np(_np64(L["x"]), _np64(L["W_gate"][0]), _np64(L["W_up"][0]), _np64(L["W_down"][0]))
    np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-7)
    assert np.all(ex["w"] == 1.0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_layer_matches_numpy_per_token_sum(orc, dtype):
    """out_t = sum_j w_tj Expert_{idx_tj}(x_t) + Shared(x_t), with non-square shapes so that a
    transposed operand or a wrong expert index cannot go unnoticed."""
    spec = moe_synth.LayerSpec("t", N=20, d=24, d_ff=40, E=6, k=2, n_shared=1, d_ff_shared=56,
                               dtype=dtype)
    L = moe_synth.make_layer(spec, seed=2)
    code = orc.BF16 if dtype == "bf16" else orc.F32
    out, ex = orc.forward_naive(L, 2, code)
    x = _np64(L["x"])
    ref = np.zeros_like(x)
    for t in range(spec.N):
        for j in range(2):
            e = ex["idx"][t, j]
            g = x[t] @ _np64(L["W_gate"][e]).T
            u = x[t] @ _np64(L["W_up"][e]).T
            h = g / (1 + np.exp(-g)) * u
            if dtype == "bf16":
                h = _bf16_round_torch(h)
            ref[t] += float(ex["w"][t, j]) * (h @ _np64(L["W_down"][e]).T)
        g = x[t] @ _np64(L["Ws_gate"][0]).T
        u = x[t] @ _np64(L["Ws_up"][0]).T
        h = g / (1 + np.exp(-g)) * u
        if dtype == "bf16":
            h = _bf16_round_torch(h)
        ref[t] += h @ _np64(L["Ws_down"][0]).T
    if dtype == "bf16":
        got = orc.bf16_bits_to_f32(out).astype(np.float64)
        # one bf16 rounding of the output (+ fp64 summation-order noise)
        np.testing.assert_allclose(got, ref, rtol=2 ** -8, atol=1e-6)
    else:
        np.testing.assert_allclose(out, ref, rtol=1e-6, atol=1e-6)


def test_naive_equals_grouped_page_shape(orc):
    L = moe_synth.make_layer(moe_synth.PAGE_SELFTEST, seed=0)
    a, _ = orc.forward_naive(L, 4, orc.F32)
    b = orc.forward_grouped(L, 4, orc.F32)
    np.testing.assert_allclose(a, b, atol=1e-5, rtol=0)


@pytest.mark.parametrize("spec,cf", [
    (moe_synth.TINY, 0.0),
    (moe_synth.LayerSpec("cap", N=96, d=32, d_ff=48, E=8, k=3, n_shared=1, d_ff_shared=16,
                         dtype="bf16", zipf_bias=1.2), 0.75),
])
def test_naive_equals_grouped(orc, spec, cf):
    L = moe_synth.make_layer(spec, seed=1)
    code = orc.BF16 if spec.dtype == "bf16" else orc.F32
    a, ex = orc.forward_naive(L, spec.k, code, cf=cf)
    b = orc.forward_grouped(L, spec.k, code, cf=cf)
    if code == orc.BF16:
        a, b = orc.bf16_bits_to_f32(a), orc.bf16_bits_to_f32(b)
        np.testing.assert_allclose(a, b, atol=1e-5, rtol=2 ** -8)
        assert ex["keep"].min() == 0          # the capacity case really drops
    else:
        np.testing.assert_allclose(a, b, atol=1e-5, rtol=0)


def test_identical_experts_make_routing_irrelevant(orc):
    """All experts equal => out_t = Expert(x_t) + Shared(x_t), since the weights sum to 1."""
    spec = moe_synth.LayerSpec("same", N=30, d=16, d_ff=24, E=5, k=3, n_shared=1, d_ff_shared=8,
                               dtype="f32")
    L = moe_synth.make_layer(spec, seed=6)
    for n in ("W_gate", "W_up", "W_down"):
        L[n] = L[n][:1].repeat(5, 1, 1).contiguous()
    out, _ = orc.forward_naive(L, 3, orc.F32)
    x = _np64(L["x"])
    ref = _swiglu_np(x, _np64(L["W_gate"][0]), _np64(L["W_up"][0]), _np64(L["W_down"][0])) + \
        _swiglu_np(x, _np64(L["Ws_gate"][0]), _np64(L["Ws_up"][0]), _np64(L["Ws_down"][0]))
    np.testing.assert_allclose(out, ref, rtol=1e-5, atol=1e-6)


def test_zero_weights_give_zero(orc):
    spec = moe_synth.LayerSpec("z", N=10, d=16, d_ff=8, E=4, k=2, n_shared=1, d_ff_shared=8,
                               dtype="bf16")
    L = moe_synth.make_layer(spec, seed=3)
    for n in ("W_down", "Ws_down"):
        L[n] = torch.zeros_like(L[n])
    out, _ = orc.forward_naive(L, 2, orc.BF16)
    assert np.all(orc.bf16_bits_to_f32(out) == 0.0)


def test_fully_dropped_token_keeps_only_shared(orc):
    """Capacity 0 drops every routed assignment: output = shared expert alone; without a
    shared expert it is exactly 0 (only the residual path remains)."""
    spec = moe_synth.LayerSpec("drop", N=8, d=16, d_ff=8, E=4, k=2, n_shared=1, d_ff_shared=12,
                               dtype="f32")
    L = moe_synth.make_layer(spec, seed=8)
    out, ex = orc.forward_naive(L, 2, orc.F32, cf=1e-9)   # C = 1: first token per expert only
    x = _np64(L["x"])
    sh = _swiglu_np(x, _np64(L["Ws_gate"][0]), _np64(L["Ws_up"][0]), _np64(L["Ws_down"][0]))
    routed = out - sh
    for t in range(8):
        if ex["keep"][t].sum() == 0:
            np.testing.assert_allclose(out[t], sh[t], rtol=1e-6, atol=1e-7)
    L2 = dict(L, Ws_gate=None, Ws_up=None, Ws_down=None)
    out2, ex2 = orc.forward_naive(L2, 2, orc.F32, cf=1e-9)
    dropped_rows = ex2["keep"].sum(1) == 0
    assert dropped_rows.any()
    assert np.all(out2[dropped_rows] == 0.0)
    del routed


def test_moe_token_matches_forward_naive(orc):
    spec = moe_synth.LayerSpec("tok", N=6, d=32, d_ff=16, E=5, k=2, n_shared=1, d_ff_shared=24,
                               dtype="bf16")
    L = moe_synth.make_layer(spec, seed=9)
    out, ex = orc.forward_naive(L, 2, orc.BF16)
    for t in range(6):
        experts = [(L["W_gate"][e], L["W_up"][e], L["W_down"][e]) for e in ex["idx"][t]]
        shared = [(L["Ws_gate"][0], L["Ws_up"][0], L["Ws_down"][0])]
        o = orc.moe_token(L["x"][t], ex["w"][t], ex["keep"][t], experts, shared, orc.BF16, 1)
        np.testing.assert_array_equal(o, out[t])
