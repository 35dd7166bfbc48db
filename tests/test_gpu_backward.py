"""GPU parity of moe_backward against the oracle's backward, through the C ABI.

The GPU runs the expert products on bf16 operands (dout, dh, dG, dU and w h rounded to bf16,
fp32 accumulation) where the oracle stays in fp64 with only h rounded (the forward's rounding
point); each rounding adds ~2^-9 relative error with random sign, so the bar is a relative L2
error <= 2e-2 per row: every token's dx, every row of dW_r and of every touched expert's
matrices (a row that nearly cancels is held to 2e-2 of 5 % of the rms row norm instead of its
own), untouched experts exactly 0, and the selection-only bias's gradient exactly 0.  The routing must
be the oracle's bit for bit on these seeds (no near ties), else the gradients are not comparable.
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import to_dev

pytestmark = pytest.mark.gpu

REL = 2e-2

LAYERS = [
    (moe_synth.LayerSpec("bwd_shared", N=96, d=128, d_ff=128, E=4, k=2, n_shared=1,
                         d_ff_shared=128), 0.01, 0.001),
    (moe_synth.LayerSpec("bwd_capacity_bias", N=160, d=256, d_ff=256, E=8, k=2,
                         capacity_factor=0.75, zipf_bias=1.2), 0.02, 0.0),
    (moe_synth.LayerSpec("bwd_selection_bias", N=64, d=192, d_ff=384, E=16, k=4, n_shared=1,
                         d_ff_shared=128, zipf_bias=1.2, bias_mode=2), 0.0, 0.01),
    (moe_synth.LayerSpec("bwd_many_experts", N=40, d=128, d_ff=128, E=64, k=6), 0.05, 0.0),
]


def rel(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / nb if nb > 0 else np.linalg.norm(a)


def rows_close(got, ref, what, floor=0.05):
    """Row by row: ||got_r - ref_r|| <= REL * max(||ref_r||, floor * rms row norm).  The floor
    keeps rows that nearly cancel (their bf16 rounding error scales with the terms, not with
    the small sum) from failing on their own magnitude; every other row is held to REL."""
    got = np.asarray(got, np.float64).reshape(got.shape[0], -1)
    ref = np.asarray(ref, np.float64).reshape(ref.shape[0], -1)
    nref = np.linalg.norm(ref, axis=1)
    scale = np.maximum(nref, floor * np.sqrt(np.mean(nref ** 2)))
    err = np.linalg.norm(got - ref, axis=1)
    bad = np.nonzero(err > REL * scale)[0]
    assert bad.size == 0, (what, bad[:8], (err[bad] / np.maximum(scale[bad], 1e-300))[:8])


@pytest.mark.parametrize("case", LAYERS, ids=lambda c: c[0].name)
def test_backward_matches_oracle(case):
    spec, aux, zc = case
    L = moe_synth.make_layer(spec, seed=17)
    dev = to_dev(L)
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev)
    lay.forward(dev["x"])
    gen = torch.Generator().manual_seed(5)
    dout = torch.randn((spec.N, spec.d), generator=gen).to(torch.bfloat16)
    g = lay.backward(dout.cuda(), aux_coef=aux, z_coef=zc)
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    bm = spec.bias_mode if spec.zipf_bias > 0 else None
    idx_o, _, _, gap_o = oracle.route(L["x"], L["W_r"], L["b_r"], spec.k, oracle.BF16, bias_mode=bm)
    assert np.array_equal(lay.buffers()["idx"].cpu().numpy(), idx_o), "routing differs"
    ref = oracle.backward(L, spec.k, oracle.BF16, dout.double().numpy(), cf=spec.capacity_factor,
                          bias_mode=bm, aux_coef=aux, z_coef=zc)
    got = {k: v.cpu().numpy() for k, v in g.items()}
    rows_close(got["dx"], ref["dx"], "dx")                 # every token
    rows_close(got["dW_r"], ref["dW_r"], "dW_r")           # every expert's router row
    if bm == 1:
        assert rel(got["db"], ref["db"]) <= REL
    else:
        assert np.all(got["db"] == 0)
    touched = np.unique(idx_o)
    for e in range(spec.E):
        for name in ("dW_gate", "dW_up", "dW_down"):
            if e in touched and np.any(ref[name][e] != 0):
                rows_close(got[name][e], ref[name][e], (name, e))   # every row of the matrix
            elif e not in touched:
                assert np.all(got[name][e] == 0), (name, e)
    if spec.n_shared:
        for name in ("dWs_gate", "dWs_up", "dWs_down"):
            for s_ in range(spec.n_shared):
                rows_close(got[name][s_], ref[name][s_], (name, s_))


def test_backward_is_deterministic():
    spec, aux, zc = LAYERS[0]
    dev = to_dev(moe_synth.make_layer(spec, seed=3))
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev)
    lay.forward(dev["x"])
    dout = torch.randn((spec.N, spec.d), device="cuda").to(torch.bfloat16)
    g1 = lay.backward(dout, aux, zc)
    g2 = lay.backward(dout, aux, zc)
    torch.cuda.synchronize()
    for k in g1:
        assert torch.equal(g1[k], g2[k]), k


def test_backward_rejects_unsupported_layers():
    spec = moe_synth.LayerSpec("odd", N=8, d=136, d_ff=128, E=4, k=2)
    cfg = moe.cfg_from_spec(spec)
    with pytest.raises(moe.MoeError):
        moe.moe_backward_workspace_size(cfg)


def test_backward_full_size_mixtral_sampled_tokens():
    """At the Mixtral-shaped size (no capacity, aux and z off) a token's dx depends on that token
    alone, so the oracle's backward of a sampled sub-batch gives its exact reference."""
    spec = moe_synth.MIXTRAL
    torch.cuda.empty_cache()
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev)
    lay.forward(dev["x"])
    gen = torch.Generator(device="cuda").manual_seed(7)
    dout = torch.randn((spec.N, spec.d), generator=gen, device="cuda").to(torch.bfloat16)
    g = lay.backward(dout)
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    for name in ("dW_gate", "dW_up", "dW_down", "dW_r"):
        assert torch.isfinite(g[name]).all()
    assert all(g["dW_down"][e].abs().max() > 0 for e in range(spec.E))
    tok = moe_synth.sample_tokens(spec.N, 6, seed=2).numpy()
    host = {n: (None if dev[n] is None else dev[n].cpu()) for n in dev}
    sub = dict(host)
    sub["x"] = host["x"][tok]
    idx_o, _, _, gap_o = oracle.route(sub["x"], host["W_r"], None, spec.k, oracle.BF16)
    assert np.all(gap_o > 1e-6)
    assert np.array_equal(lay.buffers()["idx"].cpu().numpy()[tok], idx_o)
    ref = oracle.backward(sub, spec.k, oracle.BF16, dout.cpu()[tok].double().numpy())
    got = g["dx"].cpu().numpy()[tok]
    for i in range(len(tok)):
        assert rel(got[i], ref["dx"][i]) <= REL, (int(tok[i]), rel(got[i], ref["dx"][i]))
    del dev, lay, g
    torch.cuda.empty_cache()
