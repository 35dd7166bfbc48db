"""GPU parity of moe_route (router logits, softmax, top-k, renormalisation) against the oracle,
through the C ABI.  Shapes cover every padded-expert tiling of the router kernel, ragged token
tails, k = 1 and k = E, a router bias, and fp32 / bf16 activations."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import check_routing, dtype_code

pytestmark = pytest.mark.gpu

CASES = [
    # N, d, E, k, dtype, zipf
    (64, 128, 8, 2, "f32", 0.0),
    (1, 64, 8, 1, "bf16", 0.0),
    (33, 256, 16, 4, "bf16", 0.0),
    (130, 512, 64, 6, "bf16", 0.0),
    (300, 2048, 128, 8, "bf16", 1.2),
    (257, 7168, 256, 8, "bf16", 0.0),
    (100, 1024, 1000, 16, "bf16", 0.0),
    (50, 64, 5, 5, "f32", 0.0),
    (77, 4096, 8, 2, "bf16", 0.0),
    (40, 96, 512, 3, "f32", 0.0),
]


def _route(spec, L):
    cfg = moe.cfg_from_spec(spec)
    ws = moe.workspace(cfg)
    N, k, E = spec.N, spec.k, spec.E
    dev = {n: (v.cuda() if v is not None else None) for n, v in L.items()}
    idx = torch.empty((N, k), dtype=torch.int32, device="cuda")
    w = torch.empty((N, k), dtype=torch.float32, device="cuda")
    P = torch.empty((E,), dtype=torch.float32, device="cuda")
    gap = torch.empty((N,), dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dev["x"], dev["W_r"], dev["b_r"], idx, w, P, gap, ws)
    assert moe.moe_device_error(ws) == 0
    return idx.cpu().numpy(), w.cpu().numpy(), P.cpu().double().numpy(), gap.cpu().numpy()


@pytest.mark.parametrize("N,d,E,k,dt,zipf", CASES)
def test_route_matches_oracle(N, d, E, k, dt, zipf):
    spec = moe_synth.LayerSpec("r", N=N, d=d, d_ff=64, E=E, k=k, dtype=dt, zipf_bias=zipf)
    L = moe_synth.make_layer(spec, seed=N + E, x_only=True)
    idx, w, P, gap = _route(spec, L)
    idx_o, w_o, probs_o, gap_o = oracle.route(L["x"], L["W_r"], L["b_r"], k, dtype_code(spec))
    excl, differs = check_routing(idx, w, gap, idx_o, w_o, probs_o, gap_o)
    np.testing.assert_allclose(P, probs_o.astype(np.float64).sum(0), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=2e-6)


def test_route_is_deterministic():
    spec = moe_synth.LayerSpec("r", N=500, d=1024, d_ff=64, E=256, k=8)
    L = moe_synth.make_layer(spec, seed=3, x_only=True)
    a = _route(spec, L)
    b = _route(spec, L)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


def test_route_empty_batch():
    spec = moe_synth.LayerSpec("r", N=0, d=64, d_ff=64, E=8, k=2)
    L = moe_synth.make_layer(spec, seed=0, x_only=True)
    cfg = moe.cfg_from_spec(spec)
    ws = moe.workspace(cfg)
    P = torch.full((8,), 7.0, device="cuda")
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dummy, L["W_r"].cuda(), None, dummy, dummy, P, None, ws)
    assert torch.all(P.cpu() == 0)


@pytest.mark.parametrize("N,d,E,k,dt", [
    (96, 256, 16, 4, "bf16"),      # GEMV router
    (300, 2048, 128, 8, "bf16"),   # tensor-core router
    (257, 7168, 256, 8, "bf16"),
    (64, 128, 64, 6, "f32"),       # fp32 tiled router
])
def test_route_selection_only_bias(N, d, E, k, dt):
    """bias_mode 2 (DeepSeek-V3 balancing bias): top-k chosen on p + b, weights unbiased."""
    spec = moe_synth.LayerSpec("r2", N=N, d=d, d_ff=64, E=E, k=k, dtype=dt, zipf_bias=1.2,
                               bias_mode=2)
    L = moe_synth.make_layer(spec, seed=N + 3 * E, x_only=True)
    L["b_r"] = L["b_r"] * 0.02          # a bias on the scale of the probabilities
    idx, w, P, gap = _route(spec, L)
    idx_o, w_o, probs_o, gap_o = oracle.route(L["x"], L["W_r"], L["b_r"], k, dtype_code(spec),
                                              bias_mode=2)
    check_routing(idx, w, gap, idx_o, w_o, probs_o, gap_o,
                  scores_o=probs_o + L["b_r"].numpy()[None, :])
    np.testing.assert_allclose(P, probs_o.astype(np.float64).sum(0), rtol=1e-5, atol=1e-6)
    # the bias really changed the selection on this layer
    idx_nb = oracle.route(L["x"], L["W_r"], None, k, dtype_code(spec))[0]
    assert np.any(np.sort(idx_nb, 1) != np.sort(idx_o, 1))


# Batches of more than 1024 tokens do not split d; with 192 < E <= 512 the bf16 router then runs
# fused: the ceil(E/64) expert-block CTAs of a 128-token tile form a cluster (sizes 4 to 8 below)
# and finish the tokens from each other's shared memory.  Smaller E (and d-split small batches)
# take the separate top-k kernel, covered above and by the layer tests.
FUSED = [
    # N, d, E, k, zipf, bias_mode
    (1100, 512, 200, 3, 0.0, 1),      # cluster of 4, last expert block 8 wide
    (2049, 1024, 320, 6, 1.2, 1),     # cluster of 5, ragged last token tile, logit bias
    (1500, 7168, 256, 8, 0.0, 1),     # cluster of 4, the DeepSeek-V3-shaped router
    (1025, 256, 512, 16, 0.0, 1),     # cluster of 8, k = 16
    (1300, 2048, 448, 1, 0.0, 1),     # cluster of 7, k = 1
    (1200, 2048, 256, 8, 1.2, 2),     # selection-only bias through the fused finish
]


@pytest.mark.parametrize("N,d,E,k,zipf,bm", FUSED)
def test_fused_router_matches_oracle(N, d, E, k, zipf, bm):
    spec = moe_synth.LayerSpec("rf", N=N, d=d, d_ff=64, E=E, k=k, zipf_bias=zipf, bias_mode=bm)
    L = moe_synth.make_layer(spec, seed=N + E, x_only=True)
    if bm == 2:
        L["b_r"] = L["b_r"] * 0.02
    idx, w, P, gap = _route(spec, L)
    idx_o, w_o, probs_o, gap_o = oracle.route(L["x"], L["W_r"], L["b_r"], k, dtype_code(spec),
                                              bias_mode=bm if L["b_r"] is not None else None)
    scores = probs_o + L["b_r"].numpy()[None, :] if bm == 2 else None
    check_routing(idx, w, gap, idx_o, w_o, probs_o, gap_o, scores_o=scores)
    np.testing.assert_allclose(P, probs_o.astype(np.float64).sum(0), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(w.astype(np.float64).sum(1), 1.0, atol=2e-6)


def test_prepared_router_split_is_never_stale():
    """moe_router_prepare caches the exact split of one W_r in the workspace: routes with that
    pointer reuse it, a route with another W_r splits its own (and retires the cached one), and
    the first W_r is split again afterwards -- every result matches the oracle for the weight
    actually passed."""
    spec = moe_synth.LayerSpec("rp", N=1536, d=1024, d_ff=64, E=128, k=4)
    La = moe_synth.make_layer(spec, seed=5, x_only=True)
    Lb = moe_synth.make_layer(spec, seed=6, x_only=True)
    cfg = moe.cfg_from_spec(spec)
    ws = moe.workspace(cfg)
    x = La["x"].cuda()
    Wa, Wb = La["W_r"].cuda(), Lb["W_r"].cuda()
    N, k, E = spec.N, spec.k, spec.E

    def route(W):
        idx = torch.empty((N, k), dtype=torch.int32, device="cuda")
        w = torch.empty((N, k), dtype=torch.float32, device="cuda")
        P = torch.empty((E,), dtype=torch.float32, device="cuda")
        gap = torch.empty((N,), dtype=torch.float32, device="cuda")
        moe.moe_route(cfg, x, W, None, idx, w, P, gap, ws)
        assert moe.moe_device_error(ws) == 0
        return idx.cpu().numpy(), w.cpu().numpy(), gap.cpu().numpy()

    want = {}
    for name, W in (("a", La["W_r"]), ("b", Lb["W_r"])):
        want[name] = oracle.route(La["x"], W, None, k, dtype_code(spec))
    moe.moe_router_prepare(cfg, Wa, ws)
    for name, W in (("a", Wa), ("a", Wa), ("b", Wb), ("a", Wa)):
        idx, w, gap = route(W)
        idx_o, w_o, probs_o, gap_o = want[name]
        check_routing(idx, w, gap, idx_o, w_o, probs_o, gap_o)


@pytest.mark.parametrize("label,N,d,E,k,dt", [
    ("gemv (E <= 32)", 4096, 4096, 8, 2, "bf16"),
    ("tensor cores, d split (N <= 1024)", 1024, 7168, 256, 8, "bf16"),
    ("tensor cores + top-k kernel", 4096, 2048, 128, 8, "bf16"),
    ("tensor cores, fused", 4096, 7168, 256, 8, "bf16"),
    ("fp32 tiled", 2048, 1024, 128, 8, "f32"),
])
def test_weight_error_per_router_path(label, N, d, E, k, dt):
    """Measured max |w - w_oracle| and max |gap - gap_oracle| of each router path on a large
    batch (printed for the record; held to the stated 2e-6)."""
    spec = moe_synth.LayerSpec("rw", N=N, d=d, d_ff=64, E=E, k=k, dtype=dt)
    L = moe_synth.make_layer(spec, seed=29, x_only=True)
    idx, w, P, gap = _route(spec, L)
    idx_o, w_o, probs_o, gap_o = oracle.route(L["x"], L["W_r"], None, k, dtype_code(spec))
    excl, differs = check_routing(idx, w, gap, idx_o, w_o, probs_o, gap_o)
    same = np.all(idx == idx_o, axis=1) & ~excl
    dw = np.abs(w[same].astype(np.float64) - w_o[same]).max()
    fin = np.isfinite(gap_o)
    dg = np.abs(gap[fin].astype(np.float64) - gap_o[fin]).max()
    print(f"\nrouter weight error [{label}] N={N} d={d} E={E} k={k}: max|dw| = {dw:.3e}, "
          f"max|dgap| = {dg:.3e}, tokens compared {int(same.sum())}")
    assert dw <= 2e-6 and dg <= 2e-6
