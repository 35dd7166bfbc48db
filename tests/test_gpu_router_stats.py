"""GPU parity of the router statistics (moe_router_stats and the log-sum-exp the router writes)
against the oracle, through the C ABI.

Tolerances: the GPU log-sum-exp is m + log(sum exp(l - m)) in fp32 on logits that carry the
router's ~3e-7 rounding, so |lse - lse*| <= 1e-5 + 1e-6 |lse*|; the z-loss, a mean of squares,
within 1e-5 relative; importance, sums of fp32 weights accumulated in fp64 (each weight within
2e-6 of the oracle's), within 2e-6 per assignment; CV^2 within 1e-4 relative (plus 1e-9).
Tokens whose expert set is not numerically unique (near ties) move one assignment each; where a
layer has any, importance is compared with that slack.
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import check_routing, dtype_code, run_layer, to_dev

pytestmark = pytest.mark.gpu

LAYERS = [
    moe_synth.TINY,
    moe_synth.LayerSpec("bf16_many_experts", N=200, d=512, d_ff=256, E=64, k=6),
    moe_synth.LayerSpec("bf16_capacity_bias", N=600, d=256, d_ff=128, E=16, k=4,
                        capacity_factor=0.6, zipf_bias=1.2, n_shared=1, d_ff_shared=64),
    moe_synth.LayerSpec("bf16_selection_bias", N=256, d=512, d_ff=256, E=64, k=6,
                        zipf_bias=1.2, bias_mode=2),
    moe_synth.LayerSpec("f32_wide_router", N=100, d=64, d_ff=96, E=300, k=3, dtype="f32"),
]


def _bias_mode(spec):
    return spec.bias_mode if spec.zipf_bias > 0 else None


def _check(spec, lay, x_host, W_r, b_r):
    b = lay.buffers()
    got = lay.router_stats()
    idx_o, w_o, probs_o, gap_o, lse_o = oracle.route(x_host, W_r, b_r, spec.k, dtype_code(spec),
                                                     bias_mode=_bias_mode(spec), with_lse=True)
    scores = probs_o + b_r.numpy()[None, :] if _bias_mode(spec) == 2 else None
    excl, differs = check_routing(b["idx"].cpu().numpy(), b["w"].cpu().numpy(), None, idx_o,
                                  w_o, probs_o, gap_o, scores_o=scores)
    lse_g = b["lse"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(lse_g - lse_o) <= 1e-5 + 1e-6 * np.abs(lse_o))
    ref = oracle.router_stats(idx_o, w_o, lse_o, spec.E)
    assert abs(got["z_loss"] - ref["z_loss"]) <= 1e-5 * abs(ref["z_loss"])
    slack = 2e-6 * spec.N * spec.k + 2.0 * differs.size
    np.testing.assert_allclose(got["importance"], ref["importance"], rtol=0, atol=slack)
    if differs.size == 0:
        assert abs(got["importance_cv2"] - ref["importance_cv2"]) <= \
            1e-4 * ref["importance_cv2"] + 1e-9
    return got, ref


@pytest.mark.parametrize("spec", LAYERS, ids=lambda s: s.name)
def test_router_stats_small_layers(spec):
    L = moe_synth.make_layer(spec, seed=5)
    lay, out = run_layer(spec, to_dev(L))
    _check(spec, lay, L["x"], L["W_r"], L["b_r"])


@pytest.mark.parametrize("spec", [moe_synth.MIXTRAL, moe_synth.DSV3_PREFILL,
                                  moe_synth.QWEN3_SKEWED], ids=lambda s: s.name)
def test_router_stats_full_size(spec):
    torch.cuda.empty_cache()
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    lay, out = run_layer(spec, dev)
    b_host = None if dev["b_r"] is None else dev["b_r"].cpu()
    got, ref = _check(spec, lay, dev["x"].cpu(), dev["W_r"].cpu(), b_host)
    if spec.zipf_bias > 0:
        assert ref["importance_cv2"] > 1.0     # the skewed router really is unbalanced
    del dev, lay, out
    torch.cuda.empty_cache()


def test_router_stats_standalone_route_and_permute():
    """The step calls: moe_route writes lse to the workspace, moe_permute gives perm/offsets."""
    spec = LAYERS[1]
    L = moe_synth.make_layer(spec, seed=9)
    dev = to_dev(L)
    cfg = moe.cfg_from_spec(spec)
    ws = moe.workspace(cfg)
    N, k, E = spec.N, spec.k, spec.E
    idx = torch.empty((N, k), dtype=torch.int32, device="cuda")
    w = torch.empty((N, k), dtype=torch.float32, device="cuda")
    P_sum = torch.empty(E, dtype=torch.float32, device="cuda")
    moe.moe_route(cfg, dev["x"], dev["W_r"], None, idx, w, P_sum, None, ws)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    kept = torch.empty(E, dtype=torch.int32, device="cuda")
    kept_off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    perm = torch.empty(N * k, dtype=torch.int32, device="cuda")
    pos = torch.empty(N * k, dtype=torch.int32, device="cuda")
    R = moe.moe_grouped_rows(cfg)
    row_token = torch.empty(R, dtype=torch.int32, device="cuda")
    row_weight = torch.empty(R, dtype=torch.float32, device="cuda")
    x_perm = torch.empty((R, spec.d), dtype=torch.bfloat16, device="cuda")
    moe.moe_permute(cfg, idx, w, dev["x"], counts, offsets, kept, kept_off, perm, pos, row_token,
                    row_weight, x_perm, ws)
    lse = moe.moe_forward_buffers(cfg, ws)["lse"]
    got = moe.moe_router_stats(cfg, lse, w, perm, offsets, ws)
    idx_o, w_o, _, _, lse_o = oracle.route(L["x"], L["W_r"], None, k, oracle.BF16, with_lse=True)
    ref = oracle.router_stats(idx_o, w_o, lse_o, E)
    assert abs(got["z_loss"] - ref["z_loss"]) <= 1e-5 * ref["z_loss"]
    np.testing.assert_allclose(got["importance"], ref["importance"], atol=2e-6 * N * k + 2.0)
