"""Pins for the oracle's router (softmax, top-k, renormalisation).

Page: "混合专家 MoE", section "实现：逐 token 与按专家分组", MoE.route in moe.py
(router linear d->E, softmax over E, top-k, renormalise the k weights).
Each check compares against something other than the oracle's own formula:
brute-force enumeration of k-subsets, numpy's matmul/argsort, or a
mathematical identity.
"""
import itertools

import numpy as np
import pytest
import torch

import moe_synth


def _tiny(seed, N=8, d=16, E=6, dtype="f32", bias=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(N, d, generator=g)
    W = torch.randn(E, d, generator=g) * d ** -0.5
    if dtype == "bf16":
        x = x.to(torch.bfloat16)
    return x, W, bias


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("k", [1, 2, 3])
def test_topk_is_best_k_subset_by_enumeration(orc, seed, k):
    x, W, _ = _tiny(seed)
    idx, w, probs, gap = orc.route(x, W, None, k, orc.F32)
    for t in range(x.shape[0]):
        p = probs[t].astype(np.float64)
        best = max(itertools.combinations(range(p.size), k), key=lambda s: sum(p[list(s)]))
        assert sorted(best) == sorted(idx[t].tolist())
        # slot order: descending probability
        assert all(p[idx[t, j]] >= p[idx[t, j + 1]] for j in range(k - 1))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_selection_follows_numpy_logits(orc, dtype):
    """Softmax is monotone: the top-k set is the top-k of x @ W_r^T (numpy, fp64)."""
    x, W, _ = _tiny(11, N=64, d=96, E=32, dtype=dtype)
    code = orc.BF16 if dtype == "bf16" else orc.F32
    idx, w, probs, gap = orc.route(x, W, None, 4, code)
    logits = x.to(torch.float64).numpy() @ W.to(torch.float64).numpy().T
    for t in range(64):
        order = np.argsort(-logits[t], kind="stable")
        if gap[t] >= 1e-6:
            assert sorted(order[:4].tolist()) == sorted(idx[t].tolist())


def test_probabilities_are_a_distribution(orc):
    x, W, _ = _tiny(3, N=32, d=64, E=64)
    _, _, probs, _ = orc.route(x, W, None, 8, orc.F32)
    assert np.all(probs > 0)
    np.testing.assert_allclose(probs.astype(np.float64).sum(1), 1.0, atol=1e-6)


def test_renormalised_weights_equal_softmax_over_selected_logits(orc):
    """Identity: p_j / sum_selected p = exp(l_j) / sum_selected exp(l)."""
    x, W, _ = _tiny(5, N=40, d=48, E=16)
    idx, w, probs, gap = orc.route(x, W, None, 4, orc.F32)
    logits = x.to(torch.float64).numpy() @ W.to(torch.float64).numpy().T
    for t in range(40):
        sel = logits[t, idx[t]]
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()
        np.testing.assert_allclose(w[t], ref, atol=1e-6, rtol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6
        assert len(set(idx[t].tolist())) == 4
        assert np.all((idx[t] >= 0) & (idx[t] < 16))


def test_k_equals_E_gives_dense_mixing(orc):
    """k = E: every expert is used and the renormalised weights are the probabilities."""
    x, W, _ = _tiny(7, N=10, d=12, E=5)
    idx, w, probs, gap = orc.route(x, W, None, 5, orc.F32)
    for t in range(10):
        np.testing.assert_allclose(w[t], probs[t, idx[t]], atol=1e-7)
        assert sorted(idx[t].tolist()) == list(range(5))
    assert np.all(np.isinf(gap))


def test_no_renorm_keeps_raw_probabilities(orc):
    x, W, _ = _tiny(8, N=10, d=12, E=5)
    idx, w, probs, _ = orc.route(x, W, None, 2, orc.F32, renorm=0)
    for t in range(10):
        np.testing.assert_array_equal(w[t], probs[t, idx[t]])


def test_bias_moves_selection_and_weights(orc):
    """A large logit bias on one expert puts it in slot 0 of every token."""
    x, W, _ = _tiny(9, N=20, d=16, E=8)
    b = torch.zeros(8)
    b[5] = 50.0
    idx, w, probs, _ = orc.route(x, W, b, 2, orc.F32)
    assert np.all(idx[:, 0] == 5)
    assert np.all(probs[:, 5] > 0.999)


def test_ties_go_to_lower_index(orc):
    """W_r with identical rows gives identical logits; order is by index."""
    x = torch.randn(4, 8, generator=torch.Generator().manual_seed(1))
    W = torch.randn(1, 8, generator=torch.Generator().manual_seed(2)).repeat(6, 1)
    idx, w, probs, gap = orc.route(x, W, None, 3, orc.F32)
    assert np.all(idx == np.array([0, 1, 2], np.int32))
    assert np.all(gap == 0.0)
    np.testing.assert_allclose(w, 1.0 / 3.0, atol=1e-7)


def test_gap_is_kth_minus_next(orc):
    x, W, _ = _tiny(12, N=16, d=32, E=10)
    idx, w, probs, gap = orc.route(x, W, None, 3, orc.F32)
    for t in range(16):
        s = np.sort(probs[t].astype(np.float64))[::-1]
        assert abs(gap[t] - (s[2] - s[3])) <= 1e-9


def test_zipf_bias_values():
    """ln of a Zipf(1.2) law over 128 ranks: b_0 = ln(1/H), b_127 = ln(128^-1.2 / H)."""
    b = moe_synth.zipf_bias(128, 1.2).double()
    H = sum(r ** -1.2 for r in range(1, 129))
    assert abs(H - 3.6984) < 1e-3
    assert abs(float(b[0]) - np.log(1 / H)) < 1e-6
    assert abs(float(b[127]) - np.log(128 ** -1.2 / H)) < 1e-5
    np.testing.assert_allclose(np.exp(b.numpy()).sum(), 1.0, atol=1e-6)


# ---------------------------------------------------------------- selection-only bias
# Page "混合专家 MoE", section "负载均衡": DeepSeek-V3's balancing adds a per-expert bias to
# the routing score that only decides the top-k and does not change the weights.

def test_selection_bias_picks_by_p_plus_b_weights_stay_unbiased(orc):
    x, W, _ = _tiny(21, N=30, d=24, E=8)
    b = torch.tensor([0.0, 0.3, -0.2, 0.05, 0.0, 0.6, -1.0, 0.1])
    idx, w, probs, gap = orc.route(x, W, b, 3, orc.F32, bias_mode=2)
    idx0, w0, probs0, gap0 = orc.route(x, W, None, 3, orc.F32)
    np.testing.assert_array_equal(probs, probs0)            # probabilities unbiased
    logits = x.to(torch.float64).numpy() @ W.to(torch.float64).numpy().T
    for t in range(30):
        score = probs[t].astype(np.float64) + b.double().numpy()
        best = max(itertools.combinations(range(8), 3), key=lambda s: sum(score[list(s)]))
        assert sorted(best) == sorted(idx[t].tolist())
        assert all(score[idx[t, j]] >= score[idx[t, j + 1]] for j in range(2))
        sel = logits[t, idx[t]]                               # weights: softmax over the
        ref = np.exp(sel - sel.max()) / np.exp(sel - sel.max()).sum()   # selected logits
        np.testing.assert_allclose(w[t], ref, atol=1e-6, rtol=0)
        s = np.sort(score)[::-1]
        assert abs(gap[t] - (s[2] - s[3])) <= 1e-6


def test_selection_bias_zero_equals_no_bias(orc):
    x, W, _ = _tiny(22, N=20, d=16, E=6)
    a = orc.route(x, W, torch.zeros(6), 2, orc.F32, bias_mode=2)
    b = orc.route(x, W, None, 2, orc.F32)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_large_selection_bias_forces_expert_but_not_its_weight(orc):
    x, W, _ = _tiny(23, N=25, d=16, E=8)
    b = torch.zeros(8)
    b[6] = 10.0
    idx, w, probs, _ = orc.route(x, W, b, 2, orc.F32, bias_mode=2)
    assert np.all(idx[:, 0] == 6)
    # the forced expert's weight is its unbiased share, not ~1 as a logit bias would give
    np.testing.assert_allclose(w[:, 0], probs[:, 6] / (probs[:, 6] + probs[np.arange(25), idx[:, 1]]),
                               rtol=1e-6)
    assert w[:, 0].max() < 0.99
