"""Pins of the oracle's router statistics: the z-loss term and the importance CV^2.

The pages keep only the words ("混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践", sections
二.2 Importance Loss and 三.3 Z-Loss; the formulas are lost): the importance loss penalises the
spread of the gate weight the experts receive, the z-loss acts on the raw gate logits before the
top-k.  Readings: z = mean_t (log sum_e exp l_te)^2; Imp_e = sum of the renormalised top-k
weights assigned to e (before any capacity drop); CV^2 = population Var(Imp) / Mean(Imp)^2.
Every expected value below is a closed form.
"""
import math

import numpy as np
import pytest
import torch

import oracle


def _route(x, W_r, b_r=None, k=1, bias_mode=None):
    return oracle.route(torch.as_tensor(np.asarray(x, np.float32)),
                        torch.as_tensor(np.asarray(W_r, np.float32)),
                        None if b_r is None else torch.as_tensor(np.asarray(b_r, np.float32)),
                        k, oracle.F32, bias_mode=bias_mode, with_lse=True)


def test_uniform_logits_give_log_E_squared():
    N, d, E = 12, 16, 8
    x = np.random.default_rng(0).standard_normal((N, d))
    idx, w, p, gap, lse = _route(x, np.zeros((E, d)), k=2)
    np.testing.assert_allclose(lse, math.log(E), rtol=0, atol=1e-15)
    st = oracle.router_stats(idx, w, lse, E)
    assert abs(st["z_loss"] - math.log(E) ** 2) < 1e-14


def test_log_probability_bias_gives_zero_and_selection_bias_does_not_enter():
    E, N, d = 5, 7, 4
    probs = np.array([0.4, 0.25, 0.2, 0.1, 0.05])
    b = np.log(probs)
    x = np.ones((N, d))
    idx, w, p, gap, lse = _route(x, np.zeros((E, d)), b, k=2, bias_mode=1)
    assert np.all(np.abs(lse) < 1e-6)                    # log sum p = log 1 (fp32 bias)
    assert oracle.router_stats(idx, w, lse, E)["z_loss"] < 1e-12
    # the selection-only bias is not part of the logits
    idx2, w2, p2, gap2, lse2 = _route(x, np.zeros((E, d)), b, k=2, bias_mode=2)
    np.testing.assert_allclose(lse2, math.log(E), atol=1e-15)


def test_lse_of_known_logits():
    # d = 1, x = 1: the logits are the weights themselves (2, 0, 0, 0)
    idx, w, p, gap, lse = _route(np.ones((3, 1)), [[2.0], [0.0], [0.0], [0.0]], k=1)
    np.testing.assert_allclose(lse, math.log(math.exp(2.0) + 3.0), rtol=1e-15)
    st = oracle.router_stats(idx, w, lse, 4)
    assert abs(st["z_loss"] - math.log(math.exp(2.0) + 3.0) ** 2) < 1e-12


@pytest.mark.parametrize("E,k", [(8, 2), (16, 1), (6, 3)])
def test_importance_all_on_the_first_k_experts(E, k):
    """Equal logits: every token takes experts 0..k-1 (ties to the lower index) with weight
    1/k, so Imp = (N/k, ..., N/k, 0, ...) and CV^2 = E/k - 1."""
    N, d = 10, 4
    idx, w, p, gap, lse = _route(np.ones((N, d)), np.zeros((E, d)), k=k)
    st = oracle.router_stats(idx, w, lse, E)
    np.testing.assert_allclose(st["importance"][:k], N / k, rtol=1e-7)
    assert np.all(st["importance"][k:] == 0)
    assert abs(st["importance_cv2"] - (E / k - 1)) < 1e-6


def test_importance_uniform_when_every_expert_is_chosen():
    N, d, E = 9, 4, 6
    idx, w, p, gap, lse = _route(np.ones((N, d)), np.zeros((E, d)), k=E)
    st = oracle.router_stats(idx, w, lse, E)
    np.testing.assert_allclose(st["importance"], N / E, rtol=1e-7)
    assert st["importance_cv2"] < 1e-12


def test_importance_uses_renormalised_weights():
    """Logits (ln 3, 0, -20, -20), k = 2: weights (3/4, 1/4), Imp = (3N/4, N/4, 0, 0),
    CV^2 = 1.5 (counting assignments would give 1)."""
    N = 8
    W = [[math.log(3.0)], [0.0], [-20.0], [-20.0]]
    idx, w, p, gap, lse = _route(np.ones((N, 1)), W, k=2)
    st = oracle.router_stats(idx, w, lse, 4)
    np.testing.assert_allclose(st["importance"][:2], [0.75 * N, 0.25 * N], rtol=1e-6)
    assert abs(st["importance_cv2"] - 1.5) < 1e-5


def test_importance_is_sparse_not_dense_probabilities():
    """k = 1, logits (ln 2, 0, 0, 0): Imp = (N, 0, 0, 0), CV^2 = 3 (the dense mean
    probability (0.4, 0.2, 0.2, 0.2) would give 0.12)."""
    idx, w, p, gap, lse = _route(np.ones((5, 1)), [[math.log(2.0)], [0.0], [0.0], [0.0]], k=1)
    st = oracle.router_stats(idx, w, lse, 4)
    assert abs(st["importance_cv2"] - 3.0) < 1e-6


def test_router_stats_reject_bad_index():
    with pytest.raises(ValueError):
        oracle.router_stats(np.array([[4]]), np.array([[1.0]]), np.array([0.0]), 4)
