"""Pins for the oracle's load-balance statistics.

Page: "混合专家 MoE", section "负载均衡": L_aux = E * sum_i f_i P_i with f_i the
fraction of assignments routed to expert i (bincount / idx.numel()) and P_i
the mean router probability of expert i; minimal when perfectly balanced; the
page's extreme-skew example (all 50 tokens pick experts 0..3 with probability
0.25 each, 16 experts) must exceed the random-router value.
"""
import json
import os

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_page_skew_example_closed_form(orc):
    g = json.load(open(os.path.join(GOLDEN, "page_aux_loss_skew.json")))
    N, E, hot = g["N"], g["E"], g["hot_experts"]
    probs = np.zeros((N, E), np.float32)
    probs[:, hot] = g["prob"]
    idx = np.tile(np.array(hot, np.int32), (N, 1))
    s = orc.stats(idx, probs)
    assert s["aux"] == pytest.approx(g["expected_aux"], abs=1e-12)
    np.testing.assert_allclose(s["f"][hot], 0.25)


def test_all_tokens_on_one_expert_gives_E_times_Pj(orc):
    rng = np.random.default_rng(0)
    N, E, j = 37, 9, 4
    probs = rng.dirichlet(np.ones(E), size=N).astype(np.float32)
    idx = np.full((N, 1), j, np.int32)
    s = orc.stats(idx, probs)
    Pj = probs[:, j].astype(np.float64).mean()
    assert s["aux"] == pytest.approx(E * Pj, rel=1e-12)


def test_uniform_f_gives_one(orc):
    """Each expert gets exactly 1/E of the assignments => L_aux = sum_i P_i = 1."""
    rng = np.random.default_rng(1)
    E, k = 8, 2
    N = 4 * E
    probs = rng.dirichlet(np.ones(E), size=N).astype(np.float32)
    idx = np.stack([np.arange(N) % E, (np.arange(N) + 3) % E], axis=1).astype(np.int32)
    s = orc.stats(idx, probs)
    np.testing.assert_allclose(s["f"], 1.0 / E)
    assert s["aux"] == pytest.approx(probs.astype(np.float64).sum(1).mean(), rel=1e-12)
    assert s["aux"] == pytest.approx(1.0, abs=1e-6)


def test_uniform_P_gives_one(orc):
    rng = np.random.default_rng(2)
    N, E, k = 25, 5, 2
    probs = np.full((N, E), 0.2, np.float32)
    idx = np.stack([rng.choice(E, 2, replace=False) for _ in range(N)]).astype(np.int32)
    s = orc.stats(idx, probs)
    assert s["aux"] == pytest.approx(E * 0.2 * 1.0, abs=1e-6)


def test_random_router_below_skew(orc):
    """The page's comparison: a random router scores lower than the extreme skew (4.0)."""
    import moe_synth
    L = moe_synth.make_layer(moe_synth.PAGE_SELFTEST, seed=0, x_only=True)
    idx, w, probs, gap = orc.route(L["x"], L["W_r"], None, 4, orc.F32)
    s = orc.stats(idx, probs)
    assert 0.8 < s["aux"] < 4.0


def test_counters(orc):
    N, E, k = 4, 3, 2
    idx = np.array([[0, 1], [0, 2], [0, 1], [2, 1]], np.int32)
    probs = np.full((N, E), 1 / 3, np.float32)
    keep = np.array([[1, 1], [1, 0], [0, 0], [1, 1]], np.int32)
    gap = np.array([0.5, 1e-7, 0.0, 2e-6], np.float32)
    s = orc.stats(idx, probs, keep, gap)
    assert (s["dropped"], s["fully_dropped"], s["near_tie"]) == (3, 1, 2)
    np.testing.assert_allclose(s["f"], [3 / 8, 3 / 8, 2 / 8])
