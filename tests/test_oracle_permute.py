"""Pins for the oracle's grouping by expert and the capacity limit.

Pages: "混合专家 MoE", section "实现：逐 token 与按专家分组" (forward_grouped:
flatten, stable argsort, bincount, segment starts) and the closing remark that
the counts are a histogram and the segment starts a prefix sum;
"混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践", section 三.1
(static expert capacity, overflow tokens skip the experts).
Checks compare with numpy's stable argsort/bincount, a brute-force comparison
sort, and the per-token "seen so far" reading of the capacity rule.
"""
import numpy as np
import pytest


def _idx(seed, N, k, E, skew=False):
    rng = np.random.default_rng(seed)
    out = np.zeros((N, k), np.int32)
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
    for t in range(N):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return out


@pytest.mark.parametrize("N,k,E", [(1, 1, 1), (7, 2, 5), (50, 4, 16), (64, 8, 64), (333, 3, 7)])
def test_grouping_matches_numpy(orc, N, k, E):
    idx = _idx(N * 31 + E, N, k, E)
    g = orc.permute(idx, E)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(g["counts"], np.bincount(flat, minlength=E))
    np.testing.assert_array_equal(g["offsets"], np.concatenate([[0], np.cumsum(g["counts"])]))
    np.testing.assert_array_equal(g["perm"], np.argsort(flat, kind="stable"))
    assert g["offsets"][-1] == N * k
    np.testing.assert_array_equal(g["kept"], g["counts"])
    # without capacity every slot keeps its place in the sorted order
    inv = np.empty_like(g["perm"])
    inv[g["perm"]] = np.arange(N * k)
    np.testing.assert_array_equal(g["pos"], inv)


def test_grouping_matches_brute_force_sort(orc):
    idx = _idx(3, 20, 3, 6)
    g = orc.permute(idx, 6)
    flat = idx.reshape(-1).tolist()
    ref = sorted(range(len(flat)), key=lambda f: (flat[f], f))
    assert g["perm"].tolist() == ref
    for e in range(6):
        seg = g["perm"][g["offsets"][e]:g["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)          # stable: increasing slot index
        assert np.all(idx.reshape(-1)[seg] == e)


def test_empty_experts_and_empty_batch(orc):
    idx = np.array([[2, 5]], np.int32)
    g = orc.permute(idx, 8)
    assert g["counts"].tolist() == [0, 0, 1, 0, 0, 1, 0, 0]
    assert g["offsets"].tolist() == [0, 0, 0, 1, 1, 1, 2, 2, 2]
    g0 = orc.permute(np.zeros((0, 2), np.int32), 4)
    assert g0["counts"].tolist() == [0] * 4 and g0["perm"].size == 0


def test_out_of_range_index_rejected(orc):
    with pytest.raises(ValueError):
        orc.permute(np.array([[0, 9]], np.int32), 8)


def test_capacity_formula(orc):
    # C = ceil(CF * N * k / E): the skewed 128-expert layer gets exactly 1280
    assert orc.capacity(16384, 8, 128, 1.25) == 1280
    assert orc.capacity(10, 2, 3, 1.0) == 7          # ceil(20/3)
    assert orc.capacity(10, 2, 3, 0.0) == -1


@pytest.mark.parametrize("cap", [0, 1, 3, 10, 10 ** 9])
def test_capacity_keeps_first_C_in_stable_order(orc, cap):
    N, k, E = 200, 4, 16
    idx = _idx(17, N, k, E, skew=True)
    g = orc.permute(idx, E, cap)
    flat = idx.reshape(-1)
    np.testing.assert_array_equal(g["kept"], np.minimum(g["counts"], cap))
    kept_total = int(g["kept"].sum())
    assert kept_total + int((g["pos"] < 0).sum()) == N * k
    # kept rows form a bijection onto [0, sum kept)
    kp = np.sort(g["pos"][g["pos"] >= 0])
    np.testing.assert_array_equal(kp, np.arange(kept_total))
    # the per-token reading of the rule ("fewer than C earlier assignments") agrees
    keep = orc.keep_naive(idx, E, cap)
    np.testing.assert_array_equal(keep.reshape(-1), (g["pos"] >= 0).astype(np.int32))
    # brute force: slot f is kept iff its rank among same-expert slots is < C
    for f in range(N * k):
        rank = int(np.sum(flat[:f] == flat[f]))
        assert (g["pos"][f] >= 0) == (rank < cap)
        if rank < cap:
            assert g["pos"][f] == g["kept_offsets"][flat[f]] + rank


def test_huge_capacity_equals_no_capacity(orc):
    idx = _idx(5, 100, 2, 8, skew=True)
    a = orc.permute(idx, 8, -1)
    b = orc.permute(idx, 8, 10 ** 9)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key])


def test_one_hot_expert_keeps_exactly_C(orc):
    N, k, E = 64, 1, 4
    idx = np.zeros((N, k), np.int32)
    C = orc.capacity(N, k, E, 1.0)
    g = orc.permute(idx, E, C)
    assert C == 16 and g["kept"].tolist() == [16, 0, 0, 0]
    assert np.all(g["pos"][:16] == np.arange(16)) and np.all(g["pos"][16:] == -1)
