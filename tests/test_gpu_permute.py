"""GPU parity of moe_permute (histogram, prefix sums, stable scatter, capacity, row gather)
against the oracle's counting sort, through the C ABI.  All outputs are integers or copies, so
every comparison is bit-exact.  The routing fed in is the oracle's own (or a synthetic one).
The grouping runs as one cooperative kernel when its blocks fit on the GPU at once (every case
here); the three-launch form is run on the same cases in a child process (MOE_PERMUTE=unfused)."""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import oracle
from sparse_conditional_moe_b300 import moe

pytestmark = pytest.mark.gpu


def _random_idx(seed, N, k, E, skew=0.0):
    rng = np.random.default_rng(seed)
    p = None
    if skew > 0:
        p = 1.0 / np.arange(1, E + 1) ** skew
        p /= p.sum()
    idx = np.zeros((N, k), np.int32)
    for t in range(N):
        idx[t] = rng.choice(E, size=k, replace=False, p=p)
    return idx


def _permute(N, k, E, idx, cf=0.0, d=64, dtype=moe.MOE_BF16, seed=0):
    cfg = moe.make_cfg(N=N, d=d, d_ff=64, E=E, k=k, capacity_factor=cf, act_dtype=dtype)
    ws = moe.workspace(cfg)
    R = moe.moe_grouped_rows(cfg)
    g = torch.Generator().manual_seed(seed)
    act = torch.bfloat16 if dtype == moe.MOE_BF16 else torch.float32
    x = torch.randn((N, d), generator=g).to(act)
    w = torch.rand((N, k), generator=g)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(counts=torch.empty(E, **i32), offsets=torch.empty(E + 1, **i32),
             kept=torch.empty(E, **i32), kept_offsets=torch.empty(E + 1, **i32),
             perm=torch.empty(max(N * k, 1), **i32), pos=torch.empty(max(N * k, 1), **i32),
             row_token=torch.full((max(R, 1),), -7, **i32),
             row_weight=torch.empty(max(R, 1), dtype=torch.float32, device="cuda"),
             x_perm=torch.empty((max(R, 1), d), dtype=act, device="cuda"))
    xd, wd, idd = x.cuda(), w.cuda(), torch.from_numpy(idx).cuda()
    moe.moe_permute(cfg, idd, wd, xd, o["counts"], o["offsets"], o["kept"], o["kept_offsets"],
                    o["perm"], o["pos"], o["row_token"], o["row_weight"], o["x_perm"], ws)
    err = moe.moe_device_error(ws)
    host = {n: v.cpu() for n, v in o.items()}
    return host, x, w, R, err, cfg


@pytest.mark.parametrize("N,k,E,cf,skew", [
    (1, 1, 1, 0.0, 0.0),
    (50, 4, 16, 0.0, 0.0),
    (64, 2, 8, 0.0, 0.0),
    (3001, 3, 7, 0.0, 0.0),            # several blocks, ragged tail
    (4096, 8, 256, 0.0, 0.0),
    (2500, 16, 1024, 0.0, 0.0),
    (64, 8, 256, 0.0, 0.0),            # many empty experts
    (2000, 8, 128, 1.25, 1.2),         # capacity with a skewed router
    (700, 2, 8, 0.3, 1.0),             # most assignments dropped
    (5, 3, 3, 0.0, 0.0),               # k = E
    (1025, 2, 16, 0.0, 0.0),           # last block of 2 slots: most of its warps get none
    (4101, 2, 64, 1.0, 1.0),           # 4 full blocks and a 10-slot one, with capacity
    (16384, 8, 128, 1.25, 1.2),        # the Qwen-shaped layer's grouping: 64 blocks
    (65536, 8, 256, 0.0, 0.0),         # 256 blocks in one cooperative grid
])
def test_permute_matches_oracle(N, k, E, cf, skew):
    idx = _random_idx(N * 7 + E, N, k, E, skew)
    got, x, w, R, err, cfg = _permute(N, k, E, idx, cf)
    assert err == 0
    cap = oracle.capacity(N, k, E, cf)
    ref = oracle.permute(idx, E, cap)
    A = N * k
    for key in ("counts", "offsets", "kept", "kept_offsets"):
        assert np.array_equal(got[key].numpy(), ref[key]), key
    assert np.array_equal(got["perm"].numpy()[:A], ref["perm"])
    assert np.array_equal(got["pos"].numpy()[:A], ref["pos"])
    M = int(ref["kept_offsets"][-1])
    assert M <= R
    # row r holds slot f with pos[f] = r: its token, its weight, its x row
    flat_w = w.reshape(-1).numpy()
    rt = np.full(M, -1, np.int64)
    rw = np.zeros(M, np.float32)
    for f in range(A):
        if ref["pos"][f] >= 0:
            rt[ref["pos"][f]] = f // k
            rw[ref["pos"][f]] = flat_w[f]
    assert np.array_equal(got["row_token"].numpy()[:M], rt)
    assert np.array_equal(got["row_weight"].numpy()[:M], rw)
    assert torch.equal(got["x_perm"][:M], x[torch.from_numpy(rt)])


def test_permute_fp32_rows_and_empty_batch():
    idx = _random_idx(1, 40, 2, 6)
    got, x, w, R, err, cfg = _permute(40, 2, 6, idx, d=36, dtype=moe.MOE_F32)
    ref = oracle.permute(idx, 6)
    assert np.array_equal(got["perm"].numpy(), ref["perm"])
    rt = torch.from_numpy(ref["perm"] // 2)
    assert torch.equal(got["x_perm"][:80], x[rt])
    got0, *_ = _permute(0, 2, 6, np.zeros((0, 2), np.int32))
    assert got0["counts"].sum() == 0 and got0["offsets"].sum() == 0


def test_out_of_range_index_sets_error_word_without_faulting():
    """The kernels bounds-check every expert index: a bad one is skipped and reported."""
    idx = _random_idx(2, 30, 2, 8)
    idx[3, 1] = 8
    idx[7, 0] = -1
    got, x, w, R, err, cfg = _permute(30, 2, 8, idx)
    assert err & moe.MOE_DEVERR_BOUNDS
    assert got["pos"][3 * 2 + 1] == -1 and got["pos"][7 * 2] == -1
    assert int(got["counts"].sum()) == 58


def test_permute_is_deterministic():
    idx = _random_idx(5, 4096, 8, 256)
    a = _permute(4096, 8, 256, idx)[0]
    b = _permute(4096, 8, 256, idx)[0]
    for key in a:
        assert torch.equal(a[key], b[key]), key


def test_three_launch_form_matches_oracle():
    """The count / scan / scatter kernels the cooperative kernel replaces, on the same cases."""
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, MOE_PERMUTE="unfused")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(here, "test_gpu_permute.py"),
                        "-q", "-x", "-m", "gpu", "-k", "not three_launch"],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
