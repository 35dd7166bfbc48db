"""moe_permute_noalloc: the grouping step for callers that cannot give the library a
workspace (their device memory is owned by another allocator, or their interface has no place
for one).  Its per-block tables live in a fixed device array inside the library, shared by all
calls.  These tests call it through the C ABI and require its outputs to be identical to
moe_permute's and to the oracle's grouping (integer and copy outputs: bit-exact) on two
different calls in a row, so whatever the first call left in the shared array cannot leak into
the second."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from sparse_conditional_moe_b300 import moe

pytestmark = pytest.mark.gpu


def _idx(seed, N, k, E, skew):
    rng = np.random.default_rng(seed)
    p = None
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
    return np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(N)]).astype(np.int32)


def _outputs(cfg, N, k, E, d):
    R = moe.moe_grouped_rows(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    return dict(counts=torch.full((E,), -1, **i32), offsets=torch.full((E + 1,), -1, **i32),
                kept=torch.full((E,), -1, **i32), kept_offsets=torch.full((E + 1,), -1, **i32),
                perm=torch.full((N * k,), -1, **i32), pos=torch.full((N * k,), -9, **i32),
                row_token=torch.full((R,), -1, **i32),
                row_weight=torch.full((R,), -1.0, dtype=torch.float32, device="cuda"),
                x_perm=torch.zeros((R, d), dtype=torch.bfloat16, device="cuda"))


def _both(N, k, E, d, cf, skew, seed):
    cfg = moe.make_cfg(N=N, d=d, d_ff=64, E=E, k=k, capacity_factor=cf)
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((N, d), generator=g).to(torch.bfloat16).cuda()
    w = torch.rand((N, k), generator=g).cuda()
    idx = torch.from_numpy(_idx(seed, N, k, E, skew)).cuda()
    ref = _outputs(cfg, N, k, E, d)
    ws = moe.workspace(cfg)
    moe.moe_permute(cfg, idx, w, x, ref["counts"], ref["offsets"], ref["kept"],
                    ref["kept_offsets"], ref["perm"], ref["pos"], ref["row_token"],
                    ref["row_weight"], ref["x_perm"], ws)
    got = _outputs(cfg, N, k, E, d)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_permute_noalloc(cfg, idx, w, x, got["counts"], got["offsets"], got["kept"],
                            got["kept_offsets"], got["perm"], got["pos"], got["row_token"],
                            got["row_weight"], got["x_perm"], err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0 and moe.moe_device_error(ws) == 0
    _oracle_check(N, k, E, cf, idx.cpu().numpy(), w.cpu().numpy(), x.cpu(), got)
    return ref, got


def _oracle_check(N, k, E, cf, idx, w, x, got):
    """The oracle's grouping (counting sort, keep the first C of each expert in slot order) and
    the rows it implies: row r holds slot f, token f // k, weight w[f], activations x[f // k]."""
    ref = oracle.permute(idx, E, oracle.capacity(N, k, E, cf))
    for key in ("counts", "offsets", "kept", "kept_offsets", "perm", "pos"):
        assert np.array_equal(got[key].cpu().numpy(), ref[key]), key
    M = int(ref["kept_offsets"][-1])
    pos = ref["pos"].reshape(-1)
    live = np.nonzero(pos >= 0)[0]
    row_slot = np.empty(M, np.int64)
    row_slot[pos[live]] = live
    assert np.array_equal(got["row_token"][:M].cpu().numpy(), row_slot // k)
    assert np.array_equal(got["row_weight"][:M].cpu().numpy(), w.reshape(-1)[row_slot])
    assert torch.equal(got["x_perm"][:M].cpu(), x[torch.from_numpy(row_slot // k)])


def test_noalloc_matches_moe_permute_on_two_calls_in_a_row():
    # first call: several blocks, skewed routing with capacity drops
    ref1, got1 = _both(N=3001, k=4, E=64, d=256, cf=1.1, skew=True, seed=1)
    # second call right after, other sizes: leftovers from the first must not matter
    ref2, got2 = _both(N=500, k=8, E=128, d=128, cf=0.0, skew=False, seed=2)
    for ref, got in ((ref1, got1), (ref2, got2)):
        for key in ref:
            assert torch.equal(ref[key], got[key]), key
    assert int((ref1["pos"] < 0).sum()) > 0   # the first call really exercised the capacity


def test_noalloc_rejects_sizes_beyond_its_table():
    """ceil(N*k/2048) * E above 131072 entries is refused before anything runs."""
    L = moe.lib()
    cfg = moe.make_cfg(N=600000, d=64, d_ff=64, E=1024, k=1)   # 293 blocks x 1024 experts
    P = ctypes.c_void_p(256)
    rc = L.moe_permute_noalloc(ctypes.byref(cfg), P, P, P, P, P, P, P, P, P, P, P, P, None, None)
    assert rc == 6   # MOE_ERR_WORKSPACE
