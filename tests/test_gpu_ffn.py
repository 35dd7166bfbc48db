"""GPU parity of moe_grouped_ffn (grouped gate/up SwiGLU GEMM + grouped down GEMM with the
routing weight applied) through the C ABI.  Row r of expert e must equal
row_weight[r] * Expert_e(x_perm[r]) as the oracle computes it for one token and one expert.
Group sizes span several 128-row tiles and ragged tails (1, 127, 128, 129, 300 rows), empty
experts, d and d_ff that are not multiples of the 64-wide k-blocks or the output tiles."""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import ExpertCache, compare_rows, dtype_code, out_f64

pytestmark = pytest.mark.gpu


def _grouped(spec, rows_per_expert, seed=0, check_rows=None):
    E = spec.E
    L = moe_synth.make_layer(spec.with_(N=1), seed=seed)
    R = int(sum(rows_per_expert))
    g = torch.Generator().manual_seed(seed + 1)
    act = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    x_perm = torch.randn((max(R, 1), spec.d), generator=g).to(act)
    row_w = torch.rand((max(R, 1),), generator=g)
    kept = torch.tensor(rows_per_expert, dtype=torch.int32)
    kept_off = torch.zeros(E + 1, dtype=torch.int32)
    kept_off[1:] = torch.cumsum(kept, 0)
    # a config whose grouped-row capacity covers R rows
    cfg = moe.make_cfg(N=max(R, 1), d=spec.d, d_ff=spec.d_ff, E=E, k=1,
                       act_dtype=moe.MOE_BF16 if spec.dtype == "bf16" else moe.MOE_F32)
    ws = moe.workspace(cfg)
    dev = {n: L[n].cuda() for n in ("W_gate", "W_up", "W_down")}
    y = torch.empty((max(R, 1), spec.d), dtype=act, device="cuda")
    moe.moe_grouped_ffn(cfg, x_perm.cuda(), kept.cuda(), kept_off.cuda(), row_w.cuda(),
                        dev["W_gate"], dev["W_up"], dev["W_down"], y, ws)
    assert moe.moe_device_error(ws) == 0
    # oracle: one expert, one token, weight row_w[r]
    cache = ExpertCache(dev)
    code = dtype_code(spec)
    rows = range(R) if check_rows is None else check_rows
    ref = np.zeros((len(rows), spec.d))
    for i, r in enumerate(rows):
        e = int(np.searchsorted(kept_off.numpy(), r, side="right") - 1)
        o = oracle.moe_token(x_perm[r], np.array([row_w[r]], np.float32), np.array([1]),
                             [cache.routed(e)], [], code, 1 if code == oracle.BF16 else 0)
        ref[i] = out_f64(o, spec)
    return out_f64(y[torch.as_tensor(list(rows), dtype=torch.long)], spec), ref


@pytest.mark.parametrize("d,F,rows", [
    (256, 384, [1, 127, 128, 129, 300, 0]),       # several m-tiles, ragged, empty expert
    (520, 200, [5, 0, 131, 64]),                    # ragged k-block, ragged n-tiles
    (128, 128, [128]),                              # exactly one tile
    (1024, 1024, [256, 257, 3]),
])
def test_grouped_ffn_bf16(d, F, rows):
    _check_grouped_ffn_bf16(d, F, rows)


def test_grouped_ffn_more_tiles_than_pairs():
    """More tiles than CTA pairs in both GEMMs (120 gate/up and 160 down tiles of 130-row chunks
    over 74 pairs), so every pair runs several tiles: both TMEM accumulators, their full/empty
    phases and the rings' phases across tiles.  Checked rows: each chunk's first and last row
    and a seeded sample."""
    spec = moe_synth.LayerSpec("g", N=1, d=2048, d_ff=768, E=10, k=1)
    rows = [260] * 10                       # two chunks of 130 rows (MMA N = 144) per expert
    rng = np.random.default_rng(7)
    check = set()
    for e in range(10):
        base = 260 * e
        check.update((base, base + 129, base + 130, base + 259))
    check.update(rng.choice(2600, 24, replace=False).tolist())
    check = sorted(check)
    got, ref = _grouped(spec, rows, seed=3, check_rows=check)
    compare_rows(got, ref, spec, what="grouped ffn, several tiles per pair")


def test_grouped_ffn_decode_variant_many_tiles():
    """The decode-sized variant (at most 64 rows in all, 32-row token slots) with 1024 tiles per
    GEMM: 64 one-row experts, d = 4096, d_ff = 2048 (16 weight tiles per chunk in both GEMMs),
    every row checked."""
    spec = moe_synth.LayerSpec("g", N=1, d=4096, d_ff=2048, E=64, k=1)
    got, ref = _grouped(spec, [1] * 64, seed=5)
    compare_rows(got, ref, spec, what="grouped ffn, decode variant")


def _chunk_bounds(n, chunk_rows=256):
    """First and last row (within the group) of every chunk of a group of n rows: the group splits
    evenly into ceil(n / chunk_rows) chunks, the first n % chunks one row longer."""
    if n == 0:
        return []
    c = -(-n // chunk_rows)
    base, rem = divmod(n, c)
    out, start = [], 0
    for i in range(c):
        r = base + (1 if i < rem else 0)
        out += [start, start + r - 1]
        start += r
    return out


def test_grouped_ffn_chunk_boundaries():
    """Groups on both sides of the CTA-pair GEMMs' chunk boundaries (256, 512, 768 rows; chunks
    split evenly and rounded up to 16 for the MMA's N), an empty and a one-row group.  Checked
    rows: every chunk's first and last row and a seeded sample."""
    rows = [255, 256, 257, 300, 0, 511, 512, 513, 777, 1, 1100, 258]
    spec = moe_synth.LayerSpec("g", N=1, d=512, d_ff=384, E=len(rows), k=1)
    off = np.concatenate([[0], np.cumsum(rows)])
    check = set()
    for e, n in enumerate(rows):
        check.update(int(off[e] + r) for r in _chunk_bounds(n))
    rng = np.random.default_rng(17)
    check.update(rng.choice(int(off[-1]), 40, replace=False).tolist())
    got, ref = _grouped(spec, rows, seed=19, check_rows=sorted(check))
    compare_rows(got, ref, spec, what="grouped ffn, chunk boundaries")


def _check_grouped_ffn_bf16(d, F, rows):
    spec = moe_synth.LayerSpec("g", N=1, d=d, d_ff=F, E=len(rows), k=1)
    got, ref = _grouped(spec, rows, seed=d + F)
    compare_rows(got, ref, spec, what="grouped ffn")


def test_grouped_ffn_tail_tile_boundaries():
    """Every boundary of the tail handling: a last m-tile of at most 96 rows is computed with the
    operands swapped (N = its rows rounded up to 16, stored transposed through 32-row chunks),
    97..127 rows as a masked 128-row tile; groups below, at and above 16, 32, 96, 128 rows."""
    rows = [1, 15, 16, 17, 31, 32, 33, 95, 96, 97, 127, 128, 129, 144, 160, 223, 224, 225]
    spec = moe_synth.LayerSpec("g", N=1, d=192, d_ff=320, E=len(rows), k=1)
    got, ref = _grouped(spec, rows, seed=11)
    compare_rows(got, ref, spec, what="grouped ffn tail tiles")


@pytest.mark.parametrize("d,F,rows", [(128, 256, [16, 0, 65, 1]), (36, 20, [3, 70])])
def test_grouped_ffn_fp32(d, F, rows):
    spec = moe_synth.LayerSpec("g", N=1, d=d, d_ff=F, E=len(rows), k=1, dtype="f32")
    got, ref = _grouped(spec, rows, seed=d)
    compare_rows(got, ref, spec, what="grouped ffn fp32")


def test_grouped_ffn_long_reduction():
    """K = 7168 (112 k-blocks through the 4-stage ring) on a few rows of two experts."""
    spec = moe_synth.LayerSpec("g", N=1, d=7168, d_ff=256, E=2, k=1)
    got, ref = _grouped(spec, [130, 7], seed=5)
    compare_rows(got, ref, spec, what="grouped ffn K=7168")
