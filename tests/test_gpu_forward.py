"""End-to-end GPU parity of moe_forward against the oracle, through the C ABI.

Small layers (the oracle finishes in seconds) are compared on every token: routing bit-exact
(near-ties excluded), counts / offsets / permutation / positions bit-exact, outputs within the
stated tolerance.  The five workload layers are compared at their full sizes in the launch
configuration the benchmark uses: routing and grouping on every token, outputs on the tokens the
oracle computes one by one -- every token of the small-batch layers, and on the prefill-sized
layers a token on every tile of the grouped GEMMs (each expert's first grouped row and the last
row of each of its 256-row chunks) plus a seeded sample.
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import (ExpertCache, check_routing, compare_rows, dtype_code, oracle_tokens,
                      out_f64, run_layer, to_dev)

pytestmark = pytest.mark.gpu

SMALL = [
    moe_synth.TINY,
    moe_synth.PAGE_SELFTEST,
    moe_synth.LayerSpec("bf16_small", N=300, d=256, d_ff=384, E=8, k=2, n_shared=1,
                        d_ff_shared=128),
    moe_synth.LayerSpec("bf16_many_experts", N=200, d=512, d_ff=256, E=64, k=6),
    moe_synth.LayerSpec("bf16_capacity", N=600, d=256, d_ff=128, E=16, k=4,
                        capacity_factor=0.6, zipf_bias=1.2, n_shared=1, d_ff_shared=64),
    moe_synth.LayerSpec("bf16_capacity_no_shared", N=400, d=128, d_ff=256, E=8, k=2,
                        capacity_factor=0.25, zipf_bias=2.0),
    moe_synth.LayerSpec("bf16_k1", N=129, d=192, d_ff=136, E=4, k=1),
    moe_synth.LayerSpec("bf16_dense_k_eq_E", N=70, d=128, d_ff=128, E=4, k=4, n_shared=2,
                        d_ff_shared=64),
    moe_synth.LayerSpec("f32_capacity", N=100, d=64, d_ff=96, E=8, k=3, capacity_factor=0.5,
                        dtype="f32", n_shared=1, d_ff_shared=32),
    moe_synth.LayerSpec("bf16_selection_bias", N=256, d=512, d_ff=256, E=64, k=6, n_shared=1,
                        d_ff_shared=128, zipf_bias=1.2, bias_mode=2, capacity_factor=1.5),
]


def _bias_mode(spec):
    return spec.bias_mode if spec.zipf_bias > 0 else 0


def _by_expert(idx, pos):
    """Each token's grouped rows listed in expert order (independent of slot order)."""
    o = np.argsort(idx, axis=1, kind="stable")
    return np.take_along_axis(idx, o, 1), np.take_along_axis(pos.reshape(idx.shape), o, 1)


def _grouping_checks(spec, bufs, idx_o, differs, probs_o=None):
    cap = oracle.capacity(spec.N, spec.k, spec.E, spec.capacity_factor)
    ref = oracle.permute(idx_o, spec.E, cap)
    if differs.size:          # a near-tie token went to another expert: grouping not unique
        return ref
    for key in ("counts", "offsets", "kept", "kept_offsets"):
        assert np.array_equal(bufs[key].cpu().numpy(), ref[key]), key
    perm, pos = bufs["perm"].cpu().numpy(), bufs["pos"].cpu().numpy()
    idx_g = bufs["idx"].cpu().numpy()
    if np.array_equal(idx_g, idx_o):
        assert np.array_equal(perm, ref["perm"])
        assert np.array_equal(pos, ref["pos"])
    else:
        # Tokens with two selected experts within 1e-6 may list them in either slot order;
        # what is unique is the token order inside each expert segment and the grouped row of
        # every (token, expert) pair.
        assert np.array_equal(perm // spec.k, ref["perm"] // spec.k)
        ge, gp = _by_expert(idx_g, pos)
        oe, op = _by_expert(idx_o, ref["pos"])
        assert np.array_equal(ge, oe) and np.array_equal(gp, op)
    return ref


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_forward_small_layers_every_token(spec):
    L = moe_synth.make_layer(spec, seed=11)
    dev = to_dev(L)
    lay, out = run_layer(spec, dev)
    assert lay.device_error() == 0
    bufs = lay.buffers()
    code = dtype_code(spec)
    ref, ex = oracle.forward_naive(L, spec.k, code, cf=spec.capacity_factor,
                                   bias_mode=_bias_mode(spec))
    scores = ex["probs"] + L["b_r"].numpy()[None, :] if _bias_mode(spec) == 2 else None
    excl, differs = check_routing(bufs["idx"].cpu().numpy(), bufs["w"].cpu().numpy(),
                                  bufs["gap"].cpu().numpy(), ex["idx"], ex["w"], ex["probs"],
                                  ex["gap"], scores_o=scores)
    _grouping_checks(spec, bufs, ex["idx"], differs)
    rows = np.ones(spec.N, bool) if differs.size == 0 else ~excl
    compare_rows(out_f64(out, spec), out_f64(ref, spec), spec, rows=rows)
    # fully dropped tokens without shared experts are exactly zero
    if spec.capacity_factor > 0 and spec.n_shared == 0:
        dropped = ex["keep"].sum(1) == 0
        assert dropped.any()
        assert torch.all(out[torch.from_numpy(dropped).cuda()] == 0)


def test_forward_is_deterministic_and_repeatable():
    spec = SMALL[4]
    dev = to_dev(moe_synth.make_layer(spec, seed=2))
    lay, out1 = run_layer(spec, dev)
    out2 = lay.forward(dev["x"]).clone()
    out3 = lay.forward(dev["x"]).clone()
    assert torch.equal(out1, out2) and torch.equal(out2, out3)


@pytest.mark.parametrize("spec", [s for s in SMALL if s.dtype == "bf16"], ids=lambda s: s.name)
def test_forward_grouped_rows_match_the_step_path(spec):
    """moe_forward's grouped outputs equal those of the step path fed with x_perm built here from
    x and row_token (torch indexing): the same kernels in the same order, so bit-identical."""
    dev = to_dev(moe_synth.make_layer(spec, seed=5))
    lay, _ = run_layer(spec, dev)
    b = lay.buffers()
    cfg = moe.cfg_from_spec(spec)
    R = moe.moe_grouped_rows(cfg)
    M = int(b["kept_offsets"][spec.E].item())
    x_perm = torch.zeros((max(R, 1), spec.d), dtype=torch.bfloat16, device="cuda")
    x_perm[:M] = dev["x"][b["row_token"][:M].long()]
    y = torch.full((max(R, 1), spec.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn(cfg, x_perm, b["kept"], b["kept_offsets"], b["row_weight"],
                        dev["W_gate"], dev["W_up"], dev["W_down"], y, lay.ws)
    torch.cuda.synchronize()
    assert M > 0 and torch.equal(y[:M], b["y_perm"][:M])


def test_forward_empty_batch():
    spec = moe_synth.LayerSpec("empty", N=0, d=128, d_ff=128, E=8, k=2, n_shared=1,
                               d_ff_shared=128)
    dev = to_dev(moe_synth.make_layer(spec.with_(N=4), seed=0))
    dev["x"] = dev["x"][:0]
    lay, out = run_layer(spec, dev)
    assert out.shape == (0, 128) and lay.device_error() == 0


def test_stats_match_oracle():
    spec = SMALL[4]
    L = moe_synth.make_layer(spec, seed=4)
    lay, out = run_layer(spec, to_dev(L))
    st = lay.stats()
    ref, ex = oracle.forward_naive(L, spec.k, dtype_code(spec), cf=spec.capacity_factor)
    so = oracle.stats(ex["idx"], ex["probs"], ex["keep"], ex["gap"])
    np.testing.assert_allclose(st["f"], so["f"], rtol=0, atol=1e-7)
    np.testing.assert_allclose(st["P"], so["P"], rtol=1e-5, atol=1e-7)
    assert abs(st["aux"] - so["aux"]) <= 1e-5 * max(1.0, so["aux"])
    assert st["dropped"] == so["dropped"] and st["fully_dropped"] == so["fully_dropped"]
    assert st["near_tie"] == so["near_tie"] and st["device_error"] == 0
    assert st["kept_rows"] == int(ex["keep"].sum())


# ------------------------------------------------------------------ full-size workloads

FULL = [moe_synth.TINY, moe_synth.MIXTRAL, moe_synth.DSV3_PREFILL, moe_synth.DSV3_DECODE,
        moe_synth.QWEN3_SKEWED]
CHUNK = 256   # token rows per tile of the CTA-pair grouped GEMMs


def chunk_cover_tokens(spec, idx_o, cap):
    """Tokens whose grouped rows cover every tile of the grouped GEMMs: for every expert the
    first grouped row, and the last row of each of its chunks (a group of n kept rows is cut into
    ceil(n / 256) chunks split evenly, the MMA's N rounded up to 16: the last row sits next to
    the chunk's padding).  Returns sorted token indices."""
    ref = oracle.permute(idx_o, spec.E, cap)
    pos = ref["pos"].reshape(-1)
    kept, koff = ref["kept"], ref["kept_offsets"]
    row_slot = np.full(int(koff[-1]), -1, np.int64)
    live = np.nonzero(pos >= 0)[0]
    row_slot[pos[live]] = live
    rows = []
    for e in range(spec.E):
        n = int(kept[e])
        if n == 0:
            continue
        base = int(koff[e])
        nch = -(-n // CHUNK)
        b, rem = divmod(n, nch)
        start = 0
        rows.append(base)
        for c in range(nch):
            rc = b + (1 if c < rem else 0)
            rows.append(base + start + rc - 1)
            start += rc
    slots = row_slot[np.array(rows, np.int64)]
    assert np.all(slots >= 0)
    return np.unique(slots // spec.k)


@pytest.mark.parametrize("spec", FULL, ids=lambda s: s.name)
def test_forward_full_size_workloads(spec):
    torch.cuda.empty_cache()
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    lay, out = run_layer(spec, dev)
    assert lay.device_error() == 0
    bufs = lay.buffers()
    x_host = dev["x"].cpu()
    b_host = None if dev["b_r"] is None else dev["b_r"].cpu()
    code = dtype_code(spec)
    idx_o, w_o, probs_o, gap_o = oracle.route(x_host, dev["W_r"].cpu(), b_host, spec.k, code)
    excl, differs = check_routing(bufs["idx"].cpu().numpy(), bufs["w"].cpu().numpy(),
                                  bufs["gap"].cpu().numpy(), idx_o, w_o, probs_o, gap_o)
    _grouping_checks(spec, bufs, idx_o, differs)
    cap = oracle.capacity(spec.N, spec.k, spec.E, spec.capacity_factor)
    keep_o = oracle.keep_naive(idx_o, spec.E, cap)
    if spec.capacity_factor > 0:
        assert keep_o.min() == 0       # the skewed layer really overflows some experts
    if spec.N <= 64:                   # the tiny and decode layers: every token
        tok = np.arange(spec.N)
    else:                              # a token on every tile of the grouped GEMMs + a sample
        tok = np.union1d(chunk_cover_tokens(spec, idx_o, cap),
                         moe_synth.sample_tokens(spec.N, 12, seed=1).numpy())
    tok = tok[~excl[tok]] if differs.size else tok
    if spec.capacity_factor > 0:       # include tokens that lost assignments
        lost = np.nonzero(keep_o.sum(1) < spec.k)[0]
        tok = np.unique(np.concatenate([tok, lost[:: max(1, lost.size // 6)][:6]]))
    cache = ExpertCache(dev)
    ref = oracle_tokens(spec, x_host, tok, idx_o, w_o, keep_o, cache)
    got = out_f64(out[torch.from_numpy(tok).cuda()], spec)
    compare_rows(got, ref, spec, what=spec.name)
    del dev, lay, out
    torch.cuda.empty_cache()
