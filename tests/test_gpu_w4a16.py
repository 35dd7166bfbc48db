"""GPU parity of the W4A16 expert path (moe_quantize_w4, moe_grouped_ffn_w4a16,
moe_forward_w4a16) against the oracle, through the C ABI.

Quantisation is compared bit for bit: the oracle quantises the same host bf16 weights itself
(no code or scale comes from the GPU).  Layer outputs use the bf16 tolerance of the other parity
tests (per-token relative L2 <= 2e-2): the oracle takes the dequantised weights q * s exactly in
fp64 with h rounded to bf16; the GPU forms q * s in fp32 and accumulates in fp32.
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import check_routing, compare_rows, to_dev

pytestmark = pytest.mark.gpu

SMALL = [
    moe_synth.LayerSpec("w4_small", N=300, d=256, d_ff=384, E=8, k=2, n_shared=1,
                        d_ff_shared=128, w4a16=True),
    moe_synth.LayerSpec("w4_decode_many_experts", N=48, d=512, d_ff=256, E=64, k=6, n_shared=1,
                        d_ff_shared=256, w4a16=True),
    moe_synth.LayerSpec("w4_capacity_bias", N=600, d=256, d_ff=128, E=16, k=4,
                        capacity_factor=0.6, zipf_bias=1.2, w4a16=True),
    moe_synth.LayerSpec("w4_k1_wide", N=33, d=1152, d_ff=1280, E=4, k=1, w4a16=True),
]


class W4Oracle:
    """The oracle's own W4A16 copies of host bf16 expert matrices, made on first use."""

    def __init__(self, layer_host: dict):
        self.L = layer_host
        self.cache = {}

    def _trip(self, names, e):
        return tuple(oracle.quantize_w4(self.L[n][e]) for n in names)

    def routed(self, e: int):
        if ("r", e) not in self.cache:
            self.cache[("r", e)] = self._trip(("W_gate", "W_up", "W_down"), e)
        return self.cache[("r", e)]

    def shared(self):
        if self.L.get("Ws_gate") is None:
            return []
        S = self.L["Ws_gate"].shape[0]
        for s in range(S):
            if ("s", s) not in self.cache:
                self.cache[("s", s)] = self._trip(("Ws_gate", "Ws_up", "Ws_down"), s)
        return [self.cache[("s", s)] for s in range(S)]


def oracle_w4_tokens(x_host, tokens, idx_o, w_o, keep_o, q: W4Oracle) -> np.ndarray:
    shared = q.shared()
    for t in tokens:
        for e in idx_o[t]:
            q.routed(int(e))

    def one(t):
        experts = [q.routed(int(e)) for e in idx_o[t]]
        o = oracle.moe_token_w4(x_host[t], w_o[t], keep_o[t], experts, shared, 1)
        return oracle.bf16_bits_to_f32(o).astype(np.float64)

    with cf.ThreadPoolExecutor(max(1, min(32, os.cpu_count() or 1))) as ex:
        rows = list(ex.map(one, tokens))
    return np.stack(rows) if rows else np.zeros((0, x_host.shape[1]))


def _bias_mode(spec):
    return spec.bias_mode if spec.zipf_bias > 0 else None


def _gpu_out(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


# ------------------------------------------------------------------ quantiser

def test_quantize_bit_exact_against_oracle():
    gen = torch.Generator().manual_seed(5)
    W = (torch.randn(3, 256, 384, generator=gen) * 0.05).to(torch.bfloat16)
    W[0, 5, :128] = 0                                   # an all-zero group
    W[1, 7, :128] = 0                                   # exact halves: ties go to even
    W[1, 7, :9] = torch.tensor([7.0, 2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 6.5, 1.5])
    W[2, 9, 128:256] *= 1e-37                           # subnormal weights and scale
    q, s = moe.moe_quantize_w4(W.cuda())
    torch.cuda.synchronize()
    qo, so = oracle.quantize_w4(W)
    np.testing.assert_array_equal(q.cpu().numpy(), qo)
    np.testing.assert_array_equal(s.cpu().numpy(), so)


def test_quantize_full_size_expert_bit_exact():
    spec = moe_synth.DSV3_DECODE
    gen = torch.Generator(device="cuda").manual_seed(3)
    W = (torch.randn((2 * spec.d_ff, spec.d), generator=gen, device="cuda") * spec.d ** -0.5)
    W = W.to(torch.bfloat16)
    q, s = moe.moe_quantize_w4(W)
    torch.cuda.synchronize()
    qo, so = oracle.quantize_w4(W.cpu())
    assert np.array_equal(q.cpu().numpy(), qo) and np.array_equal(s.cpu().numpy(), so)


# ------------------------------------------------------------------ whole layer

def _run(spec, L, seed_dev=None):
    dev = to_dev(L)
    w4 = moe.quantize_layer_w4(dev)
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev, w4=w4)
    out = lay.forward(dev["x"]).clone()
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    return dev, w4, lay, out


@pytest.mark.parametrize("spec", SMALL, ids=lambda s: s.name)
def test_w4_forward_small_layers_every_token(spec):
    L = moe_synth.make_layer(spec, seed=13)
    dev, w4, lay, out = _run(spec, L)
    bufs = lay.buffers()
    idx_o, w_o, probs_o, gap_o = oracle.route(L["x"], L["W_r"], L["b_r"], spec.k, oracle.BF16,
                                              bias_mode=_bias_mode(spec))
    excl, differs = check_routing(bufs["idx"].cpu().numpy(), bufs["w"].cpu().numpy(),
                                  bufs["gap"].cpu().numpy(), idx_o, w_o, probs_o, gap_o)
    cap = oracle.capacity(spec.N, spec.k, spec.E, spec.capacity_factor)
    keep_o = oracle.keep_naive(idx_o, spec.E, cap)
    tok = np.arange(spec.N) if differs.size == 0 else np.nonzero(~excl)[0]
    ref = oracle_w4_tokens(L["x"], tok, idx_o, w_o, keep_o, W4Oracle(L))
    compare_rows(_gpu_out(out[torch.from_numpy(tok).cuda()]), ref, spec, what=spec.name)
    if spec.capacity_factor > 0 and spec.n_shared == 0:
        dropped = keep_o.sum(1) == 0
        assert dropped.any()
        assert torch.all(out[torch.from_numpy(dropped).cuda()] == 0)


def test_w4_grouped_ffn_step_rows_against_oracle():
    """The grouped step alone: every grouped row r of expert e is w_r * Expert_e(x_token)."""
    spec = SMALL[1]
    L = moe_synth.make_layer(spec, seed=21)
    dev, w4, lay, out = _run(spec, L)
    b = lay.buffers()
    cfg = moe.cfg_from_spec(spec)
    R = moe.moe_grouped_rows(cfg)
    y = torch.full((R, spec.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn_w4a16(cfg, b["x_perm"], b["kept"], b["kept_offsets"], b["row_weight"],
                              w4, y, lay.ws)
    torch.cuda.synchronize()
    assert torch.equal(y, b["y_perm"])            # the step and the layer run the same kernels
    idx_o, w_o, _, gap_o = oracle.route(L["x"], L["W_r"], None, spec.k, oracle.BF16)
    assert np.array_equal(b["idx"].cpu().numpy(), idx_o)      # this seed has no near-ties
    ref = oracle.permute(idx_o, spec.E)
    q = W4Oracle(L)
    rows = np.arange(0, R, 7)
    want = []
    for r in rows:
        f = int(ref["perm"][r])
        t, j = divmod(f, spec.k)
        e = int(idx_o[t, j])
        o = oracle.moe_token_w4(L["x"][t], np.array([w_o[t, j]], np.float32),
                                np.array([1], np.int32), [q.routed(e)], [], 1)
        want.append(oracle.bf16_bits_to_f32(o).astype(np.float64))
    compare_rows(_gpu_out(y[torch.from_numpy(rows).cuda()]), np.stack(want), spec, what="y_perm")


def test_w4_grouped_ffn_extreme_activation_scales():
    """The kernel stages activations as fp16 with a power-of-two scale per token (bf16 values
    leave fp16's range).  Grouped rows scaled by 2^-50 .. 2^50, a row mixing 2^40 and 1, and a
    zero row, against the oracle row by row through the grouped step (no router involved)."""
    spec = moe_synth.LayerSpec("w4_scales", N=64, d=1024, d_ff=512, E=4, k=1, w4a16=True)
    L = moe_synth.make_layer(spec, seed=31)
    dev = to_dev(L)
    w4 = moe.quantize_layer_w4(dev)
    cfg = moe.cfg_from_spec(spec)
    ws = moe.workspace(cfg)
    counts = np.array([20, 0, 33, 11], np.int32)          # rows per expert, 64 in all
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = moe.moe_grouped_rows(cfg)
    assert R >= 64
    x = L["x"].float().clone()
    exps = [-50, -24, -8, 0, 8, 24, 50]
    for r in range(64):
        x[r] *= 2.0 ** exps[r % len(exps)]
    x[5] = L["x"][5].float()                               # one row spanning 2^40 within itself
    x[5, : spec.d // 2] *= 2.0 ** 40                       # (h ~ 2^80 stays inside bf16)
    x[6] = 0                                               # a zero row gives exactly zero
    x_perm = torch.zeros((R, spec.d), dtype=torch.bfloat16)
    x_perm[:64] = x.to(torch.bfloat16)
    assert torch.equal(x_perm[:64].float(), x)             # the scaled rows are exact in bf16
    row_w = torch.ones(R, dtype=torch.float32)
    y = torch.full((R, spec.d), float("nan"), dtype=torch.bfloat16, device="cuda")
    moe.moe_grouped_ffn_w4a16(cfg, x_perm.cuda(), torch.from_numpy(counts).cuda(),
                              torch.from_numpy(offs).cuda(), row_w.cuda(), w4, y, ws)
    torch.cuda.synchronize()
    assert moe.moe_device_error(ws) == 0
    q = W4Oracle(L)
    want = []
    for r in range(64):
        e = int(np.searchsorted(offs, r, side="right") - 1)
        o = oracle.moe_token_w4(x_perm[r], np.array([1.0], np.float32), np.array([1], np.int32),
                                [q.routed(e)], [], 1)
        want.append(oracle.bf16_bits_to_f32(o).astype(np.float64))
    got = _gpu_out(y[:64])
    assert np.all(np.isfinite(got))
    compare_rows(got, np.stack(want), spec, what="scaled rows")
    assert np.all(got[6] == 0)


def test_w4_forward_empty_batch_and_repeatable():
    spec = SMALL[0]
    L = moe_synth.make_layer(spec, seed=1)
    dev, w4, lay, out1 = _run(spec, L)
    out2 = lay.forward(dev["x"]).clone()
    assert torch.equal(out1, out2)
    empty = spec.with_(N=0)
    lay0 = moe.MoELayer(moe.cfg_from_spec(empty), dev, w4=w4)
    o = lay0.forward(dev["x"][:0])
    torch.cuda.synchronize()
    assert o.shape == (0, spec.d) and lay0.device_error() == 0


def test_w4_forward_full_size_decode_sampled():
    spec = moe_synth.DSV3_DECODE_W4
    torch.cuda.empty_cache()
    dev = moe_synth.make_layer(spec, seed=0, device="cuda")
    w4 = moe.quantize_layer_w4(dev)
    lay = moe.MoELayer(moe.cfg_from_spec(spec), dev, w4=w4)
    out = lay.forward(dev["x"]).clone()
    torch.cuda.synchronize()
    assert lay.device_error() == 0
    b = lay.buffers()
    x_host = dev["x"].cpu()
    idx_o, w_o, probs_o, gap_o = oracle.route(x_host, dev["W_r"].cpu(), None, spec.k, oracle.BF16)
    excl, differs = check_routing(b["idx"].cpu().numpy(), b["w"].cpu().numpy(),
                                  b["gap"].cpu().numpy(), idx_o, w_o, probs_o, gap_o)
    keep_o = oracle.keep_naive(idx_o, spec.E, -1)
    tok = moe_synth.sample_tokens(spec.N, 12, seed=1).numpy()
    tok = tok[~excl[tok]]

    class HostView:                                   # host copies of just the experts used
        def __init__(self):
            self.cache = {}

        def __getitem__(self, name):
            return _Bank(dev[name])

        def get(self, name):
            return None if dev.get(name) is None else _Bank(dev[name])

    class _Bank:
        def __init__(self, t):
            self.t = t
            self.shape = t.shape

        def __getitem__(self, e):
            return self.t[e].cpu()

    q = W4Oracle(HostView())
    ref = oracle_w4_tokens(x_host, tok, idx_o, w_o, keep_o, q)
    compare_rows(_gpu_out(out[torch.from_numpy(tok).cuda()]), ref, spec, what=spec.name)
    # the quantised copies the layer ran on are the oracle's, bit for bit (one used expert)
    e = int(idx_o[tok[0], 0])
    F = spec.d_ff
    qg, sg = w4["W_gate"]
    qo, so = q.routed(e)[0]
    assert np.array_equal(qg[e * F:(e + 1) * F].cpu().numpy(), qo)
    assert np.array_equal(sg[:, e * F:(e + 1) * F].cpu().numpy(), so)
    del dev, w4, lay, out
    torch.cuda.empty_cache()
