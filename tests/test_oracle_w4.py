"""Pins of the oracle's W4A16 weight format and of the layer with W4A16 weights.

The format is the library's reading of "混合专家模型 (MoE)：大规模稀疏条件计算的架构与工程实践",
section 五.1 (INT4 expert weights, 16-bit activations, arithmetic on dequantised values): per
row, each group of 128 consecutive columns has the fp32 scale s = max|w| / 7, stored
group-major ([cols/128, rows]); a code is round-half-even(w / s) clamped to [-8, 7];
two's-complement nibbles, even column in the low nibble; the weight's value is q * s.  The pins fix every part of that from outside the oracle:
exact round trips for weights on the code grid, the packing written out bit by bit in numpy,
the half-to-even rule on exact halves, the error bound s/2 on random weights, and a layer whose
W4 weights hold exactly the values of bf16 weights giving the bf16 oracle's output bit for bit.
"""
import numpy as np
import pytest
import torch

import moe_synth
import oracle

G = oracle.W4_GROUP


def bf16(a) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, np.float32)).to(torch.bfloat16)


def grid_weights(rows, cols, seed, exps=(-6, -3, 0, 2)):
    """Weights q * 2^e with integer q in [-7, 7], every group holding a +-7 (so s = 2^e exactly)."""
    rng = np.random.default_rng(seed)
    q = rng.integers(-7, 8, size=(rows, cols))
    e = rng.choice(exps, size=(rows, cols // G))
    for r in range(rows):
        for g in range(cols // G):
            q[r, g * G + rng.integers(0, G)] = 7 if rng.random() < 0.5 else -7
    W = q * np.ldexp(1.0, np.repeat(e, G, axis=1))
    return q, e, W


def pack_reference(q: np.ndarray) -> np.ndarray:
    """The packing written out: byte b of a row holds column 2b in bits 0-3, 2b+1 in bits 4-7."""
    u = (q & 15).astype(np.uint8)
    return (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)


def test_grid_weights_round_trip_exactly():
    q, e, W = grid_weights(6, 3 * G, seed=1)
    qq, s = oracle.quantize_w4(bf16(W))
    np.testing.assert_array_equal(s, np.ldexp(1.0, e).astype(np.float32).T)
    np.testing.assert_array_equal(qq, pack_reference(q))
    np.testing.assert_array_equal(oracle.dequantize_w4(qq, s, 3 * G), W)


def test_packing_of_known_codes():
    """Codes -8..7 in order along a row: bytes are (c_{2b} & 15) | (c_{2b+1} & 15) << 4."""
    codes = np.tile(np.arange(-8, 8), G // 16)[None, :]           # one row, one group
    s = np.ones((1, 1), np.float32) * 0.25
    q = pack_reference(codes)
    assert q[0, 0] == 0x98 and q[0, 7] == 0x76                     # (-8, -7) and (6, 7)
    np.testing.assert_array_equal(oracle.dequantize_w4(q, s, G)[0], codes[0] * 0.25)


def test_half_to_even_and_max_to_seven():
    row = np.zeros(G)
    row[0] = 7.0                                   # s = 1
    row[1:9] = [2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 6.5, 1.5]
    qq, s = oracle.quantize_w4(bf16(row[None, :]))
    assert s[0, 0] == 1.0
    got = oracle.dequantize_w4(qq, s, G)[0, :9]
    np.testing.assert_array_equal(got, [7, 2, 4, -2, -4, 0, -0.0, 6, 2])


def test_negative_maximum_and_zero_group():
    W = np.zeros((2, 2 * G))
    W[0, :G] = np.linspace(-3.5, 1.0, G)            # max |w| = 3.5 at a negative weight
    qq, s = oracle.quantize_w4(bf16(W))
    assert s[0, 0] == np.float32(3.5) / np.float32(7.0)
    assert s.shape == (2, 2)                                   # [groups, rows]
    assert s[1, 0] == 0 and s[0, 1] == 0 and s[1, 1] == 0      # all-zero groups
    D = oracle.dequantize_w4(qq, s, 2 * G)
    assert D[0, 0] == -7 * s[0, 0]
    np.testing.assert_array_equal(D[0, G:], 0)
    np.testing.assert_array_equal(D[1], 0)


@pytest.mark.parametrize("seed", [0, 1])
def test_random_weights_error_within_half_step(seed):
    rng = np.random.default_rng(seed)
    W = bf16(rng.standard_normal((16, 4 * G)) * 0.02)
    Wd = W.float().numpy().astype(np.float64)
    qq, s = oracle.quantize_w4(W)
    D = oracle.dequantize_w4(qq, s, 4 * G)
    half = np.repeat(s.T.astype(np.float64), G, axis=1) / 2
    assert np.all(np.abs(D - Wd) <= half * (1 + 1e-6))
    # the largest weight of every group is reproduced to within fp32 rounding of 7 * s
    for r in range(16):
        for g in range(4):
            blk = Wd[r, g * G:(g + 1) * G]
            i = int(np.argmax(np.abs(blk)))
            assert abs(D[r, g * G + i]) == 7 * np.float64(s[g, r])


def test_w4_layer_equals_bf16_layer_on_grid_weights():
    """Expert weights on the code grid are exactly representable in both formats, so the token
    output with W4 weights equals the bf16-weight oracle's bit for bit."""
    d, F, k = 2 * G, G, 2
    rng = np.random.default_rng(7)
    mats = []
    for e in range(3):                              # two routed experts + one shared
        trip = []
        for shape in ((F, d), (F, d), (d, F)):
            _, _, W = grid_weights(shape[0], shape[1], seed=100 + 10 * e + len(trip),
                                   exps=(-8, -7, -6))
            trip.append(W)
        mats.append(trip)
    x = bf16(rng.standard_normal(d))
    w_t = np.array([0.7, 0.3], np.float32)
    keep = np.array([1, 1], np.int32)
    ref = oracle.moe_token(x, w_t, keep, [tuple(bf16(m) for m in mats[i]) for i in range(k)],
                           [tuple(bf16(m) for m in mats[2])], oracle.BF16, 1)
    q4 = [tuple(oracle.quantize_w4(bf16(m)) for m in trip) for trip in mats]
    got = oracle.moe_token_w4(x, w_t, keep, q4[:k], q4[2:], 1)
    np.testing.assert_array_equal(got, ref)
    assert np.any(ref != 0)


def test_w4_layer_drops_like_bf16_layer():
    """A dropped slot contributes nothing in the W4 path either."""
    d, F = G, G
    _, _, Wg = grid_weights(F, d, 3)
    _, _, Wu = grid_weights(F, d, 4)
    _, _, Wd = grid_weights(d, F, 5)
    x = bf16(np.random.default_rng(2).standard_normal(d))
    trip = tuple(oracle.quantize_w4(bf16(m)) for m in (Wg, Wu, Wd))
    out = oracle.moe_token_w4(x, np.array([1.0], np.float32), np.array([0], np.int32), [trip], [], 1)
    np.testing.assert_array_equal(out, 0)


def test_quantize_rejects_ragged_columns():
    with pytest.raises(ValueError):
        oracle.quantize_w4(bf16(np.ones((2, 100))))
