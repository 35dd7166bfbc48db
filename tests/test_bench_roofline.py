"""The benchmark's phase rooflines: a GEMM phase is reported against whichever of its two bounds
binds (tensor: algorithmic flops / the bf16 peak; HBM: touched experts' weights + rows read and
written / HBM bandwidth), with the other bound's fraction beside it."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import moe_synth  # noqa: E402
from sparse_conditional_moe_b300 import accounting  # noqa: E402

PEAKS = {"bf16_tflops": 1808.6, "hbm_gbs": 6425.0}


def _phases(spec, kept_rows, touched, ms, w_b=2.0):
    return bench.phase_rooflines(spec, 2, w_b, kept_rows, touched,
                                 {"gateup": ms, "down": ms / 2, "route": 0.1, "permute": 0.1,
                                  "combine": 0.1}, PEAKS)


def test_prefill_layer_with_many_experts_is_hbm_bound():
    # DeepSeek-V3-shaped prefill: 256 experts x 2*7168*2048 bf16 weights (15 GB) against
    # 3.85 TFLOP: 2.53 ms of HBM vs 2.13 ms of tensor work at the peaks above
    spec = moe_synth.DSV3_PREFILL
    kept = spec.N * spec.k
    ph = _phases(spec, kept, 256, 3.3)
    g = ph["gateup"]
    assert g["bound"] == "hbm" and g["unit"] == "GB/s"
    nbytes = 2.0 * 2 * spec.d * spec.d_ff * 256 + kept * (spec.d + spec.d_ff) * 2
    assert g["bytes"] == pytest.approx(nbytes)
    assert g["achieved"] == pytest.approx(nbytes / 3.3e-3 / 1e9)
    assert g["frac"] == pytest.approx(g["achieved"] / PEAKS["hbm_gbs"])
    flops = accounting.gateup_flops(spec.d, spec.d_ff, kept)
    assert g["tensor_frac"] == pytest.approx(flops / 3.3e-3 / 1e12 / PEAKS["bf16_tflops"])
    assert flops / (PEAKS["bf16_tflops"] * 1e12) < nbytes / (PEAKS["hbm_gbs"] * 1e9)


def test_few_large_experts_are_tensor_bound():
    spec = moe_synth.MIXTRAL      # 8 experts, ~1024 rows each
    kept = spec.N * spec.k
    ph = _phases(spec, kept, 8, 1.2)
    for name in ("gateup", "down"):
        assert ph[name]["bound"] == "tensor" and ph[name]["unit"] == "TFLOP/s"
        assert 0 < ph[name]["hbm_frac"] < ph[name]["frac"]


def test_decode_layer_is_hbm_bound_and_w4_counts_code_bytes():
    spec = moe_synth.DSV3_DECODE
    kept = spec.N * spec.k
    bf = _phases(spec, kept, 220, 1.9)
    w4 = _phases(spec, kept, 220, 1.9, w_b=accounting.W4_BYTES_PER_WEIGHT)
    assert bf["gateup"]["bound"] == "hbm" and w4["gateup"]["bound"] == "hbm"
    assert w4["gateup"]["bytes"] < 0.3 * bf["gateup"]["bytes"]


def test_data_movement_phases_are_hbm_bound_and_zero_times_skipped():
    spec = moe_synth.QWEN3_SKEWED
    ph = bench.phase_rooflines(spec, 2, 2.0, spec.N * spec.k, 120,
                               {"route": 0.05, "permute": 0.0, "combine": 0.02, "gateup": 0.2},
                               PEAKS)
    assert "permute" not in ph
    for name in ("route", "combine"):
        assert ph[name]["bound"] == "hbm" and ph[name]["unit"] == "GB/s"
