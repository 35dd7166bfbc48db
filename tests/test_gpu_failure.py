"""Failure detection without a GPU fault: a device wait that can never be satisfied must give
up after its limit, report MOE_DEVERR_TIMEOUT through the workspace error word, and leave the
context usable (a layer forward pass right after it still matches the oracle).  An expert index
outside [0, E) is covered in test_gpu_permute.py (reported, skipped, no fault)."""
import time

import numpy as np
import pytest
import torch

import moe_synth
import oracle
from sparse_conditional_moe_b300 import moe

from gpu_util import compare_rows, out_f64, run_layer, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    cfg = moe.make_cfg(N=64, d=128, d_ff=128, E=8, k=2)
    ws = moe.workspace(cfg)
    assert moe.moe_device_error(ws) == 0
    t0 = time.perf_counter()
    moe.moe_selftest_wait_timeout(ws, 50_000)          # 50 ms
    code = moe.moe_device_error(ws)                    # synchronises
    dt = time.perf_counter() - t0
    assert code & moe.MOE_DEVERR_TIMEOUT
    assert 0.04 < dt < 5.0
    moe.moe_workspace_init(cfg, ws)                    # the word is sticky until cleared
    assert moe.moe_device_error(ws) == 0


def test_context_usable_after_timeout():
    cfg = moe.make_cfg(N=64, d=128, d_ff=128, E=8, k=2)
    ws = moe.workspace(cfg)
    moe.moe_selftest_wait_timeout(ws, 20_000)
    assert moe.moe_device_error(ws) & moe.MOE_DEVERR_TIMEOUT
    spec = moe_synth.LayerSpec("after_timeout", N=200, d=256, d_ff=256, E=8, k=2)
    L = moe_synth.make_layer(spec, seed=3)
    lay, out = run_layer(spec, to_dev(L))
    assert lay.device_error() == 0
    ref, _ = oracle.forward_naive(L, 2, oracle.BF16)
    compare_rows(out_f64(out, spec), out_f64(ref, spec), spec)


def test_selftest_rejects_bad_arguments():
    cfg = moe.make_cfg(N=64, d=128, d_ff=128, E=8, k=2)
    ws = moe.workspace(cfg)
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(ws, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_selftest_wait_timeout(ws, 3_000_000)
