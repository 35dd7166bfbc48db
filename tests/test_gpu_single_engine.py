"""The single-CTA grouped GEMM engine (grouped_gemm_tc.cu: 128 token rows x 256 weight rows per
tile on one SM, ragged last m-tiles of at most 96 rows computed with swapped operands), selected
with MOE_GROUPED_GEMM=single (read once per process), runs in a child process on layers with
ragged groups and a shared expert; outputs must match the oracle as in the other parity tests.
The default engine (CTA pairs, grouped_gemm_pair.cu) is covered by every other GPU test."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, numpy as np
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import moe_synth, oracle
from gpu_util import check_routing, compare_rows, out_f64, run_layer, to_dev, dtype_code
for spec in (moe_synth.LayerSpec("single_even", N=1024, d=256, d_ff=256, E=4, k=2, n_shared=1,
                                 d_ff_shared=128),
             moe_synth.LayerSpec("single_ragged_tails", N=1500, d=384, d_ff=136, E=5, k=2),
             moe_synth.LayerSpec("single_capacity", N=700, d=192, d_ff=320, E=6, k=3,
                                 capacity_factor=0.8)):
    L = moe_synth.make_layer(spec, seed=21)
    lay, out = run_layer(spec, to_dev(L))
    assert lay.device_error() == 0
    ref, ex = oracle.forward_naive(L, spec.k, dtype_code(spec), cf=spec.capacity_factor)
    b = lay.buffers()
    check_routing(b["idx"].cpu().numpy(), b["w"].cpu().numpy(), b["gap"].cpu().numpy(),
                  ex["idx"], ex["w"], ex["probs"], ex["gap"])
    compare_rows(out_f64(out, spec), out_f64(ref, spec), spec, what=spec.name)
print("single ok")
"""


def test_single_cta_engine_matches_oracle():
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    env = dict(os.environ, MOE_GROUPED_GEMM="single")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "single ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
