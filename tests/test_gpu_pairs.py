"""The CTA-pair (tcgen05 cta_group::2) grouped GEMMs, which are opt-in (MOE_TC_PAIRS=1, read once
per process), run in a child process on layers whose groups are large enough to use them,
including groups with an odd number of 128-row m-tiles (their tail m-tile goes to the single-CTA
kernel) and a shared expert; outputs must match the oracle as in the other parity tests."""
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
for spec in (moe_synth.LayerSpec("pairs_even", N=1024, d=256, d_ff=256, E=4, k=2, n_shared=1,
                                 d_ff_shared=128),
             moe_synth.LayerSpec("pairs_odd_tails", N=1500, d=384, d_ff=136, E=5, k=2)):
    L = moe_synth.make_layer(spec, seed=21)
    lay, out = run_layer(spec, to_dev(L))
    assert lay.device_error() == 0
    ref, ex = oracle.forward_naive(L, spec.k, dtype_code(spec))
    b = lay.buffers()
    check_routing(b["idx"].cpu().numpy(), b["w"].cpu().numpy(), b["gap"].cpu().numpy(),
                  ex["idx"], ex["w"], ex["probs"], ex["gap"])
    compare_rows(out_f64(out, spec), out_f64(ref, spec), spec, what=spec.name)
print("pairs ok")
"""


def test_cta_pair_kernels_match_oracle():
    code = CHILD.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    env = dict(os.environ, MOE_TC_PAIRS="1")
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "pairs ok" in r.stdout, r.stdout[-3000:] + r.stderr[-3000:]
