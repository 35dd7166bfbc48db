"""The FLOP/byte/parameter accounting used by the benchmark, pinned to the page's
exercise ("混合专家 MoE", section 练习, exercise 1: 64 experts, top-8,
3 x 2048 x 1408 parameters per expert, 24 MoE layers -> 13.29B total, 1.66B active)."""
import json
import os

from sparse_conditional_moe_b300 import accounting

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_page_exercise_param_counts():
    g = json.load(open(os.path.join(GOLDEN, "page_exercise_params.json")))
    total, active = accounting.moe_param_counts(g["n_experts"], g["top_k"], g["d"], g["d_ff"],
                                                g["moe_layers"])
    assert round(total / 1e9, 2) == g["expected_total_B_2dp"]
    assert round(active / 1e9, 2) == g["expected_active_B_2dp"]


def test_layer_work_mixtral_shape():
    # N=4096, d=4096, F=14336, E=8, k=2: all 8192 assignments kept, all 8 experts touched
    w = accounting.layer_work(4096, 4096, 14336, 8, 2, 0, 0, 2, 8192, 8)
    assert abs(w.flops - 2.887e12) / 2.887e12 < 1e-3
    assert abs(w.bytes - 2.886e9) / 2.886e9 < 1e-3
    assert w.bound(1815.6e12, 6509.1e9) == "tensor"


def test_layer_work_decode_is_hbm_bound():
    w = accounting.layer_work(64, 7168, 2048, 256, 8, 1, 2048, 2, 512, 222)
    assert w.bound(1815.6e12, 6509.1e9) == "hbm"
    assert abs(w.bytes - (3 * 7168 * 2048 * 2 * 223 + 4 * 7168 * 256 + 2 * 64 * 7168 * 2)) < 1
