"""The benchmark fills roofline.traffic from the committed ncu table only while the table's
source hash matches the kernel source, only for the layer it was captured for, and scaled from
the captured case to a full launch by the table's factor."""
import hashlib
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = ("grouped_gemm_pair.cu", "tc_ptx.cuh")
HEAD = ("| kernel | workload | source hash | dram bytes per captured launch | scale to full launch |\n"
        "|---|---|---|---|---|\n")


def _tree(tmp_path):
    csrc = tmp_path / "sparse_conditional_moe_b300" / "csrc"
    csrc.mkdir(parents=True)
    for f in SRC:
        shutil.copy(os.path.join(ROOT, "sparse_conditional_moe_b300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return csrc


def _hash(csrc):
    h = hashlib.sha256()
    for f in SRC:
        h.update((csrc / f).read_bytes())
    return h.hexdigest()[:16]


def test_traffic_read_only_for_current_source_and_its_layer(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    good = _hash(csrc)
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        HEAD + f"| gateup | layer_a | {good} | 1.5e9 | 8 |\n"
               f"| gateup | layer_c | {'0' * 16} | 2.0e9 | 1 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("gateup", "layer_a") == 1.5e9 * 8
    assert bench.read_traffic("gateup", "layer_b") is None
    assert bench.read_traffic("gateup", "layer_c") is None      # stale hash
    # any change to the kernel source retires the captured number
    (csrc / "grouped_gemm_pair.cu").write_text((csrc / "grouped_gemm_pair.cu").read_text() + "\n")
    assert bench.read_traffic("gateup", "layer_a") is None
