"""The benchmark fills roofline.traffic from the committed per-layer ncu table only while the
table's source hash matches the kernel source, and only for the layer it was captured on."""
import hashlib
import os
import shutil
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

SRC = ("grouped_gemm_tc.cu", "tc_ptx.cuh")


def _tree(tmp_path, table_hash):
    csrc = tmp_path / "sparse_conditional_moe_b300" / "csrc"
    csrc.mkdir(parents=True)
    for f in SRC:
        shutil.copy(os.path.join(ROOT, "sparse_conditional_moe_b300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        "| kernel | workload | source hash | dram bytes per launch |\n|---|---|---|---|\n"
        f"| gateup | layer_a | {table_hash} | 1.5e9 |\n")
    return csrc


def _hash(csrc):
    h = hashlib.sha256()
    for f in SRC:
        h.update((csrc / f).read_bytes())
    return h.hexdigest()[:16]


def test_traffic_read_only_for_current_source_and_its_layer(tmp_path, monkeypatch):
    csrc = _tree(tmp_path, "0" * 16)
    good = _hash(csrc)
    (tmp_path / "profiles" / "ncu_traffic.md").write_text(
        "| kernel | workload | source hash | dram bytes per launch |\n|---|---|---|---|\n"
        f"| gateup | layer_a | {good} | 1.5e9 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.read_traffic("gateup", "layer_a") == 1.5e9
    assert bench.read_traffic("gateup", "layer_b") is None
    # any change to the kernel source retires the captured number
    (csrc / "grouped_gemm_tc.cu").write_text((csrc / "grouped_gemm_tc.cu").read_text() + "\n")
    assert bench.read_traffic("gateup", "layer_a") is None

