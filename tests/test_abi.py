"""The C-ABI library loads, exports every function include/moe.h declares, and validates
arguments on the host (these calls return before touching CUDA, so no GPU is needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from sparse_conditional_moe_b300 import build as moe_build
from sparse_conditional_moe_b300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    moe_build.build()
    return moe.lib()


def header_functions():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_every_declared_function_is_exported(L):
    names = header_functions()
    assert len(names) >= 13
    out = subprocess.check_output(["nm", "-D", "--defined-only", moe.LIB_PATH], text=True)
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert set(names) <= exported, set(names) - exported
    assert set(moe.EXPORTS) == set(names)
    for n in names:
        assert hasattr(L, n)


def test_struct_layouts_match_c(tmp_path):
    prog = tmp_path / "layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moe.h"\n'
                    "int main(){printf(\"%zu %zu %zu %zu %zu %zu\\n\", sizeof(moe_cfg),"
                    " offsetof(moe_cfg, capacity_factor), offsetof(moe_cfg, act_dtype),"
                    " sizeof(moe_buffers), sizeof(moe_stats_summary),"
                    " offsetof(moe_stats_summary, dropped));return 0;}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)], text=True).split()]
    want = [ctypes.sizeof(moe.MoeCfg), moe.MoeCfg.capacity_factor.offset,
            moe.MoeCfg.act_dtype.offset, ctypes.sizeof(moe.MoeBuffers),
            ctypes.sizeof(moe.MoeStatsSummary), moe.MoeStatsSummary.dropped.offset]
    assert got == want


def test_status_strings(L):
    assert moe.status_string(0) == "ok"
    assert "workspace" in moe.status_string(6)


def _cfg(**kw):
    base = dict(N=64, d=128, d_ff=256, E=8, k=2, n_shared=1, d_ff_shared=256,
                act_dtype=moe.MOE_BF16)
    base.update(kw)
    return moe.make_cfg(**base)


def _status(L, cfg):
    n = ctypes.c_size_t(0)
    return L.moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n))


@pytest.mark.parametrize("kw,code", [
    (dict(k=9), 1), (dict(E=0), 1), (dict(k=0), 1), (dict(N=-1), 1), (dict(d=100), 1),
    (dict(d_ff=12), 1), (dict(act_dtype=7), 1), (dict(renorm=2), 1), (dict(n_shared=1, d_ff_shared=0), 1),
    (dict(E=2048, k=2), 2), (dict(k=17, E=64), 2), (dict(bias_mode=3), 1), (dict(n_shared=9), 2),
    (dict(bias_mode=2), 0),
    (dict(), 0), (dict(N=0), 0), (dict(act_dtype=moe.MOE_F32, d=100, d_ff=12, d_ff_shared=12), 0),
])
def test_cfg_validation(L, kw, code):
    assert _status(L, _cfg(**kw)) == code


def test_workspace_size_grows_with_N_and_capacity_shrinks_rows(L):
    small = moe.moe_workspace_size(_cfg(N=64))
    big = moe.moe_workspace_size(_cfg(N=4096))
    assert big > small > 0
    # E*C = 128*1280 exceeds N*k = 131072, so the grouped buffers hold N*k rows ...
    assert moe.moe_grouped_rows(_cfg(N=16384, d=2048, d_ff=768, E=128, k=8, n_shared=0,
                                     capacity_factor=1.25)) == 16384 * 8
    # ... while CF 0.5 (C = 512) bounds them by E*C
    assert moe.moe_grouped_rows(_cfg(N=16384, d=2048, d_ff=768, E=128, k=8, n_shared=0,
                                     capacity_factor=0.5)) == 128 * 512
    assert moe.moe_grouped_rows(_cfg(N=100, k=2, E=8, capacity_factor=100.0)) == 200


def test_calls_reject_bad_workspace_and_pointers_without_launching(L):
    cfg = _cfg()
    need = moe.moe_workspace_size(cfg)
    fake_ws = ctypes.c_void_p(1 << 20)           # never dereferenced: validation fails first
    P = ctypes.c_void_p
    # missing / misaligned / short workspace
    assert L.moe_route(ctypes.byref(cfg), P(256), P(256), None, P(256), P(256), P(256), None,
                       None, need, None) == 6
    assert L.moe_route(ctypes.byref(cfg), P(256), P(256), None, P(256), P(256), P(256), None,
                       P((1 << 20) + 16), need, None) == 6
    assert L.moe_route(ctypes.byref(cfg), P(256), P(256), None, P(256), P(256), P(256), None,
                       fake_ws, need - 1, None) == 6
    # null / misaligned tensors
    assert L.moe_route(ctypes.byref(cfg), None, P(256), None, P(256), P(256), P(256), None,
                       fake_ws, need, None) == 1
    assert L.moe_route(ctypes.byref(cfg), P(264), P(256), None, P(256), P(256), P(256), None,
                       fake_ws, need, None) == 1
    assert L.moe_forward(ctypes.byref(cfg), P(256), P(256), None, P(256), P(256), P(256),
                         None, P(256), P(256), P(256), fake_ws, need, None) == 1   # shared missing
    bias_cfg = _cfg(bias_mode=1)
    need_b = moe.moe_workspace_size(bias_cfg)
    assert L.moe_route(ctypes.byref(bias_cfg), P(256), P(256), None, P(256), P(256), P(256), None,
                       fake_ws, need_b, None) == 1                                   # bias missing
    assert L.moe_grouped_ffn(ctypes.byref(cfg), P(256), P(256), P(256), None, P(256), P(264),
                             P(256), P(256), fake_ws, need, None) == 1                # misaligned W_up


def _w4_layer(ptr=256, bad=None):
    st = moe.MoeW4Layer()
    for n in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down"):
        setattr(st, n, moe.MoeW4(ptr, ptr))
    if bad:
        setattr(st, bad[0], moe.MoeW4(*bad[1]))
    return st


def test_w4a16_calls_validate_without_launching(L):
    P = ctypes.c_void_p
    # quantiser: columns must be a positive multiple of 128; empty input is a no-op
    assert L.moe_quantize_w4(P(256), 4, 100, P(256), P(256), None) == 1
    assert L.moe_quantize_w4(P(256), 4, 0, P(256), P(256), None) == 1
    assert L.moe_quantize_w4(P(256), -1, 128, P(256), P(256), None) == 1
    assert L.moe_quantize_w4(None, 0, 128, None, None, None) == 0
    assert L.moe_quantize_w4(P(256), 4, 128, P(264), P(256), None) == 1          # misaligned q
    cfg = _cfg()
    need = moe.moe_workspace_size(cfg)
    fake_ws = P(1 << 20)
    st = _w4_layer()
    args = (P(256), P(256), None, ctypes.byref(st), P(256), fake_ws, need, None, None)
    # fp32 activations, or dims that are not multiples of 128, are not supported
    f32 = _cfg(act_dtype=moe.MOE_F32)
    assert L.moe_forward_w4a16(ctypes.byref(f32), *args[:5], fake_ws,
                               moe.moe_workspace_size(f32), None, None) == 2
    odd = _cfg(d=136)
    assert L.moe_forward_w4a16(ctypes.byref(odd), *args[:5], fake_ws,
                               moe.moe_workspace_size(odd), None, None) == 2
    odd_ff = _cfg(d_ff=200)
    assert L.moe_forward_w4a16(ctypes.byref(odd_ff), *args[:5], fake_ws,
                               moe.moe_workspace_size(odd_ff), None, None) == 2
    # missing struct, missing / misaligned matrices, short workspace
    assert L.moe_forward_w4a16(ctypes.byref(cfg), P(256), P(256), None, None, P(256), fake_ws,
                               need, None, None) == 1
    bad_q = _w4_layer(bad=("down", (264, 256)))
    assert L.moe_forward_w4a16(ctypes.byref(cfg), P(256), P(256), None, ctypes.byref(bad_q),
                               P(256), fake_ws, need, None, None) == 1
    no_shared = _w4_layer(bad=("shared_up", (None, None)))
    assert L.moe_forward_w4a16(ctypes.byref(cfg), P(256), P(256), None, ctypes.byref(no_shared),
                               P(256), fake_ws, need, None, None) == 1
    assert L.moe_forward_w4a16(ctypes.byref(cfg), *args[:5], fake_ws, need - 1, None, None) == 6
    # the grouped step does not read the shared matrices
    assert L.moe_grouped_ffn_w4a16(ctypes.byref(cfg), P(256), P(256), P(256), None,
                                   ctypes.byref(no_shared), P(256), fake_ws, need - 1, None) == 6
    assert L.moe_grouped_ffn_w4a16(ctypes.byref(f32), P(256), P(256), P(256), None,
                                   ctypes.byref(st), P(256), fake_ws,
                                   moe.moe_workspace_size(f32), None) == 2


def test_w4_struct_layout_matches_c(tmp_path):
    prog = tmp_path / "w4layout.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "moe.h"\n'
                    "int main(){printf(\"%zu %zu %zu %zu %zu\\n\", sizeof(moe_w4), sizeof(moe_w4_layer),"
                    " offsetof(moe_w4_layer, shared_down), sizeof(moe_router_summary),"
                    " offsetof(moe_buffers, lse));return 0;}\n")
    exe = tmp_path / "w4layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)], text=True).split()]
    assert got == [ctypes.sizeof(moe.MoeW4), ctypes.sizeof(moe.MoeW4Layer),
                   moe.MoeW4Layer.shared_down.offset, ctypes.sizeof(moe.MoeRouterSummary),
                   moe.MoeBuffers.lse.offset]


def test_router_stats_validate_without_launching(L):
    P = ctypes.c_void_p
    cfg = _cfg()
    need = moe.moe_workspace_size(cfg)
    fake_ws = P(1 << 20)
    summ = moe.MoeRouterSummary()
    assert L.moe_router_stats(ctypes.byref(cfg), P(256), P(256), P(256), P(256), None, None,
                              fake_ws, need, None) == 1                       # no summary
    assert L.moe_router_stats(ctypes.byref(cfg), P(256), P(256), P(256), P(256), None,
                              ctypes.byref(summ), fake_ws, need - 1, None) == 6
    assert L.moe_router_stats(ctypes.byref(cfg), None, P(256), P(256), P(256), None,
                              ctypes.byref(summ), fake_ws, need, None) == 1   # no lse
    assert L.moe_router_stats(ctypes.byref(cfg), P(256), P(256), P(256), P(258), None,
                              ctypes.byref(summ), fake_ws, need, None) == 1   # misaligned offsets
