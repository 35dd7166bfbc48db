"""ctypes binding of libmoe.so: the same entry points as include/moe.h, taking torch tensors.

Argument marshalling only: every step of the layer runs in the library's CUDA kernels.
There is no fallback: if libmoe.so is missing or no GPU is present, calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
# MOE_LIB: load another build of the same library (e.g. one compiled with other tile sizes)
LIB_PATH = os.environ.get("MOE_LIB") or os.path.join(_PKG, "libmoe.so")

MOE_F32, MOE_BF16 = 0, 1
MOE_DEVERR_BOUNDS, MOE_DEVERR_TIMEOUT = 1, 2
MOE_TRACE_EVENTS = 7
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_DEVICE_BOUNDS", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_WORKSPACE"}

# Every function the header declares (checked against the library's exports by the tests).
EXPORTS = ("moe_workspace_size", "moe_workspace_init", "moe_grouped_rows", "moe_route",
           "moe_permute", "moe_permute_noalloc", "moe_grouped_ffn", "moe_combine", "moe_forward",
           "moe_forward_traced", "moe_forward_buffers", "moe_stats", "moe_device_error",
           "moe_selftest_wait_timeout", "moe_status_string", "moe_status_str", "moe_quantize_w4",
           "moe_grouped_ffn_w4a16", "moe_forward_w4a16", "moe_router_stats",
           "moe_selftest_gemm", "moe_backward_workspace_size", "moe_backward",
           "moe_router_prepare")
MOE_W4_GROUP = 128


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}")
        self.status = status


class MoeCfg(ctypes.Structure):
    _fields_ = [("N", ctypes.c_int64), ("d", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("E", ctypes.c_int32), ("k", ctypes.c_int32), ("n_shared", ctypes.c_int32),
                ("d_ff_shared", ctypes.c_int32), ("capacity_factor", ctypes.c_double),
                ("renorm", ctypes.c_int32), ("bias_mode", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32)]


class MoeBuffers(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("idx", "w", "gap", "P_sum", "counts", "offsets", "kept", "kept_offsets", "perm",
                 "pos", "row_token", "row_weight", "x_perm", "y_perm", "lse")]


class MoeRouterSummary(ctypes.Structure):
    _fields_ = [("z_loss", ctypes.c_double), ("importance_cv2", ctypes.c_double),
                ("importance_mean", ctypes.c_double)]


class MoeStatsSummary(ctypes.Structure):
    _fields_ = [("aux", ctypes.c_float), ("device_error", ctypes.c_int32),
                ("dropped", ctypes.c_int64), ("fully_dropped", ctypes.c_int64),
                ("near_tie", ctypes.c_int64), ("touched_experts", ctypes.c_int64),
                ("kept_rows", ctypes.c_int64)]


class MoeW4(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p)]


class MoeW4Layer(ctypes.Structure):
    _fields_ = [(n, MoeW4) for n in ("gate", "up", "down", "shared_gate", "shared_up", "shared_down")]


_lib = None


def lib():
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m sparse_conditional_moe_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
        C = ctypes.POINTER(MoeCfg)
        sig = {
            "moe_workspace_size": [C, ctypes.POINTER(SZ)],
            "moe_workspace_init": [C, P, SZ, P],
            "moe_router_prepare": [C, P, P, SZ, P],
            "moe_route": [C, P, P, P, P, P, P, P, P, SZ, P],
            "moe_permute": [C, P, P, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_permute_noalloc": [C, P, P, P, P, P, P, P, P, P, P, P, P, P, P],
            "moe_grouped_ffn": [C, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_combine": [C, P, P, P, P, P, P, P, P, SZ, P],
            "moe_forward": [C, P, P, P, P, P, P, P, P, P, P, P, SZ, P],
            "moe_forward_traced": [C, P, P, P, P, P, P, P, P, P, P, P, SZ, P, P],
            "moe_forward_buffers": [C, P, SZ, ctypes.POINTER(MoeBuffers)],
            "moe_stats": [C, P, P, P, P, P, P, P, ctypes.POINTER(MoeStatsSummary), P, SZ, P],
            "moe_device_error": [P, SZ, ctypes.POINTER(ctypes.c_int32), P],
            "moe_selftest_wait_timeout": [P, SZ, ctypes.c_uint32, P],
            "moe_quantize_w4": [P, I64, ctypes.c_int32, P, P, P],
            "moe_grouped_ffn_w4a16": [C, P, P, P, P, ctypes.POINTER(MoeW4Layer), P, P, SZ, P],
            "moe_forward_w4a16": [C, P, P, P, ctypes.POINTER(MoeW4Layer), P, P, SZ, P, P],
            "moe_router_stats": [C, P, P, P, P, P, ctypes.POINTER(MoeRouterSummary), P, SZ, P],
            "moe_selftest_gemm": [ctypes.c_int32] * 5 + [P, P, P, P, SZ, P],
            "moe_backward_workspace_size": [C, ctypes.POINTER(SZ)],
            "moe_backward": [C] + [P] * 10 + [ctypes.c_double, ctypes.c_double] + [P] * 9
                            + [P, SZ, P, SZ, P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.moe_grouped_rows.argtypes = [C]
        L.moe_grouped_rows.restype = I64
        L.moe_status_string.argtypes = [ctypes.c_int]
        L.moe_status_string.restype = ctypes.c_char_p
        _lib = L
    return _lib


def _check(rc: int, where: str):
    if rc != 0:
        raise MoeError(rc, where)


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _s(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_cfg(N: int, d: int, d_ff: int, E: int, k: int, n_shared: int = 0, d_ff_shared: int = 0,
             capacity_factor: float = 0.0, renorm: int = 1, bias_mode: int = 0,
             act_dtype: int = MOE_BF16) -> MoeCfg:
    return MoeCfg(N, d, d_ff, E, k, n_shared, d_ff_shared if n_shared else 0, capacity_factor,
                  renorm, bias_mode, act_dtype)


def cfg_from_spec(spec, N: Optional[int] = None) -> MoeCfg:
    """MoeCfg of a moe_synth.LayerSpec (its bias_mode when the layer has a router bias)."""
    return make_cfg(spec.N if N is None else N, spec.d, spec.d_ff, spec.E, spec.k, spec.n_shared,
                    spec.d_ff_shared, spec.capacity_factor, spec.renorm,
                    getattr(spec, "bias_mode", 1) if getattr(spec, "zipf_bias", 0) > 0 else 0,
                    MOE_BF16 if spec.dtype == "bf16" else MOE_F32)


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


# ------------------------------------------------------------------ workspace

def moe_workspace_size(cfg: MoeCfg) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_workspace_size(ctypes.byref(cfg), ctypes.byref(n)), "moe_workspace_size")
    return n.value


def moe_grouped_rows(cfg: MoeCfg) -> int:
    r = lib().moe_grouped_rows(ctypes.byref(cfg))
    if r < 0:
        raise MoeError(1, "moe_grouped_rows")
    return r


def moe_router_prepare(cfg: MoeCfg, W_r: torch.Tensor, ws: torch.Tensor, stream=None):
    """Write the router weight's exact bf16 split into the workspace once (see include/moe.h);
    later calls with this workspace and this W_r tensor skip the split.  Call again after
    changing W_r in place."""
    _check(lib().moe_router_prepare(ctypes.byref(cfg), _p(W_r), _p(ws), ws.numel(), _s(stream)),
           "moe_router_prepare")


def moe_workspace_init(cfg: MoeCfg, ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(ctypes.byref(cfg), _p(ws), ws.numel(), _s(stream)),
           "moe_workspace_init")


def workspace(cfg: MoeCfg, device="cuda", stream=None) -> torch.Tensor:
    """Allocate (torch) and initialise a workspace of moe_workspace_size bytes."""
    ws = torch.empty(moe_workspace_size(cfg), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("torch returned a workspace that is not 256-byte aligned")
    moe_workspace_init(cfg, ws, stream)
    return ws


# ------------------------------------------------------------------ steps

def moe_route(cfg, x, W_r, b_r, idx, w, P_sum, gap, ws, stream=None):
    _check(lib().moe_route(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(idx), _p(w), _p(P_sum),
                           _p(gap), _p(ws), ws.numel(), _s(stream)), "moe_route")


def moe_permute(cfg, idx, w, x, counts, offsets, kept, kept_offsets, perm, pos, row_token,
                row_weight, x_perm, ws, stream=None):
    _check(lib().moe_permute(ctypes.byref(cfg), _p(idx), _p(w), _p(x), _p(counts), _p(offsets),
                             _p(kept), _p(kept_offsets), _p(perm), _p(pos), _p(row_token),
                             _p(row_weight), _p(x_perm), _p(ws), ws.numel(), _s(stream)),
           "moe_permute")


def moe_permute_noalloc(cfg, idx, w, x, counts, offsets, kept, kept_offsets, perm, pos,
                        row_token, row_weight, x_perm, err=None, stream=None):
    """moe_permute for callers that cannot provide a workspace: the library keeps the per-block
    tables in a fixed device array of its own (see include/moe.h for its size limit and the
    rule that overlapping calls race on it)."""
    _check(lib().moe_permute_noalloc(ctypes.byref(cfg), _p(idx), _p(w), _p(x), _p(counts),
                                     _p(offsets), _p(kept), _p(kept_offsets), _p(perm), _p(pos),
                                     _p(row_token), _p(row_weight), _p(x_perm), _p(err),
                                     _s(stream)), "moe_permute_noalloc")


def moe_grouped_ffn(cfg, x_perm, kept, kept_offsets, row_weight, W_gate, W_up, W_down, y_perm, ws,
                    stream=None):
    _check(lib().moe_grouped_ffn(ctypes.byref(cfg), _p(x_perm), _p(kept), _p(kept_offsets),
                                 _p(row_weight), _p(W_gate), _p(W_up), _p(W_down), _p(y_perm),
                                 _p(ws), ws.numel(), _s(stream)), "moe_grouped_ffn")


def moe_combine(cfg, y_perm, pos, x, Ws_gate, Ws_up, Ws_down, out, ws, stream=None):
    _check(lib().moe_combine(ctypes.byref(cfg), _p(y_perm), _p(pos), _p(x), _p(Ws_gate),
                             _p(Ws_up), _p(Ws_down), _p(out), _p(ws), ws.numel(), _s(stream)),
           "moe_combine")


def moe_forward(cfg, x, W_r, b_r, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, out, ws,
                stream=None, events=None):
    if events is None:
        _check(lib().moe_forward(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(W_gate), _p(W_up),
                                 _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down), _p(out), _p(ws),
                                 ws.numel(), _s(stream)), "moe_forward")
    else:
        arr = _event_array(events, stream)
        _check(lib().moe_forward_traced(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(W_gate),
                                        _p(W_up), _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down),
                                        _p(out), _p(ws), ws.numel(), _s(stream), arr),
               "moe_forward_traced")


# ------------------------------------------------------------------ W4A16 expert weights

def moe_quantize_w4(W: torch.Tensor, stream=None):
    """bf16 W [..., cols] (device) -> (q uint8 [rows, cols/2], s float32 [cols/128, rows]) in the
    library's W4A16 format (rows = W.numel() / cols; scales group-major)."""
    cols = W.shape[-1]
    rows = W.numel() // cols if cols else 0
    q = torch.empty((rows, cols // 2), dtype=torch.uint8, device=W.device)
    s = torch.empty((max(cols // MOE_W4_GROUP, 1), rows), dtype=torch.float32, device=W.device)
    _check(lib().moe_quantize_w4(_p(W), rows, cols, _p(q), _p(s), _s(stream)), "moe_quantize_w4")
    return q, s


def quantize_layer_w4(weights: dict, stream=None) -> dict:
    """W4A16 copies of a layer's expert weights: {name: (q, s)} for W_gate, W_up, W_down and,
    when present, Ws_gate, Ws_up, Ws_down."""
    out = {}
    for n in ("W_gate", "W_up", "W_down", "Ws_gate", "Ws_up", "Ws_down"):
        if weights.get(n) is not None:
            out[n] = moe_quantize_w4(weights[n], stream)
    return out


def w4_layer_struct(w4: dict) -> MoeW4Layer:
    def m(name):
        qs = w4.get(name)
        return MoeW4(None, None) if qs is None else MoeW4(qs[0].data_ptr(), qs[1].data_ptr())
    return MoeW4Layer(m("W_gate"), m("W_up"), m("W_down"), m("Ws_gate"), m("Ws_up"), m("Ws_down"))


def moe_grouped_ffn_w4a16(cfg, x_perm, kept, kept_offsets, row_weight, w4: dict, y_perm, ws,
                          stream=None):
    st = w4_layer_struct(w4)
    _check(lib().moe_grouped_ffn_w4a16(ctypes.byref(cfg), _p(x_perm), _p(kept), _p(kept_offsets),
                                       _p(row_weight), ctypes.byref(st), _p(y_perm), _p(ws),
                                       ws.numel(), _s(stream)), "moe_grouped_ffn_w4a16")


def _event_array(events, stream):
    """MOE_TRACE_EVENTS torch events (None entries are not recorded) as a void* array."""
    if events is None:
        return None
    for e in events:                  # torch creates the CUDA event on its first record
        if e is not None and e.cuda_event == 0:
            e.record(stream if stream is not None else torch.cuda.current_stream())
    return (ctypes.c_void_p * MOE_TRACE_EVENTS)(
        *[ctypes.c_void_p(e.cuda_event if e is not None else 0) for e in events])


def moe_forward_w4a16(cfg, x, W_r, b_r, w4: dict, out, ws, stream=None, events=None):
    st = w4_layer_struct(w4)
    _check(lib().moe_forward_w4a16(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), ctypes.byref(st),
                                   _p(out), _p(ws), ws.numel(), _s(stream),
                                   _event_array(events, stream)), "moe_forward_w4a16")


# ------------------------------------------------------------------ backward

def moe_backward_workspace_size(cfg: MoeCfg) -> int:
    n = ctypes.c_size_t(0)
    _check(lib().moe_backward_workspace_size(ctypes.byref(cfg), ctypes.byref(n)),
           "moe_backward_workspace_size")
    return n.value


def moe_backward(cfg, x, W_r, b_r, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, dout, grads: dict,
                 ws, bws, aux_coef: float = 0.0, z_coef: float = 0.0, stream=None):
    """grads: dict of fp32 device tensors dx, dW_r, db (optional), dW_gate, dW_up, dW_down and,
    with shared experts, dWs_gate, dWs_up, dWs_down (see include/moe.h)."""
    g = grads
    _check(lib().moe_backward(ctypes.byref(cfg), _p(x), _p(W_r), _p(b_r), _p(W_gate), _p(W_up),
                              _p(W_down), _p(Ws_gate), _p(Ws_up), _p(Ws_down), _p(dout),
                              float(aux_coef), float(z_coef), _p(g["dx"]), _p(g["dW_r"]),
                              _p(g.get("db")), _p(g["dW_gate"]), _p(g["dW_up"]), _p(g["dW_down"]),
                              _p(g.get("dWs_gate")), _p(g.get("dWs_up")), _p(g.get("dWs_down")),
                              _p(ws), ws.numel(), _p(bws), bws.numel(), _s(stream)),
           "moe_backward")


def moe_forward_buffers(cfg, ws) -> dict:
    """Device tensors viewing the intermediates moe_forward leaves in the workspace."""
    b = MoeBuffers()
    _check(lib().moe_forward_buffers(ctypes.byref(cfg), _p(ws), ws.numel(), ctypes.byref(b)),
           "moe_forward_buffers")
    N, k, E, d = cfg.N, cfg.k, cfg.E, cfg.d
    R = moe_grouped_rows(cfg)
    act = torch.bfloat16 if cfg.act_dtype == MOE_BF16 else torch.float32
    esz = 2 if cfg.act_dtype == MOE_BF16 else 4
    base = ws.data_ptr()

    def view(ptr, n, dtype, esize):
        off = ptr - base
        return ws[off:off + n * esize].view(dtype)

    return dict(
        idx=view(b.idx, N * k, torch.int32, 4).view(N, k),
        w=view(b.w, N * k, torch.float32, 4).view(N, k),
        gap=view(b.gap, N, torch.float32, 4),
        P_sum=view(b.P_sum, E, torch.float32, 4),
        counts=view(b.counts, E, torch.int32, 4),
        offsets=view(b.offsets, E + 1, torch.int32, 4),
        kept=view(b.kept, E, torch.int32, 4),
        kept_offsets=view(b.kept_offsets, E + 1, torch.int32, 4),
        perm=view(b.perm, N * k, torch.int32, 4),
        pos=view(b.pos, N * k, torch.int32, 4),
        row_token=view(b.row_token, R, torch.int32, 4),
        row_weight=view(b.row_weight, R, torch.float32, 4),
        x_perm=view(b.x_perm, R * d, act, esz).view(R, d),
        y_perm=view(b.y_perm, R * d, act, esz).view(R, d),
        lse=view(b.lse, N, torch.float32, 4),
    )


def moe_stats(cfg, counts, kept, P_sum, pos, gap, ws, stream=None):
    """Returns dict(f, P, aux, dropped, fully_dropped, near_tie, touched_experts, kept_rows,
    device_error).  Synchronises the stream."""
    E = cfg.E
    f = (ctypes.c_float * E)()
    P = (ctypes.c_float * E)()
    s = MoeStatsSummary()
    _check(lib().moe_stats(ctypes.byref(cfg), _p(counts), _p(kept), _p(P_sum), _p(pos), _p(gap),
                           f, P, ctypes.byref(s), _p(ws), ws.numel(), _s(stream)), "moe_stats")
    return dict(f=list(f), P=list(P), aux=s.aux, dropped=s.dropped, fully_dropped=s.fully_dropped,
                near_tie=s.near_tie, touched_experts=s.touched_experts, kept_rows=s.kept_rows,
                device_error=s.device_error)


def moe_router_stats(cfg, lse, w, perm, offsets, ws, stream=None) -> dict:
    """z-loss, per-expert importance and its CV^2 (see include/moe.h).  Synchronises."""
    imp = (ctypes.c_float * cfg.E)()
    s = MoeRouterSummary()
    _check(lib().moe_router_stats(ctypes.byref(cfg), _p(lse), _p(w), _p(perm), _p(offsets), imp,
                                  ctypes.byref(s), _p(ws), ws.numel(), _s(stream)),
           "moe_router_stats")
    return dict(z_loss=s.z_loss, importance_cv2=s.importance_cv2,
                importance_mean=s.importance_mean, importance=list(imp))


def moe_selftest_gemm(A, B, M: int, N: int, K: int, a_mn: bool, b_mn: bool, ws, stream=None):
    """C [M,N] fp32 = sum_k A(m,k) B(n,k) through the backward GEMM engine (see include/moe.h)."""
    C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _check(lib().moe_selftest_gemm(int(a_mn), int(b_mn), M, N, K, _p(A), _p(B), _p(C), _p(ws),
                                   ws.numel(), _s(stream)), "moe_selftest_gemm")
    return C


def moe_selftest_wait_timeout(ws, timeout_us: int, stream=None):
    """Launch the bounded-wait failure check (see include/moe.h); asynchronous."""
    _check(lib().moe_selftest_wait_timeout(_p(ws), ws.numel(), timeout_us, _s(stream)),
           "moe_selftest_wait_timeout")


def moe_device_error(ws, stream=None) -> int:
    """Synchronises and returns the sticky device error word (MOE_DEVERR_* bits)."""
    code = ctypes.c_int32(0)
    lib().moe_device_error(_p(ws), ws.numel(), ctypes.byref(code), _s(stream))
    return code.value


# ------------------------------------------------------------------ convenience

class MoELayer:
    """Holds device weights, a workspace and an output buffer for one layer shape."""

    def __init__(self, cfg: MoeCfg, weights: dict, device="cuda", w4: Optional[dict] = None):
        """w4: W4A16 expert weights (quantize_layer_w4); the forward then reads them instead of
        the bf16 expert matrices (only W_r and b_r are taken from weights)."""
        self.cfg = cfg
        self.w = weights
        self.w4 = w4
        self.device = torch.device(device)
        self.ws = workspace(cfg, self.device)
        act = torch.bfloat16 if cfg.act_dtype == MOE_BF16 else torch.float32
        self.out = torch.empty((cfg.N, cfg.d), dtype=act, device=self.device)
        self.prepare_router()

    def prepare_router(self, stream=None):
        """(Re)write the router weight's split into the workspace: call after changing
        weights["W_r"] in place."""
        moe_router_prepare(self.cfg, self.w["W_r"], self.ws, stream)

    def forward(self, x: torch.Tensor, stream=None, events=None,
                out: Optional[torch.Tensor] = None) -> torch.Tensor:
        """out: where to write the layer output (default: the layer's own buffer)."""
        w = self.w
        self.last_x = x
        out = self.out if out is None else out
        if self.w4 is not None:
            moe_forward_w4a16(self.cfg, x, w["W_r"], w.get("b_r"), self.w4, out, self.ws,
                              stream, events)
            return out
        moe_forward(self.cfg, x, w["W_r"], w.get("b_r"), w["W_gate"], w["W_up"], w["W_down"],
                    w.get("Ws_gate"), w.get("Ws_up"), w.get("Ws_down"), out, self.ws,
                    stream, events)
        return out

    def capture(self, x: torch.Tensor) -> "torch.cuda.CUDAGraph":
        """Capture the forward on the static input buffer x into a CUDA graph (on a side stream,
        as capture requires); each replay() recomputes self.out from x's current contents.  Run
        one eager forward first so that the library's own streams exist before the capture."""
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g):
                self.forward(x)
        torch.cuda.current_stream().wait_stream(side)
        return g

    def buffers(self) -> dict:
        return moe_forward_buffers(self.cfg, self.ws)

    def stats(self, stream=None) -> dict:
        b = self.buffers()
        return moe_stats(self.cfg, b["counts"], b["kept"], b["P_sum"], b["pos"], b["gap"],
                         self.ws, stream)

    def router_stats(self, stream=None) -> dict:
        b = self.buffers()
        return moe_router_stats(self.cfg, b["lse"], b["w"], b["perm"], b["offsets"], self.ws,
                                stream)

    def backward(self, dout: torch.Tensor, aux_coef: float = 0.0, z_coef: float = 0.0,
                 stream=None) -> dict:
        """Gradients (fp32) of <dout, out> + aux_coef L_aux + z_coef L_z for the last forward."""
        c, w = self.cfg, self.w
        if self.w4 is not None:
            raise MoeError(2, "backward with W4A16 weights")
        if getattr(self, "bws", None) is None:
            self.bws = torch.empty(moe_backward_workspace_size(c), dtype=torch.uint8,
                                   device=self.device)
        f = lambda *shape: torch.empty(shape, dtype=torch.float32, device=self.device)
        E, d, F, S, Fs = c.E, c.d, c.d_ff, c.n_shared, c.d_ff_shared
        g = dict(dx=f(c.N, d), dW_r=f(E, d), db=f(E), dW_gate=f(E, F, d), dW_up=f(E, F, d),
                 dW_down=f(E, d, F))
        if S > 0:
            g.update(dWs_gate=f(S, Fs, d), dWs_up=f(S, Fs, d), dWs_down=f(S, d, Fs))
        moe_backward(c, self.last_x, w["W_r"], w.get("b_r"), w["W_gate"], w["W_up"], w["W_down"],
                     w.get("Ws_gate"), w.get("Ws_up"), w.get("Ws_down"), dout, g, self.ws, self.bws,
                     aux_coef, z_coef, stream)
        return g

    def device_error(self, stream=None) -> int:
        return moe_device_error(self.ws, stream)
