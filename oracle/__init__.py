"""CPU oracle for the top-k routed MoE SwiGLU FFN layer (forward pass).

TEST INFRASTRUCTURE ONLY: imported by the test suite, the smoke check and the
benchmark's CPU-baseline leg, never by the CUDA path.  The arithmetic lives in
``moe_oracle.c`` (plain C loops, fp32 router, fp64 experts); this file only
marshals numpy arrays into it.  Every function cites the page passage it
follows in the C source.  Parity pins for each function are in
``tests/test_oracle_*.py``; none of them is unpinned.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
# A prebuilt copy may be substituted (the mutation test loads planted-mistake builds this way).
_OVERRIDE = os.environ.get("MOE_ORACLE_LIB")
_lib = None

F32, BF16, W4 = 0, 1, 2
W4_GROUP = 128
TIE_EPS = 1e-6


class W4Mat(ctypes.Structure):
    """A W4A16 weight matrix as the oracle reads it: packed 4-bit codes and fp32 group scales."""
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("rows", ctypes.c_int64)]


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into liboracle.so with gcc (OpenMP over tokens).  Rebuilt when the
    SHA-256 of the source and the compile line differs from the one stored beside the library."""
    if _OVERRIDE:
        return _OVERRIDE
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]
    h = hashlib.sha256(" ".join(cmd).encode())
    with open(_SRC, "rb") as f:
        h.update(f.read())
    key = h.hexdigest()
    key_path = _LIB_PATH + ".key"
    try:
        with open(key_path) as f:
            stored = f.read().strip()
    except OSError:
        stored = ""
    if force or not os.path.exists(_LIB_PATH) or stored != key:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(cmd + ["-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
        with open(key_path + f".tmp{os.getpid()}", "w") as f:
            f.write(key + "\n")
        os.replace(key_path + f".tmp{os.getpid()}", key_path)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        L.oracle_round_bf16.argtypes = [D]
        L.oracle_round_bf16.restype = ctypes.c_uint16
        L.oracle_route.argtypes = [I64, I32, I32, I32, I32, P, P, P, I32, I32, P, P, P, P, P]
        L.oracle_router_stats.argtypes = [I64, I32, I32, P, P, P, P, P, P]
        L.oracle_capacity.argtypes = [I64, I32, I32, D]
        L.oracle_capacity.restype = I64
        L.oracle_permute.argtypes = [I64, I32, I32, P, I64, P, P, P, P, P, P]
        L.oracle_keep_naive.argtypes = [I64, I32, I32, P, I64, P]
        L.oracle_keep_naive.restype = None
        L.oracle_moe_token.argtypes = [I32, I32, I32, I32, I32, I32, I32, P, P, P,
                                       P, P, P, P, P, P, P]
        L.oracle_moe_token_w.argtypes = [I32, I32, I32, I32, I32, I32, I32, I32, P, P, P,
                                         P, P, P, P, P, P, P]
        L.oracle_quantize_w4.argtypes = [P, I64, I32, P, P]
        L.oracle_dequantize_w4.argtypes = [P, P, I64, I32, P]
        L.oracle_dequantize_w4.restype = None
        L.oracle_forward_naive.argtypes = [I64, I32, I32, I32, I32, I32, I32, I32, D, I32, I32,
                                           P, P, P, I32, P, P, P, P, P, P, P, P, P, P, P, P]
        L.oracle_forward_grouped.argtypes = [I64, I32, I32, I32, I32, I32, I32, I32, D, I32, I32,
                                             P, P, P, I32, P, P, P, P, P, P, P]
        L.oracle_backward.argtypes = [I64, I32, I32, I32, I32, I32, I32, I32, D, I32, I32,
                                      P, P, P, I32, P, P, P, P, P, P, P, D, D,
                                      P, P, P, P, P, P, P, P, P]
        L.oracle_stats.argtypes = [I64, I32, I32, P, P, P, P, D, P, P, P, P]
        for fn in ("oracle_route", "oracle_router_stats", "oracle_backward", "oracle_permute", "oracle_moe_token", "oracle_moe_token_w",
                   "oracle_quantize_w4", "oracle_forward_naive",
                   "oracle_forward_grouped", "oracle_stats"):
            getattr(L, fn).restype = I32
        _lib = L
    return _lib


# ---------------------------------------------------------------- helpers

def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def as_host(a, dtype_code: int) -> np.ndarray:
    """torch tensor / numpy array -> contiguous numpy (bf16 as uint16 bits)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return a.view(torch.int16).numpy().view(np.uint16)
            return a.numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if dtype_code == BF16 and a.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns")
    return a


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def round_bf16(v: float) -> int:
    return int(lib().oracle_round_bf16(float(v)))


def capacity(N: int, k: int, E: int, cf: float) -> int:
    return int(lib().oracle_capacity(N, k, E, float(cf)))


# ---------------------------------------------------------------- steps

def route(x, W_r, b_r, k: int, dtype: int, renorm: int = 1, bias_mode: Optional[int] = None,
          with_lse: bool = False):
    """Router: returns idx [N,k] int32, w [N,k] f32, probs [N,E] f32, gap [N] f32 (and, with
    with_lse, lse [N] f64: log-sum-exp of each token's raw logits).
    bias_mode: 1 = b_r added to the logits (default when b_r is given), 2 = b_r added to the
    probabilities for the top-k choice only."""
    bias_mode = (0 if b_r is None else 1) if bias_mode is None else bias_mode
    x = as_host(x, dtype)
    W_r = np.ascontiguousarray(as_host(W_r, F32), dtype=np.float32)
    b = None if b_r is None else np.ascontiguousarray(as_host(b_r, F32), dtype=np.float32)
    N, d = x.shape
    E = W_r.shape[0]
    idx = np.zeros((N, k), np.int32)
    w = np.zeros((N, k), np.float32)
    probs = np.zeros((N, E), np.float32)
    gap = np.zeros((N,), np.float32)
    lse = np.zeros((N,), np.float64) if with_lse else None
    rc = lib().oracle_route(N, d, E, k, dtype, _p(x), _p(W_r), _p(b), bias_mode, renorm,
                            _p(idx), _p(w), _p(probs), _p(gap), _p(lse))
    if rc:
        raise ValueError("oracle_route rejected its arguments")
    return (idx, w, probs, gap, lse) if with_lse else (idx, w, probs, gap)


def router_stats(idx: np.ndarray, w: np.ndarray, lse: np.ndarray, E: int):
    """z-loss, per-expert importance and its CV^2 (see oracle_router_stats)."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    w = np.ascontiguousarray(w, dtype=np.float32)
    lse = np.ascontiguousarray(lse, dtype=np.float64)
    N, k = idx.shape
    z = ctypes.c_double(0)
    cv2 = ctypes.c_double(0)
    imp = np.zeros(E, np.float64)
    if lib().oracle_router_stats(N, E, k, _p(idx), _p(w), _p(lse), ctypes.byref(z), _p(imp),
                                 ctypes.byref(cv2)):
        raise ValueError("oracle_router_stats rejected its arguments")
    return dict(z_loss=z.value, importance=imp, importance_cv2=cv2.value)


def permute(idx: np.ndarray, E: int, cap: int = -1):
    """Grouping by expert: counts, offsets, kept, kept_offsets, perm, pos."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, k = idx.shape
    A = N * k
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    kept = np.zeros(E, np.int32)
    kept_offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(max(A, 1), np.int32)
    pos = np.zeros(max(A, 1), np.int32)
    rc = lib().oracle_permute(N, k, E, _p(idx), cap, _p(counts), _p(offsets), _p(kept),
                              _p(kept_offsets), _p(perm), _p(pos))
    if rc:
        raise ValueError("oracle_permute: expert index out of range")
    return dict(counts=counts, offsets=offsets, kept=kept, kept_offsets=kept_offsets,
                perm=perm[:A], pos=pos[:A])


def keep_naive(idx: np.ndarray, E: int, cap: int) -> np.ndarray:
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    N, k = idx.shape
    keep = np.zeros((N, k), np.int32)
    lib().oracle_keep_naive(N, k, E, _p(idx), cap, _p(keep))
    return keep


def moe_token(x_t, w_t, keep_t, experts: Sequence, shared: Sequence, dtype: int,
              round_h: int) -> np.ndarray:
    """One token's layer output.  experts: k tuples (Wg [F,d], Wu [F,d], Wd [d,F]) of the
    chosen experts in slot order; shared: S such tuples.  Arrays in the layer dtype."""
    x_t = as_host(x_t, dtype)
    d = x_t.shape[-1]
    k, S = len(experts), len(shared)
    mats = [[as_host(m, dtype) for m in trip] for trip in experts]
    smats = [[as_host(m, dtype) for m in trip] for trip in shared]
    F = mats[0][0].shape[0] if k else 0
    Fs = smats[0][0].shape[0] if S else 0

    def ptrs(ms, i):
        arr = (ctypes.c_void_p * max(len(ms), 1))()
        for j, trip in enumerate(ms):
            arr[j] = trip[i].ctypes.data
        return arr

    w_t = np.ascontiguousarray(w_t, dtype=np.float32)
    keep_t = np.ascontiguousarray(keep_t, dtype=np.int32)
    out = np.zeros(d, np.uint16 if dtype == BF16 else np.float32)
    rc = lib().oracle_moe_token(d, F, k, S, Fs, dtype, round_h, _p(x_t), _p(w_t), _p(keep_t),
                                ptrs(mats, 0), ptrs(mats, 1), ptrs(mats, 2),
                                ptrs(smats, 0), ptrs(smats, 1), ptrs(smats, 2), _p(out))
    if rc:
        raise ValueError("oracle_moe_token rejected its arguments")
    return out


def quantize_w4(W, cols: Optional[int] = None):
    """bf16 weight rows -> (q uint8 [rows, cols/2], s float32 [cols/128, rows]) (W4A16 format,
    scales group-major)."""
    Wb = as_host(W, BF16)
    cols = Wb.shape[-1] if cols is None else cols
    Wb = np.ascontiguousarray(Wb.reshape(-1, cols))
    rows = Wb.shape[0]
    q = np.zeros((rows, cols // 2), np.uint8)
    s = np.zeros((cols // W4_GROUP, rows), np.float32)
    if lib().oracle_quantize_w4(_p(Wb), rows, cols, _p(q), _p(s)):
        raise ValueError("oracle_quantize_w4: cols must be a multiple of 128")
    return q, s


def dequantize_w4(q, s, cols: int) -> np.ndarray:
    """(q [rows, cols/2], s [cols/128, rows]) -> W [rows, cols] float64, exactly q * s."""
    q = np.ascontiguousarray(q, np.uint8).reshape(-1, cols // 2)
    s = np.ascontiguousarray(s, np.float32).reshape(cols // W4_GROUP, q.shape[0])
    W = np.zeros((q.shape[0], cols), np.float64)
    lib().oracle_dequantize_w4(_p(q), _p(s), q.shape[0], cols, _p(W))
    return W


def moe_token_w4(x_t, w_t, keep_t, experts: Sequence, shared: Sequence, round_h: int = 1):
    """One token's layer output (bf16 bits) with W4A16 weights.  experts / shared: tuples of
    ((q, s) gate, (q, s) up, (q, s) down) per chosen / shared expert, in slot order."""
    x_t = as_host(x_t, BF16)
    d = x_t.shape[-1]
    keep = []

    def mats(trips, i):
        arr = (ctypes.c_void_p * max(len(trips), 1))()
        for j, trip in enumerate(trips):
            q, sc = (np.ascontiguousarray(a) for a in trip[i])
            m = W4Mat(q.ctypes.data, sc.ctypes.data, q.shape[0])
            keep.extend([q, sc, m])
            arr[j] = ctypes.addressof(m)
        return arr

    k, S = len(experts), len(shared)
    F = np.asarray(experts[0][0][0]).shape[0] if k else 0
    Fs = np.asarray(shared[0][0][0]).shape[0] if S else 0
    w_t = np.ascontiguousarray(w_t, dtype=np.float32)
    keep_t = np.ascontiguousarray(keep_t, dtype=np.int32)
    out = np.zeros(d, np.uint16)
    rc = lib().oracle_moe_token_w(d, F, k, S, Fs, BF16, W4, round_h, _p(x_t), _p(w_t), _p(keep_t),
                                  mats(experts, 0), mats(experts, 1), mats(experts, 2),
                                  mats(shared, 0), mats(shared, 1), mats(shared, 2), _p(out))
    if rc:
        raise ValueError("oracle_moe_token_w rejected its arguments")
    return out


def _layer_arrays(layer, dtype):
    g = lambda n: None if layer.get(n) is None else as_host(layer[n], dtype)
    x = as_host(layer["x"], dtype)
    W_r = np.ascontiguousarray(as_host(layer["W_r"], F32), dtype=np.float32)
    b_r = None if layer.get("b_r") is None else np.ascontiguousarray(as_host(layer["b_r"], F32),
                                                                     dtype=np.float32)
    return x, W_r, b_r, g("W_gate"), g("W_up"), g("W_down"), g("Ws_gate"), g("Ws_up"), g("Ws_down")


def forward_naive(layer: dict, k: int, dtype: int, cf: float = 0.0, renorm: int = 1,
                  round_h: Optional[int] = None, bias_mode: Optional[int] = None):
    """The whole layer token by token.  Returns (out, extras dict)."""
    x, W_r, b_r, Wg, Wu, Wd, Wsg, Wsu, Wsd = _layer_arrays(layer, dtype)
    bias_mode = (0 if b_r is None else 1) if bias_mode is None else bias_mode
    round_h = (1 if dtype == BF16 else 0) if round_h is None else round_h
    N, d = x.shape
    E, F = Wg.shape[0], Wg.shape[1]
    S = 0 if Wsg is None else Wsg.shape[0]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    out = np.zeros_like(x)
    idx = np.zeros((N, k), np.int32)
    w = np.zeros((N, k), np.float32)
    keep = np.zeros((N, k), np.int32)
    probs = np.zeros((N, E), np.float32)
    gap = np.zeros((N,), np.float32)
    rc = lib().oracle_forward_naive(N, d, F, E, k, S, Fs, dtype, float(cf), renorm, round_h,
                                    _p(x), _p(W_r), _p(b_r), bias_mode, _p(Wg), _p(Wu), _p(Wd),
                                    _p(Wsg), _p(Wsu), _p(Wsd), _p(out), _p(idx), _p(w),
                                    _p(keep), _p(probs), _p(gap))
    if rc:
        raise ValueError("oracle_forward_naive rejected its arguments")
    return out, dict(idx=idx, w=w, keep=keep, probs=probs, gap=gap)


def backward(layer: dict, k: int, dtype: int, dout, cf: float = 0.0, renorm: int = 1,
             round_h: Optional[int] = None, bias_mode: Optional[int] = None,
             aux_coef: float = 0.0, z_coef: float = 0.0) -> dict:
    """Gradients of sum <dout, out> + aux_coef L_aux + z_coef L_z (see oracle_backward), fp64:
    dx [N,d], dW_r [E,d], db [E], dW_gate, dW_up [E,F,d], dW_down [E,d,F] and the shared
    dWs_gate, dWs_up [S,F_s,d], dWs_down [S,d,F_s] (None without shared experts)."""
    x, W_r, b_r, Wg, Wu, Wd, Wsg, Wsu, Wsd = _layer_arrays(layer, dtype)
    bias_mode = (0 if b_r is None else 1) if bias_mode is None else bias_mode
    round_h = (1 if dtype == BF16 else 0) if round_h is None else round_h
    N, d = x.shape
    E, F = Wg.shape[0], Wg.shape[1]
    S = 0 if Wsg is None else Wsg.shape[0]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    dout = np.ascontiguousarray(np.asarray(dout, np.float64).reshape(N, d))
    z = lambda *shape: np.zeros(shape, np.float64)
    g = dict(dx=z(N, d), dW_r=z(E, d), db=z(E), dW_gate=z(E, F, d), dW_up=z(E, F, d),
             dW_down=z(E, d, F), dWs_gate=z(max(S, 1), Fs, d), dWs_up=z(max(S, 1), Fs, d),
             dWs_down=z(max(S, 1), d, Fs))
    rc = lib().oracle_backward(N, d, F, E, k, S, Fs, dtype, float(cf), renorm, round_h, _p(x),
                               _p(W_r), _p(b_r), bias_mode, _p(Wg), _p(Wu), _p(Wd), _p(Wsg),
                               _p(Wsu), _p(Wsd), _p(dout), float(aux_coef), float(z_coef),
                               _p(g["dx"]), _p(g["dW_r"]), _p(g["db"]), _p(g["dW_gate"]),
                               _p(g["dW_up"]), _p(g["dW_down"]), _p(g["dWs_gate"]),
                               _p(g["dWs_up"]), _p(g["dWs_down"]))
    if rc:
        raise ValueError("oracle_backward rejected its arguments")
    if S == 0:
        g["dWs_gate"] = g["dWs_up"] = g["dWs_down"] = None
    return g


def forward_grouped(layer: dict, k: int, dtype: int, cf: float = 0.0, renorm: int = 1,
                    round_h: Optional[int] = None, bias_mode: Optional[int] = None):
    x, W_r, b_r, Wg, Wu, Wd, Wsg, Wsu, Wsd = _layer_arrays(layer, dtype)
    bias_mode = (0 if b_r is None else 1) if bias_mode is None else bias_mode
    round_h = (1 if dtype == BF16 else 0) if round_h is None else round_h
    N, d = x.shape
    E, F = Wg.shape[0], Wg.shape[1]
    S = 0 if Wsg is None else Wsg.shape[0]
    Fs = 0 if Wsg is None else Wsg.shape[1]
    out = np.zeros_like(x)
    rc = lib().oracle_forward_grouped(N, d, F, E, k, S, Fs, dtype, float(cf), renorm, round_h,
                                      _p(x), _p(W_r), _p(b_r), bias_mode, _p(Wg), _p(Wu), _p(Wd),
                                      _p(Wsg), _p(Wsu), _p(Wsd), _p(out))
    if rc:
        raise ValueError("oracle_forward_grouped rejected its arguments")
    return out


def stats(idx: np.ndarray, probs: np.ndarray, keep: Optional[np.ndarray] = None,
          gap: Optional[np.ndarray] = None, tie_eps: float = TIE_EPS):
    """Load-balance statistics: f [E], P [E], aux, dropped, fully_dropped, near_tie."""
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    probs = np.ascontiguousarray(probs, dtype=np.float32)
    N, k = idx.shape
    E = probs.shape[1]
    keep = None if keep is None else np.ascontiguousarray(keep, dtype=np.int32)
    gap = None if gap is None else np.ascontiguousarray(gap, dtype=np.float32)
    f = np.zeros(E, np.float64)
    P = np.zeros(E, np.float64)
    aux = ctypes.c_double(0.0)
    cnt = np.zeros(3, np.int64)
    rc = lib().oracle_stats(N, E, k, _p(idx), _p(probs), _p(keep), _p(gap), tie_eps,
                            _p(f), _p(P), ctypes.byref(aux), _p(cnt))
    if rc:
        raise ValueError("oracle_stats rejected its arguments")
    return dict(f=f, P=P, aux=aux.value, dropped=int(cnt[0]), fully_dropped=int(cnt[1]),
                near_tie=int(cnt[2]))
