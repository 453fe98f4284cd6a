"""Python harness around the CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  The product library never imports this module; only
tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference legs of
``bench.py`` do.  It compiles ``oracle.c`` with the host C compiler on first use
(or via :func:`build`) and exposes numpy-level wrappers.

Arrays of bf16 values are passed as ``numpy.uint16`` bit patterns.  Floating
results come back as fp64 (the oracle accumulates in fp64); :func:`round_bf16`
rounds them to bf16 with ties-to-even in one step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_u16p = np.ctypeslib.ndpointer(dtype=np.uint16, flags="C_CONTIGUOUS")
_f32p = np.ctypeslib.ndpointer(dtype=np.float32, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain C, OpenMP over rows)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        sig = {
            "oracle_round_bf16": (None, [_f64p, _i64, _u16p]),
            "oracle_widen_bf16": (None, [_u16p, _i64, _f64p]),
            "oracle_route": (_int, [_i32p, _i64, _int, _int, _int, _i32p, _i32p, _vp, _i32p, _vp]),
            "oracle_n_blocks": (_i64, [_i64, _int, _int]),
            "oracle_ragged_k_starts": (None, [_i32p, _int, _int, _int, _i32p]),
            "oracle_permute": (None, [_u16p, _i32p, _i64, _int, _i64, _u16p]),
            "oracle_unpermute_combine": (None, [_u16p, _vp, _vp, _i64, _int, _i64, _f64p]),
            "oracle_unpermute_combine_bwd": (None, [_u16p, _vp, _vp, _vp, _i64, _int, _i64, _f64p,
                                                    _vp]),
            "oracle_swiglu": (None, [_f64p, _i64, _i64, _f64p]),
            "oracle_swiglu_bwd": (None, [_u16p, _u16p, _i64, _i64, _f64p]),
            "oracle_swiglu_bwd_f64": (None, [_u16p, _f64p, _i64, _i64, _f64p]),
            "oracle_forward": (None, [_u16p, _u16p, _i32p, _vp, _vp, _i64, _int, _int, _i64, _i64,
                                      _int, _int, _int, _f64p]),
            "oracle_forward_rows": (None, [_u16p, _u16p, _i32p, _vp, _vp, _int, _int, _i64, _i64,
                                           _int, _int, _int, _i64p, _i64, _f64p, _i64p]),
            "oracle_backward_dX": (None, [_u16p, _u16p, _i32p, _vp, _i64, _int, _int, _i64, _i64,
                                          _int, _int, _f64p]),
            "oracle_backward_dX_rows": (None, [_u16p, _u16p, _i32p, _vp, _int, _i64, _i64, _int,
                                               _int, _i64p, _i64, _f64p, _i64p]),
            "oracle_topk_sum": (None, [_u16p, _i64, _int, _i64, _f64p]),
            "oracle_backward_dW": (None, [_u16p, _u16p, _i32p, _vp, _i64, _int, _int, _i64, _i64,
                                          _int, _int, _f64p]),
            "oracle_backward_dW_rows": (None, [_u16p, _u16p, _i32p, _vp, _int, _int, _i64, _i64,
                                               _int, _int, _i32p, _i64p, _i64, _f64p]),
            "oracle_dual_asym": (None, [_u16p, _u16p, _u16p, _u16p, _i64, _i64, _i64, _i64, _i64,
                                        _int, _int, _f64p, _f64p]),
            "oracle_dual_asym_rows": (None, [_u16p, _u16p, _i64, _i64, _i64, _int, _int, _i64p,
                                             _i64, _f64p]),
            "oracle_num_threads": (_int, []),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- helpers --

def round_bf16(x) -> np.ndarray:
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_round_bf16(x.reshape(-1), x.size, out.reshape(-1))
    return out


def widen_bf16(h) -> np.ndarray:
    h = _c(h, np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    _load().oracle_widen_bf16(h.reshape(-1), h.size, out.reshape(-1))
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ------------------------------------------------------------------- route --

def route(ids, T: int, topk: int, E: int, pad_block: int = 0):
    """Returns dict(m_sizes, offsets, padded_offsets|None, gather_idx, row_id_map)."""
    ids = _c(ids, np.int32).reshape(-1)
    R = T * topk
    assert ids.size == R
    m = np.empty(E, np.int32)
    off = np.empty(E + 1, np.int32)
    poff = np.empty(E + 1, np.int32) if pad_block > 0 else None
    g = np.empty(R, np.int32)
    rim = np.empty(R, np.int32)
    rc = _load().oracle_route(ids, T, topk, E, pad_block, m, off, _ptr(poff), g, _ptr(rim))
    if rc != 0:
        raise ValueError("expert id out of range")
    return dict(m_sizes=m, offsets=off, padded_offsets=poff, gather_idx=g, row_id_map=rim)


def n_blocks(n_rows: int, E: int, block_m: int) -> int:
    return int(_load().oracle_n_blocks(n_rows, E, block_m))


def ragged_k_starts(hist, block_k: int, padded: bool) -> np.ndarray:
    hist = _c(hist, np.int32)
    out = np.empty(hist.size + 1, np.int32)
    _load().oracle_ragged_k_starts(hist, hist.size, block_k, int(padded), out)
    return out


# ---------------------------------------------------------- permute/combine --

def permute(X, gather_idx, topk: int) -> np.ndarray:
    X = _c(X, np.uint16)
    g = _c(gather_idx, np.int32)
    R, K = g.size, X.shape[1]
    Xp = np.empty((R, K), np.uint16)
    _load().oracle_permute(X, g, R, topk, K, Xp)
    return Xp


def _weights(topk_w, R: int):
    """The [T, topk] routing weights as contiguous fp32, or None; the C oracle
    reads R = T * topk of them, so any other size is refused here."""
    if topk_w is None:
        return None
    w = _c(topk_w, np.float32)
    if w.size != R:
        raise ValueError("topk_w must have T*topk = %d elements, got %d" % (R, w.size))
    return w


def unpermute_combine(Y, row_id_map, topk_w, T: int, topk: int) -> np.ndarray:
    Y = _c(Y, np.uint16)
    N = Y.shape[1]
    rim = None if row_id_map is None else _c(row_id_map, np.int32)
    w = _weights(topk_w, T * topk)
    out = np.empty((T, N), np.float64)
    _load().oracle_unpermute_combine(Y, _ptr(rim), _ptr(w), T, topk, N, out)
    return out


def unpermute_combine_bwd(G, Y, row_id_map, topk_w, T: int, topk: int, want_dw: bool = True):
    """(dY [R, N] fp64, dw [T, topk] fp64 or None) for the combine's backward."""
    G = _c(G, np.uint16)
    N = G.shape[1]
    R = T * topk
    Yc = None if (Y is None or not want_dw) else _c(Y, np.uint16)
    rim = None if row_id_map is None else _c(row_id_map, np.int32)
    w = _weights(topk_w, T * topk)
    dY = np.empty((R, N), np.float64)
    dw = np.empty((T, topk), np.float64) if want_dw else None
    _load().oracle_unpermute_combine_bwd(G, _ptr(Yc), _ptr(rim), _ptr(w), T, topk, N, dY, _ptr(dw))
    return dY, dw


def swiglu(h) -> np.ndarray:
    """act [rows, I] from interleaved gate/up columns h [rows, 2I] (fp64)."""
    h = _c(h, np.float64)
    rows, two_i = h.shape
    assert two_i % 2 == 0
    act = np.empty((rows, two_i // 2), np.float64)
    _load().oracle_swiglu(h, rows, two_i // 2, act)
    return act


def swiglu_bwd(H, dA) -> np.ndarray:
    """dH [rows, 2I] (fp64) from the stored bf16 H [rows, 2I] and dA [rows, I]."""
    H = _c(H, np.uint16)
    dA = _c(dA, np.uint16)
    rows, two_i = H.shape
    assert dA.shape == (rows, two_i // 2)
    dH = np.empty((rows, two_i), np.float64)
    _load().oracle_swiglu_bwd(H, dA, rows, two_i // 2, dH)
    return dH


def swiglu_bwd_f64(H, dA) -> np.ndarray:
    """dH [rows, 2I] fp64 from stored H (bf16) and an exact upstream dA (fp64)."""
    H = _c(H, np.uint16)
    dA = _c(dA, np.float64)
    rows, two_i = H.shape
    assert dA.shape == (rows, two_i // 2)
    dH = np.empty((rows, two_i), np.float64)
    _load().oracle_swiglu_bwd_f64(H, dA, rows, two_i // 2, dH)
    return dH


# ----------------------------------------------------------- grouped GEMMs --

def forward(X, W, m_sizes, gather_idx, topk_w, T, topk, permute_x, permute_y, fuse_mul_post):
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    E, N, K = W.shape
    m = _c(m_sizes, np.int32)
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    w = _weights(topk_w, T * topk)
    Y = np.zeros((T * topk, N), np.float64)
    _load().oracle_forward(X, W, m, _ptr(g), _ptr(w), T, topk, E, N, K, int(permute_x),
                           int(permute_y), int(fuse_mul_post), Y)
    return Y


def forward_combine(X, W, m_sizes, gather_idx, topk_w, T, topk, permute_x):
    """out [T, N] fp64: the forward with the weighted top-k combine fused
    (matmul_ogs.py, the scatter path with several active experts per token:
    token row t is the sum over its slots f = t*topk + j of w[f] * y_f).
    Composed from the forward in token-slot order (scaled by w when given),
    then a sum over each token's slots in ascending j."""
    fm = 0 if topk_w is None else 1
    Y = forward(X, W, m_sizes, gather_idx, topk_w, T, topk, permute_x, 1, fm)
    N = Y.shape[1]
    Y = Y.reshape(T, topk, N)
    out = np.zeros((T, N), np.float64)
    for j in range(topk):
        out += Y[:, j, :]
    return out


def forward_rows(X, W, m_sizes, gather_idx, topk_w, topk, permute_x, permute_y, fuse_mul_post,
                 rows):
    """Expert-order rows computed one by one -> (values [n, N], destination rows [n])."""
    X = _c(X, np.uint16)
    W = _c(W, np.uint16)
    E, N, K = W.shape
    m = _c(m_sizes, np.int32)
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    w = _weights(topk_w, int(m.sum()))
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, N), np.float64)
    dest = np.empty(rows.size, np.int64)
    _load().oracle_forward_rows(X, W, m, _ptr(g), _ptr(w), topk, E, N, K, int(permute_x),
                                int(permute_y), int(fuse_mul_post), rows, rows.size, out, dest)
    return out, dest


def backward_dX(dY, W, m_sizes, gather_idx, T, topk, permute_x, permute_y):
    dY = _c(dY, np.uint16)
    W = _c(W, np.uint16)
    E, N, K = W.shape
    m = _c(m_sizes, np.int32)
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    dX = np.zeros((T * topk, K), np.float64)
    _load().oracle_backward_dX(dY, W, m, _ptr(g), T, topk, E, N, K, int(permute_x),
                               int(permute_y), dX)
    return dX


def backward_dX_swiglu(dY, W, m_sizes, gather_idx, T, topk, permute_y, H):
    """dH [R, 2K] fp64: the dX pass (expert-order rows, no scatter) followed by
    the SwiGLU backward on its unrounded output dA [R, K] with the stored H."""
    dA = backward_dX(dY, W, m_sizes, gather_idx, T, topk, 0, permute_y)
    return swiglu_bwd_f64(H, dA)


def backward_dX_rows(dY, W, m_sizes, gather_idx, permute_x, permute_y, rows):
    dY = _c(dY, np.uint16)
    W = _c(W, np.uint16)
    E, N, K = W.shape
    m = _c(m_sizes, np.int32)
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, K), np.float64)
    dest = np.empty(rows.size, np.int64)
    _load().oracle_backward_dX_rows(dY, W, m, _ptr(g), E, N, K, int(permute_x), int(permute_y),
                                    rows, rows.size, out, dest)
    return out, dest


def topk_sum(dX_bf16, T, topk) -> np.ndarray:
    d = _c(dX_bf16, np.uint16)
    K = d.shape[1]
    out = np.empty((T, K), np.float64)
    _load().oracle_topk_sum(d, T, topk, K, out)
    return out


def backward_dW(X, dY, m_sizes, gather_idx, T, topk, permute_x, permute_y):
    X = _c(X, np.uint16)
    dY = _c(dY, np.uint16)
    m = _c(m_sizes, np.int32)
    E = m.size
    N, K = dY.shape[1], X.shape[1]
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    dW = np.zeros((E, N, K), np.float64)
    _load().oracle_backward_dW(X, dY, m, _ptr(g), T, topk, E, N, K, int(permute_x),
                               int(permute_y), dW)
    return dW


def backward_dW_rows(X, dY, m_sizes, gather_idx, topk, permute_x, permute_y, es, ns):
    X = _c(X, np.uint16)
    dY = _c(dY, np.uint16)
    m = _c(m_sizes, np.int32)
    E = m.size
    N, K = dY.shape[1], X.shape[1]
    g = None if gather_idx is None else _c(gather_idx, np.int32)
    es = _c(es, np.int32)
    ns = _c(ns, np.int64)
    out = np.empty((es.size, K), np.float64)
    _load().oracle_backward_dW_rows(X, dY, m, _ptr(g), topk, E, N, K, int(permute_x),
                                    int(permute_y), es, ns, es.size, out)
    return out


def dual_asym(X0, X1, W0, W1, trans_a=False, trans_b=False):
    X0, X1, W0, W1 = (_c(a, np.uint16) for a in (X0, X1, W0, W1))
    k = X0.shape[0] if trans_a else X0.shape[1]
    m0 = X0.shape[1] if trans_a else X0.shape[0]
    m1 = X1.shape[1] if trans_a else X1.shape[0]
    n0 = W0.shape[0] if trans_b else W0.shape[1]
    n1 = W1.shape[0] if trans_b else W1.shape[1]
    Y0 = np.empty((m0, n0), np.float64)
    Y1 = np.empty((m1, n1), np.float64)
    _load().oracle_dual_asym(X0, X1, W0, W1, m0, m1, k, n0, n1, int(trans_a), int(trans_b), Y0, Y1)
    return Y0, Y1


def dual_asym_rows(Xs, Ws, m, k, n, trans_a, trans_b, rows):
    Xs, Ws = _c(Xs, np.uint16), _c(Ws, np.uint16)
    rows = _c(rows, np.int64)
    out = np.empty((rows.size, n), np.float64)
    _load().oracle_dual_asym_rows(Xs, Ws, m, k, n, int(trans_a), int(trans_b), rows, rows.size,
                                  out)
    return out
