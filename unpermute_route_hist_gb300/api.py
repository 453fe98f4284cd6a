"""Python binding of the C ABI with the same names (minus the ``gg_`` prefix).

Argument marshalling only: torch CUDA tensors provide device memory and the
current stream; every step of the computation runs in libgg.so's kernels.
Outputs may be passed in (``out=``) or are allocated here with ``torch.empty``.
bf16 tensors are ``torch.bfloat16``; index tensors ``torch.int32``; routing
weights ``torch.float32``.
"""
from __future__ import annotations

import torch

from . import _lib
from ._lib import GGError  # noqa: F401  (re-export)


def _p(t):
    return None if t is None else t.data_ptr()


def _stream(device=None):
    return torch.cuda.current_stream(device).cuda_stream


def _need(t, dtype, name, shape=None):
    if t is None:
        raise ValueError("%s is required" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    return t


def _opt(t, dtype, name, shape=None):
    return None if t is None else _need(t, dtype, name, shape)


def _out(out, shape, dtype, device, name):
    if out is None:
        return torch.empty(shape, dtype=dtype, device=device)
    return _need(out, dtype, name, shape)


def route_workspace_size(T: int, topk: int, E: int) -> int:
    return int(_lib.load().gg_route_workspace_size(T, topk, E))


def workspace_size(op: int, T: int, topk: int, E: int, N: int = 0, K: int = 0, flags: int = 0) -> int:
    """Bytes of workspace for gg_* entry point `op` (_lib.GG_OP_*) on this problem."""
    return int(_lib.load().gg_workspace_size(op, T, topk, E, N, K, flags))


def set_gemm_schedule(mode: int) -> int:
    """Process-wide tile schedule of the GEMM launches (_lib.GG_SCHEDULE_*); returns the previous mode."""
    rc = _lib.load().gg_set_gemm_schedule(int(mode))
    if rc < 0:
        _lib.check("gg_set_gemm_schedule", rc)
    return rc


def read_status(status):
    """(rc, code): synchronise the current stream, read the device status word;
    rc is GG_OK, GG_ERR_DEVICE_CHECK or GG_ERR_TIMEOUT, code the GG_DEV_* value."""
    import ctypes
    _need(status, torch.int32, "status", (1,))
    code = ctypes.c_int32(0)
    rc = _lib.load().gg_read_status(_p(status), ctypes.addressof(code), _stream(status.device))
    if rc == _lib.GG_ERR_CUDA:
        _lib.check("gg_read_status", rc)
    return rc, int(code.value)


def _workspace(ws, nbytes, device):
    """A caller's workspace tensor, False (none), or None: allocate one of nbytes."""
    if ws is False or nbytes == 0:
        return None
    if ws is None:
        return torch.empty(nbytes, dtype=torch.uint8, device=device)
    if not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return ws


def _nbytes(t):
    return 0 if t is None else t.numel() * t.element_size()


def route_hist_offsets(topk_ids, E: int, pad_block: int = 0, *, workspace=None, status=None,
                       row_id_map: bool = True, outs: dict | None = None) -> dict:
    """m_sizes, offsets, padded_offsets (pad_block > 0), gather_idx, row_id_map."""
    T, topk = topk_ids.shape
    _need(topk_ids, torch.int32, "topk_ids")
    dev = topk_ids.device
    R = T * topk
    o = dict(outs or {})
    m = _out(o.get("m_sizes"), (E,), torch.int32, dev, "m_sizes")
    off = _out(o.get("offsets"), (E + 1,), torch.int32, dev, "offsets")
    poff = _out(o.get("padded_offsets"), (E + 1,), torch.int32, dev, "padded_offsets") if pad_block > 0 else None
    g = _out(o.get("gather_idx"), (R,), torch.int32, dev, "gather_idx")
    rim = _out(o.get("row_id_map"), (R,), torch.int32, dev, "row_id_map") if row_id_map else None
    need = route_workspace_size(T, topk, E)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    rc = _lib.load().gg_route_hist_offsets(_p(topk_ids), T, topk, E, pad_block, _p(m), _p(off),
                                           _p(poff), _p(g), _p(rim), _p(workspace),
                                           workspace.numel() * workspace.element_size(), _p(status),
                                           _stream(dev))
    _lib.check("gg_route_hist_offsets", rc)
    return dict(m_sizes=m, offsets=off, padded_offsets=poff, gather_idx=g, row_id_map=rim)


def permute(X, row_id_map, topk: int, *, out=None, status=None):
    _need(X, torch.bfloat16, "X")
    T, K = X.shape
    _need(row_id_map, torch.int32, "row_id_map", (T * topk,))
    Xp = _out(out, (T * topk, K), torch.bfloat16, X.device, "out")
    rc = _lib.load().gg_permute(_p(X), _p(row_id_map), T, topk, K, _p(Xp), _p(status), _stream(X.device))
    _lib.check("gg_permute", rc)
    return Xp


def unpermute_combine(Y, row_id_map, topk_w, T: int, topk: int, *, out=None, status=None):
    _need(Y, torch.bfloat16, "Y", (T * topk, Y.shape[1]))
    N = Y.shape[1]
    _opt(row_id_map, torch.int32, "row_id_map", (T * topk,))
    _opt(topk_w, torch.float32, "topk_w")
    if topk_w is not None and topk_w.numel() != T * topk:
        raise ValueError("topk_w must have T*topk elements")
    o = _out(out, (T, N), torch.bfloat16, Y.device, "out")
    rc = _lib.load().gg_unpermute_combine(_p(Y), _p(row_id_map), _p(topk_w), T, topk, N, _p(o),
                                          _p(status), _stream(Y.device))
    _lib.check("gg_unpermute_combine", rc)
    return o


def unpermute_combine_bwd(G, Y, row_id_map, topk_w, T: int, topk: int, *, want_dw=True, out=None,
                          out_dw=None, status=None):
    """(dY [T*topk, N] bf16, dw [T, topk] fp32 or None): the combine's backward."""
    _need(G, torch.bfloat16, "G", (T, G.shape[1]))
    N = G.shape[1]
    R = T * topk
    if want_dw:
        _need(Y, torch.bfloat16, "Y", (R, N))
    _opt(row_id_map, torch.int32, "row_id_map", (R,))
    _opt(topk_w, torch.float32, "topk_w")
    if topk_w is not None and topk_w.numel() != R:
        raise ValueError("topk_w must have T*topk elements")
    dY = _out(out, (R, N), torch.bfloat16, G.device, "out")
    dw = _out(out_dw, (T, topk), torch.float32, G.device, "out_dw") if want_dw else None
    rc = _lib.load().gg_unpermute_combine_bwd(_p(G), _p(Y) if want_dw else None, _p(row_id_map),
                                              _p(topk_w), T, topk, N, _p(dY), _p(dw), _p(status),
                                              _stream(G.device))
    _lib.check("gg_unpermute_combine_bwd", rc)
    return dY, dw


def forward(X, W, m_sizes, gather_idx, topk_w, topk: int, permute_x=False, permute_y=False,
            fuse_mul_post=False, *, out=None, status=None):
    _need(X, torch.bfloat16, "X")
    _need(W, torch.bfloat16, "W")
    E, N, K = W.shape
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    rows = X.shape[0]
    T = rows if permute_x else rows // topk
    R = T * topk
    if not permute_x and rows != R:
        raise ValueError("X must have T*topk rows without permute_x")
    _opt(gather_idx, torch.int32, "gather_idx", (R,))
    _opt(topk_w, torch.float32, "topk_w")
    if topk_w is not None and topk_w.numel() != R:
        raise ValueError("topk_w must have T*topk elements")
    Y = _out(out, (R, N), torch.bfloat16, X.device, "out")
    rc = _lib.load().gg_forward(_p(X), _p(W), _p(m_sizes), _p(gather_idx), _p(topk_w), T, topk, E, N,
                                K, int(permute_x), int(permute_y), int(fuse_mul_post), _p(Y),
                                _p(status), _stream(X.device))
    _lib.check("gg_forward", rc)
    return Y


def forward_combine(X, W, m_sizes, gather_idx, topk_w, topk: int, permute_x=False, *, out=None,
                    workspace=None, status=None):
    """out [T, N]: forward with the weighted top-k combine fused (atomic adds,
    not bit-deterministic); topk_w [T, topk] fp32 or None (unit weights).
    workspace: None allocates the T*N fp32 accumulator, a tensor is used as it,
    False selects bf16 accumulation in out (topk <= GG_COMBINE_BF16_MAX_TOPK)."""
    _need(X, torch.bfloat16, "X")
    _need(W, torch.bfloat16, "W")
    E, N, K = W.shape
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    rows = X.shape[0]
    T = rows if permute_x else rows // topk
    R = T * topk
    if not permute_x and rows != R:
        raise ValueError("X must have T*topk rows without permute_x")
    _need(gather_idx, torch.int32, "gather_idx", (R,))
    _opt(topk_w, torch.float32, "topk_w")
    if topk_w is not None and topk_w.numel() != R:
        raise ValueError("topk_w must have T*topk elements")
    out = _out(out, (T, N), torch.bfloat16, X.device, "out")
    ws = _workspace(workspace, workspace_size(_lib.GG_OP_FORWARD_COMBINE, T, topk, E, N, K), X.device)
    rc = _lib.load().gg_forward_combine(_p(X), _p(W), _p(m_sizes), _p(gather_idx), _p(topk_w), T, topk,
                                        E, N, K, int(permute_x), _p(out), _p(ws), _nbytes(ws),
                                        _p(status), _stream(X.device))
    _lib.check("gg_forward_combine", rc)
    return out


def forward_swiglu(X, W, m_sizes, gather_idx, topk: int, permute_x=False, *, store_y=True, out=None,
                   out_act=None, status=None):
    """(Y [R, N] or None, A [R, N/2]): forward with the SwiGLU of interleaved gate/up columns."""
    _need(X, torch.bfloat16, "X")
    _need(W, torch.bfloat16, "W")
    E, N, K = W.shape
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    rows = X.shape[0]
    T = rows if permute_x else rows // topk
    R = T * topk
    if not permute_x and rows != R:
        raise ValueError("X must have T*topk rows without permute_x")
    _opt(gather_idx, torch.int32, "gather_idx", (R,))
    Y = _out(out, (R, N), torch.bfloat16, X.device, "out") if store_y else None
    A = _out(out_act, (R, N // 2), torch.bfloat16, X.device, "out_act")
    rc = _lib.load().gg_forward_swiglu(_p(X), _p(W), _p(m_sizes), _p(gather_idx), T, topk, E, N, K,
                                       int(permute_x), _p(Y), _p(A), _p(status), _stream(X.device))
    _lib.check("gg_forward_swiglu", rc)
    return Y, A


def swiglu_bwd(H, dA, *, out=None):
    _need(H, torch.bfloat16, "H")
    rows, two_i = H.shape
    _need(dA, torch.bfloat16, "dA", (rows, two_i // 2))
    dH = _out(out, (rows, two_i), torch.bfloat16, H.device, "out")
    rc = _lib.load().gg_swiglu_bwd(_p(H), _p(dA), rows, two_i // 2, _p(dH), _stream(H.device))
    _lib.check("gg_swiglu_bwd", rc)
    return dH


def backward_dX(dY, W, m_sizes, gather_idx, T: int, topk: int, permute_x=False, permute_y=False,
                *, token_sum=False, out=None, out_tok=None, status=None):
    _need(dY, torch.bfloat16, "dY")
    _need(W, torch.bfloat16, "W")
    E, N, K = W.shape
    R = T * topk
    _need(dY, torch.bfloat16, "dY", (R, N))
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    _opt(gather_idx, torch.int32, "gather_idx", (R,))
    dX = _out(out, (R, K), torch.bfloat16, dY.device, "out")
    dXt = _out(out_tok, (T, K), torch.bfloat16, dY.device, "out_tok") if token_sum else None
    rc = _lib.load().gg_backward_dX(_p(dY), _p(W), _p(m_sizes), _p(gather_idx), T, topk, E, N, K,
                                    int(permute_x), int(permute_y), _p(dX), _p(dXt), _p(status),
                                    _stream(dY.device))
    _lib.check("gg_backward_dX", rc)
    return (dX, dXt) if token_sum else dX


def backward_dX_swiglu(dY, W, m_sizes, topk: int, H, *, out=None, status=None):
    """dH [R, 2K]: dX of the GEMM on the SwiGLU output (dY in expert order),
    with the SwiGLU backward on the stored H fused into the epilogue."""
    _need(dY, torch.bfloat16, "dY")
    _need(W, torch.bfloat16, "W")
    E, N, K = W.shape
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    R = dY.shape[0]
    if R % topk:
        raise ValueError("dY must have T*topk rows")
    _need(dY, torch.bfloat16, "dY", (R, N))
    _need(H, torch.bfloat16, "H", (R, 2 * K))
    dH = _out(out, (R, 2 * K), torch.bfloat16, dY.device, "out")
    rc = _lib.load().gg_backward_dX_swiglu(_p(dY), _p(W), _p(m_sizes), R // topk, topk, E, N, K, _p(H),
                                           _p(dH), _p(status), _stream(dY.device))
    _lib.check("gg_backward_dX_swiglu", rc)
    return dH


def backward_dW(X, dY, m_sizes, gather_idx, T: int, topk: int, permute_x=False, permute_y=False,
                *, out=None, workspace=None, status=None):
    """dW [E, N, K].  With a permute flag, workspace None allocates the buffer
    for the expert-order copies of the gathered operands (the fast path), a
    tensor is used as it, False fuses the row gathers into the operand loads."""
    _need(X, torch.bfloat16, "X")
    _need(dY, torch.bfloat16, "dY")
    E = m_sizes.shape[0]
    _need(m_sizes, torch.int32, "m_sizes", (E,))
    R = T * topk
    K = X.shape[1]
    N = dY.shape[1]
    if X.shape[0] != (T if permute_x else R) or dY.shape[0] != R:
        raise ValueError("X must have T (permute_x) or T*topk rows; dY T*topk rows")
    _opt(gather_idx, torch.int32, "gather_idx", (R,))
    dW = _out(out, (E, N, K), torch.bfloat16, X.device, "out")
    flags = (_lib.GG_PERMUTE_X if permute_x else 0) | (_lib.GG_PERMUTE_Y if permute_y else 0)
    ws = _workspace(workspace, workspace_size(_lib.GG_OP_BACKWARD_DW, T, topk, E, N, K, flags), X.device)
    rc = _lib.load().gg_backward_dW(_p(X), _p(dY), _p(m_sizes), _p(gather_idx), T, topk, E, N, K,
                                    int(permute_x), int(permute_y), _p(dW), _p(ws), _nbytes(ws),
                                    _p(status), _stream(X.device))
    _lib.check("gg_backward_dW", rc)
    return dW


def dual_asym(X0, X1, W0, W1, trans_a=False, trans_b=False, *, out0=None, out1=None, status=None):
    for t, n in ((X0, "X0"), (X1, "X1"), (W0, "W0"), (W1, "W1")):
        _need(t, torch.bfloat16, n)
    k = X0.shape[0] if trans_a else X0.shape[1]
    m0 = X0.shape[1] if trans_a else X0.shape[0]
    m1 = X1.shape[1] if trans_a else X1.shape[0]
    n0 = W0.shape[0] if trans_b else W0.shape[1]
    n1 = W1.shape[0] if trans_b else W1.shape[1]
    Y0 = _out(out0, (m0, n0), torch.bfloat16, X0.device, "out0")
    Y1 = _out(out1, (m1, n1), torch.bfloat16, X0.device, "out1")
    rc = _lib.load().gg_dual_asym(_p(X0), _p(X1), _p(W0), _p(W1), _p(Y0), _p(Y1), m0, m1, k, n0, n1,
                                  int(trans_a), int(trans_b), _p(status), _stream(X0.device))
    _lib.check("gg_dual_asym", rc)
    return Y0, Y1
