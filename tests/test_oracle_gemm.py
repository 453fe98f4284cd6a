"""Pins for the oracle's grouped GEMMs (forward, dX, dW) and the dual GEMM.

The oracle computes each result row by row with explicit gather/scatter
loops.  These tests tie it to independent computations:
  * integer-valued inputs: every product and sum is exact, compared with
    numpy int64 matrix products of every expert's full block;
  * E = 1 with identity routing: a plain dense matmul;
  * torch autograd (CPU, fp64) through a dense per-expert formulation gives
    the backward dX and dW without any hand-written backward formula;
  * structural cases: empty experts contribute no rows and a zero dW;
    dropping an empty expert changes nothing;
  * the sampled-row entry points agree with the full ones."""
import itertools

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from unpermute_route_hist_gb300 import synth

FLAGS = [(px, py, fm) for px, py, fm in itertools.product([0, 1], [0, 1], [0, 1]) if not (fm and not py)]


def _int_bf16(rng, shape, lo=-3, hi=4):
    return orc.round_bf16(rng.integers(lo, hi, size=shape).astype(np.float64))


def _setup(T, topk, E, K, N, seed, empty=()):
    rng = np.random.default_rng(seed)
    choices = [e for e in range(E) if e not in empty]
    ids = rng.choice(choices, size=(T, topk)).astype(np.int32)
    r = orc.route(ids, T, topk, E)
    return rng, ids, r


def _dense_expected_forward(X, W, r, topk, px, py, fm, w):
    """Every expert's full product via int64 matmul, then the rows it owns."""
    Xi = orc.widen_bf16(X).astype(np.int64)
    Wi = orc.widen_bf16(W).astype(np.int64)
    E = W.shape[0]
    R = r["gather_idx"].size
    g = r["gather_idx"]
    A = Xi[g // topk] if px else Xi                     # expert-order input rows
    full = np.stack([A @ Wi[e].T for e in range(E)])    # [E, R, N]
    expert = np.searchsorted(r["offsets"], np.arange(R), side="right") - 1
    Yexp = full[expert, np.arange(R)].astype(np.float64)
    if fm:
        Yexp = Yexp * w.reshape(-1)[g].astype(np.float64)[:, None]
    if py:
        Y = np.zeros_like(Yexp)
        Y[g] = Yexp
        return Y
    return Yexp


@pytest.mark.parametrize("px,py,fm", FLAGS)
def test_forward_integer_exact_all_flags(px, py, fm):
    T, topk, E, K, N = 24, 2, 5, 16, 12
    rng, ids, r = _setup(T, topk, E, K, N, 100 + 4 * px + 2 * py + fm, empty=(3,))
    X = _int_bf16(rng, (T if px else T * topk, K))
    W = _int_bf16(rng, (E, N, K))
    w = (rng.integers(1, 5, size=(T, topk)) / 4.0).astype(np.float32)  # dyadic: exact
    Y = orc.forward(X, W, r["m_sizes"], r["gather_idx"], w, T, topk, px, py, fm)
    np.testing.assert_array_equal(Y, _dense_expected_forward(X, W, r, topk, px, py, fm, w))


@pytest.mark.parametrize("px,use_w", [(0, True), (1, True), (1, False)])
def test_forward_combine_integer_exact(px, use_w):
    """Fused combine: every token row is the (weighted) sum of its slots' rows,
    checked against int64 products of every expert's full block."""
    T, topk, E, K, N = 20, 3, 5, 16, 12
    rng, ids, r = _setup(T, topk, E, K, N, 300 + px, empty=(2,))
    X = _int_bf16(rng, (T if px else T * topk, K))
    W = _int_bf16(rng, (E, N, K))
    w = (rng.integers(1, 5, size=(T, topk)) / 4.0).astype(np.float32) if use_w else None
    out = orc.forward_combine(X, W, r["m_sizes"], r["gather_idx"], w, T, topk, px)
    slots = _dense_expected_forward(X, W, r, topk, px, 1, 1 if use_w else 0, w)
    np.testing.assert_array_equal(out, slots.reshape(T, topk, N).sum(axis=1))


def test_forward_combine_single_slot_is_scatter_forward():
    T, topk, E, K, N = 40, 1, 4, 24, 16
    rng, ids, r = _setup(T, topk, E, K, N, 17)
    X = orc.round_bf16(rng.standard_normal((T, K)))
    W = orc.round_bf16(rng.standard_normal((E, N, K)))
    out = orc.forward_combine(X, W, r["m_sizes"], r["gather_idx"], None, T, topk, 1)
    np.testing.assert_array_equal(out, orc.forward(X, W, r["m_sizes"], r["gather_idx"], None, T, topk,
                                                   1, 1, 0))


def test_forward_E1_identity_is_dense_matmul():
    rng = np.random.default_rng(1)
    R, K, N = 70, 48, 40
    X = orc.round_bf16(rng.standard_normal((R, K)))
    W = orc.round_bf16(rng.standard_normal((1, N, K)))
    Y = orc.forward(X, W, np.array([R], np.int32), None, None, R, 1, 0, 0, 0)
    ref = orc.widen_bf16(X) @ orc.widen_bf16(W)[0].T
    np.testing.assert_allclose(Y, ref, rtol=1e-13, atol=1e-13)


def test_forward_empty_expert_is_inert():
    T, topk, E, K, N = 30, 2, 6, 16, 8
    rng, ids, r = _setup(T, topk, E, K, N, 7, empty=(0, 4))
    assert r["m_sizes"][0] == 0 and r["m_sizes"][4] == 0
    X = orc.round_bf16(rng.standard_normal((T, K)))
    W = orc.round_bf16(rng.standard_normal((E, N, K)))
    Y = orc.forward(X, W, r["m_sizes"], r["gather_idx"], None, T, topk, 1, 1, 0)
    # remove the empty experts entirely: same routing of every slot
    keep = [e for e in range(E) if e not in (0, 4)]
    remap = {e: i for i, e in enumerate(keep)}
    ids2 = np.vectorize(remap.get)(ids).astype(np.int32)
    r2 = orc.route(ids2, T, topk, len(keep))
    np.testing.assert_array_equal(r2["gather_idx"], r["gather_idx"])
    Y2 = orc.forward(X, W[keep], r2["m_sizes"], r2["gather_idx"], None, T, topk, 1, 1, 0)
    np.testing.assert_array_equal(Y, Y2)
    # and changing the empty experts' weights changes nothing
    W3 = W.copy()
    W3[[0, 4]] = orc.round_bf16(rng.standard_normal((2, N, K)) * 100)
    np.testing.assert_array_equal(Y, orc.forward(X, W3, r["m_sizes"], r["gather_idx"], None, T,
                                                 topk, 1, 1, 0))


def _torch_reference_grads(X, W, dY, r, topk, px, py):
    """Dense per-expert forward in torch fp64; autograd gives dX and dW."""
    g = torch.from_numpy(r["gather_idx"].astype(np.int64))
    off = r["offsets"]
    Xt = torch.from_numpy(orc.widen_bf16(X)).requires_grad_(True)
    Wt = torch.from_numpy(orc.widen_bf16(W)).requires_grad_(True)
    A = Xt[g // topk] if px else Xt
    parts = [A[off[e]:off[e + 1]] @ Wt[e].T for e in range(W.shape[0])]
    Yexp = torch.cat(parts, 0)
    if py:
        Y = torch.zeros_like(Yexp).index_copy(0, g, Yexp)
    else:
        Y = Yexp
    loss = (Y * torch.from_numpy(orc.widen_bf16(dY))).sum()
    loss.backward()
    return Xt.grad.numpy(), Wt.grad.numpy()


@pytest.mark.parametrize("px,py", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_backward_matches_autograd(px, py):
    T, topk, E, K, N = 40, 3, 6, 24, 20
    rng, ids, r = _setup(T, topk, E, K, N, 20 + 2 * px + py, empty=(2,))
    X = orc.round_bf16(rng.standard_normal((T if px else T * topk, K)))
    W = orc.round_bf16(rng.standard_normal((E, N, K)))
    dY = orc.round_bf16(rng.standard_normal((T * topk, N)))
    gX, gW = _torch_reference_grads(X, W, dY, r, topk, px, py)
    dX = orc.backward_dX(dY, W, r["m_sizes"], r["gather_idx"], T, topk, px, py)
    dW = orc.backward_dW(X, dY, r["m_sizes"], r["gather_idx"], T, topk, px, py)
    np.testing.assert_allclose(dW, gW, rtol=1e-12, atol=1e-12)
    assert (dW[2] == 0).all()  # the empty expert
    if px:
        # dX is stored per token slot; the token gradient sums a token's slots
        np.testing.assert_allclose(dX.reshape(T, topk, K).sum(1), gX, rtol=1e-12, atol=1e-12)
    else:
        np.testing.assert_allclose(dX, gX, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("px,py", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_backward_integer_exact(px, py):
    T, topk, E, K, N = 18, 2, 4, 12, 10
    rng, ids, r = _setup(T, topk, E, K, N, 50 + 2 * px + py)
    X = _int_bf16(rng, (T if px else T * topk, K))
    W = _int_bf16(rng, (E, N, K))
    dY = _int_bf16(rng, (T * topk, N))
    g = r["gather_idx"]
    Xi, Wi, Gi = (orc.widen_bf16(a).astype(np.int64) for a in (X, W, dY))
    A = Xi[g // topk] if px else Xi             # expert-order inputs
    Gexp = Gi[g] if py else Gi                  # expert-order output grads
    dX = orc.backward_dX(dY, W, r["m_sizes"], g, T, topk, px, py)
    dW = orc.backward_dW(X, dY, r["m_sizes"], g, T, topk, px, py)
    off = r["offsets"]
    for e in range(E):
        lo, hi = off[e], off[e + 1]
        np.testing.assert_array_equal(dW[e], Gexp[lo:hi].T @ A[lo:hi])
        rows = Gexp[lo:hi] @ Wi[e]
        dest = g[lo:hi] if px else np.arange(lo, hi)
        np.testing.assert_array_equal(dX[dest], rows)


def test_dW_E1_is_dense_and_empty_is_zero():
    rng = np.random.default_rng(3)
    R, K, N = 50, 16, 24
    X = orc.round_bf16(rng.standard_normal((R, K)))
    dY = orc.round_bf16(rng.standard_normal((R, N)))
    dW = orc.backward_dW(X, dY, np.array([R], np.int32), None, R, 1, 0, 0)
    np.testing.assert_allclose(dW[0], orc.widen_bf16(dY).T @ orc.widen_bf16(X), rtol=1e-13, atol=1e-13)
    dW0 = orc.backward_dW(X, dY, np.array([0, R, 0], np.int32), None, R, 1, 0, 0)
    assert (dW0[0] == 0).all() and (dW0[2] == 0).all()
    np.testing.assert_array_equal(dW0[1], dW[0])


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_dual_matches_library_matmul(ta, tb):
    cfg = synth.DualConfig(m0=24, m1=16, k=40, n0=32, n1=8, seed=3)
    d = synth.dual_tensors(cfg, bool(ta), bool(tb))
    Y0, Y1 = orc.dual_asym(d["X0"], d["X1"], d["W0"], d["W1"], bool(ta), bool(tb))
    for Y, Xs, Ws in ((Y0, d["X0"], d["W0"]), (Y1, d["X1"], d["W1"])):
        A = orc.widen_bf16(Xs)
        B = orc.widen_bf16(Ws)
        ref = (A.T if ta else A) @ (B.T if tb else B)
        np.testing.assert_allclose(Y, ref, rtol=1e-12, atol=1e-12)


def test_sampled_rows_agree_with_full():
    T, topk, E, K, N = 40, 2, 5, 24, 16
    rng, ids, r = _setup(T, topk, E, K, N, 77, empty=(1,))
    _, w = synth.topk_softmax_route(rng.standard_normal((T, E)), topk)
    X = orc.round_bf16(rng.standard_normal((T, K)))
    W = orc.round_bf16(rng.standard_normal((E, N, K)))
    dY = orc.round_bf16(rng.standard_normal((T * topk, N)))
    rows = np.array([0, 5, 17, 79, 33], np.int64)
    for px, py, fm in FLAGS:
        Xin = X if px else orc.permute(X, r["gather_idx"], topk)
        Y = orc.forward(Xin, W, r["m_sizes"], r["gather_idx"], w, T, topk, px, py, fm)
        vals, dest = orc.forward_rows(Xin, W, r["m_sizes"], r["gather_idx"], w, topk, px, py, fm, rows)
        np.testing.assert_array_equal(vals, Y[dest])
        np.testing.assert_array_equal(dest, r["gather_idx"][rows] if py else rows)
    for px, py in [(0, 0), (1, 0), (0, 1), (1, 1)]:
        Xin = X if px else orc.permute(X, r["gather_idx"], topk)
        dX = orc.backward_dX(dY, W, r["m_sizes"], r["gather_idx"], T, topk, px, py)
        vals, dest = orc.backward_dX_rows(dY, W, r["m_sizes"], r["gather_idx"], px, py, rows)
        np.testing.assert_array_equal(vals, dX[dest])
        dW = orc.backward_dW(Xin, dY, r["m_sizes"], r["gather_idx"], T, topk, px, py)
        es = np.array([0, 2, 4, 1], np.int32)
        ns = np.array([3, 0, 15, 7], np.int64)
        np.testing.assert_array_equal(
            orc.backward_dW_rows(Xin, dY, r["m_sizes"], r["gather_idx"], topk, px, py, es, ns),
            dW[es, ns])
    d = synth.dual_tensors(synth.DualConfig(m0=12, m1=8, k=16, n0=24, n1=8), True, False)
    Y0, Y1 = orc.dual_asym(d["X0"], d["X1"], d["W0"], d["W1"], True, False)
    np.testing.assert_array_equal(orc.dual_asym_rows(d["X1"], d["W1"], 8, 16, 8, True, False,
                                                     np.array([7, 0, 3])), Y1[[7, 0, 3]])


def test_swiglu_matches_library_silu_and_closed_forms():
    rng = np.random.default_rng(8)
    h = rng.standard_normal((37, 2 * 24)) * 3
    act = orc.swiglu(h)
    g, u = h[:, 0::2], h[:, 1::2]
    ref = torch.nn.functional.silu(torch.from_numpy(g)).numpy() * u
    np.testing.assert_allclose(act, ref, rtol=1e-13, atol=1e-15)
    # closed forms: silu(0) = 0, silu(large) -> g, silu(very negative) -> 0, u = 0 -> 0
    hh = np.array([[0.0, 5.0, 50.0, 2.0, -60.0, 3.0, 1.5, 0.0]])
    a = orc.swiglu(hh)[0]
    assert a[0] == 0.0 and abs(a[1] - 100.0) < 1e-12 and abs(a[2]) < 1e-20 and a[3] == 0.0


def test_swiglu_bwd_matches_autograd():
    rng = np.random.default_rng(9)
    rows, I = 29, 20
    H = orc.round_bf16(rng.standard_normal((rows, 2 * I)) * 2)
    dA = orc.round_bf16(rng.standard_normal((rows, I)))
    dH = orc.swiglu_bwd(H, dA)
    Ht = torch.from_numpy(orc.widen_bf16(H)).requires_grad_(True)
    act = torch.nn.functional.silu(Ht[:, 0::2]) * Ht[:, 1::2]
    (act * torch.from_numpy(orc.widen_bf16(dA))).sum().backward()
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-12, atol=1e-13)


def test_swiglu_bwd_f64_agrees_with_stored_bf16_form():
    """With an upstream gradient that is exactly representable in bf16 the
    fp64-input form gives the stored-input form's values bit for bit."""
    rng = np.random.default_rng(21)
    rows, I = 17, 24
    H = orc.round_bf16(rng.standard_normal((rows, 2 * I)) * 2)
    dA = orc.round_bf16(rng.standard_normal((rows, I)))
    np.testing.assert_array_equal(orc.swiglu_bwd_f64(H, orc.widen_bf16(dA)), orc.swiglu_bwd(H, dA))


@pytest.mark.parametrize("py", [0, 1])
def test_backward_dX_swiglu_matches_autograd(py):
    """dX followed by the SwiGLU backward, against torch autograd (CPU, fp64)
    through the dense per-expert product and the activation."""
    T, topk, E, K, N = 18, 2, 4, 16, 12
    rng, ids, r = _setup(T, topk, E, K, N, 40 + py, empty=(1,))
    R = T * topk
    dY = orc.round_bf16(rng.standard_normal((R, N)))
    W = orc.round_bf16(rng.standard_normal((E, N, K)))
    H = orc.round_bf16(rng.standard_normal((R, 2 * K)) * 2)
    dH = orc.backward_dX_swiglu(dY, W, r["m_sizes"], r["gather_idx"], T, topk, py, H)
    g = r["gather_idx"]
    expert = np.searchsorted(r["offsets"], np.arange(R), side="right") - 1
    dYt = torch.from_numpy(orc.widen_bf16(dY))
    Wt = torch.from_numpy(orc.widen_bf16(W))
    rows_dy = dYt[torch.from_numpy(g.astype(np.int64))] if py else dYt
    dA = torch.stack([rows_dy[i] @ Wt[expert[i]] for i in range(R)])
    Ht = torch.from_numpy(orc.widen_bf16(H)).requires_grad_(True)
    act = torch.nn.functional.silu(Ht[:, 0::2]) * Ht[:, 1::2]
    (act * dA).sum().backward()
    np.testing.assert_allclose(dH, Ht.grad.numpy(), rtol=1e-11, atol=1e-11)


def test_weights_of_the_wrong_size_are_refused():
    """The C oracle reads T*topk routing weights; the harness refuses any other
    size instead of letting it read past the array."""
    T, topk, E, K, N = 6, 2, 3, 8, 8
    rng = np.random.default_rng(3)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    ro = orc.route(ids, T, topk, E)
    X = synth.normal_bf16(1, "ww", (T * topk, K), 0.5)
    W = synth.normal_bf16(2, "ww", (E, N, K), 0.5)
    short = np.ones((T, 1), np.float32)
    with pytest.raises(ValueError):
        orc.forward(X, W, ro["m_sizes"], ro["gather_idx"], short, T, topk, 0, 1, 1)
    with pytest.raises(ValueError):
        orc.forward_rows(X, W, ro["m_sizes"], ro["gather_idx"], short, topk, 0, 1, 1, np.arange(4))
    with pytest.raises(ValueError):
        orc.unpermute_combine(X, ro["row_id_map"], short, T, topk)
    ok = np.full((T, topk), 0.5, np.float32)
    orc.forward(X, W, ro["m_sizes"], ro["gather_idx"], ok, T, topk, 0, 1, 1)
