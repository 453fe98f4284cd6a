"""Pins for the oracle's permute, unpermute-combine, top-k sum and bf16
rounding: round trips, a dense combine-matrix formulation evaluated with a
library matmul, integer-valued inputs whose sums are exact, and known bf16
encodings."""
import numpy as np
import pytest

from oracle import oracle as orc
from unpermute_route_hist_gb300 import synth


def _route(T, topk, E, seed):
    rng = np.random.default_rng(seed)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    return ids, orc.route(ids, T, topk, E)


def test_bf16_rounding_known_values():
    vals = np.array([0.0, 1.0, -2.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -8 + 2.0 ** -30,
                     3.4e38, 1e-45, -0.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -134])
    expect = [0x0000, 0x3F80, 0xC000,
              0x3F80,  # exactly halfway between 1 and 1+2^-7: ties to even -> 1
              0x3F82,  # halfway between 1+2^-7 and 1+2^-6: ties to even -> 1+2^-6
              0x3F81,  # just above halfway: rounds up
              0x7F80,  # beyond the largest finite bf16 -> inf
              0x0000,  # far below the smallest subnormal
              0x8000,
              0x0001,  # smallest bf16 subnormal
              0x0000,  # half of it: ties to even -> 0
              0x0002]  # 1.5 quanta: ties to even -> 2 quanta
    assert orc.round_bf16(vals).tolist() == expect
    # widening is exact and inverts rounding on representable values
    h = np.arange(0, 65536, 7, dtype=np.uint16)
    h = h[(h & 0x7F80) != 0x7F80]  # drop inf/nan encodings
    np.testing.assert_array_equal(orc.round_bf16(orc.widen_bf16(h)), h)
    # agrees with the synthetic generator's fp32 rounding on fp32 inputs
    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    np.testing.assert_array_equal(orc.round_bf16(x.astype(np.float64)), synth.f32_to_bf16_bits(x))


@pytest.mark.parametrize("T,topk,E,K", [(5, 1, 2, 8), (64, 2, 4, 128), (37, 8, 16, 24)])
def test_permute_is_row_gather(T, topk, E, K):
    ids, r = _route(T, topk, E, T)
    X = synth.normal_bf16(1, "x", (T, K), 1.0)
    Xp = orc.permute(X, r["gather_idx"], topk)
    # library fancy indexing
    np.testing.assert_array_equal(Xp, X[r["gather_idx"] // topk])
    # brute force: every token's row appears exactly topk times, under its experts
    for t in range(T):
        rows = [i for i in range(T * topk) if r["gather_idx"][i] // topk == t]
        assert len(rows) == topk
        for i in rows:
            np.testing.assert_array_equal(Xp[i], X[t])


def test_unpermute_inverts_permute_topk1():
    T, K = 77, 40
    ids, r = _route(T, 1, 6, 3)
    X = synth.normal_bf16(2, "x", (T, K), 1.0)
    Xp = orc.permute(X, r["gather_idx"], 1)
    back = orc.unpermute_combine(Xp, r["row_id_map"], None, T, 1)
    np.testing.assert_array_equal(orc.round_bf16(back), X)


def test_combine_of_permute_with_normalised_weights_is_identity():
    cfg = synth.TINY
    ids, w = synth.route_choices(cfg)
    r = orc.route(ids, cfg.T, cfg.topk, cfg.E)
    X = synth.normal_bf16(0, "x", (cfg.T, 64), 1.0)
    Xp = orc.permute(X, r["gather_idx"], cfg.topk)
    back = orc.unpermute_combine(Xp, r["row_id_map"], w, cfg.T, cfg.topk)
    # sum_j w_tj * x_t = x_t * sum_j w_tj, and the weights sum to 1 in fp32
    np.testing.assert_allclose(back, orc.widen_bf16(X) * w.astype(np.float64).sum(1, keepdims=True),
                               rtol=1e-15, atol=0)
    np.testing.assert_allclose(back, orc.widen_bf16(X), rtol=1e-6, atol=0)


@pytest.mark.parametrize("topk,use_map,use_w", [(1, True, True), (2, True, False), (4, False, True),
                                                (3, True, True)])
def test_combine_equals_dense_combine_matrix(topk, use_map, use_w):
    T, E, N = 29, 5, 16
    ids, r = _route(T, topk, E, 7 + topk)
    R = T * topk
    rng = np.random.default_rng(5)
    # integer-valued rows and dyadic weights: every product and sum is exact
    Y = orc.round_bf16(rng.integers(-8, 9, size=(R, N)).astype(np.float64))
    w = (rng.integers(1, 8, size=(T, topk)) / 8.0).astype(np.float32) if use_w else None
    rim = r["row_id_map"] if use_map else None
    out = orc.unpermute_combine(Y, rim, w, T, topk)
    C = np.zeros((T, R))
    for t in range(T):
        for j in range(topk):
            f = t * topk + j
            C[t, rim[f] if use_map else f] += (w[t, j] if use_w else 1.0)
    np.testing.assert_array_equal(out, C @ orc.widen_bf16(Y))


def test_combine_adjoint_identity():
    T, topk, E, N = 40, 3, 7, 12
    ids, r = _route(T, topk, E, 9)
    rng = np.random.default_rng(1)
    Y = orc.round_bf16(rng.standard_normal((T * topk, N)))
    w = rng.random((T, topk)).astype(np.float32)
    G = rng.standard_normal((T, N))
    lhs = (orc.unpermute_combine(Y, r["row_id_map"], w, T, topk) * G).sum()
    # combine^T: token gradient G[t] scaled by w[f] lands on row row_id_map[f]
    GT = np.zeros((T * topk, N))
    for f in range(T * topk):
        GT[r["row_id_map"][f]] += w.reshape(-1)[f] * G[f // topk]
    rhs = (orc.widen_bf16(Y) * GT).sum()
    assert abs(lhs - rhs) <= 1e-12 * max(1.0, abs(lhs))


def test_topk_sum_integer_exact():
    T, topk, K = 31, 4, 20
    rng = np.random.default_rng(3)
    d = orc.round_bf16(rng.integers(-50, 51, size=(T * topk, K)).astype(np.float64))
    out = orc.topk_sum(d, T, topk)
    exact = orc.widen_bf16(d).reshape(T, topk, K).sum(axis=1)
    np.testing.assert_array_equal(out, exact)
    # brute force one entry
    t, k = 17, 9
    assert out[t, k] == sum(orc.widen_bf16(d)[t * topk + j, k] for j in range(topk))


@pytest.mark.parametrize("topk,use_map,use_w", [(2, True, True), (4, False, True), (1, True, False),
                                                (8, True, True)])
def test_combine_bwd_matches_autograd(topk, use_map, use_w):
    """The combine's backward (dY and the routing-weight gradient) equals torch
    autograd through a dense formulation of the forward combine."""
    import torch
    T, E, N = 23, 6, 16
    ids, r = _route(T, topk, E, 40 + topk)
    rng = np.random.default_rng(topk)
    Y = orc.round_bf16(rng.standard_normal((T * topk, N)))
    G = orc.round_bf16(rng.standard_normal((T, N)))
    w = rng.random((T, topk)).astype(np.float32) if use_w else None
    rim = r["row_id_map"] if use_map else None
    dY, dw = orc.unpermute_combine_bwd(G, Y, rim, w, T, topk)
    Yt = torch.from_numpy(orc.widen_bf16(Y)).requires_grad_(True)
    wt = torch.from_numpy(w.astype(np.float64) if use_w else np.ones((T, topk))).requires_grad_(True)
    rows = torch.from_numpy((rim if use_map else np.arange(T * topk)).astype(np.int64))
    out = (wt.reshape(-1, 1) * Yt[rows]).reshape(T, topk, N).sum(1)
    (out * torch.from_numpy(orc.widen_bf16(G))).sum().backward()
    np.testing.assert_allclose(dY, Yt.grad.numpy(), rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(dw, wt.grad.numpy(), rtol=1e-12, atol=1e-12)


def test_combine_bwd_is_the_adjoint_of_combine_integer_exact():
    T, topk, E, N = 31, 3, 5, 12
    ids, r = _route(T, topk, E, 77)
    rng = np.random.default_rng(3)
    Y = orc.round_bf16(rng.integers(-6, 7, size=(T * topk, N)).astype(np.float64))
    G = orc.round_bf16(rng.integers(-6, 7, size=(T, N)).astype(np.float64))
    w = (rng.integers(1, 9, size=(T, topk)) / 8.0).astype(np.float32)  # dyadic: exact
    fwd = orc.unpermute_combine(Y, r["row_id_map"], w, T, topk)
    dY, dw = orc.unpermute_combine_bwd(G, Y, r["row_id_map"], w, T, topk)
    # <combine(Y), G> == <Y, dY>, exactly on integers
    assert (fwd * orc.widen_bf16(G)).sum() == (orc.widen_bf16(Y) * dY).sum()
    # d<combine(Y), G>/dw[t, j] == <G[t], Y[row]>: brute force one entry
    t, j = 13, 2
    row = r["row_id_map"][t * topk + j]
    assert dw[t, j] == (orc.widen_bf16(G)[t] * orc.widen_bf16(Y)[row]).sum()
    # without Y, only dY comes back and it equals the weighted broadcast
    dY2, dw2 = orc.unpermute_combine_bwd(G, None, r["row_id_map"], w, T, topk, want_dw=False)
    assert dw2 is None
    np.testing.assert_array_equal(dY2, dY)
