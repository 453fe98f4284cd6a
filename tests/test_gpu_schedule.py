"""The two tile schedules of the grouped-GEMM launches: the static round-robin
and the dynamic hand-out (a device counter per launch, tile numbers passed to
both CTAs of a pair through a shared-memory queue).  Results must be bit for
bit the same under both (a tile's sums do not depend on which pair computes
it), and equal to the oracle; the per-launch counters reset themselves, so
many launches in turn, CUDA-graph replays and two streams at once all give
the same results.  The problems have more tiles than there are pairs, so
tiles past the first wave are handed out."""
import contextlib

import numpy as np
import pytest
import torch

import unpermute_route_hist_gb300 as gg
from oracle import oracle as orc
from unpermute_route_hist_gb300 import _lib, synth

from gpu_util import assert_close, dbf, df32, di32, hbf, status_of, status_tensor

pytestmark = pytest.mark.gpu

# T, topk, E, K, N, empty experts: 8192 routed rows over 9 experts (one empty),
# ragged expert sizes; forward 5 n-tiles x ~40 row pairs, dX 3 n-tiles, dW 9 x 15
SHAPE = (2048, 4, 9, 520, 1040, (4,))


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@contextlib.contextmanager
def schedule(mode):
    prev = gg.set_gemm_schedule(mode)
    try:
        yield
    finally:
        gg.set_gemm_schedule(prev)


@pytest.fixture(scope="module")
def problem():
    T, topk, E, K, N, empty = SHAPE
    rng = np.random.default_rng(17)
    choices = [e for e in range(E) if e not in empty]
    # skewed expert popularity: ragged, unequal expert sizes
    p = rng.random(len(choices)) ** 2 + 0.05
    ids = rng.choice(choices, size=(T, topk), p=p / p.sum()).astype(np.int32)
    _, w = synth.topk_softmax_route(rng.standard_normal((T, E)), topk)
    R = T * topk
    d = dict(ids=ids, w=w, ro=orc.route(ids, T, topk, E),
             X=synth.normal_bf16(71, "sx", (R, K), 0.1), Xt=synth.normal_bf16(72, "st", (T, K), 0.1),
             W=synth.normal_bf16(73, "sw", (E, N, K), 0.1), dY=synth.normal_bf16(74, "sdy", (R, N), 0.1))
    st = status_tensor()
    d["r"] = gg.route_hist_offsets(di32(ids), E, status=st)
    assert status_of(st) == 0
    return d


def _passes(d):
    """Every GEMM entry point with a pair launch, on the problem's operands."""
    T, topk, E, K, N, _ = SHAPE
    r, st = d["r"], status_tensor()
    m, gi = r["m_sizes"], r["gather_idx"]
    X, Xt, W, dY, w = dbf(d["X"]), dbf(d["Xt"]), dbf(d["W"]), dbf(d["dY"]), df32(d["w"])
    out = {}
    out["fwd"] = gg.forward(X, W, m, gi, w, topk, False, True, True, status=st)
    out["fwd_swiglu"], out["act"] = gg.forward_swiglu(X, W, m, gi, topk, status=st)
    out["dX"] = gg.backward_dX(dY, W, m, gi, T, topk, False, True, status=st)
    out["dW"] = gg.backward_dW(X, dY, m, gi, T, topk, status=st)
    out["dW_tok"] = gg.backward_dW(Xt, dY, m, gi, T, topk, True, False, status=st)
    torch.cuda.synchronize()
    assert status_of(st) == 0
    return out


def test_schedules_bit_identical_and_match_oracle(problem):
    d = problem
    T, topk, E, K, N, _ = SHAPE
    with schedule(_lib.GG_SCHEDULE_STATIC):
        ref = _passes(d)
    with schedule(_lib.GG_SCHEDULE_DYNAMIC):
        dyn = _passes(d)
    for k in ref:
        assert torch.equal(ref[k], dyn[k]), k
    ro = d["ro"]
    # the dynamic results against the oracle (every element of the forward and dW)
    assert_close(hbf(dyn["fwd"]), orc.forward(d["X"], d["W"], ro["m_sizes"], ro["gather_idx"], d["w"], T, topk,
                                              0, 1, 1), "forward, dynamic schedule")
    assert_close(hbf(dyn["dW"]), orc.backward_dW(d["X"], d["dY"], ro["m_sizes"], ro["gather_idx"], T, topk, 0, 0),
                 "dW, dynamic schedule")
    rows = np.random.default_rng(3).choice(T * topk, 64, replace=False)
    vals, dest = orc.backward_dX_rows(d["dY"], d["W"], ro["m_sizes"], ro["gather_idx"], 0, 1, rows)
    assert_close(hbf(dyn["dX"])[dest], vals, "dX rows, dynamic schedule")


def test_counters_reset_across_many_launches(problem):
    """More launches than there are counter slots, forward and dW interleaved:
    every result equals the first one."""
    d = problem
    T, topk, E, K, N, _ = SHAPE
    r = d["r"]
    m, gi = r["m_sizes"], r["gather_idx"]
    X, W, dY = dbf(d["X"]), dbf(d["W"]), dbf(d["dY"])
    st = status_tensor()
    with schedule(_lib.GG_SCHEDULE_DYNAMIC):
        y0 = gg.forward(X, W, m, gi, None, topk, status=st)
        w0 = gg.backward_dW(X, dY, m, gi, T, topk, status=st)
        y = torch.empty_like(y0)
        dw = torch.empty_like(w0)
        bad = 0
        for i in range(1100):
            gg.forward(X, W, m, gi, None, topk, out=y, status=st)
            if i % 100 == 99:
                gg.backward_dW(X, dY, m, gi, T, topk, out=dw, status=st)
                bad += int(not torch.equal(dw, w0))
            if i % 50 == 49:
                bad += int(not torch.equal(y, y0))
        torch.cuda.synchronize()
    assert status_of(st) == 0
    assert bad == 0


def test_graph_replays_and_two_streams(problem):
    """A captured forward replayed several times, and the forward and dX
    running at once on two streams, give the eager results."""
    d = problem
    T, topk, E, K, N, _ = SHAPE
    r = d["r"]
    m, gi = r["m_sizes"], r["gather_idx"]
    X, W, dY = dbf(d["X"]), dbf(d["W"]), dbf(d["dY"])
    st = status_tensor()
    with schedule(_lib.GG_SCHEDULE_DYNAMIC):
        y_ref = gg.forward(X, W, m, gi, None, topk, status=st)
        dx_ref = gg.backward_dX(dY, W, m, gi, T, topk, status=st)
        torch.cuda.synchronize()
        y = torch.empty_like(y_ref)
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            gg.forward(X, W, m, gi, None, topk, out=y, status=st)  # warm (attribute set, maps)
        torch.cuda.current_stream().wait_stream(s)
        with torch.cuda.graph(g):
            gg.forward(X, W, m, gi, None, topk, out=y, status=st)
        for _ in range(5):
            y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert torch.equal(y, y_ref)
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        y2, dx2 = torch.empty_like(y_ref), torch.empty_like(dx_ref)
        bad = 0
        for _ in range(20):
            s1.wait_stream(torch.cuda.current_stream())
            s2.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(s1):
                gg.forward(X, W, m, gi, None, topk, out=y2, status=st)
            with torch.cuda.stream(s2):
                gg.backward_dX(dY, W, m, gi, T, topk, out=dx2, status=st)
            torch.cuda.synchronize()
            bad += int(not torch.equal(y2, y_ref)) + int(not torch.equal(dx2, dx_ref))
    assert status_of(st) == 0
    assert bad == 0


def test_auto_mode_matches_static_at_a_long_reduction():
    """The default (automatic) schedule at a reduction long enough for the
    dynamic hand-out (K = 4096: 64 blocks a tile) equals the static schedule."""
    T, topk, E, K, N = 1024, 2, 4, 4096, 1024
    rng = np.random.default_rng(23)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    st = status_tensor()
    r = gg.route_hist_offsets(di32(ids), E, status=st)
    X = dbf(synth.normal_bf16(81, "ax", (T * topk, K), 0.05))
    W = dbf(synth.normal_bf16(82, "aw", (E, N, K), 0.05))
    with schedule(_lib.GG_SCHEDULE_AUTO):
        ya = gg.forward(X, W, r["m_sizes"], r["gather_idx"], None, topk, status=st)
    with schedule(_lib.GG_SCHEDULE_STATIC):
        ys = gg.forward(X, W, r["m_sizes"], r["gather_idx"], None, topk, status=st)
    torch.cuda.synchronize()
    assert status_of(st) == 0
    assert torch.equal(ya, ys)
