"""Expert-parallel MoE layer on one GPU: G ranks (2 and 4) run as threads of
one process, each with its own tokens and its share of the experts, through
the product API (ExpertParallel.dispatch / combine / combine_backward /
dispatch_backward, whose steps are libgg's kernels) and a loopback exchange
that stands in for the all-to-all: ranks post their send buffers, meet at a
host barrier, and copy their slices with stream-ordered device copies.  No
kernel waits on another rank's kernel; the only waits are the host barrier.

Checked against one routing of all ranks' tokens by the oracle: local
m_sizes and rows and the device row map bit for bit, the combined output,
the routing-weight gradient, the input gradient (summed over each token's
slots) and every expert's weight gradient within the tolerances."""
import threading

import numpy as np
import pytest
import torch

import unpermute_route_hist_gb300 as gg
from oracle import oracle as orc
from unpermute_route_hist_gb300 import ep, synth

from gpu_util import assert_close, dbf, df32, di32, hbf, status_of, status_tensor

pytestmark = pytest.mark.gpu

CASES = [
    dict(G=2, T=[300, 170], topk=2, E=8, K=128, N=256, seed=1),
    dict(G=4, T=[64, 0, 129, 77], topk=3, E=8, K=64, N=136, seed=2),  # rank 1 has no tokens
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


class LoopbackExchange:
    """All-to-all among G rank threads on one device (test stand-in for NCCL)."""

    def __init__(self, G):
        self.G = G
        self.barrier = threading.Barrier(G, timeout=120)
        self.posted = [None] * G

    def view(self, rank):
        lb = self

        class _Rank:
            def all_to_all_equal(self, out, inp):
                n = inp.shape[0] // lb.G
                self.all_to_all(out, inp, [n] * lb.G, [n] * lb.G)

            def all_to_all(self, out, inp, out_splits, in_splits):
                lb.posted[rank] = (inp, [int(x) for x in in_splits])
                lb.barrier.wait()
                off = 0
                for s in range(lb.G):
                    src, sp = lb.posted[s]
                    start, n = sum(sp[:rank]), sp[rank]
                    assert n == int(out_splits[s])
                    if n:
                        out[off:off + n].copy_(src[start:start + n])
                    off += n
                lb.barrier.wait()  # every rank has read the posted buffers

        return _Rank()


def _data(c):
    rng = np.random.default_rng(c["seed"])
    Tt = sum(c["T"])
    choices = [e for e in range(c["E"]) if e != 5]  # expert 5 never chosen
    ids = rng.choice(choices, size=(Tt, c["topk"])).astype(np.int32)
    w = (rng.random((Tt, c["topk"])) + 0.25).astype(np.float32)
    X = synth.normal_bf16(c["seed"], "gep/X", (Tt, c["K"]), 0.2)
    W = synth.normal_bf16(c["seed"], "gep/W", (c["E"], c["N"], c["K"]), 0.1)
    Gr = synth.normal_bf16(c["seed"], "gep/G", (Tt, c["N"]), 0.2)
    return ids, w, X, W, Gr


@pytest.mark.parametrize("c", CASES, ids=["G2", "G4"])
def test_expert_parallel_layer_on_thread_ranks(c):
    G, E, k, K, N = c["G"], c["E"], c["topk"], c["K"], c["N"]
    E_loc = E // G
    ids, w, X, W, Gr = _data(c)
    Wd = dbf(W)
    lb = LoopbackExchange(G)
    results, errors = [None] * G, []

    def rank_fn(r):
        try:
            t0, T = sum(c["T"][:r]), c["T"][r]
            epr = ep.ExpertParallel(E, r, G, exchange=lb.view(r))
            st = status_tensor()
            Xr = dbf(X[t0:t0 + T].reshape(T, K))
            d = epr.dispatch(Xr, di32(ids[t0:t0 + T].reshape(T, k)), status=st)
            Wl = Wd[r * E_loc:(r + 1) * E_loc]
            R_loc = d.x.shape[0]
            wr = df32(w[t0:t0 + T].reshape(T, k))
            y_loc = gg.forward(d.x, Wl, d.m_sizes, None, None, 1, status=st)
            out = epr.combine(y_loc, d, wr, status=st)
            dy_loc, dw = epr.combine_backward(dbf(Gr[t0:t0 + T].reshape(T, N)), d, wr, status=st)
            dx_loc = gg.backward_dX(dy_loc, Wl, d.m_sizes, None, R_loc, 1, status=st)
            dX = epr.dispatch_backward(dx_loc, d, status=st)
            dW = gg.backward_dW(d.x, dy_loc, d.m_sizes, None, R_loc, 1, status=st)
            results[r] = dict(x=hbf(d.x), m=d.m_sizes.cpu().numpy(), row_map=d.row_map.cpu().numpy(),
                              out=hbf(out), dw=dw.cpu().numpy().astype(np.float64), dX=hbf(dX),
                              dW=hbf(dW), status=status_of(st))
        except BaseException as exc:  # a failing rank releases the others
            errors.append(exc)
            lb.barrier.abort()

    threads = [threading.Thread(target=rank_fn, args=(r,)) for r in range(G)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    if errors:
        raise errors[0]

    Tt = ids.shape[0]
    rg = orc.route(ids, Tt, k, E)
    m, g = rg["m_sizes"], rg["gather_idx"]
    Xp = orc.permute(X, g, k)
    Yh = orc.round_bf16(orc.forward(X, W, m, g, None, Tt, k, 1, 1, 0))
    out_ref = orc.unpermute_combine(Yh, None, w, Tt, k)
    out_mag = (np.abs(orc.widen_bf16(Yh)).reshape(Tt, k, N) * w[:, :, None]).sum(axis=1)
    dY2, dw_ref = orc.unpermute_combine_bwd(Gr, Yh, None, w, Tt, k)
    dY2h = orc.round_bf16(dY2)
    dXh = orc.round_bf16(orc.backward_dX(dY2h, W, m, g, Tt, k, 1, 1))
    dX_ref = orc.topk_sum(dXh, Tt, k)
    dX_mag = np.abs(orc.widen_bf16(dXh)).reshape(Tt, k, K).sum(axis=1)
    dW_ref = orc.backward_dW(X, dY2h, m, g, Tt, k, 1, 1)
    ranks_m = [orc.route(ids[sum(c["T"][:r]):sum(c["T"][:r + 1])], c["T"][r], k, E)["m_sizes"]
               .reshape(G, E_loc) for r in range(G)]
    for r in range(G):
        res = results[r]
        assert res["status"] == 0
        t0, T = sum(c["T"][:r]), c["T"][r]
        lo, hi = rg["offsets"][r * E_loc], rg["offsets"][(r + 1) * E_loc]
        np.testing.assert_array_equal(res["m"], m[r * E_loc:(r + 1) * E_loc])
        np.testing.assert_array_equal(res["x"], Xp[lo:hi])
        recv_m = np.stack([ranks_m[s][r] for s in range(G)])
        pl = ep.plan(ranks_m[r].reshape(-1), recv_m, G, E_loc, row_map=True)
        np.testing.assert_array_equal(res["row_map"], pl["row_map"])
        if T == 0:
            assert res["out"].shape == (0, N) and res["dX"].shape == (0, K)
        else:
            assert_close(res["out"], out_ref[t0:t0 + T], "EP G=%d rank %d out" % (G, r),
                         magnitude=out_mag[t0:t0 + T])
            assert_close(res["dX"], dX_ref[t0:t0 + T], "EP G=%d rank %d dX" % (G, r),
                         magnitude=dX_mag[t0:t0 + T])
            # each forward row element may sit one bf16 step from the oracle's
            Ga = np.abs(orc.widen_bf16(Gr[t0:t0 + T]))
            Ya = np.abs(orc.widen_bf16(Yh)).reshape(Tt, k, N)[t0:t0 + T]
            bound = 2.0 ** -7 * np.einsum("tn,tjn->tj", Ga, Ya) + 1e-6
            assert (np.abs(res["dw"] - dw_ref[t0:t0 + T]) <= bound).all(), "EP dw rank %d" % r
        assert_close(res["dW"], dW_ref[r * E_loc:(r + 1) * E_loc], "EP G=%d rank %d dW" % (G, r))
        if 5 // E_loc == r:
            assert (res["dW"][5 % E_loc] == 0).all()


@pytest.mark.parametrize("G,E_loc", [(1, 3), (2, 4), (4, 2), (8, 256)])
def test_recv_map_kernel_matches_host_plan(G, E_loc):
    """gg_ep_recv_map on the device equals gg_ep_plan's host row map, with
    empty blocks (and whole empty sources) among the received counts."""
    rng = np.random.default_rng(G * 1000 + E_loc)
    recv = rng.integers(0, 40, size=(G, E_loc)).astype(np.int32)
    recv[rng.random((G, E_loc)) < 0.35] = 0
    if G > 1:
        recv[1] = 0
    m = rng.integers(0, 5, size=G * E_loc).astype(np.int32)
    pl = ep.plan(m, recv, G, E_loc, row_map=True)
    st = status_tensor()
    rmap = ep.recv_map(di32(recv), G, E_loc, int(recv.sum()), status=st)
    assert status_of(st) == 0
    np.testing.assert_array_equal(rmap.cpu().numpy(), pl["row_map"])
    # a row count that disagrees with the matrix is reported; the extra rows map to -1
    st2 = status_tensor()
    rmap2 = ep.recv_map(di32(recv), G, E_loc, int(recv.sum()) + 3, status=st2)
    assert status_of(st2) == gg._lib.GG_DEV_SIZES_MISMATCH
    assert (rmap2.cpu().numpy()[-3:] == -1).all()


def test_expert_parallel_through_nccl_one_rank():
    """The default exchange (torch.distributed all-to-all over NCCL) on a
    one-rank group: the whole dispatch / combine / backward chain with real
    collectives (each exchange a copy to itself), against the oracle."""
    import socket

    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1,
                            device_id=torch.device("cuda:0"))
    try:
        c = dict(G=1, T=[150], topk=2, E=4, K=64, N=128, seed=5)
        ids, w, X, W, Gr = _data(c)
        T, k, K, N, E = 150, 2, 64, 128, 4
        epr = ep.ExpertParallel(E, 0, 1)  # TorchDistExchange on the default group
        st = status_tensor()
        d = epr.dispatch(dbf(X), di32(ids), status=st)
        y = gg.forward(d.x, dbf(W), d.m_sizes, None, None, 1, status=st)
        out = epr.combine(y, d, df32(w), status=st)
        dy, dw = epr.combine_backward(dbf(Gr), d, df32(w), status=st)
        dX = epr.dispatch_backward(gg.backward_dX(dy, dbf(W), d.m_sizes, None, d.x.shape[0], 1, status=st), d,
                                   status=st)
        assert status_of(st) == 0
        rg = orc.route(ids, T, k, E)
        np.testing.assert_array_equal(hbf(d.x), orc.permute(X, rg["gather_idx"], k))
        Yh = orc.round_bf16(orc.forward(X, W, rg["m_sizes"], rg["gather_idx"], None, T, k, 1, 1, 0))
        mag = (np.abs(orc.widen_bf16(Yh)).reshape(T, k, N) * w[:, :, None]).sum(axis=1)
        assert_close(hbf(out), orc.unpermute_combine(Yh, None, w, T, k), "EP over NCCL out", magnitude=mag)
        dY2, dw_ref = orc.unpermute_combine_bwd(Gr, Yh, None, w, T, k)
        dXh = orc.round_bf16(orc.backward_dX(orc.round_bf16(dY2), W, rg["m_sizes"], rg["gather_idx"], T, k, 1, 1))
        assert_close(hbf(dX), orc.topk_sum(dXh, T, k), "EP over NCCL dX",
                     magnitude=np.abs(orc.widen_bf16(dXh)).reshape(T, k, K).sum(axis=1))
        bound = 2.0 ** -7 * np.einsum("tn,tjn->tj", np.abs(orc.widen_bf16(Gr)),
                                      np.abs(orc.widen_bf16(Yh)).reshape(T, k, N)) + 1e-6
        assert (np.abs(dw.cpu().numpy() - dw_ref) <= bound).all()
    finally:
        dist.destroy_process_group()
