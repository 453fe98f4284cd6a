"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times: the whole MoE layer step (route, permute, forward, combine,
backward dX with the token sum, backward dW) runs once on the GPU, then
sampled outputs are computed one by one by the oracle from the same seeded
host inputs.  The variants with the gather fused into the operand load (the
forward's token gather, dX's slot gather, dW's token and slot gathers) are
checked on the same samples.  Samples include every expert's first and last row and rows on
both sides of each 128-row tile boundary, plus seeded random rows; for dW,
rows of every non-empty expert, its first and last, and the largest expert.
Integer outputs (routing, permute) are compared in full, bit for bit."""
import numpy as np
import pytest
import torch

import unpermute_route_hist_gb300 as gg
from oracle import oracle as orc
from unpermute_route_hist_gb300 import synth

from gpu_util import assert_close, dbf, df32, hbf, status_of, status_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


def _sample_rows(off, rng, n_random=48):
    rows = set()
    E = len(off) - 1
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi <= lo:
            continue
        for r in (lo, hi - 1, lo + 127, lo + 128, hi - 129, hi - 128):
            if lo <= r < hi:
                rows.add(r)
    rows.update(int(x) for x in rng.integers(0, int(off[-1]), size=n_random))
    return np.array(sorted(rows), np.int64)


def _sample_dw(m_sizes, n_rows, rng, per_expert=2):
    es, ns = [], []
    nz = [e for e in range(len(m_sizes)) if m_sizes[e] > 0]
    big = int(np.argmax(m_sizes))
    pick = sorted(set(nz[:2] + nz[-2:] + [big] + [int(x) for x in rng.choice(nz, size=min(6, len(nz)), replace=False)]))
    for e in pick:
        for n in [0, n_rows - 1] + [int(x) for x in rng.integers(0, n_rows, size=per_expert)]:
            es.append(e)
            ns.append(n)
    empty = [e for e in range(len(m_sizes)) if m_sizes[e] == 0]
    return np.array(es, np.int32), np.array(ns, np.int64), empty


def _run_layer(cfg):
    """The benchmark's step, once.  Returns host copies of every output."""
    dev = torch.device("cuda:0")
    ids, w = synth.route_choices(cfg)
    host = synth.moe_tensors(cfg)
    T, k, E, K, N1, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.I, cfg.R
    st = status_tensor()
    r = gg.route_hist_offsets(torch.from_numpy(ids).to(dev), E, 128, status=st)
    X, W1, dH = dbf(host["X"]), dbf(host["W1"]), dbf(host["dH"])
    res = {"ids": ids, "w": w, "host": host}
    Xp = gg.permute(X, r["row_id_map"], k, status=st)
    res["Xp"] = hbf(Xp)
    res["H"] = hbf(gg.forward(Xp, W1, r["m_sizes"], r["gather_idx"], None, k, status=st))
    res["H_fused"] = hbf(gg.forward(X, W1, r["m_sizes"], r["gather_idx"], None, k, True, status=st))
    dX1, dXt = gg.backward_dX(dH, W1, r["m_sizes"], r["gather_idx"], T, k, True, False, token_sum=True,
                              status=st)
    res["dX1"], res["dXt"] = hbf(dX1), hbf(dXt)
    res["dW1"] = hbf(gg.backward_dW(Xp, dH, r["m_sizes"], r["gather_idx"], T, k, status=st))
    res["dW1_fused"] = hbf(gg.backward_dW(X, dH, r["m_sizes"], r["gather_idx"], T, k, True, False,
                                          workspace=False, status=st))
    res["dW1_ws"] = hbf(gg.backward_dW(X, dH, r["m_sizes"], r["gather_idx"], T, k, True, False,
                                       status=st))
    if I:
        A2, W2, G = dbf(host["A2"]), dbf(host["W2"]), dbf(host["G"])
        wt = df32(w)
        Y2 = gg.forward(A2, W2, r["m_sizes"], r["gather_idx"], None, k, False, True, status=st)
        res["Y2"] = hbf(Y2)
        res["out"] = hbf(gg.unpermute_combine(Y2, None, wt, T, k, status=st))
        dY2, dw = gg.unpermute_combine_bwd(G, Y2, None, wt, T, k, status=st)
        res["dY2"], res["dw"] = hbf(dY2), dw.cpu().numpy().astype(np.float64)
        res["Y2_scaled"] = hbf(gg.forward(A2, W2, r["m_sizes"], r["gather_idx"], wt, k, False, True,
                                          True, status=st))
        dYp = gg.permute(dY2, r["row_id_map"], 1, status=st)  # token-slot -> expert order
        res["dA2"] = hbf(gg.backward_dX(dYp, W2, r["m_sizes"], r["gather_idx"], T, k, status=st))
        res["dA2_fused"] = hbf(gg.backward_dX(dY2, W2, r["m_sizes"], r["gather_idx"], T, k, False, True,
                                              status=st))
        res["dW2"] = hbf(gg.backward_dW(A2, dYp, r["m_sizes"], r["gather_idx"], T, k, status=st))
        res["dW2_fused"] = hbf(gg.backward_dW(A2, dY2, r["m_sizes"], r["gather_idx"], T, k, False, True,
                                              workspace=False, status=st))
        res["dW2_ws"] = hbf(gg.backward_dW(A2, dY2, r["m_sizes"], r["gather_idx"], T, k, False, True,
                                           status=st))
    for key in ("m_sizes", "offsets", "padded_offsets", "gather_idx", "row_id_map"):
        res[key] = r[key].cpu().numpy()
    res["status"] = status_of(st)
    return res


@pytest.mark.parametrize("name", ["mlp8", "fine128", "zipf64"])
def test_full_layer_sampled(name):
    cfg = synth.CONFIGS[name]
    T, k, E, K, N1, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.I, cfg.R
    res = _run_layer(cfg)
    assert res["status"] == 0
    host, w = res["host"], res["w"]
    ro = orc.route(res["ids"], T, k, E, pad_block=128)
    for key in ("m_sizes", "offsets", "padded_offsets", "gather_idx", "row_id_map"):
        np.testing.assert_array_equal(res[key], ro[key], err_msg=key)
    m, g, rim = ro["m_sizes"], ro["gather_idx"], ro["row_id_map"]
    np.testing.assert_array_equal(res["Xp"], orc.permute(host["X"], g, k))
    rng = np.random.default_rng(2024)
    rows = _sample_rows(ro["offsets"], rng)

    # GEMM1 forward: dense on Xp, and with the token gather fused
    vals, dest = orc.forward_rows(host["X"], host["W1"], m, g, None, k, 1, 0, 0, rows)
    assert_close(res["H"][dest], vals, name + " GEMM1 fwd")
    assert_close(res["H_fused"][dest], vals, name + " GEMM1 fwd (fused gather)")
    # GEMM1 backward: dX rows land at their token slots; token sums; dW rows
    vals, dest = orc.backward_dX_rows(host["dH"], host["W1"], m, g, 1, 0, rows)
    assert_close(res["dX1"][dest], vals, name + " dX1")
    toks = np.unique(rng.integers(0, T, size=48))
    slot_rows = rim[(toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)].astype(np.int64)
    svals, sdest = orc.backward_dX_rows(host["dH"], host["W1"], m, g, 1, 0, slot_rows)
    sub = np.empty((toks.size * k, K), np.uint16)
    order = {int(d): i for i, d in enumerate(sdest)}
    for ti, t in enumerate(toks):
        for j in range(k):
            sub[ti * k + j] = orc.round_bf16(svals[order[int(t) * k + j]])
    mag = np.abs(orc.widen_bf16(sub)).reshape(toks.size, k, K).sum(axis=1)
    assert_close(res["dXt"][toks], orc.topk_sum(sub, toks.size, k), name + " dX token sum", magnitude=mag)
    es, ns, empty = _sample_dw(m, N1, rng)
    vals = orc.backward_dW_rows(host["X"], host["dH"], m, g, k, 1, 0, es, ns)
    assert_close(res["dW1"][es, ns], vals, name + " dW1")
    assert_close(res["dW1_fused"][es, ns], vals, name + " dW1 (fused token gather)")
    assert_close(res["dW1_ws"][es, ns], vals, name + " dW1 (token gather into the workspace)")
    for e in empty:
        assert (res["dW1"][e] == 0).all() and (res["dW1_fused"][e] == 0).all()
        assert (res["dW1_ws"][e] == 0).all()

    if I:
        # GEMM2 forward with the scatter to token order (and with the top-k scale)
        vals, dest = orc.forward_rows(host["A2"], host["W2"], m, g, w, k, 0, 1, 0, rows)
        assert_close(res["Y2"][dest], vals, name + " GEMM2 fwd (scatter)")
        svals, sdest = orc.forward_rows(host["A2"], host["W2"], m, g, w, k, 0, 1, 1, rows)
        assert_close(res["Y2_scaled"][sdest], svals, name + " GEMM2 fwd (scatter + scale)")
        # combine of sampled tokens from oracle-computed rows
        slot_rows = rim[(toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)].astype(np.int64)
        yv, yd = orc.forward_rows(host["A2"], host["W2"], m, g, w, k, 0, 1, 0, slot_rows)
        order = {int(d): i for i, d in enumerate(yd)}
        ysub = np.empty((toks.size * k, K), np.uint16)
        for ti, t in enumerate(toks):
            for j in range(k):
                ysub[ti * k + j] = orc.round_bf16(yv[order[int(t) * k + j]])
        ref = orc.unpermute_combine(ysub, None, w[toks], toks.size, k)
        mag = (np.abs(orc.widen_bf16(ysub)).reshape(toks.size, k, K) * w[toks][:, :, None]).sum(axis=1)
        assert_close(res["out"][toks], ref, name + " combine", magnitude=mag)
        # combine backward: dY2 in full, dw of the sampled tokens from oracle rows
        rdY2 = orc.unpermute_combine_bwd(host["G"], None, None, w, T, k, want_dw=False)[0]
        assert_close(res["dY2"], rdY2, name + " combine bwd dY2")
        dY2h = orc.round_bf16(rdY2)
        _, rdw = orc.unpermute_combine_bwd(host["G"][toks], ysub, None, None, toks.size, k)
        # each forward row element may sit one bf16 step (<= 2^-7 of itself) from the oracle's
        Ga, Ya = np.abs(orc.widen_bf16(host["G"][toks])), np.abs(orc.widen_bf16(ysub)).reshape(toks.size, k, K)
        bound = 2.0 ** -7 * np.einsum("tn,tjn->tj", Ga, Ya) + 1e-6
        d = res["dw"][toks] - rdw
        assert (np.abs(d) <= bound).all(), name + " dw elementwise"
        assert np.linalg.norm(d) <= 1e-2 * np.linalg.norm(rdw), name + " dw rel-Frobenius"
        # GEMM2 backward on the expert-ordered dY2, and with the slot gather fused
        vals, dest = orc.backward_dX_rows(dY2h, host["W2"], m, g, 0, 1, rows)
        assert_close(res["dA2"][dest], vals, name + " dX2")
        assert_close(res["dA2_fused"][dest], vals, name + " dX2 (fused gather)")
        es, ns, empty = _sample_dw(m, K, rng)
        vals = orc.backward_dW_rows(host["A2"], dY2h, m, g, k, 0, 1, es, ns)
        assert_close(res["dW2"][es, ns], vals, name + " dW2")
        assert_close(res["dW2_fused"][es, ns], vals, name + " dW2 (fused slot gather)")
        assert_close(res["dW2_ws"][es, ns], vals, name + " dW2 (slot gather into the workspace)")
        for e in empty:
            assert (res["dW2"][e] == 0).all() and (res["dW2_fused"][e] == 0).all()
            assert (res["dW2_ws"][e] == 0).all()


def test_mlp8_gemm1_swiglu_sampled():
    """GEMM1 of mlp8 with the fused SwiGLU (the benchmark's forward), and the
    SwiGLU backward, on sampled rows."""
    cfg = synth.MLP8
    T, k, E, K, N1, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.R
    ids, w = synth.route_choices(cfg)
    host = synth.moe_tensors(cfg, ("X", "W1"))
    st = status_tensor()
    dev = torch.device("cuda:0")
    r = gg.route_hist_offsets(torch.from_numpy(ids).to(dev), E, status=st)
    Xp = gg.permute(dbf(host["X"]), r["row_id_map"], k, status=st)
    H, A = gg.forward_swiglu(Xp, dbf(host["W1"]), r["m_sizes"], r["gather_idx"], k, status=st)
    dA = synth.normal_bf16(5, "mlp8/dA", (R, N1 // 2), 0.02)
    dH = gg.swiglu_bwd(H, dbf(dA))
    Hh, Ah, dHh = hbf(H), hbf(A), hbf(dH)
    assert status_of(st) == 0
    ro = orc.route(ids, T, k, E)
    rows = _sample_rows(ro["offsets"], np.random.default_rng(7), n_random=24)
    vals, dest = orc.forward_rows(host["X"], host["W1"], ro["m_sizes"], ro["gather_idx"], None, k,
                                  1, 0, 0, rows)
    assert_close(Hh[dest], vals, "mlp8 GEMM1 fwd (swiglu kernel) H")
    assert_close(Ah[dest], orc.swiglu(vals), "mlp8 GEMM1 fwd SwiGLU act")
    # backward from the stored H (the kernel's own input here is the GPU's H; the
    # oracle gets the same stored rows only through its own forward, rounded)
    Href = orc.round_bf16(vals)
    assert_close(dHh[dest], orc.swiglu_bwd(Href, dA[dest]), "mlp8 SwiGLU bwd",
                 magnitude=np.abs(orc.swiglu_bwd(Href, dA[dest])) * 4)


@pytest.mark.parametrize("fp32", [True, False])
def test_mlp8_gemm2_fused_combine_sampled(fp32):
    """GEMM2 of mlp8 with the top-k combine fused into the epilogue (the
    inference form), on sampled tokens: each token's slots are computed one by
    one by the oracle and summed with the routing weights.  fp32: sums in the
    fp32 workspace, one rounding; else bf16 atomic adds into the output."""
    cfg = synth.MLP8
    T, k, E, K, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.I, cfg.R
    ids, w = synth.route_choices(cfg)
    host = synth.moe_tensors(cfg, ("W2", "A2"))
    st = status_tensor()
    dev = torch.device("cuda:0")
    r = gg.route_hist_offsets(torch.from_numpy(ids).to(dev), E, status=st)
    out = gg.forward_combine(dbf(host["A2"]), dbf(host["W2"]), r["m_sizes"], r["gather_idx"], df32(w),
                             k, False, workspace=None if fp32 else False, status=st)
    outh = hbf(out)
    assert status_of(st) == 0
    ro = orc.route(ids, T, k, E)
    rng = np.random.default_rng(11)
    toks = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, size=40)])).astype(np.int64)
    slots = (toks[:, None] * k + np.arange(k)[None, :]).reshape(-1)
    rows = ro["row_id_map"][slots].astype(np.int64)
    vals, dest = orc.forward_rows(host["A2"], host["W2"], ro["m_sizes"], ro["gather_idx"], w, k, 0, 1, 1,
                                  rows)
    assert (dest == slots).all()
    ref = vals.reshape(toks.size, k, K).sum(axis=1)
    mag = np.abs(vals).reshape(toks.size, k, K).sum(axis=1)
    if fp32:
        assert_close(outh[toks], ref, "mlp8 GEMM2 fused combine (fp32 sums)")
    else:
        assert_close(outh[toks], ref, "mlp8 GEMM2 fused combine (bf16 adds)", magnitude=(k + 1) / 4.0 * mag)


def test_mlp8_dX2_swiglu_sampled():
    """dX of mlp8's GEMM2 with the SwiGLU backward fused (the benchmark's
    form), on sampled expert-order rows."""
    cfg = synth.MLP8
    T, k, E, K, I, N1, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.I, cfg.N1, cfg.R
    ids, w = synth.route_choices(cfg)
    host = synth.moe_tensors(cfg, ("W2",))
    dYp = synth.normal_bf16(6, "mlp8/dYp", (R, K), 0.02)
    H = synth.normal_bf16(7, "mlp8/H", (R, N1), 1.0)
    st = status_tensor()
    dev = torch.device("cuda:0")
    r = gg.route_hist_offsets(torch.from_numpy(ids).to(dev), E, status=st)
    dH = gg.backward_dX_swiglu(dbf(dYp), dbf(host["W2"]), r["m_sizes"], k, dbf(H), status=st)
    dHh = hbf(dH)
    assert status_of(st) == 0
    ro = orc.route(ids, T, k, E)
    rows = _sample_rows(ro["offsets"], np.random.default_rng(8), n_random=24)
    dA, dest = orc.backward_dX_rows(dYp, host["W2"], ro["m_sizes"], ro["gather_idx"], 0, 0, rows)
    assert (dest == rows).all()
    assert_close(dHh[rows], orc.swiglu_bwd_f64(H[rows], dA), "mlp8 dX2 + SwiGLU bwd")


def test_tiny_full():
    """The tiny workload end to end, every element (the oracle runs it in full)."""
    cfg = synth.TINY
    res = _run_layer(cfg)
    assert res["status"] == 0
    host, w = res["host"], res["w"]
    T, k, E = cfg.T, cfg.topk, cfg.E
    ro = orc.route(res["ids"], T, k, E)
    m, g = ro["m_sizes"], ro["gather_idx"]
    assert_close(res["H"], orc.forward(host["X"], host["W1"], m, g, None, T, k, 1, 0, 0), "tiny fwd1")
    assert_close(res["Y2_scaled"], orc.forward(host["A2"], host["W2"], m, g, w, T, k, 0, 1, 1), "tiny fwd2")
    assert_close(res["dX1"], orc.backward_dX(host["dH"], host["W1"], m, g, T, k, 1, 0), "tiny dX1")
    assert_close(res["dW1"], orc.backward_dW(host["X"], host["dH"], m, g, T, k, 1, 0), "tiny dW1")
    dY2h = orc.round_bf16(orc.unpermute_combine_bwd(host["G"], None, None, w, T, k, want_dw=False)[0])
    assert_close(res["dA2"], orc.backward_dX(dY2h, host["W2"], m, g, T, k, 0, 1), "tiny dX2")
    assert_close(res["dW2"], orc.backward_dW(host["A2"], dY2h, m, g, T, k, 0, 1), "tiny dW2")


@pytest.mark.parametrize("ta,tb", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_dual_workload_full(ta, tb):
    d = synth.dual_tensors(synth.DUAL, bool(ta), bool(tb))
    st = status_tensor()
    Y0, Y1 = gg.dual_asym(dbf(d["X0"]), dbf(d["X1"]), dbf(d["W0"]), dbf(d["W1"]), bool(ta), bool(tb),
                          status=st)
    assert status_of(st) == 0
    R0, R1 = orc.dual_asym(d["X0"], d["X1"], d["W0"], d["W1"], bool(ta), bool(tb))
    assert_close(hbf(Y0), R0, "dual Y0")
    assert_close(hbf(Y1), R1, "dual Y1")


@pytest.mark.parametrize("m0,m1", [(128, 8192), (8192, 128), (8192, 8192), (1024, 256)])
def test_dual_sweep_sampled(m0, m1):
    cfg = synth.DualConfig(m0=m0, m1=m1)
    d = synth.dual_tensors(cfg)
    st = status_tensor()
    Y0, Y1 = gg.dual_asym(dbf(d["X0"]), dbf(d["X1"]), dbf(d["W0"]), dbf(d["W1"]), status=st)
    assert status_of(st) == 0
    rng = np.random.default_rng(m0 + m1)
    for Y, Xs, Ws, mm, n in ((Y0, d["X0"], d["W0"], m0, cfg.n0), (Y1, d["X1"], d["W1"], m1, cfg.n1)):
        rows = np.unique(np.concatenate([[0, mm - 1, min(127, mm - 1), min(128, mm - 1)],
                                         rng.integers(0, mm, size=24)])).astype(np.int64)
        ref = orc.dual_asym_rows(Xs, Ws, mm, cfg.k, n, False, False, rows)
        assert_close(hbf(Y)[rows], ref, "dual sweep %dx%d" % (m0, m1))
