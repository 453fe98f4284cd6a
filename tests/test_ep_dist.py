"""Expert-parallel dispatch and combine on CPU ranks (gloo), world sizes 2
and 4: the count exchange, the host plan of libgg (gg_ep_plan) and the row
exchanges run for real; the steps that are GPU kernels in the product (route,
permute, the local GEMM, the combine) are the CPU oracle's here.  Everything is
checked against one routing of all ranks' tokens (numbered rank after rank)
by the oracle: send and receive counts, local m_sizes and every local row bit
for bit, and the combined output exactly (the same fp64 sums of the same
rounded rows)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

CASES = {
    2: dict(T=[70, 45], topk=2, E=6, K=24, N=16, seed=3),
    4: dict(T=[33, 0, 51, 20], topk=3, E=8, K=16, N=24, seed=4),  # rank 1 has no tokens
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _global_data(c):
    """Every rank's tokens, expert choices and weights, and the expert weights
    (the same seeded data in every process); expert 1 is never chosen."""
    from unpermute_route_hist_gb300 import synth
    rng = np.random.default_rng(c["seed"])
    Tt = sum(c["T"])
    choices = [e for e in range(c["E"]) if e != 1]
    ids = rng.choice(choices, size=(Tt, c["topk"])).astype(np.int32)
    w = rng.random((Tt, c["topk"])).astype(np.float32)
    X = synth.normal_bf16(c["seed"], "ep/X", (Tt, c["K"]), 0.5)
    W = synth.normal_bf16(c["seed"], "ep/W", (c["E"], c["N"], c["K"]), 0.5)
    return ids, w, X, W


def _worker(rank, world, port, out):
    import torch.distributed as dist

    from oracle import oracle as orc
    from unpermute_route_hist_gb300 import ep

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    c = CASES[world]
    G, E, k = world, c["E"], c["topk"]
    E_loc = E // G
    ids_g, w_g, X_g, W = _global_data(c)
    t0 = sum(c["T"][:rank])
    T = c["T"][rank]
    ids, w, X = ids_g[t0:t0 + T], w_g[t0:t0 + T], X_g[t0:t0 + T]
    # this rank's routing and expert-order rows (GPU kernels in the product)
    ro = orc.route(ids, T, k, E)
    Xp = orc.permute(X, ro["gather_idx"], k)
    ex = ep.TorchDistExchange()
    counts = torch.from_numpy(ro["m_sizes"].reshape(G, E_loc).copy())
    recv_m = torch.empty_like(counts)
    ex.all_to_all_equal(recv_m, counts)
    pl = ep.plan(ro["m_sizes"], recv_m.numpy(), G, E_loc, row_map=True)
    R_loc = int(pl["recv_counts"].sum())
    # rows travel as bytes (gloo has no 16-bit integer type)
    x_recv = torch.empty(R_loc, 2 * c["K"], dtype=torch.uint8)
    ex.all_to_all(x_recv, torch.from_numpy(Xp.view(np.uint8)), pl["recv_counts"], pl["send_counts"])
    x_loc = np.empty((R_loc, c["K"]), np.uint16)
    x_loc[pl["row_map"]] = x_recv.numpy().view(np.uint16)
    # the local experts' GEMM, then back to received order and home
    W_loc = np.ascontiguousarray(W[rank * E_loc:(rank + 1) * E_loc])
    y_loc = orc.round_bf16(orc.forward(x_loc, W_loc, pl["local_m_sizes"], None, None, R_loc, 1, 0, 0, 0))
    y_recv = np.ascontiguousarray(y_loc[pl["row_map"]])
    y_back = torch.empty(int(pl["send_counts"].sum()), 2 * c["N"], dtype=torch.uint8)
    ex.all_to_all(y_back, torch.from_numpy(y_recv.view(np.uint8)), pl["send_counts"], pl["recv_counts"])
    res = orc.unpermute_combine(np.ascontiguousarray(y_back.numpy().view(np.uint16)), ro["row_id_map"], w, T, k)
    out[rank] = dict(send=pl["send_counts"], recv=pl["recv_counts"], m_loc=pl["local_m_sizes"],
                     x_loc=x_loc, out=res)
    dist.destroy_process_group()


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as g
    g.build()


@pytest.mark.parametrize("world", [2, 4])
def test_expert_parallel_matches_one_routing_of_all_tokens(world):
    from oracle import oracle as orc
    c = CASES[world]
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    G, E, k = world, c["E"], c["topk"]
    E_loc = E // G
    ids_g, w_g, X_g, W = _global_data(c)
    Tt = ids_g.shape[0]
    rg = orc.route(ids_g, Tt, k, E)
    Xp_g = orc.permute(X_g, rg["gather_idx"], k)
    Y_g = orc.round_bf16(orc.forward(X_g, W, rg["m_sizes"], rg["gather_idx"], None, Tt, k, 1, 1, 0))
    out_g = orc.unpermute_combine(Y_g, None, w_g, Tt, k)
    per_rank_m = []
    for r in range(G):
        t0 = sum(c["T"][:r])
        per_rank_m.append(orc.route(ids_g[t0:t0 + c["T"][r]], c["T"][r], k, E)["m_sizes"]
                          .reshape(G, E_loc).astype(np.int64))
    for r in range(G):
        got = res[r]
        lo, hi = rg["offsets"][r * E_loc], rg["offsets"][(r + 1) * E_loc]
        np.testing.assert_array_equal(got["m_loc"], rg["m_sizes"][r * E_loc:(r + 1) * E_loc])
        np.testing.assert_array_equal(got["send"], per_rank_m[r].sum(axis=1))
        np.testing.assert_array_equal(got["recv"], [per_rank_m[s][r].sum() for s in range(G)])
        np.testing.assert_array_equal(got["x_loc"], Xp_g[lo:hi])
        t0 = sum(c["T"][:r])
        np.testing.assert_array_equal(got["out"], out_g[t0:t0 + c["T"][r]])


def test_plan_against_brute_force():
    """gg_ep_plan: counts, local m_sizes and the row map from their definition,
    on random count matrices with empty blocks; bad inputs refused."""
    from unpermute_route_hist_gb300 import _lib, ep
    rng = np.random.default_rng(0)
    for G, E_loc in ((1, 5), (2, 3), (4, 4), (8, 1), (3, 7)):
        m = rng.integers(0, 4, size=G * E_loc).astype(np.int32)
        recv = rng.integers(0, 4, size=(G, E_loc)).astype(np.int32)
        recv[rng.random((G, E_loc)) < 0.3] = 0
        pl = ep.plan(m, recv, G, E_loc, row_map=True)
        np.testing.assert_array_equal(pl["send_counts"], m.reshape(G, E_loc).sum(axis=1))
        np.testing.assert_array_equal(pl["recv_counts"], recv.sum(axis=1))
        np.testing.assert_array_equal(pl["local_m_sizes"], recv.sum(axis=0))
        # brute force: list the received rows as (source, expert, q) in arrival order and
        # their places in the expert-major, source-minor order
        arrival = [(s, e, q) for s in range(G) for e in range(E_loc) for q in range(recv[s, e])]
        placed = sorted(arrival, key=lambda x: (x[1], x[0], x[2]))
        where = {a: i for i, a in enumerate(placed)}
        np.testing.assert_array_equal(pl["row_map"], [where[a] for a in arrival])
        assert sorted(pl["row_map"].tolist()) == list(range(len(arrival)))
    bad = np.array([[1, -1]], np.int32)
    with pytest.raises(_lib.GGError):
        ep.plan(np.zeros(2, np.int32), bad, 1, 2)
    with pytest.raises(ValueError):
        ep.plan(np.zeros(3, np.int32), np.zeros((1, 2), np.int32), 1, 2)
