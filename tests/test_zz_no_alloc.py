"""gg_route_hist_offsets_noalloc, the routing entry point for callers that
cannot allocate device memory (a runtime that owns all device memory in its
own arena and passes only input/output buffers, or a latency-critical path
that must not pay for an allocation).  It keeps the counting sort's scratch
in a static device array instead of a caller workspace.

Checked through the C ABI against gg_route_hist_offsets (which takes a
workspace) and against the CPU oracle's routing: two calls in a row on
different routings must both give the same integers, bit for bit; so must a
problem whose scratch is exactly the static array's size.  The file sorts last so that a stop-at-first-failure
run has already run every other test; it also passes alone in a fresh
process (it builds and loads the library itself)."""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from unpermute_route_hist_gb300 import _lib
    return _lib.load()


def _outs(T, topk, E):
    dev = torch.device("cuda:0")
    R = T * topk
    return dict(m_sizes=torch.full((E,), -7, dtype=torch.int32, device=dev),
                offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                padded_offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
                gather_idx=torch.full((R,), -7, dtype=torch.int32, device=dev),
                row_id_map=torch.full((R,), -7, dtype=torch.int32, device=dev))


def _call_noalloc(lib, ids, T, topk, E, pad, o, status, stream):
    return lib.gg_route_hist_offsets_noalloc(
        ids.data_ptr(), T, topk, E, pad, o["m_sizes"].data_ptr(), o["offsets"].data_ptr(),
        o["padded_offsets"].data_ptr(), o["gather_idx"].data_ptr(), o["row_id_map"].data_ptr(),
        status.data_ptr(), stream)


def _call_with_workspace(lib, ids, T, topk, E, pad, o, status, stream):
    need = lib.gg_route_workspace_size(T, topk, E)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=ids.device)
    return lib.gg_route_hist_offsets(
        ids.data_ptr(), T, topk, E, pad, o["m_sizes"].data_ptr(), o["offsets"].data_ptr(),
        o["padded_offsets"].data_ptr(), o["gather_idx"].data_ptr(), o["row_id_map"].data_ptr(),
        ws.data_ptr(), ws.numel(), status.data_ptr(), stream)


def test_noalloc_route_matches_workspace_route_twice(lib):
    from unpermute_route_hist_gb300 import synth
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    cases = []
    ids_a, _ = synth.route_choices(synth.FINE128)            # T=16384, top-8, E=128
    cases.append((ids_a, synth.FINE128.E, 128))
    rng = np.random.default_rng(5)
    cases.append((rng.integers(0, 37, size=(3001, 3)).astype(np.int32), 37, 64))
    for ids_np, E, pad in cases:                             # two calls in a row
        T, topk = ids_np.shape
        ids = torch.from_numpy(ids_np).to(dev)
        st_n = torch.zeros(1, dtype=torch.int32, device=dev)
        st_w = torch.zeros(1, dtype=torch.int32, device=dev)
        got, ref = _outs(T, topk, E), _outs(T, topk, E)
        assert _call_noalloc(lib, ids, T, topk, E, pad, got, st_n, stream) == 0
        assert _call_with_workspace(lib, ids, T, topk, E, pad, ref, st_w, stream) == 0
        torch.cuda.synchronize()
        assert int(st_n.item()) == 0 and int(st_w.item()) == 0
        for k in got:
            assert torch.equal(got[k], ref[k]), k
        _check_against_oracle(got, ids_np, E, pad)


def _check_against_oracle(got, ids_np, E, pad):
    from oracle import oracle as orc
    T, topk = ids_np.shape
    ro = orc.route(ids_np, T, topk, E, pad_block=pad)
    for k in ("m_sizes", "offsets", "padded_offsets", "gather_idx", "row_id_map"):
        np.testing.assert_array_equal(got[k].cpu().numpy(), ro[k], err_msg=k)


def test_noalloc_route_at_exactly_the_scratch_size(lib):
    from unpermute_route_hist_gb300 import _lib
    dev = torch.device("cuda:0")
    stream = torch.cuda.current_stream(dev).cuda_stream
    # ceil(65536/256) = 256 chunks * 1024 experts * 4 bytes = 1 MiB: the largest problem accepted
    T, topk, E, pad = 65536, 1, 1024, 32
    assert lib.gg_route_workspace_size(T, topk, E) == _lib.GG_ROUTE_NOALLOC_SCRATCH_BYTES
    ids_np = np.random.default_rng(9).integers(0, E, size=(T, topk)).astype(np.int32)
    ids = torch.from_numpy(ids_np).to(dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    got = _outs(T, topk, E)
    assert _call_noalloc(lib, ids, T, topk, E, pad, got, st, stream) == _lib.GG_OK
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _check_against_oracle(got, ids_np, E, pad)
    # one slot more needs a 257th chunk: refused on the host, nothing launched
    fake = ctypes.c_void_p(4096)
    assert lib.gg_route_hist_offsets_noalloc(fake, T + 1, 1, E, 0, fake, fake, None, fake, fake,
                                             None, None) == _lib.GG_ERR_WORKSPACE


def test_noalloc_route_rejects_problems_beyond_its_scratch(lib):
    from unpermute_route_hist_gb300 import _lib
    # ceil(65536/256) chunks * 2048 experts * 4 bytes = 2 MiB > 1 MiB of static scratch;
    # rejected on the host before any device work (the pointers are never used)
    fake = ctypes.c_void_p(4096)
    rc = lib.gg_route_hist_offsets_noalloc(fake, 65536, 1, 2048, 0, fake, fake, None, fake, fake,
                                           None, None)
    assert rc == _lib.GG_ERR_WORKSPACE
    assert lib.gg_route_workspace_size(65536, 1, 2048) > _lib.GG_ROUTE_NOALLOC_SCRATCH_BYTES
