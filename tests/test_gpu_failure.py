"""Failure detection on the GPU without a fault: a bounded wait that can never
complete runs out, reports GG_DEV_TIMEOUT through the status word, and the
context stays usable (a grouped GEMM runs correctly right after)."""
import numpy as np
import pytest
import torch

import unpermute_route_hist_gb300 as gg
from oracle import oracle as orc
from unpermute_route_hist_gb300 import _lib, synth

from gpu_util import assert_close, dbf, di32, hbf, status_of, status_tensor

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    return _lib.load()


def test_stuck_wait_times_out_with_status(lib):
    dev = torch.device("cuda:0")
    st = status_tensor()
    result = torch.full((1,), -1, dtype=torch.int32, device=dev)
    rc = lib.gg_selftest_bounded_wait(st.data_ptr(), result.data_ptr(), 2_000_000,  # 2 ms
                                      torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    assert status_of(st) == _lib.GG_DEV_TIMEOUT
    assert int(result.item()) == 0
    # gg_read_status maps the device code to the host code for a timeout
    assert gg.read_status(st) == (_lib.GG_ERR_TIMEOUT, _lib.GG_DEV_TIMEOUT)
    # the context is intact: a grouped GEMM right after is correct
    T, topk, E, K, N = 64, 2, 4, 128, 256
    ids = np.random.default_rng(0).integers(0, E, size=(T, topk)).astype(np.int32)
    ro = orc.route(ids, T, topk, E)
    r = gg.route_hist_offsets(di32(ids), E)
    X = synth.normal_bf16(0, "x", (T * topk, K), 0.1)
    W = synth.normal_bf16(1, "w", (E, N, K), 0.1)
    st2 = status_tensor()
    Y = gg.forward(dbf(X), dbf(W), r["m_sizes"], r["gather_idx"], None, topk, status=st2)
    assert gg.read_status(st2) == (_lib.GG_OK, 0)
    assert_close(hbf(Y), orc.forward(X, W, ro["m_sizes"], ro["gather_idx"], None, T, topk, 0, 0, 0),
                 "forward after timeout")


def test_selftest_rejects_bad_arguments(lib):
    assert lib.gg_selftest_bounded_wait(None, None, 1000, None) == _lib.GG_ERR_INVALID_ARG


def test_read_status_reports_bad_input_data(lib):
    """An expert id out of range is skipped by the routing kernels and reported
    through the status word; gg_read_status returns GG_ERR_DEVICE_CHECK."""
    ids = np.array([[0, 1], [2, 7]], np.int32)  # 7 is outside [0, 4)
    st = status_tensor()
    gg.route_hist_offsets(di32(ids), 4, status=st)
    assert gg.read_status(st) == (_lib.GG_ERR_DEVICE_CHECK, _lib.GG_DEV_BAD_EXPERT_ID)
