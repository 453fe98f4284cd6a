"""The C ABI library loads and exports every entry point include/gg.h
declares; host-side argument validation returns its documented codes.  No
call here reaches the GPU (each returns before any CUDA work)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "gg.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gg_[a-z_A-Z0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    from unpermute_route_hist_gb300 import _lib
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    from unpermute_route_hist_gb300 import _lib
    assert sorted(_lib.SIGNATURES) == names


def test_binding_constants_match_header(lib):
    # every integer #define of gg.h that the binding also names has the same value
    from unpermute_route_hist_gb300 import _lib
    src = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", "gg.h")).read(), flags=re.S)
    defs = {}
    for name, val in re.findall(r"^#define\s+(GG_[A-Z0-9_]+)\s+(.+?)\s*$", src, flags=re.M):
        expr = val.replace("u", "").strip()
        if re.fullmatch(r"[0-9()<\s+\-]+", expr):
            defs[name] = int(eval(expr))
    for must in ("GG_ROUTE_NOALLOC_SCRATCH_BYTES", "GG_ERR_WORKSPACE", "GG_ERR_DEVICE_CHECK", "GG_ERR_TIMEOUT",
                 "GG_COMBINE_BF16_MAX_TOPK", "GG_OP_BACKWARD_DW", "GG_PERMUTE_Y"):
        assert must in defs, must
    for name, v in defs.items():
        assert hasattr(_lib, name), name
        assert getattr(_lib, name) == v, (name, getattr(_lib, name), v)


def test_status_strings(lib):
    from unpermute_route_hist_gb300 import _lib
    assert _lib.status_string(0) == "ok"
    for c in (-1, -2, -3, -4, -5, -6):
        assert _lib.status_string(c) != "unknown status"
    for c in (1, 2, 3, 4):
        assert _lib.device_status_string(c) != "unknown device status"


def test_workspace_size(lib):
    from unpermute_route_hist_gb300 import _lib, api
    assert api.route_workspace_size(0, 1, 4) == 0
    small = api.route_workspace_size(64, 2, 4)
    assert small >= 4 * 4 and small % 256 == 0
    assert api.route_workspace_size(16384, 8, 128) >= 512 * 128 * 4
    assert api.route_workspace_size(-1, 1, 4) == 0
    ws = api.workspace_size
    assert ws(_lib.GG_OP_ROUTE, 16384, 8, 128) == api.route_workspace_size(16384, 8, 128)
    # dW: expert-order copies of the gathered operands, each rounded up to 256 bytes
    T, k, N, K = 8192, 2, 28672, 4096
    assert ws(_lib.GG_OP_BACKWARD_DW, T, k, 8, N, K, 0) == 0
    assert ws(_lib.GG_OP_BACKWARD_DW, T, k, 8, N, K, _lib.GG_PERMUTE_X) == T * k * K * 2
    assert ws(_lib.GG_OP_BACKWARD_DW, T, k, 8, N, K, _lib.GG_PERMUTE_Y) == T * k * N * 2
    assert ws(_lib.GG_OP_BACKWARD_DW, 3, 1, 8, 8, 16, 3) == 256 + 256
    # fused combine: a [T, N] fp32 accumulator
    assert ws(_lib.GG_OP_FORWARD_COMBINE, 100, 4, 8, 24, 16, 0) == 100 * 24 * 4
    assert ws(99, 100, 4, 8, 24, 16, 0) == 0 and ws(_lib.GG_OP_ROUTE, -1, 1, 4) == 0


def test_host_validation_codes(lib):
    from unpermute_route_hist_gb300 import _lib
    L = lib
    fake = ctypes.c_void_p(4096)  # never dereferenced: every call below fails validation first
    odd = ctypes.c_void_p(4096 + 2)
    # negative sizes, too many experts / topk
    assert L.gg_forward(fake, fake, fake, None, None, -1, 2, 4, 8, 8, 0, 0, 0, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    assert L.gg_forward(fake, fake, fake, None, None, 4, 2, 4096, 8, 8, 0, 0, 0, fake, None, None) == _lib.GG_ERR_UNSUPPORTED
    assert L.gg_forward(fake, fake, fake, fake, None, 4, 65, 4, 8, 8, 0, 0, 0, fake, None, None) == _lib.GG_ERR_UNSUPPORTED
    # row widths must be multiples of 8
    assert L.gg_forward(fake, fake, fake, None, None, 4, 2, 4, 12, 8, 0, 0, 0, fake, None, None) == _lib.GG_ERR_UNSUPPORTED
    assert L.gg_backward_dX(fake, fake, fake, None, 4, 2, 4, 8, 20, 0, 0, fake, None, None, None) == _lib.GG_ERR_UNSUPPORTED
    # permute flags need gather_idx; fuse_mul_post needs permute_y and weights
    assert L.gg_forward(fake, fake, fake, None, None, 4, 2, 4, 8, 8, 1, 0, 0, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    assert L.gg_forward(fake, fake, fake, fake, fake, 4, 2, 4, 8, 8, 0, 0, 1, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    assert L.gg_forward(fake, fake, fake, fake, None, 4, 2, 4, 8, 8, 0, 1, 1, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    # misaligned tensor pointer
    assert L.gg_forward(odd, fake, fake, None, None, 4, 2, 4, 8, 8, 0, 0, 0, fake, None, None) == _lib.GG_ERR_UNSUPPORTED
    # dX token sum only with permute_x
    assert L.gg_backward_dX(fake, fake, fake, fake, 4, 2, 4, 8, 8, 0, 1, fake, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    # null outputs
    assert L.gg_backward_dW(fake, fake, fake, None, 4, 2, 4, 8, 8, 0, 0, None, None, 0, None, None) == _lib.GG_ERR_INVALID_ARG
    # dW with a gathered operand: a workspace too small or misaligned is refused
    need = L.gg_workspace_size(_lib.GG_OP_BACKWARD_DW, 4, 2, 4, 8, 8, _lib.GG_PERMUTE_X)
    assert need == 256  # 8 rows x 8 columns x 2 bytes, rounded up to 256
    assert L.gg_backward_dW(fake, fake, fake, fake, 4, 2, 4, 8, 8, 1, 0, fake, fake, need - 1, None, None) == _lib.GG_ERR_WORKSPACE
    assert L.gg_backward_dW(fake, fake, fake, fake, 4, 2, 4, 8, 8, 1, 0, fake, odd, need, None, None) == _lib.GG_ERR_WORKSPACE
    # fused combine: bf16 accumulation (no workspace) refused above its topk limit; a
    # small fp32 workspace refused
    assert L.gg_forward_combine(fake, fake, fake, fake, None, 4, _lib.GG_COMBINE_BF16_MAX_TOPK + 1, 4, 8, 8, 0,
                                fake, None, 0, None, None) == _lib.GG_ERR_WORKSPACE
    assert L.gg_forward_combine(fake, fake, fake, fake, None, 4, 2, 4, 8, 8, 0, fake, fake, 4 * 8 * 4 - 1,
                                None, None) == _lib.GG_ERR_WORKSPACE
    assert L.gg_read_status(None, None, None) == _lib.GG_ERR_INVALID_ARG
    # empty problems are OK without a launch
    assert L.gg_forward(None, None, None, None, None, 0, 2, 4, 8, 8, 0, 0, 0, None, None, None) == _lib.GG_OK
    assert L.gg_permute(None, None, 0, 2, 8, None, None, None) == _lib.GG_OK
    assert L.gg_unpermute_combine(None, None, None, 5, 2, 0, None, None, None) == _lib.GG_OK
    assert L.gg_dual_asym(None, None, None, None, None, None, 0, 0, 8, 8, 8, 0, 0, None, None) == _lib.GG_OK
    # dual sizes must be multiples of 8
    assert L.gg_dual_asym(fake, fake, fake, fake, fake, fake, 12, 8, 8, 8, 8, 0, 0, None, None) == _lib.GG_ERR_UNSUPPORTED
    # combine backward: dw needs the forward input; empty problems launch nothing
    assert L.gg_unpermute_combine_bwd(fake, None, None, None, 4, 2, 8, fake, fake, None, None) == _lib.GG_ERR_INVALID_ARG
    assert L.gg_unpermute_combine_bwd(fake, fake, None, None, 4, 2, 12, fake, None, None, None) == _lib.GG_ERR_UNSUPPORTED
    assert L.gg_unpermute_combine_bwd(None, None, None, None, 0, 2, 8, None, None, None, None) == _lib.GG_OK
    # route: workspace too small, bad sizes
    ws = L.gg_route_workspace_size(64, 2, 4)
    assert L.gg_route_hist_offsets(fake, 64, 2, 4, 0, fake, fake, None, fake, fake, fake, ws - 1, None, None) == _lib.GG_ERR_WORKSPACE
    assert L.gg_route_hist_offsets(fake, 64, 2, 0, 0, fake, fake, None, fake, fake, fake, ws, None, None) == _lib.GG_ERR_INVALID_ARG
    assert L.gg_route_hist_offsets(fake, 64, 2, 4, 8, fake, fake, None, fake, fake, fake, ws, None, None) == _lib.GG_ERR_INVALID_ARG


def test_gemm_schedule_mode(lib):
    """gg_set_gemm_schedule returns the previous mode and refuses unknown ones
    (host state only: nothing is launched)."""
    from unpermute_route_hist_gb300 import _lib
    prev = lib.gg_set_gemm_schedule(_lib.GG_SCHEDULE_STATIC)
    assert prev == _lib.GG_SCHEDULE_AUTO
    assert lib.gg_set_gemm_schedule(_lib.GG_SCHEDULE_DYNAMIC) == _lib.GG_SCHEDULE_STATIC
    assert lib.gg_set_gemm_schedule(3) == _lib.GG_ERR_INVALID_ARG
    assert lib.gg_set_gemm_schedule(-1) == _lib.GG_ERR_INVALID_ARG
    assert lib.gg_set_gemm_schedule(_lib.GG_SCHEDULE_AUTO) == _lib.GG_SCHEDULE_DYNAMIC


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    from unpermute_route_hist_gb300 import _lib
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()
