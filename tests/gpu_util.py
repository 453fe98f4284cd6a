"""Helpers shared by the GPU parity tests: host<->device conversion of bf16
bit patterns and the tolerance checks."""
import numpy as np
import torch

from oracle import oracle as orc

# bf16-in / fp32-accumulate outputs vs the oracle's fp64 result
MAX_ABS = 2e-2
REL_FRO = 1e-2


def dev():
    return torch.device("cuda:0")


def dbf(u16):
    """uint16 bf16 bits (numpy) -> torch.bfloat16 on the GPU."""
    return torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16).to(dev())


def hbf(t):
    """torch.bfloat16 -> uint16 bf16 bits (numpy)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def di32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev())


def df32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(dev())


def assert_close(got_u16, ref, what, tight=True, magnitude=None, rel_fro=None):
    """Spec tolerance (max-abs <= 2e-2, rel-Frobenius <= 1e-2) and an
    elementwise bound of 2^-8 * magnitude + 1e-3 rms(ref): one bf16 rounding
    plus fp32 summation noise, small enough that any wrong, missing or
    misplaced element fails.  For a sum of rounded bf16 terms pass the sum of
    the terms' magnitudes: each term may already sit one rounding step
    (<= 2^-7 of itself) away, which adds 2^-7 * magnitude to the bound."""
    g = orc.widen_bf16(got_u16)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    if ref.size == 0:
        return
    d = g - ref
    ma = float(np.abs(d).max())
    nrm = float(np.linalg.norm(ref))
    rf = float(np.linalg.norm(d)) / nrm if nrm > 0 else float(np.linalg.norm(d))
    assert np.isfinite(g).all(), "%s: non-finite output" % what
    assert ma <= MAX_ABS, "%s: max-abs error %.4g" % (what, ma)
    # rel_fro: the limit for an output whose arithmetic is not fp32 accumulation
    # (the caller derives it from that arithmetic); default the spec limit
    lim = REL_FRO if rel_fro is None else rel_fro
    assert rf <= lim, "%s: rel-Frobenius error %.4g (limit %.4g)" % (what, rf, lim)
    if tight:
        rms = float(np.sqrt(np.mean(ref * ref)))
        bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms + 1e-30
        if magnitude is not None:
            # each rounded term may sit one bf16 step (<= 2^-7 of itself) away
            bound = bound + 2.0 ** -7 * magnitude
        bad = np.argwhere(np.abs(d) > bound)
        assert bad.size == 0, "%s: %d elements off, first %s got %r ref %r" % (
            what, len(bad), bad[0].tolist(), g[tuple(bad[0])], ref[tuple(bad[0])])


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device=dev())


def status_of(st):
    torch.cuda.synchronize()
    return int(st.item())
