"""Seeded synthetic inputs for the MoE grouped GEMM workloads.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds only input generation (random tensors, router top-k choices);
none of the grouped-GEMM arithmetic lives here.  It imports nothing else from
the package, so loading it never loads the CUDA library.

Random streams: every tensor comes from its own ``numpy.random.Generator``
(PCG64) seeded by ``SeedSequence([seed, crc32(name), block])``, generated in
row blocks so that any block can be regenerated alone.  fp32 samples are
rounded to bf16 (ties to even); bf16 tensors are carried as uint16 bit
patterns on the host.
"""
from __future__ import annotations

import dataclasses
import os
import zlib
from concurrent.futures import ThreadPoolExecutor

import numpy as np

BLOCK_ROWS = 4096  # rows per independently seeded block


def _gen(seed: int, name: str, block: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), zlib.crc32(name.encode()), int(block)])
    return np.random.Generator(np.random.PCG64(ss))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(
        np.float32)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_bf16(seed: int, name: str, shape, std: float) -> np.ndarray:
    """bf16 tensor ~ N(0, std^2), generated in blocks of BLOCK_ROWS leading rows
    (the last dimension is the contiguous one)."""
    shape = tuple(int(s) for s in shape)
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    cols = shape[-1]
    out = np.empty((rows, cols), np.uint16)
    nblk = (rows + BLOCK_ROWS - 1) // BLOCK_ROWS

    def fill(b):
        lo, hi = b * BLOCK_ROWS, min(rows, (b + 1) * BLOCK_ROWS)
        g = _gen(seed, name, b)
        x = g.standard_normal((hi - lo, cols), dtype=np.float32)
        x *= np.float32(std)
        out[lo:hi] = f32_to_bf16_bits(x)

    if nblk == 1:
        fill(0)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(fill, range(nblk)))
    return out.reshape(shape)


# ------------------------------------------------------------------ router --

def topk_softmax_route(logits: np.ndarray, topk: int):
    """Router stand-in: softmax over experts, top-k (ties to the lower expert
    id), weights renormalised to sum to 1 over the chosen k (fp32)."""
    logits = logits.astype(np.float64)
    z = logits - logits.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    order = np.argsort(-p, axis=1, kind="stable")[:, :topk]
    ids = order.astype(np.int32)
    w = np.take_along_axis(p, order, axis=1)
    w = w / w.sum(axis=1, keepdims=True)
    return ids, w.astype(np.float32)


def zipf_route(seed: int, T: int, topk: int, E: int, s: float = 1.2, n_empty: int = 4):
    """Skewed routing: each slot's expert drawn iid from a Zipf(s) law over
    ranks 1..E-n_empty; n_empty experts get probability 0; rank -> expert id
    through a seeded permutation.  Weights: uniform(0.5, 1.5) renormalised."""
    g = _gen(seed, "zipf_route", 0)
    perm = g.permutation(E)
    ranks = np.arange(1, E - n_empty + 1, dtype=np.float64)
    p = ranks ** (-s)
    p /= p.sum()
    draws = g.choice(E - n_empty, size=(T, topk), p=p)
    ids = perm[draws].astype(np.int32)
    w = g.uniform(0.5, 1.5, size=(T, topk))
    w = (w / w.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, w


# ----------------------------------------------------------------- configs --

@dataclasses.dataclass(frozen=True)
class MoEConfig:
    """One MoE layer workload.  GEMM1 (gate_up) maps hidden K -> N1 with the
    token gather; GEMM2 (down) maps I -> K with the scatter back to token
    order.  For a single-GEMM workload N2 == 0."""
    name: str
    T: int
    topk: int
    E: int
    K: int          # hidden size (GEMM1 reduction, GEMM2 output)
    N1: int         # GEMM1 output width
    I: int          # GEMM2 reduction width (0: single GEMM)
    routing: str    # "softmax_normal" | "softmax_uniform" | "softmax_normal_biased" | "zipf"
    seed: int = 0
    std: float = 0.02

    @property
    def R(self) -> int:
        return self.T * self.topk

    def gemm_flops_fwd(self) -> float:
        f = 2.0 * self.R * self.N1 * self.K
        if self.I:
            f += 2.0 * self.R * self.K * self.I
        return f


TINY = MoEConfig("tiny", T=64, topk=2, E=4, K=128, N1=256, I=128, routing="softmax_normal")
MLP8 = MoEConfig("mlp8", T=8192, topk=2, E=8, K=4096, N1=2 * 14336, I=14336,
                 routing="softmax_uniform")
FINE128 = MoEConfig("fine128", T=16384, topk=8, E=128, K=2048, N1=2 * 768, I=768,
                    routing="softmax_normal_biased")
ZIPF64 = MoEConfig("zipf64", T=32768, topk=4, E=64, K=4096, N1=1024, I=0, routing="zipf")

CONFIGS = {c.name: c for c in (TINY, MLP8, FINE128, ZIPF64)}


def route_choices(cfg: MoEConfig):
    """Expert ids int32 [T, topk] and weights fp32 [T, topk] for a config."""
    g = _gen(cfg.seed, "router", 0)
    if cfg.routing == "softmax_normal":
        logits = g.standard_normal((cfg.T, cfg.E))
    elif cfg.routing == "softmax_uniform":
        logits = g.random((cfg.T, cfg.E))
    elif cfg.routing == "softmax_normal_biased":
        logits = g.standard_normal((cfg.T, cfg.E))
        pick = _gen(cfg.seed, "router_bias", 0).permutation(cfg.E)[:8]
        bias = np.zeros(cfg.E)
        bias[pick[:4]] = -1e9   # never chosen: empty experts
        bias[pick[4:]] = -3.0   # rarely chosen: few tokens
        logits = logits + bias
    elif cfg.routing == "zipf":
        return zipf_route(cfg.seed, cfg.T, cfg.topk, cfg.E)
    else:
        raise ValueError(cfg.routing)
    return topk_softmax_route(logits, cfg.topk)


def moe_tensors(cfg: MoEConfig, which=("X", "W1", "W2", "A2", "G", "dH")) -> dict:
    """Seeded bf16 tensors of a config (uint16 bits):
      X   [T, K]        token hidden states
      W1  [E, N1, K]    GEMM1 weights (E, N, K), K contiguous
      W2  [E, K, I]     GEMM2 weights
      A2  [R, I]        GEMM2 input in expert order (stands in for act(GEMM1))
      G   [T, K]        gradient of the layer output (after the top-k combine)
      dY2 [R, K]        gradient of GEMM2's token-major output (on request)
      dH  [R, N1]       gradient of GEMM1's expert-order output
    Backward gradients use the same std (keeps dW magnitudes O(0.1))."""
    out = {}
    s, c = cfg.std, cfg
    shapes = {
        "X": (c.T, c.K),
        "W1": (c.E, c.N1, c.K),
        "W2": (c.E, c.K, c.I) if c.I else None,
        "A2": (c.R, c.I) if c.I else None,
        "dY2": (c.R, c.K) if c.I else None,
        "G": (c.T, c.K) if c.I else None,
        "dH": (c.R, c.N1),
    }
    for name in which:
        shp = shapes[name]
        if shp is None:
            continue
        out[name] = normal_bf16(c.seed, c.name + "/" + name, shp, s)
    return out


@dataclasses.dataclass(frozen=True)
class DualConfig:
    m0: int = 512
    m1: int = 256
    k: int = 1024
    n0: int = 2048
    n1: int = 4096
    seed: int = 0


DUAL = DualConfig()


def dual_tensors(cfg: DualConfig, trans_a: bool = False, trans_b: bool = False) -> dict:
    """X0 [m0,k], X1 [m1,k], W0 [k,n0], W1 [k,n1] ~ N(0,1)/sqrt(k); with trans_a
    the inputs are stored transposed ([k,m]), with trans_b the weights ([n,k])."""
    std = 1.0 / np.sqrt(cfg.k)
    tag = "dual/%d_%d_%d_%d_%d" % (cfg.m0, cfg.m1, cfg.k, cfg.n0, cfg.n1)
    X0 = normal_bf16(cfg.seed, tag + "/X0", (cfg.m0, cfg.k), std)
    X1 = normal_bf16(cfg.seed, tag + "/X1", (cfg.m1, cfg.k), std)
    W0 = normal_bf16(cfg.seed, tag + "/W0", (cfg.k, cfg.n0), std)
    W1 = normal_bf16(cfg.seed, tag + "/W1", (cfg.k, cfg.n1), std)
    if trans_a:
        X0, X1 = np.ascontiguousarray(X0.T), np.ascontiguousarray(X1.T)
    if trans_b:
        W0, W1 = np.ascontiguousarray(W0.T), np.ascontiguousarray(W1.T)
    return dict(X0=X0, X1=X1, W0=W0, W1=W1)
