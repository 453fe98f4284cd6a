"""Benchmark: one MoE layer forward + backward through the grouped-GEMM path.

A step is one pass of the whole hot path over one batch of synthetic input
(configuration "mlp8": T=8192 tokens, hidden 4096, expert intermediate 14336
(gate_up N = 28672), E=8 experts, top-2):
    route          gg_route_hist_offsets   histogram, offsets, stable permutation
    permute        gg_permute              X -> expert order (Xp)
    GEMM1 fwd      gg_forward_swiglu       Xp (dense TMA operands) -> H, and the fused
                                           SwiGLU A = silu(gate) * up (interleaved columns)
    GEMM2 fwd      gg_forward              A, permute_y (scatter to token order fused)
    combine        gg_unpermute_combine    weighted top-k combine -> [T, hidden]
    combine bwd    gg_unpermute_combine_bwd  dY2 = w * G in token-slot order, and the
                                           routing-weight gradient dw
    permute        gg_permute              dY2 (token-slot order) -> expert order
    GEMM2 bwd      gg_backward_dX -> dA, gg_backward_dW on the expert-ordered dY2
    SwiGLU bwd     gg_swiglu_bwd           dH from H and dA
    GEMM1 bwd      gg_backward_dX (permute_x scatter store + top-k token sum),
                   gg_backward_dW on Xp
Materialising the expert-ordered operands once (about 0.03-0.05 ms each) lets
every GEMM read dense TMA tiles; the fused-gather variants of the same calls
compute the same values (tests) and are timed separately under "variants".
The seeded inputs are the tokens X, the layer-output gradient G, the weights
and the router's choices; every other tensor is computed in the step; FLOPs counted are 2*R*N*K per GEMM pass (6
passes), padding rows not counted.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gg|reference]
Prints ONE JSON line (rank 0).  --only PASS times one GEMM pass alone (profiling aid);
--suite times the other workloads (fine128, zipf64, the dual GEMM and its sweep).  Under torchrun every rank runs an independent
replica of the layer on its own GPU (weak scaling, no collective on the data
path); value = FLOPs of all ranks / max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "grouped-GEMM fwd+bwd TFLOP/s and % of bf16 tensor peak; permute GB/s vs HBM"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as fh:
                d = json.load(fh)
            return d, "measured"
        except Exception:
            pass
    return dict(FALLBACK_PEAKS), "fallback"


def _peak_value(d, keys, default):
    for k in keys:
        v = d.get(k)
        if isinstance(v, (int, float)) and v > 0:
            return float(v)
        if isinstance(v, dict):
            for kk in ("value", "peak", "tflops", "gbs"):
                if isinstance(v.get(kk), (int, float)):
                    return float(v[kk])
    return default


def engine_code_sha():
    """sha256 of the GEMM engine's code (common.cuh and gemm_engine.cuh with
    comments and blank lines removed): a comment edit keeps it, any code change
    does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("common.cuh", "gemm_engine.cuh"):
        with open(os.path.join(ROOT, "unpermute_route_hist_gb300", "csrc", name)) as fh:
            src = fh.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update("\n".join(ln.rstrip() for ln in src.splitlines() if ln.strip()).encode())
    return h.hexdigest()


def _roofline_traffic():
    """Per-launch DRAM bytes of the roofline kernel from the committed ncu
    summary, or None once the engine's code differs from the captured one."""
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    try:
        kv = {}
        with open(path) as fh:
            for line in fh:
                if "=" in line and not line.startswith("#"):
                    k, v = (x.strip() for x in line.split("=", 1))
                    kv[k] = v
        if not engine_code_sha().startswith(kv["engine_code_sha256_prefix"]):
            return None
        return int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])
    except Exception:
        return None


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_step_time(ms_local: float, flops_per_rank: float, world_size: int, dist=None,
                        device=None):
    """Whole-job timing of independent replicas: the slowest rank's time, and
    throughput = all ranks' FLOPs / that time (TFLOP/s).  Returns (ms, value)."""
    ms = float(ms_local)
    if world_size > 1 and dist is not None:
        import torch
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    return ms, flops_per_rank * world_size / (ms * 1e-3) / 1e12


def _gemm_passes(cfg):
    R, K, N1, I = cfg.R, cfg.K, cfg.N1, cfg.I
    f1 = 2.0 * R * N1 * K
    f2 = 2.0 * R * K * I
    return {"fwd1": f1, "fwd2": f2, "dX2": f2, "dW2": f2, "dX1": f1, "dW1": f1}


# --------------------------------------------------------------- CPU oracle --

def oracle_sample(cfg, host, ro, rows_per_pass, rng):
    """Time the oracle as it stands on a bounded sample of the step: a few
    expert-order rows of every GEMM pass (plus the full route).  Returns
    (seconds, flops, description)."""
    from oracle import oracle as orc
    t0 = time.perf_counter()
    orc.route(host["ids"], cfg.T, cfg.topk, cfg.E)
    flops = 0.0
    R = cfg.R
    rows = np.sort(rng.choice(R, size=rows_per_pass, replace=False)).astype(np.int64)
    # GEMM1 forward (gather), GEMM2 forward (scatter)
    orc.forward_rows(host["X"], host["W1"], ro["m_sizes"], ro["gather_idx"], host["w"], cfg.topk,
                     1, 0, 0, rows)
    flops += rows.size * 2.0 * cfg.N1 * cfg.K
    orc.forward_rows(host["A2"], host["W2"], ro["m_sizes"], ro["gather_idx"], host["w"], cfg.topk,
                     0, 1, 0, rows)
    flops += rows.size * 2.0 * cfg.K * cfg.I
    # combine backward (the whole tensor): dY2 = w * G in token-slot order
    dY2 = orc.round_bf16(orc.unpermute_combine_bwd(host["G"], None, None, host["w"], cfg.T, cfg.topk,
                                                   want_dw=False)[0])
    orc.backward_dX_rows(dY2, host["W2"], ro["m_sizes"], ro["gather_idx"], 0, 1, rows)
    flops += rows.size * 2.0 * cfg.K * cfg.I
    orc.backward_dX_rows(host["dH"], host["W1"], ro["m_sizes"], ro["gather_idx"], 1, 0, rows)
    flops += rows.size * 2.0 * cfg.N1 * cfg.K
    # dW rows: row n of dW[e] reduces over all m_e rows of expert e
    es = rng.integers(0, cfg.E, size=max(1, rows_per_pass // 4)).astype(np.int32)
    es = np.array([e for e in es if ro["m_sizes"][e] > 0] or [int(np.argmax(ro["m_sizes"]))], np.int32)
    ns2 = rng.integers(0, cfg.K, size=es.size).astype(np.int64)
    orc.backward_dW_rows(host["A2"], dY2, ro["m_sizes"], ro["gather_idx"], cfg.topk, 0, 1, es, ns2)
    flops += float(sum(2.0 * ro["m_sizes"][e] * cfg.I for e in es))
    ns1 = rng.integers(0, cfg.N1, size=es.size).astype(np.int64)
    orc.backward_dW_rows(host["X"], host["dH"], ro["m_sizes"], ro["gather_idx"], cfg.topk, 1, 0, es, ns1)
    flops += float(sum(2.0 * ro["m_sizes"][e] * cfg.K for e in es))
    dt = time.perf_counter() - t0
    desc = ("full route + full combine backward + %d expert-order rows of each forward and dX "
            "pass + %d rows of each dW pass, GEMM2 input and GEMM1 output gradient seeded "
            "(oracle, fp64, OpenMP)" % (rows.size, es.size))
    return dt, flops, desc


def oracle_other_workloads():
    """The oracle timed on the other workloads: the tiny layer in full (forward
    with every flag, dX and dW of both GEMMs), the dual GEMM at its stated shape
    in full, and the zipf64 forward on a row sample (its 1.1 TFLOP in full would
    take about half a minute on the host).  TFLOP/s of what each computed."""
    from oracle import oracle as orc
    from unpermute_route_hist_gb300 import synth
    res = {}
    c = synth.TINY
    ids, w = synth.route_choices(c)
    t = synth.moe_tensors(c, ("X", "W1", "W2", "A2", "dH", "dY2"))
    t0 = time.perf_counter()
    ro = orc.route(ids, c.T, c.topk, c.E)
    m, gi = ro["m_sizes"], ro["gather_idx"]
    orc.forward(t["X"], t["W1"], m, gi, w, c.T, c.topk, 1, 1, 1)
    orc.forward(t["A2"], t["W2"], m, gi, w, c.T, c.topk, 0, 1, 1)
    orc.backward_dX(t["dH"], t["W1"], m, gi, c.T, c.topk, 1, 0)
    orc.backward_dW(t["X"], t["dH"], m, gi, c.T, c.topk, 1, 0)
    orc.backward_dX(t["dY2"], t["W2"], m, gi, c.T, c.topk, 0, 1)
    orc.backward_dW(t["A2"], t["dY2"], m, gi, c.T, c.topk, 0, 1)
    dt = time.perf_counter() - t0
    fl = 3.0 * (2.0 * c.R * c.N1 * c.K + 2.0 * c.R * c.K * c.I)
    res["tiny"] = {"seconds": dt, "tflops": fl / dt / 1e12, "sample": "full: route, both GEMMs' forward, dX and dW"}
    d = synth.DUAL
    dt_ = synth.dual_tensors(d)
    t0 = time.perf_counter()
    orc.dual_asym(dt_["X0"], dt_["X1"], dt_["W0"], dt_["W1"])
    dt = time.perf_counter() - t0
    fl = 2.0 * d.k * (d.m0 * d.n0 + d.m1 * d.n1)
    res["dual"] = {"seconds": dt, "tflops": fl / dt / 1e12, "sample": "full, stated shape"}
    c = synth.ZIPF64
    ids, w = synth.route_choices(c)
    t = synth.moe_tensors(c, ("X", "W1"))
    ro = orc.route(ids, c.T, c.topk, c.E)
    rows = np.sort(np.random.default_rng(3).choice(c.R, size=2048, replace=False)).astype(np.int64)
    t0 = time.perf_counter()
    orc.forward_rows(t["X"], t["W1"], ro["m_sizes"], ro["gather_idx"], None, c.topk, 1, 0, 0, rows)
    dt = time.perf_counter() - t0
    fl = rows.size * 2.0 * c.N1 * c.K
    res["zipf64_forward"] = {"seconds": dt, "tflops": fl / dt / 1e12,
                             "sample": "%d of %d expert-order rows (full forward: about %.0f s at this rate)"
                                       % (rows.size, c.R, 2.0 * c.R * c.N1 * c.K / (fl / dt))}
    return res


def make_host(cfg, which=("X", "W1", "W2", "G")):
    from unpermute_route_hist_gb300 import synth
    ids, w = synth.route_choices(cfg)
    host = synth.moe_tensors(cfg, which)
    host["ids"], host["w"] = ids, w
    return host


def add_oracle_operands(cfg, host):
    """Seeded stand-ins for the GEMM2 input and GEMM1's output gradient, so the
    oracle's row sample does not have to compute every row of the chain that
    produces them on the GPU (same shapes, so the same work per row)."""
    from unpermute_route_hist_gb300 import synth
    host.update(synth.moe_tensors(cfg, ("A2", "dH")))


def run_reference(args, cfg):
    """The reference arm: the CPU oracle as it stands, a bounded sample per step."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from oracle import oracle as orc
    orc.build()
    host = make_host(cfg)
    add_oracle_operands(cfg, host)
    ro = orc.route(host["ids"], cfg.T, cfg.topk, cfg.E)
    rng = np.random.default_rng(1234)
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle_sample(cfg, host, ro, rows, rng)
    times, flops, desc = [], 0.0, ""
    for _ in range(args.steps):
        dt, fl, desc = oracle_sample(cfg, host, ro, rows, rng)
        times.append(dt)
        flops += fl
    total = sum(times)
    value = flops / total / 1e12
    cores = orc.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": _config_dict(cfg, ws),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _config_dict(cfg, ws):
    return {"workload": "MoE layer fwd+bwd, %s: T=%d, hidden K=%d, gate_up N=%d, down I=%d, E=%d, "
                        "topk=%d, bf16, %s routing" % (cfg.name, cfg.T, cfg.K, cfg.N1, cfg.I, cfg.E,
                                                       cfg.topk, cfg.routing),
            "tokens_per_gpu": cfg.T, "experts": cfg.E, "topk": cfg.topk,
            "parallelism": "replicas" if ws > 1 else "single",
            "l2": "inputs larger than L2 (weights 2.6 GiB, activations > 1 GiB per step)"}


# ----------------------------------------------------------------- GPU arm --

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, mx, reasons = [], 0, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as fh:
            for line in fh:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx = max(mx, float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names[1:], parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def run_gg(args, cfg):
    import torch
    import torch.distributed as dist

    import unpermute_route_hist_gb300 as gg
    from unpermute_route_hist_gb300 import _lib

    ws, rank, local = _dist()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    _lib.load()

    host = make_host(cfg)
    T, k, E, K, N1, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.I, cfg.R

    def to_dev(u16):
        return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16).to(dev)

    def pinned(u16):
        t = torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16)
        return t.pin_memory()

    W1, W2 = to_dev(host["W1"]), to_dev(host["W2"])
    inputs_host = {"X": host["X"], "G": host["G"]}
    d = {n: to_dev(v) for n, v in inputs_host.items()}
    ids = torch.from_numpy(host["ids"]).to(dev)
    wts = torch.from_numpy(host["w"]).to(dev)
    bf = torch.bfloat16
    o = {
        "m_sizes": torch.empty(E, dtype=torch.int32, device=dev),
        "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "gather_idx": torch.empty(R, dtype=torch.int32, device=dev),
        "row_id_map": torch.empty(R, dtype=torch.int32, device=dev),
    }
    ws_buf = torch.empty(gg.route_workspace_size(T, k, E), dtype=torch.uint8, device=dev)
    Xp = torch.empty(R, K, dtype=bf, device=dev)
    H = torch.empty(R, N1, dtype=bf, device=dev)
    Y2 = torch.empty(R, K, dtype=bf, device=dev)
    out = torch.empty(T, K, dtype=bf, device=dev)
    dA2 = torch.empty(R, I, dtype=bf, device=dev)
    dW2 = torch.empty(E, K, I, dtype=bf, device=dev)
    dX1 = torch.empty(R, K, dtype=bf, device=dev)
    dXt = torch.empty(T, K, dtype=bf, device=dev)
    dW1 = torch.empty(E, N1, K, dtype=bf, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    passes = _gemm_passes(cfg)
    step_flops = sum(passes.values())

    ev_names = ["route", "permute", "fwd1", "fwd2", "combine", "combine_bwd", "permute_dY", "dX2",
                "dW2", "swiglu_bwd", "dX1", "dW1"]
    A2 = torch.empty(R, I, dtype=bf, device=dev)
    dH = torch.empty(R, N1, dtype=bf, device=dev)
    dYp = torch.empty(R, K, dtype=bf, device=dev)
    dY2 = torch.empty(R, K, dtype=bf, device=dev)
    dwt = torch.empty(T, k, dtype=torch.float32, device=dev)

    def step(src, evs=None, res=None):
        # res: the step's two [T, K] results (layer output and input gradient)
        res_out = out if res is None else res["out"]
        res_dxt = dXt if res is None else res["dXt"]

        def mark(i):
            if evs is not None:
                evs[i].record()
        mark(0)
        r = gg.route_hist_offsets(src["ids"], E, 0, workspace=ws_buf, status=status, outs=o)
        mark(1)
        gg.permute(src["X"], r["row_id_map"], k, out=Xp, status=status)
        mark(2)
        gg.forward_swiglu(Xp, W1, r["m_sizes"], r["gather_idx"], k, False, out=H, out_act=A2,
                          status=status)
        mark(3)
        gg.forward(A2, W2, r["m_sizes"], r["gather_idx"], None, k, False, True, False, out=Y2,
                   status=status)
        mark(4)
        gg.unpermute_combine(Y2, None, src["w"], T, k, out=res_out, status=status)
        mark(5)
        # backward of the combine: dY2 in token-slot order (the forward scattered
        # with permute_y) and the routing-weight gradient
        gg.unpermute_combine_bwd(src["G"], Y2, None, src["w"], T, k, out=dY2, out_dw=dwt,
                                 status=status)
        mark(6)
        gg.permute(dY2, r["row_id_map"], 1, out=dYp, status=status)
        mark(7)
        gg.backward_dX(dYp, W2, r["m_sizes"], r["gather_idx"], T, k, False, False, out=dA2,
                       status=status)
        mark(8)
        gg.backward_dW(A2, dYp, r["m_sizes"], r["gather_idx"], T, k, False, False,
                       out=dW2, status=status)
        mark(9)
        gg.swiglu_bwd(H, dA2, out=dH)
        mark(10)
        gg.backward_dX(dH, W1, r["m_sizes"], r["gather_idx"], T, k, True, False,
                       token_sum=True, out=dX1, out_tok=res_dxt, status=status)
        mark(11)
        gg.backward_dW(Xp, dH, r["m_sizes"], r["gather_idx"], T, k, False, False, out=dW1,
                       status=status)
        mark(12)

    # route(4) permute fwd fwd combine combine-bwd permute dX dW swiglu-bwd dX(+token sum) dW
    launches_per_step = 4 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 1 + 2 + 1
    src = dict(d, ids=ids, w=wts)
    for _ in range(max(args.warmup, 3)):
        step(src)
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d: %s" % (int(status.item()),
                                                      _lib.device_status_string(int(status.item()))))

    # ---- timed region: inputs resident in HBM --------------------------------
    stream = torch.cuda.current_stream(dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(ev_names) + 1)]
           for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks(local)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for s in range(args.steps):
        step(src, evs[s])
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if ws > 1:
        dist.barrier()
    ms_total = t_start.elapsed_time(t_end)
    per = {n: 0.0 for n in ev_names}
    for s in range(args.steps):
        for i, n in enumerate(ev_names):
            per[n] += evs[s][i].elapsed_time(evs[s][i + 1])
    per = {n: v / args.steps for n, v in per.items()}
    ms_step, value = aggregate_step_time(ms_total / args.steps, step_flops, ws,
                                         dist if ws > 1 else None, dev)

    # ---- end to end through the public API with host buffers ------------------
    # Every step uploads its inputs from pinned host memory and reads its two
    # [T, K] results back.  Two buffer sets and one copy stream per direction let
    # step i+1's upload and step i's download run while the GPU computes (and at
    # the same time as each other: the link carries both directions at once);
    # the timed region runs from the first upload to the last download.
    pin = {n: pinned(v) for n, v in inputs_host.items()}
    pin_ids = torch.from_numpy(host["ids"]).pin_memory()
    pin_w = torch.from_numpy(host["w"]).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in pin.values()) + pin_ids.numel() * 4 + pin_w.numel() * 4
    d2h = 2 * T * K * 2
    # as many steps as the device-timed region: both are sustained under the power cap
    e_steps = max(2, args.steps)
    up_stream, down_stream = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    srcs = [src, {n: torch.empty_like(v) for n, v in src.items()}]
    resd = [{"out": out, "dXt": dXt}, {"out": torch.empty_like(out), "dXt": torch.empty_like(dXt)}]
    res_host = [[torch.empty(T, K, dtype=bf).pin_memory() for _ in range(2)] for _ in range(2)]
    h2d_ev = [torch.cuda.Event() for _ in range(2)]
    comp_ev = [torch.cuda.Event() for _ in range(2)]
    d2h_ev = [torch.cuda.Event() for _ in range(2)]
    # copy durations (timed events around each copy; reported as a diagnostic)
    cp_ev = {"h2d": [], "d2h": []}

    def timed_copy(kind, strm, fn):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(strm)
        fn()
        b_.record(strm)
        cp_ev[kind].append((a, b_))

    def upload(b):
        with torch.cuda.stream(up_stream):
            def go():
                for n in pin:
                    srcs[b][n].copy_(pin[n], non_blocking=True)
                srcs[b]["ids"].copy_(pin_ids, non_blocking=True)
                srcs[b]["w"].copy_(pin_w, non_blocking=True)
            timed_copy("h2d", up_stream, go)
            h2d_ev[b].record(up_stream)

    def download(b):
        with torch.cuda.stream(down_stream):
            down_stream.wait_event(comp_ev[b])

            def go():
                res_host[b][0].copy_(resd[b]["out"], non_blocking=True)
                res_host[b][1].copy_(resd[b]["dXt"], non_blocking=True)
            timed_copy("d2h", down_stream, go)
            d2h_ev[b].record(down_stream)

    def e2e_run(n, cevs=None):
        upload(0)
        for i in range(n):
            b = i % 2
            stream.wait_event(h2d_ev[b])
            if i >= 2:
                stream.wait_event(d2h_ev[b])  # buffer b's results of step i-2 read back
            if cevs is not None:
                cevs[i][0].record(stream)
            step(srcs[b], res=resd[b])
            if cevs is not None:
                cevs[i][1].record(stream)
            comp_ev[b].record(stream)
            if i + 1 < n:
                if i >= 1:
                    up_stream.wait_event(comp_ev[1 - b])  # step i-1 done with its inputs
                upload(1 - b)
            download(b)

    e2e_run(2)
    torch.cuda.synchronize()
    if ws > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # compute-stream events around each step: their sum is the GPU's compute time,
    # the rest of the region is time the compute stream waited for copies
    cevs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(e_steps)]
    e_clocks = Clocks(local)
    e_clocks.start()
    time.sleep(0.3)
    for v in cp_ev.values():
        v.clear()
    e0.record(up_stream)
    e2e_run(e_steps, cevs)
    e1.record(down_stream)  # after the last download, which follows every step and upload
    torch.cuda.synchronize()
    copy_ms = {k: statistics.median(a.elapsed_time(b_) for a, b_ in v) for k, v in cp_ev.items()}
    e_clk = e_clocks.stop()
    e_compute_ms = sum(a.elapsed_time(b) for a, b in cevs) / e_steps
    e_ms, e_value = aggregate_step_time(e0.elapsed_time(e1) / e_steps, step_flops, ws,
                                        dist if ws > 1 else None, dev)
    if not (torch.equal(res_host[0][0], res_host[1][0]) and torch.equal(res_host[0][1], res_host[1][1])):
        raise RuntimeError("end-to-end steps on the two buffer sets disagree")

    # ---- the same passes with the gather fused into the GEMM (outside the step) -
    def time_call(fn, reps=5):
        # the median of single calls after one warm-up (a mean over back-to-back calls
        # swung by 20% from run to run with the clocks under the power cap)
        fn()
        times = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        return statistics.median(times)

    rr = o
    # workspaces: the larger dW gather copy (dY2 rows, R x K; X rows are R x K too)
    # and the fused combine's fp32 sums
    dw_ws = torch.empty(max(gg.workspace_size(_lib.GG_OP_BACKWARD_DW, T, k, E, K, I, _lib.GG_PERMUTE_Y),
                            gg.workspace_size(_lib.GG_OP_BACKWARD_DW, T, k, E, N1, K, _lib.GG_PERMUTE_X)),
                        dtype=torch.uint8, device=dev)
    comb_ws = torch.empty(gg.workspace_size(_lib.GG_OP_FORWARD_COMBINE, T, k, E, K, I), dtype=torch.uint8,
                          device=dev)
    variants = {
        "fwd1_fused_token_gather": (time_call(lambda: gg.forward(
            src["X"], W1, rr["m_sizes"], rr["gather_idx"], None, k, True, False, False, out=H,
            status=status)), passes["fwd1"]),
        "dX2_fused_slot_gather": (time_call(lambda: gg.backward_dX(
            dY2, W2, rr["m_sizes"], rr["gather_idx"], T, k, False, True, out=dA2,
            status=status)), passes["dX2"]),
        # dW with the slot gather: rows copied into the workspace, then the dense
        # reduction (the library's path when a workspace is given) ...
        "dW2_slot_gather_via_workspace": (time_call(lambda: gg.backward_dW(
            A2, dY2, rr["m_sizes"], rr["gather_idx"], T, k, False, True, out=dW2,
            workspace=dw_ws, status=status)), passes["dW2"]),
        # ... and fused into the reduction's operand loads (no workspace)
        "dW2_slot_gather_fused_in_loads": (time_call(lambda: gg.backward_dW(
            A2, dY2, rr["m_sizes"], rr["gather_idx"], T, k, False, True, out=dW2,
            workspace=False, status=status)), passes["dW2"]),
        # inference form of GEMM2 + combine: the combine fused into the epilogue
        # (atomic adds; the per-slot rows the training step keeps are not stored),
        # summed in an fp32 workspace, or in bf16 in the output
        "fwd2_fused_combine_fp32": (time_call(lambda: gg.forward_combine(
            A2, W2, rr["m_sizes"], rr["gather_idx"], src["w"], k, False, out=out,
            workspace=comb_ws, status=status)), passes["fwd2"]),
        "fwd2_fused_combine_bf16": (time_call(lambda: gg.forward_combine(
            A2, W2, rr["m_sizes"], rr["gather_idx"], src["w"], k, False, out=out,
            workspace=False, status=status)), passes["fwd2"]),
        # dX2 with the SwiGLU backward fused into its epilogue (no dA buffer); the
        # step runs dX2 then gg_swiglu_bwd, which measures faster
        "dX2_fused_swiglu_bwd": (time_call(lambda: gg.backward_dX_swiglu(
            dYp, W2, rr["m_sizes"], k, H, out=dH, status=status)), passes["dX2"]),
        "dW1_token_gather_via_workspace": (time_call(lambda: gg.backward_dW(
            src["X"], dH, rr["m_sizes"], rr["gather_idx"], T, k, True, False, out=dW1,
            workspace=dw_ws, status=status)), passes["dW1"]),
        "dW1_token_gather_fused_in_loads": (time_call(lambda: gg.backward_dW(
            src["X"], dH, rr["m_sizes"], rr["gather_idx"], T, k, True, False, out=dW1,
            workspace=False, status=status), reps=3), passes["dW1"]),
    }
    variants = {n: {"ms": ms, "tflops": fl / (ms * 1e-3) / 1e12} for n, (ms, fl) in variants.items()}

    # ---- HBM-bound movers: GB/s of the timed permute and combine --------------
    perm_bytes = T * K * 2 + R * K * 2 + R * 4
    comb_bytes = R * K * 2 + R * 4 + T * K * 2  # weights R*4 also read
    comb_bytes += R * 4
    permdy_bytes = 2 * R * K * 2 + R * 4
    # combine backward: read G once, write dY2, read Y2 for dw, weights, write dw
    combbwd_bytes = T * K * 2 + R * K * 2 + R * K * 2 + R * 4 + R * 4
    swbwd_bytes = R * N1 * 2 * 2 + R * I * 2  # read H, write dH, read dA

    if int(status.item()) != 0:
        raise RuntimeError("device status %d after the timed region" % int(status.item()))

    if rank == 0:
        peaks, src_kind = _peaks()
        tflops_sus = _peak_value(peaks, ["bf16_tflops_sustained", "bf16_tflops"], 1700.0)
        tflops_burst = _peak_value(peaks, ["bf16_tflops"], 1900.0)
        hbm = _peak_value(peaks, ["hbm_gbs", "hbm_GBs", "hbm"], 6800.0)
        dom = "fwd1"
        achieved = passes[dom] / (per[dom] * 1e-3) / 1e12
        gemm_ms = sum(per[n] for n in passes)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": _config_dict(cfg, ws),
            "roofline": {"bound": "tensor", "kernel": "grouped_gemm_kernel (GEMM1 forward + fused SwiGLU, dense TMA operands)",
                         "achieved": achieved, "peak": tflops_sus, "unit": "TFLOP/s",
                         "frac": achieved / tflops_sus, "peak_source": src_kind + " bf16 sustained",
                         "frac_of_burst_peak": achieved / tflops_burst, "burst_peak": tflops_burst,
                         "traffic": _roofline_traffic(), "traffic_unit": "bytes per launch",
                         "algorithmic_bytes": (R * K + E * N1 * K + R * N1 + R * N1 // 2) * 2},
            "gemm": {"tflops_all_gemm_launches": sum(passes.values()) / (gemm_ms * 1e-3) / 1e12,
                     "frac_of_peak": sum(passes.values()) / (gemm_ms * 1e-3) / 1e12 / tflops_sus,
                     "ms": {n: per[n] for n in passes}},
            "hbm_movers": {"permute_GBps": perm_bytes / (per["permute"] * 1e-3) / 1e9,
                           "permute_dY_GBps": permdy_bytes / (per["permute_dY"] * 1e-3) / 1e9,
                           "combine_bwd_GBps": combbwd_bytes / (per["combine_bwd"] * 1e-3) / 1e9,
                           "swiglu_bwd_GBps": swbwd_bytes / (per["swiglu_bwd"] * 1e-3) / 1e9,
                           "combine_GBps": comb_bytes / (per["combine"] * 1e-3) / 1e9,
                           "peak_GBps": hbm, "peak_source": src_kind,
                           "permute_frac": perm_bytes / (per["permute"] * 1e-3) / 1e9 / hbm,
                           "combine_frac": comb_bytes / (per["combine"] * 1e-3) / 1e9 / hbm,
                           "route_ms": per["route"]},
            "variants": variants,
            "e2e": {"value": e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d),
                    "d2h_bytes_per_step": int(d2h), "ms_per_step": e_ms,
                    "compute_ms_per_step": e_compute_ms, "copy_ms": copy_ms, "steps": e_steps,
                    "clocks": e_clk},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clk,
        }
        if not args.no_suite:
            line["suite"] = measure_suite(dev, tflops_sus, hbm, src_kind)
        if not args.no_cpu_baseline and ws == 1:
            from oracle import oracle as orc
            orc.build()
            add_oracle_operands(cfg, host)
            ro = orc.route(host["ids"], T, k, E)
            rng = np.random.default_rng(99)
            dt, fl, desc = oracle_sample(cfg, host, ro, args.cpu_rows, rng)
            line["cpu_baseline"] = {"value": fl / dt / 1e12, "unit": "TFLOP/s",
                                    "cores": orc.num_threads(), "kind": "oracle", "sample": desc,
                                    "seconds": dt, "other_workloads": oracle_other_workloads()}
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_only(args, cfg):
    """One GEMM pass of the step in isolation, on that pass's own operands only
    (a few GB on the device): the case the profiler captures.  Operands that
    the step computes are seeded random stand-ins of the same shape; the
    routing is the config's.  Prints one diagnostic JSON line (not a bench
    line)."""
    import torch

    import unpermute_route_hist_gb300 as gg
    from unpermute_route_hist_gb300 import _lib, synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    T, k, E, K, N1, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.I, cfg.R
    ids, _ = synth.route_choices(cfg)
    r = gg.route_hist_offsets(torch.from_numpy(ids).to(dev), E)
    m, gi = r["m_sizes"], r["gather_idx"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    bf = torch.bfloat16

    def rnd(*shape):
        return (torch.randn(*shape, device=dev, generator=gen) * 0.02).to(bf)

    name = args.only
    if name == "dual":
        # the two-expert GEMM at its stated shape, L2 flushed before each call
        d = synth.DUAL
        X0, X1 = rnd(d.m0, d.k) * 50, rnd(d.m1, d.k) * 50
        W0, W1 = rnd(d.k, d.n0) * 50, rnd(d.k, d.n1) * 50
        Y0 = torch.empty(d.m0, d.n0, dtype=bf, device=dev)
        Y1 = torch.empty(d.m1, d.n1, dtype=bf, device=dev)
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        flush = torch.empty(2 * l2 // 4, dtype=torch.int32, device=dev)
        for _ in range(max(args.warmup, 1)):
            gg.dual_asym(X0, X1, W0, W1, out0=Y0, out1=Y1)
        times = []
        for _ in range(args.steps):
            flush.fill_(1)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            gg.dual_asym(X0, X1, W0, W1, out0=Y0, out1=Y1)
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        fl = 2.0 * d.k * (d.m0 * d.n0 + d.m1 * d.n1)
        ms = statistics.median(times)
        print(json.dumps({"pass": "dual", "ms": ms, "tflops": fl / (ms * 1e-3) / 1e12,
                          "note": "diagnostic, not a bench line; L2 flushed before each call"}), flush=True)
        return
    if name == "fwd1":
        Xp, W1 = rnd(R, K), rnd(E, N1, K)
        H = torch.empty(R, N1, dtype=bf, device=dev)
        if I:
            A2 = torch.empty(R, I, dtype=bf, device=dev)
            fn = lambda: gg.forward_swiglu(Xp, W1, m, gi, k, False, out=H, out_act=A2)
        else:  # a config without the gated MLP (zipf64): the plain forward
            fn = lambda: gg.forward(Xp, W1, m, gi, None, k, out=H)
    elif name == "fwd2":
        A2, W2 = rnd(R, I), rnd(E, K, I)
        Y2 = torch.empty(R, K, dtype=bf, device=dev)
        fn = lambda: gg.forward(A2, W2, m, gi, None, k, False, True, False, out=Y2)
    elif name == "dX2":
        dYp, W2 = rnd(R, K), rnd(E, K, I)
        dA2 = torch.empty(R, I, dtype=bf, device=dev)
        fn = lambda: gg.backward_dX(dYp, W2, m, gi, T, k, False, False, out=dA2)
    elif name == "dW2":
        A2, dYp = rnd(R, I), rnd(R, K)
        dW2 = torch.empty(E, K, I, dtype=bf, device=dev)
        fn = lambda: gg.backward_dW(A2, dYp, m, gi, T, k, False, False, out=dW2)
    elif name == "dX1":
        dH, W1 = rnd(R, N1), rnd(E, N1, K)
        dX1, dXt = torch.empty(R, K, dtype=bf, device=dev), torch.empty(T, K, dtype=bf, device=dev)
        fn = lambda: gg.backward_dX(dH, W1, m, gi, T, k, True, False, token_sum=True, out=dX1,
                                    out_tok=dXt)
    elif name == "dW1":
        Xp, dH = rnd(R, K), rnd(R, N1)
        dW1 = torch.empty(E, N1, K, dtype=bf, device=dev)
        fn = lambda: gg.backward_dW(Xp, dH, m, gi, T, k, False, False, out=dW1)
    else:
        raise SystemExit("unknown pass %r" % name)
    flops = _gemm_passes(cfg)[name]
    for _ in range(max(args.warmup, 1)):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(args.steps):
        fn()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / max(args.steps, 1)
    print(json.dumps({"pass": name, "config": cfg.name, "ms": ms,
                      "tflops": flops / (ms * 1e-3) / 1e12, "note": "diagnostic, not a bench line"}),
          flush=True)


def measure_suite(dev, tflops_sus, hbm_gbs, src_kind):
    """The workloads the layer step does not cover, timed on the device:
      fine128 (E=128, top-8, empty and near-empty experts) and zipf64 (skewed
      routing): every GEMM pass of the config on its own routing (operands that
      a layer step would compute are seeded stand-ins of the same shape), and
      the permute and combine row movers; all operands exceed L2;
      dual: the two-expert GEMM at its stated shape and over the (m0, m1) sweep,
      each rep preceded by a write of a buffer twice the L2 size, so operands
      come from HBM.
    Returns a dict (the bench line's "suite")."""
    import torch

    import unpermute_route_hist_gb300 as gg
    from unpermute_route_hist_gb300 import synth

    gen = torch.Generator(device=dev)
    gen.manual_seed(11)
    bf = torch.bfloat16
    stream = torch.cuda.current_stream(dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 64 << 20) // 4, dtype=torch.int32, device=dev)

    def entry(ms, flops, nbytes):
        # per-pass roofline: algorithmic bytes (operands read once, outputs written
        # once), arithmetic intensity, and the cap min(tensor peak, AI x HBM)
        tf = flops / (ms * 1e-3) / 1e12
        ai = flops / nbytes
        cap = min(tflops_sus, ai * hbm_gbs / 1e3)
        return {"ms": ms, "tflops": tf, "bytes": nbytes, "flop_per_byte": ai, "cap_tflops": cap,
                "frac_of_cap": tf / cap}

    def rnd(*shape, std=0.02):
        return (torch.randn(*shape, device=dev, generator=gen) * std).to(bf)

    def timed(fn, reps=10):
        # back-to-back reps; every operand here is larger than L2
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps

    def timed_flushed(fn, reps=20):
        # median of reps, each after an L2-sized write; the flush keeps the GPU
        # busy while the host enqueues the timed call, so no launch gap is timed
        for _ in range(3):
            fn()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush_buf.fill_(1)
            a.record(stream)
            fn()
            b.record(stream)
        torch.cuda.synchronize()
        return statistics.median(a.elapsed_time(b) for a, b in evs)

    out = {"peak_tflops": tflops_sus, "hbm_gbs": hbm_gbs, "peak_source": src_kind + " bf16 sustained"}
    for cfg in (synth.FINE128, synth.ZIPF64):
        T, k, E, K, N1, I, R = cfg.T, cfg.topk, cfg.E, cfg.K, cfg.N1, cfg.I, cfg.R
        ids_np, w_np = synth.route_choices(cfg)
        ids, wts = torch.from_numpy(ids_np).to(dev), torch.from_numpy(w_np).to(dev)
        r = gg.route_hist_offsets(ids, E)
        m, gi, rim = r["m_sizes"], r["gather_idx"], r["row_id_map"]
        hist = m.cpu().numpy()
        X = rnd(T, K)
        Xp = gg.permute(X, rim, k)
        W1, dH = rnd(E, N1, K), rnd(R, N1)
        H = torch.empty(R, N1, dtype=bf, device=dev)
        res = {}
        # row movers: GB/s of algorithmic bytes
        perm_b = T * K * 2 + R * K * 2 + R * 4
        ms = timed(lambda: gg.permute(X, rim, k, out=Xp))
        res["permute"] = {"ms": ms, "GBps": perm_b / (ms * 1e-3) / 1e9,
                          "frac_of_hbm": perm_b / (ms * 1e-3) / 1e9 / hbm_gbs}
        # bytes: GEMM operands and output (bf16)
        g1 = 2.0 * (R * K + E * N1 * K + R * N1)
        dX1 = torch.empty(R, K, dtype=bf, device=dev)
        dXt = torch.empty(T, K, dtype=bf, device=dev)
        passes = {
            "fwd1": (lambda: gg.forward(Xp, W1, m, gi, None, k, False, False, False, out=H), 2.0 * R * N1 * K, g1),
            # dX1 GEMM with the scatter store to token-slot order
            "dX1": (lambda: gg.backward_dX(dH, W1, m, gi, T, k, True, False, out=dX1), 2.0 * R * N1 * K,
                    2.0 * (R * N1 + E * N1 * K + R * K)),
            "dW1": (lambda: gg.backward_dW(Xp, dH, m, gi, T, k, False, False), 2.0 * R * N1 * K, g1),
        }
        for name, (fn, fl, nb) in passes.items():
            res[name] = entry(timed(fn), fl, nb)
        # dX1's top-k token sum, an HBM-bound pass after the GEMM (R rows read, T
        # written), and the pair as the benchmark step runs it, against the serial
        # roofline of the two: flops / peak + token-sum bytes / HBM
        sum_b = 2.0 * (R * K + T * K)
        ms = timed(lambda: gg.unpermute_combine(dX1, None, None, T, k, out=dXt))
        res["dX1_token_sum"] = {"ms": ms, "GBps": sum_b / (ms * 1e-3) / 1e9,
                                "frac_of_hbm": sum_b / (ms * 1e-3) / 1e9 / hbm_gbs}
        fl1 = 2.0 * R * N1 * K
        ms = timed(lambda: gg.backward_dX(dH, W1, m, gi, T, k, True, False, token_sum=True, out=dX1,
                                          out_tok=dXt))
        serial_ms = fl1 / (tflops_sus * 1e12) * 1e3 + sum_b / (hbm_gbs * 1e9) * 1e3
        res["dX1_with_token_sum"] = {"ms": ms, "tflops": fl1 / (ms * 1e-3) / 1e12,
                                     "serial_cap_tflops": fl1 / (serial_ms * 1e-3) / 1e12,
                                     "frac_of_serial_cap": serial_ms / ms}
        del Xp, W1, dH, H, dX1, dXt
        if I:
            A2, W2, dYp = rnd(R, I), rnd(E, K, I), rnd(R, K)
            Y2 = torch.empty(R, K, dtype=bf, device=dev)
            fl = 2.0 * R * K * I
            g2 = 2.0 * (R * I + E * K * I + R * K)
            for name, fn in (("fwd2", lambda: gg.forward(A2, W2, m, gi, None, k, False, True, False, out=Y2)),
                             ("dX2", lambda: gg.backward_dX(dYp, W2, m, gi, T, k, False, False)),
                             ("dW2", lambda: gg.backward_dW(A2, dYp, m, gi, T, k, False, False))):
                res[name] = entry(timed(fn), fl, g2)
            comb_b = R * K * 2 + R * 4 + R * 4 + T * K * 2
            ms = timed(lambda: gg.unpermute_combine(Y2, None, wts, T, k, out=X))
            res["combine"] = {"ms": ms, "GBps": comb_b / (ms * 1e-3) / 1e9,
                              "frac_of_hbm": comb_b / (ms * 1e-3) / 1e9 / hbm_gbs}
            del A2, W2, dYp, Y2
        gemm = [n for n in res if "cap_tflops" in res[n]]
        tot_ms = sum(res[n]["ms"] for n in gemm)
        tot_fl = 3.0 * (2.0 * R * N1 * K + (2.0 * R * K * I if I else 0.0))
        out[cfg.name] = {
            "passes": res, "gemm_ms": tot_ms, "gemm_tflops": tot_fl / (tot_ms * 1e-3) / 1e12,
            "frac_of_peak": tot_fl / (tot_ms * 1e-3) / 1e12 / tflops_sus,
            "min_frac_of_cap": min(res[n]["frac_of_cap"] for n in gemm),
            "experts_empty": int((hist == 0).sum()),
            "largest_expert_share": float(hist.max() / hist.sum()),
            "workload": "T=%d, K=%d, N1=%d, I=%d, E=%d, topk=%d, %s routing" % (T, K, N1, I, E, k, cfg.routing)}
        del X, ids, wts, r, m, gi, rim
        torch.cuda.empty_cache()

    # Dual GEMM: device time per call, L2 flushed before each rep.
    sweep = {}
    ms_list = [128, 256, 512, 1024, 2048, 4096, 8192]
    kd, n0, n1 = synth.DUAL.k, synth.DUAL.n0, synth.DUAL.n1
    W0, W1 = rnd(kd, n0, std=kd ** -0.5), rnd(kd, n1, std=kd ** -0.5)
    for m0 in ms_list:
        for m1 in ms_list:
            X0, X1 = rnd(m0, kd, std=kd ** -0.5), rnd(m1, kd, std=kd ** -0.5)
            Y0 = torch.empty(m0, n0, dtype=bf, device=dev)
            Y1 = torch.empty(m1, n1, dtype=bf, device=dev)
            fn = lambda: gg.dual_asym(X0, X1, W0, W1, out0=Y0, out1=Y1)
            ms = timed_flushed(fn, reps=9 if (m0, m1) != (synth.DUAL.m0, synth.DUAL.m1) else 30)
            fl = 2.0 * kd * (m0 * n0 + m1 * n1)
            nb = 2.0 * (m0 * kd + m1 * kd + kd * n0 + kd * n1 + m0 * n0 + m1 * n1)
            sweep["%d,%d" % (m0, m1)] = entry(ms, fl, nb)
    del flush_buf
    torch.cuda.empty_cache()
    base = sweep["%d,%d" % (synth.DUAL.m0, synth.DUAL.m1)]
    out["dual"] = {"stated_shape": base, "sweep_m0_m1": sweep,
                   "largest_tflops": max(v["tflops"] for v in sweep.values()),
                   "timing": "device events per call, median of reps, L2 flushed (2x L2 written) before each",
                   "workload": "X0 [m0,%d] X1 [m1,%d] W0 [%d,%d] W1 [%d,%d], stated m0=%d m1=%d; sweep m0,m1 in %s"
                               % (kd, kd, kd, n0, kd, n1, synth.DUAL.m0, synth.DUAL.m1, ms_list)}
    return out


def run_suite(args):
    """--suite: the suite alone, one diagnostic JSON line (not the bench line)."""
    import torch

    from unpermute_route_hist_gb300 import _lib

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    _lib.load()
    peaks, src_kind = _peaks()
    tflops_sus = _peak_value(peaks, ["bf16_tflops_sustained", "bf16_tflops"], 1700.0)
    hbm_gbs = _peak_value(peaks, ["hbm_gbs", "hbm_GBs", "hbm"], 6800.0)
    print(json.dumps({"suite": measure_suite(dev, tflops_sus, hbm_gbs, src_kind),
                      "note": "diagnostic, not a bench line"}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gg", choices=["gg", "reference"])
    ap.add_argument("--config", default="mlp8")
    ap.add_argument("--ref-rows", type=int, default=128,
                    help="oracle rows per pass in each step of the reference arm")
    ap.add_argument("--cpu-rows", type=int, default=640,
                    help="oracle rows per pass in the cpu_baseline sample (about 10 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-suite", action="store_true",
                    help="leave fine128, zipf64 and the dual GEMM out of the bench line")
    ap.add_argument("--only", choices=["fwd1", "fwd2", "dX2", "dW2", "dX1", "dW1", "dual"],
                    help="time one GEMM pass alone on its own operands (for profiling)")
    ap.add_argument("--suite", action="store_true",
                    help="time only fine128, zipf64 and the dual GEMM (a diagnostic line, not the bench line)")
    args = ap.parse_args()
    from unpermute_route_hist_gb300 import synth
    cfg = synth.CONFIGS[args.config]
    if args.suite:
        run_suite(args)
    elif args.only:
        run_only(args, cfg)
    elif args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_gg(args, cfg)


if __name__ == "__main__":
    main()
