"""Benchmark of the PaTH attention forward pass on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference]

One step is one full forward (chunk preparation + attention scan) over one
batch of seeded synthetic inputs of the named workload, inputs resident in
HBM.  With a decoding workload (``--workload decode_t16k_d128``) one step is
one decoding step of every (b, h) at the last position of a full key/value
cache (keys rewritten in place); that line reports GB/s of algorithmic HBM
traffic against the measured copy bandwidth.  With ``--workload bwd_<name>``
one step is the forward and the backward of workload <name> (the pages time
PaTH forward + backward together) and the line reports ms per step;
``--workload bwd_grid`` times forward + backward on every B x T x d row of
the pages' latency table; ``--workload partial_<name>`` times partial PaTH
(r = d/2) beside full PaTH; ``--workload forms_<name>`` times the dense and
the low-rank transition forms (d = 64).  The
JSON line reports issued TFLOP/s (formulas in ``step_flops``), ms per step,
the roofline of the attention kernel (against the measured bf16 burst peak,
the stated spec peak and, for a second-long back-to-back loop, the measured
sustained peak), an end-to-end number through the host-buffer C-ABI entry
with the host link's own copy bandwidth beside it, sampled SM clocks, the
d = 64 (H = 32) and FoX variants of the headline shape, and a CPU-oracle
baseline.  ``--impl reference`` times the fp64 CPU oracle instead, on a
bounded sample of the same workload.  Under torchrun (N > 1) every rank runs
the full workload on its own GPU (independent replicas; weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "PaTH-attn fwd ms & TFLOP/s at B=2,T=16384,H=16,d=128 bf16; % of BF16 peak"
UNIT = "TFLOP/s"
DEFAULT_WORKLOAD = "t16k_d128"
L2_BYTES = 129 * 1024 * 1024


# ------------------------------------------------------------------ FLOP model
def step_flops(B, H, T, d, C=128):
    """Issued FLOPs of one forward, by kernel.

    Per (b, h) with N = ceil(T / C) chunks:
      attention kernel (tensor cores):
        S = Qw kr^T     2 C^2 d * N(N-1)/2     (every off-diagonal chunk pair)
        O += P V        2 C^2 d * N(N+1)/2     (diagonal chunk included)
        Qm += Qw ngt^T  2 C d^2 * (N-1)(N-2)/2 (crossings of chunks 1 .. b-1)
      chunk preparation, per chunk:
        4 Gram blocks 8 C^2 d, U W / kr / ql 6 C^2 d, ngt 2 C d^2,
        U strictLower(W K^T) and the diagonal correction 4 C^3,
        triangular solve C^3 / 3
    """
    N = -(-T // C)
    BH = B * H
    qk = 2 * C * C * d * N * (N - 1) // 2
    pv = 2 * C * C * d * N * (N + 1) // 2
    tr = 2 * C * d * d * (N - 1) * (N - 2) // 2 if N >= 2 else 0
    prep = N * (14 * C * C * d + 2 * C * d * d + 4 * C ** 3 + C ** 3 // 3)
    return {"attn": BH * (qk + pv + tr), "prep": BH * prep,
            "flash_equiv": 2 * BH * T * T * d}


# ------------------------------------------------------------------ helpers
def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p.get("bf16_tflops"), p.get("hbm_gbs"), "measured"
    except Exception:
        return 1900.0, 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            # the timed region starts only once sampling is running
            t0 = time.time()
            while time.time() - t0 < 5.0 and os.path.getsize(self.path) == 0:
                time.sleep(0.01)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def traffic_record():
    """DRAM bytes per attention launch from the committed ncu record, or None
    when the kernel sources have changed since that capture."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "attn_tc_traffic.json")) as f:
            rec = json.load(f)["attn_tc_kernel"]
        h = hashlib.sha256()
        for src in rec["sources"]:
            with open(os.path.join(ROOT, src), "rb") as f:
                h.update(f.read())
        if h.hexdigest() != rec["sources_sha256"]:
            return None
        return rec["dram_bytes_per_launch"]
    except Exception:
        return None


def dist_setup():
    """(rank, world, local_rank); initialises torch.distributed under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(x: float, world: int) -> float:
    """Max of a host float over ranks (identity for one rank)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ CPU oracle
def oracle_sample(wl, budget_s, threads, seed=0):
    """Time the fp64 oracle on a seeded row sample of one (b, h) problem of the
    workload; returns (seconds per unit of row work, description, threads).
    Row i costs i + 1 path steps, so the full workload is sum over rows."""
    import numpy as np
    import torch

    from oracle import path_oracle_fwd
    from seeded_inputs import make_inputs

    one = wl.with_(B=1, H=1)
    x = make_inputs(one)
    f = lambda t: None if t is None else t.float().numpy()
    q, k, v, w, b, lf = (f(x[n]) for n in ("q", "k", "v", "w", "beta", "logf"))
    g = np.random.default_rng(seed)
    rows, units, spent = [], 0, 0.0
    # grow the sample until the time budget is used
    batch = max(threads, 8)
    while spent < budget_s:
        r = g.integers(0, wl.T, size=batch).tolist()
        t0 = time.perf_counter()
        path_oracle_fwd(q, k, v, w, b, lf, x["scale"], rows=r, threads=threads)
        spent += time.perf_counter() - t0
        rows += r
        units += sum(i + 1 for i in r)
    desc = (f"{len(rows)} random query rows of one (b,h) problem of {wl.name}, "
            f"{spent:.1f} s; extrapolated by row cost (i+1) to all B*H*T rows")
    return spent / units, desc


def full_units(wl):
    return wl.B * wl.H * wl.T * (wl.T + 1) // 2


# ------------------------------------------------------------------ decoding
DECODE_METRIC = "PaTH decode step (keys rewritten in place) GB/s at B=2,T=16384,H=16,d=128 bf16"


def decode_bytes(wl):
    """Algorithmic HBM bytes of one decoding step at position T - 1: every
    cached key read and written back (fp32), every cached value read, the
    gate prefixes read (gated only), plus the new token in and out."""
    es = 2 if wl.dtype == "bf16" else 4
    t = wl.T - 1
    per_head = t * wl.d * (4 + 4 + es) + (t * 4 if wl.fox else 0)
    per_head += 5 * wl.d * es + wl.d * (4 + es) + 16  # q k v w in, out, cache row, scalars
    return wl.B * wl.H * per_head


def oracle_decode_sample(wl, budget_s):
    """Seconds per (b, h) decoding step of the fp64 oracle, timed on a sample
    of heads of the workload; returns (seconds per head, description)."""
    import numpy as np

    from oracle import path_oracle_decode_step
    from seeded_inputs import make_decode_inputs

    x = make_decode_inputs(wl.with_(B=1, H=1))
    f = lambda t: None if t is None else t.double().numpy()[0, 0]
    kc0, vc0, lam0 = f(x["kcache"]), f(x["vcache"]), f(x["lamcache"])
    one = {n: f(x[n]) for n in ("q", "k", "v", "w", "beta", "logf")}
    n, spent = 0, 0.0
    while spent < budget_s or n == 0:
        kc, vc = kc0.copy(), vc0.copy()
        lam = None if lam0 is None else lam0.copy()
        t0 = time.perf_counter()
        path_oracle_decode_step(kc, vc, lam, one["q"], one["k"], one["v"], one["w"],
                                float(one["beta"]), None if one["logf"] is None else float(one["logf"]),
                                wl.T - 1, scale=x["scale"])
        spent += time.perf_counter() - t0
        n += 1
    return spent / n, (f"{n} single-head decoding steps at position {wl.T - 1} of {wl.name}, "
                       f"{spent:.1f} s on one core; extrapolated to all B*H heads")


def run_decode(args, wl):
    import torch

    import householder_softmax_attention_gb300 as pa
    from seeded_inputs import make_decode_inputs

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    x = make_decode_inputs(wl, device=dev)
    cache = pa.DecodeCache.wrap(x["kcache"], x["vcache"], x["lamcache"])
    q, k, v, w, beta, logf, scale = (x[n] for n in ("q", "k", "v", "w", "beta", "logf", "scale"))
    pos = torch.full((wl.B,), wl.T - 1, dtype=torch.int32, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty(beta.shape, device=dev, dtype=torch.float32)
    st = torch.cuda.current_stream(dev)

    def step(stream=st):
        pa.path_attn_decode_step(q, k, v, w, beta, logf, cache, pos, wl.T, scale, out=out,
                                 lse=lse, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert pa.path_attn_device_status(local, True) == 0, "a decoding kernel reported an error"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timed(n, run):
        barrier(world)
        torch.cuda.synchronize(dev)
        e0.record(st)
        run(n)
        e1.record(st)
        torch.cuda.synchronize(dev)
        barrier(world)
        return e0.elapsed_time(e1) / n

    # steps are short: capture them in a CUDA graph so that host-side launch
    # cost does not set the pace; the eager loop is reported beside it
    G = max(1, min(args.steps, 50))
    graph = None
    if not args.no_graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(G):
                    step(torch.cuda.current_stream(dev))
            graph.replay()
            torch.cuda.synchronize(dev)
        except Exception as exc:  # capture unsupported: eager loop only
            graph = None
            print(f"decode graph capture failed ({exc}); timing the eager loop", file=sys.stderr)
    n_rep = -(-args.steps // G)
    with ClockSampler(local) as clk:
        eager_ms = timed(args.steps, lambda n: [step() for _ in range(n)])
        ms = timed(n_rep * G, lambda n: [graph.replay() for _ in range(n // G)]) \
            if graph is not None else eager_ms
    ms = reduce_max(ms, world)
    eager_ms = reduce_max(eager_ms, world)
    assert pa.path_attn_device_status(local, True) == 0, "a decoding kernel reported an error"
    nbytes = decode_bytes(wl)
    value = world * nbytes / (ms * 1e-3) / 1e9
    _, hbm, peak_src = _peaks()
    roofline = {"bound": "hbm", "achieved": nbytes / (ms * 1e-3) / 1e9, "peak": hbm,
                "unit": "GB/s", "frac": nbytes / (ms * 1e-3) / 1e9 / hbm,
                "traffic": args.traffic, "kernel": "decode_split_kernel",
                "peak_source": f"{peak_src} copy bandwidth",
                "avg_launch_ms": ms, "algorithmic_bytes": nbytes}

    # end to end through the Python API: the new token from pinned host memory,
    # the step, out and lse back to the host, every step
    hx = {n: x[n].cpu().pin_memory() for n in ("q", "k", "v", "w", "beta") }
    if logf is not None:
        hx["logf"] = logf.cpu().pin_memory()
    dx = {n: torch.empty_like(t, device=dev) for n, t in hx.items()}
    hout = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hlse = torch.empty(beta.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        for n, t in hx.items():
            dx[n].copy_(t, non_blocking=True)
        pa.path_attn_decode_step(dx["q"], dx["k"], dx["v"], dx["w"], dx["beta"], dx.get("logf"),
                                 cache, pos, wl.T, scale, out=out, lse=lse, stream=st)
        hout.copy_(out, non_blocking=True)
        hlse.copy_(lse, non_blocking=True)
        st.synchronize()

    for _ in range(3):
        e2e_step()
    barrier(world)
    t0 = time.perf_counter()
    n_e2e = max(1, args.steps)
    for _ in range(n_e2e):
        e2e_step()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / n_e2e, world)
    h2d = sum(t.numel() * t.element_size() for t in hx.values())
    line = {
        "metric": DECODE_METRIC if wl.name == "decode_t16k_d128" else f"PaTH decode step GB/s, {wl.name}",
        "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": n_rep * G if graph is not None else args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "cuda_graph": graph is not None, "eager_ms_per_step": eager_ms,
        "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "cache_rows": wl.T, "d": wl.d,
                   "fox": wl.fox, "position": wl.T - 1, "parallelism": f"replicas x{world}",
                   "l2": f"cache larger than L2: {nbytes / 2**20:.0f} MiB moved per step"},
        "roofline": roofline,
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": hout.numel() * hout.element_size() + hlse.numel() * 4},
        "gpu_launches": n_rep * G if graph is not None else args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        sec, desc = oracle_decode_sample(wl, min(args.cpu_budget_s, 10.0))
        est = sec * wl.B * wl.H
        line["cpu_baseline"] = {"value": nbytes / est / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": desc, "est_full_step_s": est}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_decode_reference(args, wl):
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    per_step = []
    for s in range(args.warmup + args.steps):
        sec, desc = oracle_decode_sample(wl, min(args.ref_step_s, 2.0))
        if s >= args.warmup:
            per_step.append(sec * wl.B * wl.H)
    est = statistics.median(per_step)
    value = decode_bytes(wl) / est / 1e9
    line = {
        "impl": "reference", "metric": DECODE_METRIC if wl.name == "decode_t16k_d128"
        else f"PaTH decode step GB/s, {wl.name}", "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": est * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "H": wl.H, "cache_rows": wl.T, "d": wl.d},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ producer
def producer_bytes(wl):
    """Algorithmic HBM bytes of one producer step: x read, w and beta written,
    the weights read once."""
    es = 2 if wl.dtype == "bf16" else 4
    BT = wl.B * wl.T
    return (BT * wl.Dm * es + BT * wl.H * wl.d * es + BT * wl.H * 4
            + ((wl.R + wl.H) * wl.Dm + wl.H * wl.d * wl.R) * es + wl.H * wl.d * 12 + wl.H * 4)


def oracle_producer_sample(wl, budget_s):
    """Seconds per token of the fp64 producer oracle, timed on windows of
    consecutive tokens of the workload; returns (seconds per token, text)."""
    import numpy as np

    from oracle.producer import producer_fwd
    from seeded_inputs import make_producer_inputs

    x = make_producer_inputs(wl)
    W = [x[n].double().numpy() for n in ("Wd", "Wu", "cw", "Ub", "bb")]
    xs = x["x"].double().numpy()
    n, spent, t = 0, 0.0, 0
    while spent < budget_s or n == 0:
        win = xs[:1, t:t + 256]
        t0 = time.perf_counter()
        producer_fwd(win, *W, wl.H, wl.d)
        spent += time.perf_counter() - t0
        n += win.shape[1]
        t = (t + 256) % max(1, wl.T - 256)
    return spent / n, f"{n} tokens of {wl.name} in 256-token windows, {spent:.1f} s; per token"


def run_producer(args, wl):
    import torch

    import householder_softmax_attention_gb300 as pa
    from seeded_inputs import make_producer_inputs

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    x = make_producer_inputs(wl, device=dev)
    w = torch.empty((wl.B, wl.H, wl.T, wl.d), device=dev, dtype=x["x"].dtype)
    beta = torch.empty((wl.B, wl.H, wl.T), device=dev, dtype=torch.float32)
    st = torch.cuda.current_stream(dev)
    args_ = [x[n] for n in ("x", "Wd", "Wu", "cw", "Ub", "bb")]

    def step():
        pa.path_producer_fwd(*args_, wl.H, wl.d, w=w, beta=beta, stream=st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0.record(st)
        for _ in range(args.steps):
            step()
        e1.record(st)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, world)
    nbytes = producer_bytes(wl)
    _, hbm, peak_src = _peaks()
    gbs = nbytes / (ms * 1e-3) / 1e9

    hx = x["x"].cpu().pin_memory()
    dx = torch.empty_like(x["x"])
    hw = torch.empty(w.shape, dtype=w.dtype).pin_memory()
    hb = torch.empty(beta.shape, dtype=torch.float32).pin_memory()

    def e2e_step():
        dx.copy_(hx, non_blocking=True)
        pa.path_producer_fwd(dx, *args_[1:], wl.H, wl.d, w=w, beta=beta, stream=st)
        hw.copy_(w, non_blocking=True)
        hb.copy_(beta, non_blocking=True)
        st.synchronize()

    for _ in range(2):
        e2e_step()
    n_e2e = max(1, min(args.steps, 10))
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / n_e2e, world)
    line = {
        "metric": f"PaTH w/beta producer GB/s, {wl.name}", "value": world * gbs, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "Dm": wl.Dm, "H": wl.H, "d": wl.d,
                   "R": wl.R, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {nbytes / 2**20:.0f} MiB moved per step"},
        "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": args.traffic,
                     "kernel": "producer_proj + producer_mix (the whole step)",
                     "peak_source": f"{peak_src} copy bandwidth", "avg_launch_ms": ms,
                     "algorithmic_bytes": nbytes},
        "e2e": {"value": world * nbytes / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": hx.numel() * hx.element_size(),
                "d2h_bytes_per_step": hw.numel() * hw.element_size() + hb.numel() * 4},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        sec, desc = oracle_producer_sample(wl, min(args.cpu_budget_s, 10.0))
        est = sec * wl.B * wl.T
        line["cpu_baseline"] = {"value": nbytes / est / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": desc, "est_full_step_s": est}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_producer_reference(args, wl):
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    per_step = []
    for s in range(args.warmup + args.steps):
        sec, desc = oracle_producer_sample(wl, min(args.ref_step_s, 2.0))
        if s >= args.warmup:
            per_step.append(sec * wl.B * wl.T)
    est = statistics.median(per_step)
    value = producer_bytes(wl) / est / 1e9
    print(json.dumps({
        "impl": "reference", "metric": f"PaTH w/beta producer GB/s, {wl.name}", "value": value,
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "Dm": wl.Dm, "H": wl.H, "d": wl.d,
                   "R": wl.R},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)
    return 0


# ------------------------------------------------------------------ backward
BWD_PAGES_MS = {  # PaTH-triton fwd+bwd latency on the pages (hardware unstated)
    ("t2k_d128"): 17.59, ("t2k_d64"): 11.95, ("t4k_d128_refl"): 21.88, ("t4k_d64_refl"): 16.64,
    ("t16k_d128"): 48.49, ("t16k_d64"): 43.89,
}


def bwd_flops(B, H, T, d, C=128):
    """Issued tensor-core FLOPs of one backward, by phase.  Per (b, h) with
    N = ceil(T / C) chunks, P = N(N-1)/2 chunk pairs, X = (N-1)(N-2)/2
    chunk crossings:
      X walk    X += Xw ngt^T                  2 C d^2 * X
      key pass  S^T, dP^T, dV, dKr per pair    8 C^2 d * P;  dP^T, dV per diagonal 4 C^2 d * N
      G walk    dS Kr per pair, Gw ngt per crossing   2 C^2 d * P + 2 C d^2 * X
      dF        G^T X per crossing             2 C d^2 * X
      chunk pass  30 products of 128-row operands (C x C or C x d), counted once
                  (the kernel issues each as three bf16 products)
    """
    N = -(-T // C)
    P, X = N * (N - 1) // 2, max(N - 1, 0) * max(N - 2, 0) // 2
    BH = B * H
    f = {
        "xwalk": 2 * C * d * d * X,
        "key": 8 * C * C * d * P + 4 * C * C * d * N,
        "gwalk": 2 * C * C * d * P + 2 * C * d * d * X,
        "dF": 2 * C * d * d * X,
        "chunk": N * 30 * 2 * C * C * max(C, d) * min(C, d) // C,
    }
    return {k: BH * v for k, v in f.items()}


def oracle_bwd_sample(wl, budget_s, threads):
    """Seconds of the fp64 oracle's forward + blockwise backward for one
    (b, h) problem of the workload, timed on its first Ts tokens (a causal
    prefix is itself a valid problem) and extrapolated by (T / Ts)^2."""
    import numpy as np

    from oracle import path_oracle_fwd
    from oracle.chunked_bwd import path_chunked_bwd
    from seeded_inputs import make_grad_inputs, make_inputs

    Ts = min(wl.T, 1024)
    one = wl.with_(B=1, H=1, T=Ts)
    x = make_inputs(one)
    gi = make_grad_inputs(one)
    f = lambda t: None if t is None else t[0, 0].double().numpy()
    q, k, v, w, b, lf = (f(x[n]) for n in ("q", "k", "v", "w", "beta", "logf"))
    per, spent = [], 0.0
    while spent < budget_s or not per:
        t0 = time.perf_counter()
        path_oracle_fwd(x["q"][0, 0].float().numpy(), x["k"][0, 0].float().numpy(),
                        x["v"][0, 0].float().numpy(), x["w"][0, 0].float().numpy(),
                        x["beta"][0, 0].numpy(),
                        None if lf is None else x["logf"][0, 0].numpy(), x["scale"],
                        threads=threads)
        path_chunked_bwd(q, k, v, w, b, f(gi["dout"]), 64, logf=lf, scale=x["scale"],
                         dlse=f(gi["dlse"]))
        dt = time.perf_counter() - t0
        spent += dt
        per.append(dt)
    sec = statistics.median(per) * (wl.T / Ts) ** 2
    desc = (f"fp64 oracle forward + blockwise backward of one (b,h) problem of {wl.name} "
            f"on its first {Ts} tokens, {len(per)} runs in {spent:.1f} s; extrapolated by "
            f"(T/{Ts})^2 to a head and by B*H to the workload")
    return sec, desc


def run_bwd(args, wl):
    """One step = the forward and the backward of the workload (the pages time
    PaTH fwd+bwd together); value = ms per step."""
    import torch

    import householder_softmax_attention_gb300 as pa
    from seeded_inputs import make_grad_inputs, make_inputs

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    x = make_inputs(wl, device=dev)
    gi = make_grad_inputs(wl, device=dev)
    q, k, v, w, beta, logf, scale = (x[n] for n in ("q", "k", "v", "w", "beta", "logf", "scale"))
    dout, dlse = gi["dout"], gi["dlse"]
    out = torch.empty_like(q)
    lse = torch.empty(beta.shape, device=dev, dtype=torch.float32)
    grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v), torch.empty_like(w),
             torch.empty_like(beta), torch.empty_like(logf) if logf is not None else None)
    st = torch.cuda.current_stream(dev)

    def step():
        pa.path_attn_fwd(q, k, v, w, beta, logf, scale, out=out, lse=lse, stream=st)
        pa.path_attn_bwd(q, k, v, w, beta, out, lse, dout, logf=logf, scale=scale, dlse=dlse,
                         grads=grads, stream=st)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    assert pa.path_attn_device_status(local, True) == 0, "a kernel wait expired"
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pa.path_attn_timing_enable(True)
    barrier(world)
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        e0.record(st)
        for _ in range(args.steps):
            step()
        e1.record(st)
        torch.cuda.synchronize(dev)
    barrier(world)
    ms = reduce_max(e0.elapsed_time(e1) / args.steps, world)
    prep_ms, attn_ms, fcalls = pa.path_attn_timing_read()
    phases, bcalls = pa.path_attn_bwd_timing_read()
    pa.path_attn_timing_enable(False)
    assert fcalls == args.steps and bcalls == args.steps
    assert pa.path_attn_device_status(local, True) == 0, "a kernel wait expired"
    phase_ms = {n: t / bcalls for n, t in phases.items()}
    fwd_ms = (prep_ms + attn_ms) / fcalls

    ff = step_flops(wl.B, wl.H, wl.T, wl.d)
    bf = bwd_flops(wl.B, wl.H, wl.T, wl.d)
    total = ff["attn"] + ff["prep"] + ff["prep"] + sum(bf.values())  # bwd reruns the prep
    peak, hbm, peak_src = _peaks()
    # dominant backward kernel: the key pass
    key_ms = phase_ms["key"]
    achieved = bf["key"] / (key_ms * 1e-3) / 1e12
    N, C = -(-wl.T // 128), 128
    P = N * (N - 1) // 2
    key_bytes = wl.B * wl.H * (P * (2 * C * wl.d * 2 + C * C * 2 + 2 * C * 4)
                               + N * (2 * C * wl.d * 2 + C * wl.d * 2 + C * wl.d * 4
                                      + 2 * C * C * 4 + C * wl.d * 2))
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": args.traffic, "kernel": "bwd_key_tc_kernel",
                "peak_source": f"{peak_src} bf16 burst", "avg_launch_ms": key_ms,
                "algorithmic_bytes": key_bytes,
                "hbm_frac": key_bytes / (key_ms * 1e-3) / 1e9 / hbm}

    # end to end through the Python API: inputs and upstream gradients from
    # pinned host memory, forward + backward, every gradient back to the host
    names = ("q", "k", "v", "w", "beta") + (("logf",) if logf is not None else ())
    hin = {n: x[n].cpu().pin_memory() for n in names}
    hin["dout"], hin["dlse"] = dout.cpu().pin_memory(), dlse.cpu().pin_memory()
    din = {n: torch.empty_like(t, device=dev) for n, t in hin.items()}
    hgr = [torch.empty(g.shape, dtype=g.dtype).pin_memory() for g in grads if g is not None]

    def e2e_step():
        for n, t in hin.items():
            din[n].copy_(t, non_blocking=True)
        pa.path_attn_fwd(din["q"], din["k"], din["v"], din["w"], din["beta"], din.get("logf"),
                         scale, out=out, lse=lse, stream=st)
        pa.path_attn_bwd(din["q"], din["k"], din["v"], din["w"], din["beta"], out, lse,
                         din["dout"], logf=din.get("logf"), scale=scale, dlse=din["dlse"],
                         grads=grads, stream=st)
        for h, g in zip(hgr, [g for g in grads if g is not None]):
            h.copy_(g, non_blocking=True)
        st.synchronize()

    for _ in range(2):
        e2e_step()
    n_e2e = max(1, min(args.steps, 5))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / n_e2e, world)
    h2d = sum(t.numel() * t.element_size() for t in hin.values())
    d2h = sum(t.numel() * t.element_size() for t in hgr)
    pages = BWD_PAGES_MS.get(wl.name)
    dt = 1 if wl.dtype == "bf16" else 0
    line = {
        "metric": f"PaTH-attn fwd+bwd ms, {wl.name}", "value": ms, "unit": "ms",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": False, "scaling": "weak",
        "vs_baseline": (ms / pages) if pages else None,
        "pages_triton_fwd_bwd_ms": pages, "pages_hardware": "unstated",
        "dtype": "bf16" if wl.dtype == "bf16" else "f32", "data": "synthetic",
        "config": {"workload": "bwd_" + wl.name, "B": wl.B, "H": wl.H, "T": wl.T, "d": wl.d,
                   "fox": wl.fox, "parallelism": f"replicas x{world}",
                   "l2": "inputs and pair buffers larger than L2"},
        "tflops": world * total / (ms * 1e-3) / 1e12,
        "fwd_ms": fwd_ms, "bwd_ms": sum(phase_ms.values()), "bwd_phase_ms": phase_ms,
        "flops_per_step": {"fwd": ff["attn"] + ff["prep"], "bwd": sum(bf.values()) + ff["prep"]},
        "roofline": roofline,
        "e2e": {"value": e2e_ms, "unit": "ms", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * (
            pa.path_attn_launches_per_call(wl.d, dt, logf is not None)
            + pa.path_attn_bwd_launches_per_call(wl.T, wl.d, dt, logf is not None)),
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        sec, desc = oracle_bwd_sample(wl, min(args.cpu_budget_s, 10.0), threads)
        est = sec * wl.B * wl.H
        line["cpu_baseline"] = {"value": est * 1e3, "unit": "ms", "cores": threads,
                                "kind": "oracle", "sample": desc, "est_full_step_s": est}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def run_partial(args, wl):
    """Partial PaTH (transitions on the first r = d/2 coordinates, plain dot
    products on the rest) against full PaTH on the same inputs, timed in one
    process; value = partial ms per step."""
    import torch

    import householder_softmax_attention_gb300 as pa
    from seeded_inputs import make_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pa.load_library()
    st = torch.cuda.current_stream(dev)
    x = make_inputs(wl, device=dev)
    r = wl.d // 2
    g = torch.Generator(device=dev).manual_seed(wl.seed + 5)
    u = torch.randn((wl.B, wl.H, wl.T, r), generator=g, device=dev)
    u = (u / u.norm(dim=-1, keepdim=True).clamp_min(1e-30)).to(x["q"].dtype).contiguous()
    out = torch.empty_like(x["q"])
    lse = torch.empty(x["beta"].shape, device=dev, dtype=torch.float32)

    def full():
        pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["logf"], x["scale"],
                         out=out, lse=lse, stream=st)

    def partial():
        pa.path_attn_fwd_partial(x["q"], x["k"], x["v"], u, x["beta"], x["logf"], x["scale"],
                                 out=out, lse=lse, stream=st)

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize(dev)
        assert pa.path_attn_device_status(0, True) == 0, "a kernel wait expired"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pa.path_attn_timing_enable(True)
        with ClockSampler(0) as clk:
            e0.record(st)
            for _ in range(args.steps):
                fn()
            e1.record(st)
            torch.cuda.synchronize(dev)
        p, a, n = pa.path_attn_timing_read()
        pa.path_attn_timing_enable(False)
        assert pa.path_attn_device_status(0, True) == 0, "a kernel wait expired"
        return {"ms_per_step": e0.elapsed_time(e1) / args.steps, "prep_ms": p / n,
                "attn_ms": a / n, "clocks": clk.summary()}

    tf, tp = timed(full), timed(partial)
    line = {"metric": f"partial PaTH (r = d/2) fwd ms, {wl.name}", "value": tp["ms_per_step"],
            "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": tp["ms_per_step"], "higher_is_better": False, "dtype": wl.dtype,
            "data": "synthetic",
            "config": {"workload": "partial_" + wl.name, "B": wl.B, "H": wl.H, "T": wl.T,
                       "d": wl.d, "r": r, "fox": wl.fox},
            "partial": tp, "full": tf, "speedup_vs_full": tf["ms_per_step"] / tp["ms_per_step"],
            "gpu_launches": args.steps * pa.path_attn_launches_per_call(
                wl.d, 1 if wl.dtype == "bf16" else 0, wl.fox)}
    print(json.dumps(line), flush=True)
    return 0


def run_transition_forms(args, wl):
    """The dense and the low-rank transition forms (d = 64) on the same inputs,
    timed in one process; value = low-rank ms per step."""
    import torch

    import householder_softmax_attention_gb300 as pa

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pa.load_library()
    run = ForwardRun(pa, wl, dev, torch.cuda.current_stream(dev))
    peak, _, _ = _peaks()
    res = {}
    try:
        for name, form in (("dense", 0), ("low_rank", 1), ("dense_again", 0)):
            pa.path_attn_set_transition_form(form)
            res[name] = run.summary(run.timed(args.steps, args.warmup), peak)
    finally:
        pa.path_attn_set_transition_form(0)
    N, C, d = -(-wl.T // 128), 128, wl.d
    X = (N - 1) * (N - 2) // 2
    line = {"metric": f"transition forms, PaTH fwd ms, {wl.name}",
            "value": res["low_rank"]["ms_per_step"], "unit": "ms", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "higher_is_better": False,
            "dtype": wl.dtype, "data": "synthetic", "config": {"workload": "forms_" + wl.name},
            "dense": res["dense"], "low_rank": res["low_rank"], "dense_again": res["dense_again"],
            "transition_flops_per_head": {"dense": 2 * C * d * d * X,
                                          "low_rank": 2 * (2 * C * C * d) * X},
            "attn_ratio_low_rank_over_dense": res["low_rank"]["attn_ms"] / res["dense"]["attn_ms"]}
    print(json.dumps(line), flush=True)
    return 0


# The pages' latency grid (rebuttal, "Efficiency Evaluation": PaTH Triton
# forward + backward, hardware unstated), B x T x d with H = 16 at d = 128 and
# H = 32 at d = 64; plain PaTH (the table's PaTH column).
BWD_GRID = [(16, 2048, 128, 17.59), (16, 2048, 64, 11.95), (8, 4096, 128, 21.88),
            (8, 4096, 64, 16.64), (4, 8192, 128, 30.90), (4, 8192, 64, 26.06),
            (2, 16384, 128, 48.49), (2, 16384, 64, 43.89)]


def run_bwd_grid(args):
    """Forward + backward of every row of the pages' grid, one JSON line with
    a row per configuration (ms per fwd+bwd step, the pages' Triton figure
    beside it as context)."""
    import torch

    import householder_softmax_attention_gb300 as pa
    from seeded_inputs import Workload, make_grad_inputs, make_inputs

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    pa.load_library()
    st = torch.cuda.current_stream(dev)
    rows = []
    for B, T, d, pages in BWD_GRID:
        H = 16 if d == 128 else 32
        wl = Workload(f"t{T // 1024}k_d{d}", B, H, T, d)
        x = make_inputs(wl, device=dev)
        gi = make_grad_inputs(wl, device=dev)
        q, k, v, w, beta, scale = (x[n] for n in ("q", "k", "v", "w", "beta", "scale"))
        out = torch.empty_like(q)
        lse = torch.empty(beta.shape, device=dev, dtype=torch.float32)
        grads = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v),
                 torch.empty_like(w), torch.empty_like(beta), None)

        def fwd():
            pa.path_attn_fwd(q, k, v, w, beta, None, scale, out=out, lse=lse, stream=st)

        def bwd():
            pa.path_attn_bwd(q, k, v, w, beta, out, lse, gi["dout"], scale=scale,
                             dlse=gi["dlse"], grads=grads, stream=st)

        for _ in range(max(args.warmup, 3)):
            fwd()
            bwd()
        torch.cuda.synchronize(dev)
        assert pa.path_attn_device_status(0, True) == 0, "a kernel wait expired"
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        fms, bms = [], []
        for _ in range(args.steps):
            ev[0].record(st)
            fwd()
            ev[1].record(st)
            bwd()
            ev[2].record(st)
            torch.cuda.synchronize(dev)
            fms.append(ev[0].elapsed_time(ev[1]))
            bms.append(ev[1].elapsed_time(ev[2]))
        assert pa.path_attn_device_status(0, True) == 0, "a kernel wait expired"
        fm, bm = statistics.median(fms), statistics.median(bms)
        rows.append({"B": B, "H": H, "T": T, "d": d, "fwd_ms": fm, "bwd_ms": bm,
                     "fwd_bwd_ms": fm + bm, "pages_triton_fwd_bwd_ms": pages,
                     "ratio_to_pages": (fm + bm) / pages})
        print(f"B={B} T={T} d={d} H={H}: fwd {fm:.3f} ms + bwd {bm:.3f} ms = {fm + bm:.3f} ms "
              f"(pages {pages} ms)", file=sys.stderr, flush=True)
        del x, gi, q, k, v, w, beta, out, lse, grads
        torch.cuda.empty_cache()
    line = {"metric": "PaTH-attn fwd+bwd ms over the pages' B x T x d grid", "unit": "ms",
            "value": sum(r["fwd_bwd_ms"] for r in rows), "n_gpus": 1, "steps": args.steps,
            "warmup": max(args.warmup, 3), "higher_is_better": False, "dtype": "bf16",
            "data": "synthetic", "config": {"workload": "bwd_grid"}, "rows": rows,
            "note": "value = sum over the rows; the pages' figures are Triton on unstated hardware"}
    print(json.dumps(line), flush=True)
    return 0


def run_bwd_reference(args, wl):
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    per_step, desc = [], ""
    for _ in range(args.warmup + args.steps):
        sec, desc = oracle_bwd_sample(wl, min(args.ref_step_s, 2.0), threads)
        per_step.append(sec * wl.B * wl.H)
    est = statistics.median(per_step[args.warmup:])
    line = {
        "impl": "reference", "metric": f"PaTH-attn fwd+bwd ms, {wl.name}", "value": est * 1e3,
        "unit": "ms", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": est * 1e3, "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "bwd_" + wl.name, "B": wl.B, "H": wl.H, "T": wl.T, "d": wl.d},
        "cpu_baseline": {"value": est * 1e3, "unit": "ms", "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": est * 1e3, "unit": "ms", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ arms
def run_reference(args, wl, flops):
    rank, world, _ = dist_setup()
    if rank != 0:
        return 0
    threads = os.cpu_count() or 1
    per_step = []
    for s in range(args.warmup + args.steps):
        sec_per_unit, desc = oracle_sample(wl, args.ref_step_s, threads, seed=s)
        if s >= args.warmup:
            per_step.append(sec_per_unit * full_units(wl))
    est = statistics.median(per_step)
    value = (flops["attn"] + flops["prep"]) / est / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": est * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": _config(wl, world),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def _config(wl, world):
    """The workload description both arms print (the reference arm's line
    carries the same config)."""
    es = 2 if wl.dtype == "bf16" else 4
    C = 128 if wl.dtype == "bf16" else 64
    BH, N = wl.B * wl.H, -(-wl.T // C)
    in_bytes = 4 * BH * wl.T * wl.d * es + BH * wl.T * 4 * (2 if wl.fox else 1)
    ws_bytes = BH * N * (C * wl.d * es + C * wl.d * 4 + wl.d * wl.d * es + C * C * 4)
    return {"workload": wl.name, "B": wl.B, "H": wl.H, "T": wl.T, "d": wl.d,
            "fox": wl.fox, "parallelism": f"replicas x{world}",
            "l2": f"inputs larger than L2: {in_bytes / 2**20:.0f} MiB inputs + "
                  f"{ws_bytes / 2**20:.0f} MiB workspace per step"}


# Dense BF16 tensor peak of one GB300 as NVIDIA states it (the stricter
# denominator of the two spec figures in circulation; the other is 2250).
SPEC_BF16_TFLOPS = 2500.0
NOMINAL_BF16_TFLOPS = 2250.0
# Workloads timed beside the headline one in the default run: the d = 64
# variant of the long-context shape (H = 32) and the same shape with the FoX gate.
VARIANTS = ("t16k_d64", "fox_t16k_d128")


def _sustained_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f).get("bf16_tflops_sustained")
    except Exception:
        return None


def _host_placement():
    """Where pinned host buffers can live: this process's CPU set and the
    host's NUMA nodes (read from sysfs; empty where absent)."""
    info = {"cpus": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None}
    try:
        nodes = sorted(n for n in os.listdir("/sys/devices/system/node") if n.startswith("node"))
        info["numa_nodes"] = len(nodes)
        with open("/proc/self/status") as fh:
            for line in fh:
                if line.startswith("Mems_allowed_list"):
                    info["mems_allowed"] = line.split(":", 1)[1].strip()
    except Exception:
        pass
    return info


class ForwardRun:
    """Inputs of one workload resident on the device and the timed forward."""

    def __init__(self, pa, wl, dev, st):
        import torch
        from seeded_inputs import make_inputs
        self.pa, self.wl, self.dev, self.st = pa, wl, dev, st
        self.x = make_inputs(wl, device=dev)
        x = self.x
        self.q = x["q"]
        self.out = torch.empty_like(x["q"])
        self.lse = torch.empty(x["beta"].shape, device=dev, dtype=torch.float32)
        self.flops = step_flops(wl.B, wl.H, wl.T, wl.d)

    def step(self):
        x = self.x
        self.pa.path_attn_fwd(x["q"], x["k"], x["v"], x["w"], x["beta"], x["logf"], x["scale"],
                              out=self.out, lse=self.lse, stream=self.st)

    def timed(self, steps, warmup, world=1, local=0):
        """Device time of `steps` forwards after `warmup`; per-kernel times
        from the library's own events.  Returns a dict."""
        import torch
        pa = self.pa
        for _ in range(warmup):
            self.step()
        torch.cuda.synchronize(self.dev)
        assert pa.path_attn_device_status(local, True) == 0, "a kernel wait expired"
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        pa.path_attn_timing_enable(True)
        barrier(world)
        torch.cuda.synchronize(self.dev)
        with ClockSampler(local) as clk:
            e0.record(self.st)
            for _ in range(steps):
                self.step()
            e1.record(self.st)
            torch.cuda.synchronize(self.dev)
        barrier(world)
        ms = e0.elapsed_time(e1) / steps
        prep_ms, attn_ms, calls = pa.path_attn_timing_read()
        pa.path_attn_timing_enable(False)
        assert calls == steps
        assert pa.path_attn_device_status(local, True) == 0, "a kernel wait expired"
        return {"ms": ms, "prep_ms": prep_ms / calls, "attn_ms": attn_ms / calls,
                "clocks": clk.summary(), "steps": steps}

    def summary(self, t, peak):
        f = self.flops
        total = f["attn"] + f["prep"]
        attn_tf = f["attn"] / (t["attn_ms"] * 1e-3) / 1e12
        return {"workload": self.wl.name, "B": self.wl.B, "H": self.wl.H, "T": self.wl.T,
                "d": self.wl.d, "fox": self.wl.fox, "ms_per_step": t["ms"],
                "tflops": total / (t["ms"] * 1e-3) / 1e12,
                "attn_ms": t["attn_ms"], "attn_tflops": attn_tf,
                "attn_frac_measured": attn_tf / peak, "attn_frac_spec": attn_tf / SPEC_BF16_TFLOPS,
                "prep_ms": t["prep_ms"], "steps": t["steps"], "clocks": t["clocks"]}


def run_gpu(args, wl, flops):
    import torch

    import householder_softmax_attention_gb300 as pa

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.load_library()
    st = torch.cuda.current_stream(dev)
    run = ForwardRun(pa, wl, dev, st)
    x = run.x
    q, beta, logf, scale = x["q"], x["beta"], x["logf"], x["scale"]
    t = run.timed(args.steps, args.warmup, world, local)
    ms_max = reduce_max(t["ms"], world)
    total = flops["attn"] + flops["prep"]
    value = world * total / (ms_max * 1e-3) / 1e12
    in_bytes = sum(a.numel() * a.element_size() for a in (x["q"], x["k"], x["v"], x["w"], beta,
                                                          logf) if a is not None)

    # roofline of the dominant kernel (the attention scan)
    peak, _, peak_src = _peaks()
    sustained = _sustained_peak()
    achieved = flops["attn"] / (t["attn_ms"] * 1e-3) / 1e12
    roofline = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak,
                "traffic": args.traffic if args.traffic is not None else (
                    traffic_record() if wl.name == DEFAULT_WORKLOAD else None),
                "kernel": "attn_tc_kernel", "peak_source": f"{peak_src} bf16 burst",
                "frac_spec": achieved / SPEC_BF16_TFLOPS, "spec_peak": SPEC_BF16_TFLOPS,
                "frac_nominal": achieved / NOMINAL_BF16_TFLOPS,
                "nominal_peak": NOMINAL_BF16_TFLOPS,
                "step_frac": value / world / peak, "step_frac_spec": value / world / SPEC_BF16_TFLOPS,
                "avg_launch_ms": t["attn_ms"], "prep_avg_ms": t["prep_ms"]}

    # the same step back to back for about a second: the sustained regime
    n_sus = max(args.steps, int(math.ceil(args.sustain_s * 1e3 / max(t["ms"], 1e-3))))
    ts = run.timed(n_sus, 1, world, local)
    sus = {"ms_per_step": ts["ms"], "steps": n_sus, "seconds": ts["ms"] * n_sus * 1e-3,
           "value": total / (ts["ms"] * 1e-3) / 1e12, "attn_ms": ts["attn_ms"],
           "prep_ms": ts["prep_ms"], "clocks": ts["clocks"]}
    if sustained:
        sus["step_frac_sustained_peak"] = sus["value"] / sustained
        sus["attn_frac_sustained_peak"] = flops["attn"] / (ts["attn_ms"] * 1e-3) / 1e12 / sustained
        sus["sustained_peak"] = sustained

    # end to end through the host-buffer entry: H2D of the inputs from pinned
    # memory, the forward, D2H of out and lse, every step
    hx = {n: (a.cpu().pin_memory() if torch.is_tensor(a) else a) for n, a in x.items()}
    hout = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    hlse = torch.empty(beta.shape, dtype=torch.float32).pin_memory()

    # the host link on its own: one copy of q in and of out back, best of three
    def copy_gbs(dst, src):
        best = float("inf")
        for _ in range(3):
            c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            c0.record(st)
            dst.copy_(src, non_blocking=True)
            c1.record(st)
            torch.cuda.synchronize(dev)
            best = min(best, c0.elapsed_time(c1))
        return src.numel() * src.element_size() / (best * 1e-3) / 1e9

    h2d_gbs = copy_gbs(run.out, hx["q"])
    d2h_gbs = copy_gbs(hout, run.out)

    def e2e_step():
        pa.path_attn_fwd_host(hx["q"], hx["k"], hx["v"], hx["w"], hx["beta"], hx["logf"],
                              scale, out=hout, lse=hlse, stream=st)

    for _ in range(max(1, min(args.warmup, 3))):
        e2e_step()
    n_e2e = max(1, min(args.steps, 10))
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(n_e2e):
        e2e_step()
    e2e_ms = reduce_max((time.perf_counter() - t0) * 1e3 / n_e2e, world)
    d2h = hout.numel() * hout.element_size() + hlse.numel() * 4
    del hx, hout, hlse

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic",
        "config": _config(wl, world),
        "flops_per_step": {"attn": flops["attn"], "prep": flops["prep"]},
        "flash_equiv_tflops": world * flops["flash_equiv"] / (ms_max * 1e-3) / 1e12,
        "roofline": roofline,
        "sustained": sus,
        "e2e": {"value": world * total / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": d2h,
                "link": {"h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                         "copy_floor_ms": (in_bytes / h2d_gbs + d2h / d2h_gbs) * 1e-6,
                         "host": _host_placement()}},
        "gpu_launches": args.steps * pa.path_attn_launches_per_call(
            wl.d, 1 if wl.dtype == "bf16" else 0, logf is not None),
        "clocks": t["clocks"],
    }
    if wl.name == DEFAULT_WORKLOAD and not args.no_variants:
        from seeded_inputs import WORKLOADS
        del run
        torch.cuda.empty_cache()
        variants = {}
        for name in VARIANTS:
            vr = ForwardRun(pa, WORKLOADS[name], dev, st)
            variants[name] = vr.summary(vr.timed(max(10, min(args.steps, 20)), 3, world, local),
                                        peak)
            del vr
            torch.cuda.empty_cache()
        line["variants"] = variants
    if rank == 0 and not args.no_cpu_baseline:
        threads = os.cpu_count() or 1
        sec_per_unit, desc = oracle_sample(wl, args.cpu_budget_s, threads)
        est = sec_per_unit * full_units(wl)
        line["cpu_baseline"] = {"value": total / est / 1e12, "unit": UNIT, "cores": threads,
                                "kind": "oracle", "sample": desc,
                                "est_full_workload_s": est}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-budget-s", type=float, default=15.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-variants", action="store_true",
                    help="skip the d = 64 and FoX workloads timed beside the headline one")
    ap.add_argument("--sustain-s", type=float, default=1.0,
                    help="seconds of back-to-back steps for the sustained figure")
    ap.add_argument("--no-graph", action="store_true", help="decoding: time the eager loop only")
    ap.add_argument("--B", type=int, default=None, help="override the workload's batch")
    ap.add_argument("--H", type=int, default=None, help="override the workload's heads")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention launch from an ncu capture, if current")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    from seeded_inputs import DECODE_WORKLOADS, PRODUCER_WORKLOADS, WORKLOADS
    if args.workload in PRODUCER_WORKLOADS:
        wl = PRODUCER_WORKLOADS[args.workload]
        return run_producer_reference(args, wl) if args.impl == "reference" else run_producer(args, wl)
    if args.workload in DECODE_WORKLOADS:
        wl = DECODE_WORKLOADS[args.workload]
        if args.B or args.H:
            wl = wl.with_(B=args.B or wl.B, H=args.H or wl.H)
        return run_decode_reference(args, wl) if args.impl == "reference" else run_decode(args, wl)
    if args.workload.startswith("partial_") and args.workload[8:] in WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "partial PaTH is timed against full PaTH on the GPU only"}))
            return 0
        return run_partial(args, WORKLOADS[args.workload[8:]])
    if args.workload.startswith("forms_") and args.workload[6:] in WORKLOADS:
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the transition forms are compared on the GPU only"}))
            return 0
        return run_transition_forms(args, WORKLOADS[args.workload[6:]])
    if args.workload == "bwd_grid":
        if args.impl == "reference":
            print(json.dumps({"impl": "reference", "unavailable":
                              "the grid is a GPU timing table; use bwd_<workload> for the oracle"}))
            return 0
        return run_bwd_grid(args)
    if args.workload.startswith("bwd_") and args.workload[4:] in WORKLOADS:
        wl = WORKLOADS[args.workload[4:]]
        if args.B or args.H:
            wl = wl.with_(B=args.B or wl.B, H=args.H or wl.H,
                          name=f"{wl.name}_B{args.B or wl.B}H{args.H or wl.H}")
        return run_bwd_reference(args, wl) if args.impl == "reference" else run_bwd(args, wl)
    wl = WORKLOADS[args.workload]
    if args.B or args.H:
        wl = wl.with_(B=args.B or wl.B, H=args.H or wl.H, name=f"{wl.name}_B{args.B or wl.B}H{args.H or wl.H}")
    f = step_flops(wl.B, wl.H, wl.T, wl.d)
    if args.impl == "reference":
        return run_reference(args, wl, f)
    return run_gpu(args, wl, f)


if __name__ == "__main__":
    sys.exit(main())
