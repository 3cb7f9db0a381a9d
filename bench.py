"""Benchmark: batched KKT solves per second on one GB300 (or N replicas).

A step is one gato_solve_kkt call over the whole batch: Schur complement and
stair preconditioner formation, batched PCG with dz recovery, and the
8-candidate L1-merit line search.  The workload is the 256-solve batch of
128-knot problems (n = 14 states, m = 7 controls, fp32) with synthetic,
seeded data; inputs are resident in HBM when the timed region starts and L2
is flushed (256 MB write) before every timed step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints one JSON line (rank 0).  With --impl reference the fp64 CPU oracle is
timed on the host cores on the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "KKT solves/sec and PCG iters/sec at batch M; % of GB300 HBM/L2 roofline"
UNIT = "solves/s"
WORKLOAD_INDEX = 4  # M=256, N=128, n=14, m=7

# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) of one PCG
# solve launch at this workload, from an ncu capture; valid only for the
# kernel source it was taken on (sha256 prefix of csrc/pcg.cu and
# csrc/pcg_common.cuh), null otherwise.  Captured on 152 solves (one block
# per SM) and scaled by the solves processed to the 256-solve launch
# (89.86 MB x 256 / 152).
PCG_TRAFFIC = {"pcg_sha": "bf17afc3f87af630", "bytes_per_launch": 151340301}

FP32_LANES_PER_SM = 128  # FFMA lanes per SM (4 sub-partitions x 32)

# gato_set_pcg_kernel choices by name (the values of include/gato.h)
PCG_KERNELS = {"auto": 0, "generic": 1, "wide": 2, "tile": 3, "rows": 4, "quad": 5}

# linear solvers of S lambda = gamma (gato_params.linsys)
LINSYS = {"pcg": 1, "bdsv": 2, "bdsv_chrono": 3}


def launches_per_solve(linsys, refine_steps, refine_solver=0):
    """Kernel launches of one gato_solve_kkt call: 3 formation + 1 right-hand
    side + the linear solve (PCG: 1; direct: factor + substitution) + 1 fused
    merit, and per refinement round 1 residual + 1 right-hand side + 1 solve
    (PCG, or the direct substitution) + 1 accumulate; direct corrections after
    a PCG solve add the factorisation once."""
    solve = 1 if linsys == "pcg" else 2
    factor = 1 if (linsys == "pcg" and refine_solver and refine_steps) else 0
    return 5 + solve + 4 * refine_steps + factor


def _src_sha(*paths):
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def _peaks():
    """(HBM GB/s, kind, max SM MHz) from MEASURED_PEAKS.json, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured", float(d.get("sm_max_mhz", 2070.0))
    except Exception:
        return 6800.0, "fallback", 2070.0


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running:
    every 50 ms, the first sample taken before the region it brackets starts
    (waiting at most two seconds for it)."""

    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 50):
        self.index = index
        self.interval_ms = interval_ms
        self.rows = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            t0 = time.monotonic()
            while not self.rows and self.proc.poll() is None and time.monotonic() - t0 < 2.0:
                time.sleep(0.005)
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 6:
                self.rows.append(parts)

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if not self.rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[2 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(self.rows)}


def _fp32_probe(torch, gato, dev, local):
    """Measured fp32 FMA throughput of this GPU (TFLOP/s, 2 flops per FMA):
    the library's probe kernel (independent FMA chains in every thread of
    four 256-thread blocks per SM), scalar fma.rn.f32 and packed
    fma.rn.f32x2, best of five launches of about 3 ms each after warm-up,
    timed with CUDA events; SM clocks sampled meanwhile."""
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    blocks, threads, trips = 4 * n_sm, 256, 4096
    sink = torch.zeros(blocks, dtype=torch.float32, device=dev)
    res = {}
    with ClockSampler(local) as clk:
        for name, packed in (("ffma", 0), ("ffma2", 1)):
            best = 0.0
            for k in range(8):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                flops = gato.probe_fp32(packed, blocks, threads, trips, sink)
                b.record()
                b.synchronize()
                if k >= 3:
                    best = max(best, flops / (a.elapsed_time(b) * 1e-3) / 1e12)
            res[name] = best
    res["clocks"] = clk.summary()
    return res


def _dist_env():
    from trajectory_optimization_kkt_gb300.replicas import from_env
    r = from_env()
    return r.world, r.rank, r.local


def run_reference(args, world, rank):
    """fp64 oracle on the host cores, same workload, bounded per step."""
    if rank != 0:
        return
    import multiprocessing as mp

    import oracle
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch
    w = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    per_step = w.M  # every step solves the whole batch, as the GPU arm's step does
    prob = make_batch(w, M=per_step)
    oracle.build()
    solves = [oracle.solve_one(prob, j) for j in range(per_step)]
    kw = dict(eps=w.pcg_eps, max_iters=w.pcg_max_iters, n_alpha=w.n_alpha, beta=w.beta, mu=w.mu)
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        for _ in range(args.warmup):
            pool.starmap(_oracle_solve, [(s, kw) for s in solves])
        times, iters = [], 0
        for _ in range(args.steps):
            t0 = time.perf_counter()
            res = pool.starmap(_oracle_solve, [(s, kw) for s in solves])
            times.append(time.perf_counter() - t0)
            iters += sum(r[0] for r in res)
    sec = sum(times)
    value = per_step * args.steps / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sec / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "pcg_iters_per_sec": iters / sec,
        "config": _config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"the whole batch of {w.M} solves per step, spawn pool of "
                                   f"{cores}"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _oracle_solve(prob, kw):
    import oracle
    out = oracle.solve_kkt(prob, **kw)
    return out["iters"], out["best"]


def _config(w, **extra):
    c = {"workload": w.name, "M": w.M, "N": w.N, "n": w.n, "m": w.m, "pcg_eps": w.pcg_eps,
         "pcg_max_iters": w.pcg_max_iters, "stop_rule": "relative residual ||r||<=eps||gamma||",
         "n_alpha": w.n_alpha, "beta": w.beta, "mu": w.mu,
         "refine_steps": w.refine_steps,
         "refine_solver": "direct (cyclic-reduction factors of the same S)" if w.refine_solver
                          else f"pcg to {w.refine_eps}",
         "pcg_precision": "double-float" if w.pcg_precision else "fp32",
         "l2": "flushed before every timed step (256 MB write)"}
    c.update(extra)
    return c


def _cpu_model():
    """The host CPU's model name from /proc/cpuinfo (or the machine type)."""
    import platform
    ids = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "cpu model", "hardware"):
                    return line.split(":", 1)[1].strip()
                if key in ("cpu implementer", "cpu part") and key not in ids:
                    ids[key] = line.split(":", 1)[1].strip()
    except OSError:
        pass
    if ids:  # Arm kernels name the core by implementer and part codes
        return (f"{platform.machine()} (implementer {ids.get('cpu implementer', '?')}, "
                f"part {ids.get('cpu part', '?')})")
    return platform.machine()


def _cpu_baseline(w):
    """Oracle on a bounded sample of the workload, spawn pool on all cores."""
    import multiprocessing as mp

    import oracle
    from trajectory_optimization_kkt_gb300.workloads import make_batch
    cores = os.cpu_count() or 1
    oracle.build()
    kw = dict(eps=w.pcg_eps, max_iters=w.pcg_max_iters, n_alpha=w.n_alpha, beta=w.beta, mu=w.mu)
    # the whole batch (about 8 s of CPU work at workload 4, 34 solves/s a core);
    # for batches smaller than four solves a core, that many solves of the same
    # recipe, so that the pool's dispatch does not dominate
    sample = max(w.M, 4 * cores)
    prob = make_batch(w, M=sample)
    solves = [oracle.solve_one(prob, j) for j in range(sample)]
    ctx = mp.get_context("spawn")
    with ctx.Pool(cores) as pool:
        pool.starmap(_oracle_solve, [(s, kw) for s in solves[:cores]])  # start-up
        t0 = time.perf_counter()
        res = pool.starmap(_oracle_solve, [(s, kw) for s in solves])
        sec = time.perf_counter() - t0
    # one thread: the first two solves in this process
    t0 = time.perf_counter()
    for s_ in solves[:2]:
        _oracle_solve(s_, kw)
    one = 2 / (time.perf_counter() - t0)
    return {"value": sample / sec, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"all {sample} solves of the batch" if sample == w.M else
                       f"{sample} solves of the workload's recipe (batch of {w.M})")
                      + f", fp64 C oracle, spawn pool of {cores}",
            "pcg_iters_per_sec": sum(r[0] for r in res) / sec,
            "single_thread_solves_per_s": one, "cpu_model": _cpu_model()}


def _time_solver(torch, s, p, d, out, steps, flush, stream):
    """Device time of `steps` gato_solve_kkt calls (L2 flushed before each),
    with the library's default parts; the stages from a one-part pass of the
    same steps: (ms per step, mean stage microseconds, PCG iterations per
    step, solves with a status bit)."""
    def step():
        out["status"].zero_()
        s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"], stream)
    for _ in range(3):
        step()
    ms, stages, iters = [], {"form": [], "linsys": [], "refine": [], "merit": []}, 0
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in range(steps):
        flush.fill_(float(k))
        a.record(stream)
        step()
        b.record(stream)
        b.synchronize()
        ms.append(a.elapsed_time(b))
        iters += int(out["iters"].sum())
    _time_solver.last_parts = s.get_parts()  # the parts the timed calls ran
    s.set_parts(1)
    s.set_timing(True)
    for k in range(steps):
        flush.fill_(float(k))
        step()
        st = s.get_stats()
        stages["form"].append(st.form_us)
        stages["linsys"].append(st.pcg_us)
        stages["refine"].append(max(st.refine_us, 0.0))
        stages["merit"].append(st.merit_us)
    s.set_timing(False)
    s.set_parts(0)
    bad = int((out["status"] != 0).sum())
    _time_solver.last_stats = st
    return (statistics.mean(ms), {k: statistics.mean(v) for k, v in stages.items()},
            iters / steps, bad)


def run_sweep(args, local):
    """Horizon x batch sweep of the linear solvers (the GATO documentation's
    PCG-versus-direct comparison that sets BDSV_HORIZON), one JSON line each."""
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    base = WORKLOADS[WORKLOAD_INDEX]
    for N in (32, 64, 128, 256, 512):
        for M in (1, 16, 256):
            w = base.with_batch(M, N)
            prob = make_batch(w, M=M)
            d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
            with gato.Solver(M, N, w.n, w.m) as s:
                out = s.outputs(w.n_alpha)
                for name, ls in LINSYS.items():
                    p = gato.default_params(**{**w.solver_settings(), "pcg_max_iters": 4000},
                                            linsys=ls)
                    ms, stages, iters, bad = _time_solver(torch, s, p, d, out, args.steps,
                                                          flush, stream)
                    print(json.dumps({"sweep": "linsys", "M": M, "N": N, "n": w.n, "m": w.m,
                                      "linsys": name, "solves_per_s": M / (ms / 1000.0),
                                      "ms_per_step": ms, "stage_us": stages,
                                      "pcg_iters_per_solve": iters / M,
                                      "status_nonzero_solves": bad}), flush=True)


def run_pcg_kernel_sweep(args, local):
    """PCG-only time of the wide-tile and quad kernels and of the automatic
    choice, n in {8, 10, 12, 14, 16} x N in {16, 32, 64, 128} x M in {16, 152,
    256, 1024}, then of the register-row kernel (its cluster form where one
    CTA cannot hold a solve) against the generic kernel, n in {24, 36} x N in
    {16, 32, 64, 128} x M in {16, 128}: gato_pcg_solve after one gato_form_schur (stop rule 0, eps 1e-6),
    L2 flushed before each launch, the median of 6 launches after 2; the
    batch is 16 generated solves (workload 4's generator at these sizes)
    repeated to M, so every solve of a cell takes the iterations of one of
    16.  One JSON line per cell, with the kernel each call ran as the
    library reports it."""
    import dataclasses

    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    kinds = {"wide": gato.GATO_PCG_WIDE, "quad": gato.GATO_PCG_QUAD, "auto": gato.GATO_PCG_AUTO}
    base = WORKLOADS[WORKLOAD_INDEX]
    for n in (8, 10, 12, 14, 16):
        for N in (16, 32, 64, 128):
            w = dataclasses.replace(base, n=n, m=n // 2, N=N)
            one = make_batch(w, M=16)
            for M in (16, 152, 256, 1024):
                prob = {k: np.ascontiguousarray(np.concatenate([v] * -(-M // 16))[:M])
                        for k, v in one.items()}
                d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
                p = gato.default_params(pcg_eps=1e-6, pcg_max_iters=2000)
                row = {"sweep": "pcg_kernels", "n": n, "N": N, "M": M}
                with gato.Solver(M, N, n, n // 2) as s:
                    out = s.outputs(p.n_alpha)
                    s.form_schur(d, out["status"], stream)
                    for name, kind in kinds.items():
                        s.set_pcg_kernel(kind)
                        ts = []
                        for k in range(8):
                            flush.fill_(float(k))
                            a = torch.cuda.Event(enable_timing=True)
                            b = torch.cuda.Event(enable_timing=True)
                            a.record(stream)
                            s.pcg_solve(p, out["lam"], out["dX"], out["dU"], out["iters"],
                                        out["status"], stream=stream)
                            b.record(stream)
                            b.synchronize()
                            if k >= 2:
                                ts.append(a.elapsed_time(b))
                        row[name] = {"us": 1000.0 * statistics.median(ts),
                                     "iters_per_solve": float(out["iters"].float().mean()),
                                     "ran": _kernel_names().get(s.get_stats().pcg_kernel),
                                     "status_nonzero_solves": int((out["status"] != 0).sum())}
                row["quad_over_wide"] = row["quad"]["us"] / row["wide"]["us"]
                print(json.dumps(row), flush=True)
    # n > 16: the register-row kernel (one CTA per solve where its block fits,
    # else its cluster form) against the generic kernel
    kinds = {"rows": gato.GATO_PCG_ROWS, "generic": gato.GATO_PCG_GENERIC}
    for n in (24, 36):
        for N in (16, 32, 64, 128):
            w = dataclasses.replace(base, n=n, m=n // 3, N=N)
            one = make_batch(w, M=16)
            for M in (16, 128):
                prob = {k: np.ascontiguousarray(np.concatenate([v] * -(-M // 16))[:M])
                        for k, v in one.items()}
                d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
                p = gato.default_params(pcg_eps=1e-6, pcg_max_iters=4000)
                row = {"sweep": "pcg_rows", "n": n, "N": N, "M": M}
                with gato.Solver(M, N, n, n // 3) as s:
                    out = s.outputs(p.n_alpha)
                    s.form_schur(d, out["status"], stream)
                    for name, kind in kinds.items():
                        s.set_pcg_kernel(kind)
                        ts = []
                        for k in range(8):
                            flush.fill_(float(k))
                            a = torch.cuda.Event(enable_timing=True)
                            b = torch.cuda.Event(enable_timing=True)
                            a.record(stream)
                            s.pcg_solve(p, out["lam"], out["dX"], out["dU"], out["iters"],
                                        out["status"], stream=stream)
                            b.record(stream)
                            b.synchronize()
                            if k >= 2:
                                ts.append(a.elapsed_time(b))
                        row[name] = {"us": 1000.0 * statistics.median(ts),
                                     "iters_per_solve": float(out["iters"].float().mean()),
                                     "status_nonzero_solves": int((out["status"] != 0).sum())}
                row["generic_over_rows"] = row["generic"]["us"] / row["rows"]["us"]
                print(json.dumps(row), flush=True)


def run_throughput_sweep(args, local):
    """The benchmark workload's throughput sweep: M in {1, 8, 16, 64, 256} x
    N in {16, 32, 64, 128} at n = 14, m = 7, the default PCG path; solves/s
    and PCG iterations/s of whole calls (default parts), the merit's
    microseconds per launch and (knot, candidate) pairs per second from the
    one-part stage pass; one JSON line per cell."""
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    base = WORKLOADS[WORKLOAD_INDEX]
    for N in (16, 32, 64, 128):
        for M in (1, 8, 16, 64, 256):
            w = base.with_batch(M, N)
            prob = make_batch(w, M=M)
            d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
            with gato.Solver(M, N, w.n, w.m) as s:
                out = s.outputs(w.n_alpha)
                p = gato.default_params(**w.solver_settings(), linsys=LINSYS["pcg"])
                ms, stages, iters, bad = _time_solver(torch, s, p, d, out, args.steps, flush,
                                                      stream)
                # one part: the PCG stage over the iterations of a solve (with PCG
                # corrections also the refinement stage, its correction solve and
                # small kernels, over the iterations of both); at M = 1 this is
                # the latency of one iteration of one solve
                pcg_us_it = ((stages["linsys"] + (0.0 if w.refine_solver else stages["refine"]))
                             / max(iters / M, 1.0))
                print(json.dumps({"sweep": "throughput", "M": M, "N": N, "n": w.n, "m": w.m,
                                  "parts": _time_solver.last_parts,
                                  "solves_per_s": M / (ms / 1000.0),
                                  "pcg_us_per_iteration": pcg_us_it,
                                  "pcg_kernel": _pcg_kernel_label(
                                      _time_solver.last_stats, M, N, w.n,
                                      torch.cuda.get_device_properties(dev)
                                      .multi_processor_count),
                                  "ms_per_step": ms,
                                  "pcg_iters_per_sec": iters / (ms / 1000.0),
                                  "pcg_iters_per_solve": iters / M,
                                  "merit_us_per_launch": stages["merit"],
                                  "knot_candidates_per_s":
                                      M * N * (w.n_alpha + 1) / (stages["merit"] * 1e-6),
                                  "stage_us": stages, "status_nonzero_solves": bad}),
                      flush=True)


def _ff_kernel_name(M, N, n, n_sm):
    """The double-float kernel launch_pcg_ff picks: a cluster of two CTAs per
    solve when the batch is at most half of the SMs (n <= 16, each CTA with at
    least 256 rows, the CTAs' warps within one 32-lane butterfly), else one CTA
    per solve."""
    if n <= 16:
        Nc = -(-N // 2)
        warps = -(-(Nc * n) // 32)
        if M * 2 <= n_sm and Nc < N and 2 * warps <= 32 and Nc * n >= 256:
            return "k_pcg_ff_cluster<2>"
    return "k_pcg_ff"


def _kernel_names():
    """Kernel names of the GATO_PCG_* values gato_stats reports."""
    from trajectory_optimization_kkt_gb300 import gato
    return {gato.GATO_PCG_GENERIC: "k_pcg_generic", gato.GATO_PCG_WIDE: "k_pcg_wide",
            gato.GATO_PCG_TILE: "k_pcg_tile", gato.GATO_PCG_ROWS: "k_pcg_rows",
            gato.GATO_PCG_QUAD: "k_pcg_quad", gato.GATO_PCG_CLUSTER: "k_pcg_cluster",
            gato.GATO_PCG_DOUBLE_FLOAT: "k_pcg_ff"}


def _pcg_kernel_label(st, M, N, n, n_sm):
    """The PCG kernels a call ran, as the library reports them in its stats
    (gato_stats.pcg_kernel, refine_kernel): the main solve's, then, after a
    plus sign, the refinement corrections' when they ran another PCG kernel;
    the double-float kernel's cluster form by launch_pcg_ff's rule."""
    from trajectory_optimization_kkt_gb300 import gato
    names = _kernel_names()
    main = names.get(st.pcg_kernel, "none")
    if st.pcg_kernel == gato.GATO_PCG_DOUBLE_FLOAT:
        main = _ff_kernel_name(M, N, n, n_sm)
    ref = names.get(st.refine_kernel)
    return main if ref is None or ref == main else main + " + " + ref


def run_workloads(args, local):
    """The five synthetic workloads at their own sizes and settings: solves/s
    and PCG iterations/s of whole gato_solve_kkt calls (default parts, L2
    flushed before each), the PCG stage against the fp32 FMA roofline and the
    merit against measured HBM (from the one-part stage pass), next to the
    fp64 oracle on the host's cores for the same batch.  One JSON line per
    workload."""
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    hbm_peak, peak_kind, sm_mhz = _peaks()
    probe = _fp32_probe(torch, gato, dev, local)
    alu_peak_tf = max(probe["ffma"], probe["ffma2"])
    steps = min(args.steps, 10)
    for w in WORKLOADS:
        M, N, n, m = w.M, w.N, w.n, w.m
        prob = make_batch(w)
        d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
        p = gato.default_params(**w.solver_settings())
        with gato.Solver(M, N, n, m) as s:
            out = s.outputs(w.n_alpha)
            ms, stages, iters, bad = _time_solver(torch, s, p, d, out, steps, flush, stream)
            parts = _time_solver.last_parts
        flops_it = 2 * 2 * (3 * N - 2) * n * n + 12 * N * n
        # with direct corrections the refinement stage runs no PCG iteration
        pcg_us = stages["linsys"] + (0.0 if w.refine_solver else stages["refine"])
        achieved_tf = flops_it * iters / (pcg_us * 1e-6) / 1e12
        K = N - 1
        merit_bytes = 4 * M * (N * n * n + K * (m * m + n * n + n * m) + N * n + K * m + K * n
                               + n + N * n + K * m + (w.n_alpha + 1) + 1)
        merit_gbs = merit_bytes / (stages["merit"] * 1e-6) / 1e9
        pcg_kernel = _pcg_kernel_label(_time_solver.last_stats, M, N, n,
                                       torch.cuda.get_device_properties(dev).multi_processor_count)
        row = {"workload": w.name, "M": M, "N": N, "n": n, "m": m, "parts": parts,
               "solves_per_s": M / (ms / 1000.0), "ms_per_call": ms,
               "pcg_iters_per_sec": iters / (ms / 1000.0), "pcg_iters_per_solve": iters / M,
               "stage_us": stages, "status_nonzero_solves": bad,
               "pcg_roofline": {"bound": "alu", "kernel": pcg_kernel, "achieved": achieved_tf,
                                "peak": alu_peak_tf, "unit": "TFLOP/s",
                                "frac": achieved_tf / alu_peak_tf,
                                "peak_basis": "fp32 FMA probe in this run, of measured"},
               "merit_roofline": {"bound": "hbm", "achieved": merit_gbs, "peak": hbm_peak,
                                  "unit": "GB/s", "frac": merit_gbs / hbm_peak,
                                  "peak_kind": peak_kind,
                                  "knot_candidates_per_s":
                                      M * N * (w.n_alpha + 1) / (stages["merit"] * 1e-6)}}
        if not args.no_cpu_baseline:
            row["cpu_baseline"] = _cpu_baseline(w)
        print(json.dumps(row), flush=True)


def run_merit_sweep(args, local):
    """The merit variants (the GATO line-search table's fused / unfused
    comparison): device microseconds per gato_linesearch call for the factored
    default (one launch) and the per-candidate kernel (one block per (knot,
    candidate), then the reduction) at 32, 64, 128 and 256 threads, over
    (n, m) in {(12, 6), (14, 7), (36, 12)}, N in {16, 32, 64, 128} and M in
    {1, 8, 16, 256}.  Twenty calls are recorded in a CUDA graph and replayed,
    so the time is the device's per call without the host's call overhead;
    the inputs stay in L2 from one call to the next.  One JSON line per
    cell."""
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import normals, random_lq
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    calls, reps = 20, 5

    def per_call_us(s, p, d, dX, dU, out):
        def run():
            for _ in range(calls):
                s.linesearch(p, d, dX, dU, out["merit"], out["best"], out["status"])
        run()  # loads the kernels before the capture
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            run()
        g.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            g.replay()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) * 1000.0 / (calls * reps)

    for n, m in ((12, 6), (14, 7), (36, 12)):
        for N in (16, 32, 64, 128):
            for M in (1, 8, 16, 256):
                prob = random_lq(M, N, n, m, seed=4000 + N + M)
                d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
                # a step of the problem's size (the kernels' time does not
                # depend on its values)
                dX = torch.from_numpy(0.1 * normals(5000 + N + M, 1, M * N * n)
                                      .reshape(M, N, n).astype(np.float32)).to(dev)
                dU = torch.from_numpy(0.1 * normals(5000 + N + M, 2, M * (N - 1) * m)
                                      .reshape(M, N - 1, m).astype(np.float32)).to(dev)
                row = {"sweep": "merit", "n": n, "m": m, "N": N, "M": M, "n_alpha": 8}
                with gato.Solver(M, N, n, m) as s:
                    out = s.outputs(8)
                    p = gato.default_params(merit_kernel=gato.GATO_MERIT_FUSED)
                    row["fused_us"] = per_call_us(s, p, d, dX, dU, out)
                    row["fused_kernel"] = ("k_merit_knots" if n <= 16 and m <= 16
                                           else "k_merit_fused")
                    unf = {}
                    for t in (32, 64, 128, 256):
                        p = gato.default_params(merit_kernel=gato.GATO_MERIT_PER_CANDIDATE,
                                                merit_threads=t)
                        unf[str(t)] = per_call_us(s, p, d, dX, dU, out)
                row["per_candidate_us"] = unf
                best = min(unf.values())
                row["fused_over_unfused_256"] = row["fused_us"] / unf["256"]
                row["fused_over_best_unfused"] = row["fused_us"] / best
                row["knot_candidates_per_s_fused"] = M * N * 9 / (row["fused_us"] * 1e-6)
                print(json.dumps(row), flush=True)


def _sqp_timing(torch, gato, model_np, M, iters, linsys, use_graph, dev, stream, flush, reps=3):
    """Device ms per SQP iteration of a batch of M problems (after one
    untimed call that records the graph), and the last call's outputs."""
    N, n = model_np["Q"].shape[1:3]
    m = model_np["B"].shape[-1]
    from trajectory_optimization_kkt_gb300.workloads import rho_logspace
    d = {k: torch.from_numpy(np.ascontiguousarray(v)).to(dev) for k, v in model_np.items()}
    f = dict(device=dev, dtype=torch.float32)
    p = gato.default_params(pcg_max_iters=2000, refine_steps=1, linsys=LINSYS[linsys])
    sp = gato.default_sqp_params(iters=iters, use_graph=use_graph)
    rho0 = torch.from_numpy(rho_logspace(M)).to(dev)
    with gato.Solver(M, N, n, m) as s:
        X, U = torch.zeros(M, N, n, **f), torch.zeros(M, N - 1, m, **f)
        lam, rho = torch.zeros(M, N, n, **f), rho0.clone()
        hist = torch.zeros(M, iters + 1, **f)
        status = torch.zeros(M, device=dev, dtype=torch.int32)
        times = []
        for rep in range(reps + 1):
            for t in (X, U, lam, status):
                t.zero_()
            rho.copy_(rho0)
            flush.fill_(float(rep))
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            s.sqp_linear(p, sp, d, X, U, lam, rho, hist, status, stream=stream)
            b.record(stream)
            b.synchronize()
            if rep:
                times.append(a.elapsed_time(b) / iters)
        return statistics.median(times), hist.cpu().numpy(), status.cpu().numpy()


def run_sqp_study(args, local):
    """The rho-damping case study of the GATO paper (Sec. IV-C) on the linear
    model: each batch holds one problem M times with rho log-spaced from 1e-8
    to 10 (a single solve starts at 0.1); merit after each of 100 SQP
    iterations from the zero trajectory, best over the batch, and the time
    per iteration with graph replay and with kernel-by-kernel launches."""
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import linear_models, replicate
    torch.cuda.set_device(local)
    _build.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    N, n, m, iters, problems = 64, 14, 7, 100, 8
    models = linear_models(problems, N, n, m, seed=9000)
    for M in (1, 4, 16, 32, 64, 128):
        best, ms_graph = [], []
        for j in range(problems):
            one = {k: v[j] for k, v in models.items()}
            ms, hist, _ = _sqp_timing(torch, gato, replicate(one, M), M, iters, "pcg", 1, dev,
                                      stream, flush, reps=1)
            ms_graph.append(ms)
            best.append(hist.min(axis=0))  # best merit over the batch after each iteration
        best = np.array(best)
        first = replicate({k: v[0] for k, v in models.items()}, M)
        ms_stream, _, _ = _sqp_timing(torch, gato, first, M, iters, "pcg", 0, dev, stream,
                                      flush, reps=1)
        ms_direct, hist_d, _ = _sqp_timing(torch, gato, first, M, iters, "bdsv", 1, dev,
                                           stream, flush, reps=1)
        print(json.dumps({"sqp_study": "rho_sweep", "M": M, "N": N, "n": n, "m": m,
                          "iters": iters, "problems": problems,
                          "best_merit_over_batch_mean": {
                              str(t): float(best[:, t].mean()) for t in (0, 1, 2, 5, 10, 20,
                                                                         50, 100)},
                          "ms_per_iteration_graph": statistics.median(ms_graph),
                          "ms_per_iteration_stream": ms_stream,
                          "ms_per_iteration_direct_solve_graph": ms_direct,
                          "direct_solve_best_merit_problem0": {
                              str(t): float(hist_d.min(axis=0)[t]) for t in (0, 1, 2, 100)},
                          "pcg_best_merit_problem0": {
                              str(t): float(best[0, t]) for t in (0, 1, 2, 100)}}), flush=True)


def run_gpu(args, world, rank, local):
    import torch

    from trajectory_optimization_kkt_gb300 import _build, gato
    from trajectory_optimization_kkt_gb300.workloads import WORKLOADS, make_batch

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    _build.build()
    w = WORKLOADS[args.workload]
    if args.batch or args.horizon:
        w = w.with_batch(args.batch or w.M, args.horizon)
    M = w.M
    from trajectory_optimization_kkt_gb300.replicas import Replica, job_throughput, max_over_ranks
    replica = Replica(world, rank, local)
    prob = make_batch(w, M=M, first_solve=replica.first_solve(M))
    dev = torch.device("cuda", local)
    d = {k: torch.from_numpy(v).to(dev) for k, v in prob.items()}
    s = gato.Solver(M, w.N, w.n, w.m)
    s.set_pcg_kernel(PCG_KERNELS[args.pcg_kernel])
    out = s.outputs(w.n_alpha)
    p = gato.default_params(**w.solver_settings(), linsys=LINSYS[args.linsys])
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    launches_per_step = launches_per_solve(args.linsys, w.refine_steps, w.refine_solver)

    def step():
        out["status"].zero_()
        s.solve_kkt(p, d, out["dX"], out["dU"], out["lam"], out["iters"], out["merit"],
                    out["best"], out["status"], stream)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()

    # ---- device-resident timing: per-step events, L2 flushed in between ----
    # the step as the library runs it by default: the batch in parts that run
    # concurrently on internal streams (gato_set_parts), the events on the
    # caller's stream bracketing all of them
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    iters_total = 0
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        for k in range(args.steps):
            flush.fill_(float(k))
            starts[k].record(stream)
            step()
            ends[k].record(stream)
            ends[k].synchronize()
            iters_total += int(out["iters"].sum())
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(step_ms)
    status_bad = int((out["status"] != 0).sum())
    parts = s.get_parts()

    # ---- stage breakdown: the same steps as one part, whose stages are
    # bracketed by events on one stream; the PCG roofline uses these launches
    s.set_parts(1)
    s.set_timing(True)
    pcg_us, refine_us, form_us, merit_us = [], [], [], []
    for k in range(args.steps):
        flush.fill_(float(k))
        step()
        st = s.get_stats()  # synchronises on this step's last event
        stage_stats = st
        pcg_us.append(st.pcg_us)
        refine_us.append(max(st.refine_us, 0.0))
        form_us.append(st.form_us)
        merit_us.append(st.merit_us)
    torch.cuda.synchronize()
    s.set_timing(False)
    s.set_parts(0)

    # ---- end to end through the C ABI with host buffers ----
    # gato_solve_kkt_host on pinned host arrays: every step copies the inputs
    # (and the in/out status) in and every output back, inside the timed
    # region; the library overlaps the copies of one part of the batch with
    # the solve of another
    host = gato.to_host(prob)
    host_out = s.host_outputs(w.n_alpha)
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    h2d += host_out["status"].numel() * host_out["status"].element_size()
    d2h = sum(v.numel() * v.element_size() for v in host_out.values())

    def host_step():
        s.solve_kkt_host(p, host, host_out["dX"], host_out["dU"], host_out["lam"],
                         host_out["iters"], host_out["merit"], host_out["best"],
                         host_out["status"], stream)

    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    if not args.no_e2e:
        for _ in range(2):  # the first call sets up the staging buffers and streams
            host_out["status"].zero_()
            host_step()
        torch.cuda.synchronize()
    for k in range(0 if args.no_e2e else args.steps):
        flush.fill_(float(k))
        host_out["status"].zero_()
        e_start.record(stream)
        host_step()
        e_end.record(stream)
        e_end.synchronize()
        e2e_ms += e_start.elapsed_time(e_end)
    if not args.no_e2e:
        assert int((host_out["status"] != 0).sum()) == status_bad

    # ---- max over ranks ----
    total_ms, e2e_ms = max_over_ranks([total_ms, e2e_ms], dist, dev)
    solves = M * world * args.steps
    value = job_throughput(M * args.steps, world, total_ms)

    # ---- roofline of the dominant kernel (PCG) ----
    # The PCG kernel keeps the operator on chip (registers and shared memory),
    # so its bound is the SM's fp32 FMA throughput.  Algorithmic flops per
    # solve-iteration are those of the method's iteration on the explicit
    # block-tridiagonal S and Phi^-1: two products with 3N-2 blocks of n^2
    # (2 flops per entry each) plus 12 N n of vector updates and dots.  Every
    # PCG iteration of the step counts.  With PCG corrections the time is the
    # two PCG launches plus the refinement's small kernels; with direct
    # corrections (substitutions, no PCG iteration) it is the main PCG launch
    # alone.
    N, n = w.N, w.n
    flops_it = 2 * 2 * (3 * N - 2) * n * n + 12 * N * n
    iters_per_step = iters_total / args.steps
    # with direct corrections the refinement stage runs no PCG iteration
    pcg_stage_us = statistics.mean(a + (0.0 if w.refine_solver else b)
                                   for a, b in zip(pcg_us, refine_us))
    achieved_tf = flops_it * iters_per_step / (pcg_stage_us * 1e-6) / 1e12
    hbm_peak, peak_kind, sm_mhz = _peaks()
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    nominal_tf = n_sm * FP32_LANES_PER_SM * 2 * sm_mhz * 1e6 / 1e12
    probe = _fp32_probe(torch, gato, dev, local)
    # the roofline's peak: the faster of the two measured FMA forms
    alu_peak_tf = max(probe["ffma"], probe["ffma2"])
    # the pages' streaming model: packed S and Phi^-1 read once per iteration
    bytes_it = 2 * (N * n * (n + 1) // 2 + (N - 1) * n * n) * 4
    stream_gbs = bytes_it * iters_per_step / (pcg_stage_us * 1e-6) / 1e9
    # merit: the problem data and the step read once, A + 1 merits and the
    # argmin written, per solve
    K, m = N - 1, w.m
    merit_bytes = 4 * M * (N * n * n + K * (m * m + n * n + n * m) + N * n + K * m + K * n + n
                           + N * n + K * m + (w.n_alpha + 1) + 1)
    merit_s = statistics.mean(merit_us) * 1e-6
    merit_gbs = merit_bytes / merit_s / 1e9
    sha = _src_sha(os.path.join(_build.CSRC, "pcg.cu"), os.path.join(_build.CSRC, "pcg_common.cuh"))
    # the ncu capture behind the traffic figure is of the default workload
    traffic = (PCG_TRAFFIC["bytes_per_launch"]
               if PCG_TRAFFIC["pcg_sha"] == sha and args.workload == WORKLOAD_INDEX
               and not args.batch and not args.horizon and args.pcg_kernel == "auto"
               else None)

    # ---- SQP loop on the linear model (context, not the metric) ----
    sqp = None
    if not args.no_alternatives and rank == 0:
        from trajectory_optimization_kkt_gb300.workloads import linear_models
        sq_M, sq_N, sq_iters = 128, 64, 20
        model = linear_models(sq_M, sq_N, w.n, w.m, seed=9100)
        sqp = {"M": sq_M, "N": sq_N, "n": w.n, "m": w.m, "iters_per_call": sq_iters,
               "rho0": "log-spaced 1e-8..10", "linsys": "pcg, one refinement round"}
        for mode, g in (("graph", 1), ("stream", 0)):
            ms, _, st = _sqp_timing(torch, gato, model, sq_M, sq_iters, "pcg", g, dev, stream,
                                    flush)
            sqp[f"ms_per_iteration_{mode}"] = ms
        sqp["sqp_iterations_per_sec_graph"] = 1000.0 / sqp["ms_per_iteration_graph"]

    # ---- the same step through the direct solvers (context, not the metric) ----
    alternatives = {}
    if args.linsys == "pcg" and not args.no_alternatives and rank == 0:
        for name in ("bdsv", "bdsv_chrono"):
            pa = gato.default_params(**w.solver_settings(), linsys=LINSYS[name])
            ms, stages, _, bad = _time_solver(torch, s, pa, d, out, min(args.steps, 10), flush,
                                              stream)
            alternatives[name] = {"solves_per_s": M / (ms / 1000.0), "ms_per_step": ms,
                                  "stage_us": stages, "status_nonzero_solves": bad}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded generator, workload recipe of the benchmark configs)",
            "config": _config(w, **({} if args.pcg_kernel == "auto"
                                    else {"pcg_kernel": args.pcg_kernel})),
            "pcg_iters_per_sec": iters_per_step * world / (total_ms / args.steps / 1000.0),
            "pcg_iters_per_solve": iters_per_step / M,
            "parts": parts,
            "stage_us_note": "one-part pass of the same steps (stage events need one stream)",
            "stage_us": {"form": statistics.mean(form_us), "pcg": statistics.mean(pcg_us),
                         "refine": statistics.mean(refine_us),
                         "merit": statistics.mean(merit_us)},
            "status_nonzero_solves": status_bad,
            "linsys": args.linsys,
            "roofline": None if args.linsys != "pcg" else {
                         "bound": "alu", "achieved": achieved_tf, "peak": alu_peak_tf,
                         "unit": "TFLOP/s", "frac": achieved_tf / alu_peak_tf,
                         "traffic": traffic,
                         "kernel": _pcg_kernel_label(stage_stats, M, N, n, n_sm)
                                   + (" (main solve; direct corrections)" if w.refine_solver
                                      else " (solve + refinement launches)"),
                         "peak_basis": "measured in this run: fp32 FMA probe "
                                       "(gato_probe_fp32), faster of scalar and packed form; "
                                       "of measured",
                         "peak_probe": {"ffma_tflops": probe["ffma"],
                                        "ffma2_tflops": probe["ffma2"],
                                        "sm_mhz_median": probe["clocks"].get("sm_mhz"),
                                        "reasons": probe["clocks"].get("reasons")},
                         "peak_nominal": nominal_tf,
                         "peak_nominal_basis": f"{n_sm} SMs x {FP32_LANES_PER_SM} FFMA lanes x "
                                               f"2 flop x {sm_mhz:.0f} MHz (max SM clock)",
                         "frac_of_nominal": achieved_tf / nominal_tf,
                         "flops_per_solve_iteration": flops_it,
                         "iterations_per_step": iters_per_step},
            "merit_roofline": {"bound": "hbm", "achieved": merit_gbs, "peak": hbm_peak,
                               "unit": "GB/s", "frac": merit_gbs / hbm_peak,
                               "peak_kind": peak_kind, "bytes_per_launch": merit_bytes,
                               "kernel": "k_merit_knots" if n <= 16 and m <= 16
                                         else "k_merit_fused",
                               "knot_candidates_per_s":
                                   M * N * (w.n_alpha + 1) / merit_s},
            "hbm_stream_model": {"equivalent_gbs": stream_gbs, "hbm_gbs": hbm_peak,
                                 "equivalent_over_hbm": stream_gbs / hbm_peak,
                                 "note": "the rate at which the pages' design would have to "
                                         "stream packed S and Phi^-1 from memory to match "
                                         "this step; not a roofline fraction: the kernel "
                                         "keeps the operator on chip and moves none of "
                                         "these bytes"},
            "e2e": None if args.no_e2e else {
                "value": solves / (e2e_ms / 1000.0), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            "gpu_launches": launches_per_step * parts * args.steps,  # each part launches all
            "clocks": clk.summary(),
        }
        if alternatives:
            line["linsys_alternatives"] = alternatives
        if sqp:
            line["sqp_loop"] = sqp
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = _cpu_baseline(w)
        print(json.dumps(line), flush=True)
    s.close()
    if dist:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gato", choices=["gato", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true",
                    help="skip the host-buffer end-to-end measurement")
    ap.add_argument("--linsys", default="pcg", choices=sorted(LINSYS),
                    help="linear solver of the timed step (default pcg, the metric's)")
    ap.add_argument("--no-alternatives", action="store_true",
                    help="skip timing the same step through the direct solvers")
    ap.add_argument("--sweep", action="store_true",
                    help="horizon x batch sweep of the three linear solvers instead")
    ap.add_argument("--pcg-kernel-sweep", action="store_true",
                    help="PCG-only time of the wide and quad kernels and AUTO over n x N x M")
    ap.add_argument("--throughput-sweep", action="store_true",
                    help="the workload's M x N throughput sweep (solves/s, merit us) instead")
    ap.add_argument("--workloads", action="store_true",
                    help="the five synthetic workloads at their own sizes, each next to the "
                         "oracle on the host's cores, instead")
    ap.add_argument("--merit-sweep", action="store_true",
                    help="the merit variants' sweep (fused / per-candidate at 32-256 "
                         "threads) instead")
    ap.add_argument("--sqp-study", action="store_true",
                    help="the rho-damping SQP case study on the linear model instead")
    ap.add_argument("--workload", type=int, default=WORKLOAD_INDEX, choices=range(5),
                    help="the workload of the timed step (default 4, the metric's: "
                         "M=256, N=128, n=14, m=7); the others are parity cases, run "
                         "here for profiler captures")
    ap.add_argument("--pcg-kernel", default="auto", choices=sorted(PCG_KERNELS),
                    help="the PCG kernel of the timed step (default: the library's "
                         "automatic choice); for comparisons and profiler captures")
    ap.add_argument("--horizon", type=int, default=None,
                    help="knots N (default: the workload's); for profiler captures of "
                         "other horizons")
    ap.add_argument("--batch", type=int, default=None,
                    help="solves per GPU (default: the workload's 256); for profiler "
                         "captures of a smaller case")
    args = ap.parse_args()
    world, rank, local = _dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
    elif args.sweep:
        run_sweep(args, local)
    elif args.pcg_kernel_sweep:
        run_pcg_kernel_sweep(args, local)
    elif args.throughput_sweep:
        run_throughput_sweep(args, local)
    elif args.workloads:
        run_workloads(args, local)
    elif args.merit_sweep:
        run_merit_sweep(args, local)
    elif args.sqp_study:
        run_sqp_study(args, local)
    else:
        run_gpu(args, world, rank, local)


if __name__ == "__main__":
    main()
