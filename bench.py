"""Benchmark: FMM evaluation throughput (particles/s) on one B300 per rank.

One step = one complete FMM evaluation (keys, sort, tree, P2M/M2M, walk, lists,
M2L, L2L, L2P + P2P) of the default workload: N = 2^20 clustered particles
(64 Plummer halos + 20 % background), fp32, p = 4, theta = 0.7, leaf 64 -- the
N ~ 1e6 point of the metric. The N = 1e5 fp64 Plummer point (p = 4,
theta = 0.7, leaf 32) is timed in the same run and reported under "also".

Inputs are resident in HBM before the timed region; L2 is flushed (256 MiB
write) between timed steps, outside the per-step CUDA events. Multi-GPU runs
are independent replicas (the FMM here does not shard): every rank evaluates
its own copy, the barrier + max-over-ranks timing is the only communication.

``--impl reference`` times the CPU oracle (plain C, OpenMP) on a bounded
sample of the same workload on this machine's host cores.
"""
from __future__ import annotations

import argparse
import dataclasses
import gc
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

from body_forces_morton_b300 import workloads as W  # noqa: E402

# Peaks: HBM copy bandwidth from the driver-written measurement; FP32 / FP64
# pipe peaks derived from unit counts and the maximum SM clock: 148 SMs x 128
# FP32 lanes x 2 flop per FMA x 2.032 GHz = 77.0 TFLOP/s (38.5e12 FP32 lane
# operations/s); FP64: 148 SMs x 2 FMA per clock x 2 flop x 2.032 GHz = 1.20
# TFLOP/s (the FP64 FMA rate ncu reports per SM).
SM_CLOCK_HZ = 2.032e9
FP32_PEAK_TFLOPS = 148 * 128 * 2 * SM_CLOCK_HZ / 1e12
FP32_LANE_OPS_PEAK = 148 * 128 * SM_CLOCK_HZ  # FP32 pipe lane-operations per second (an FFMA counts once)
FP64_PEAK_TFLOPS = 148 * 2 * 2 * SM_CLOCK_HZ / 1e12
F64_ARITH = ("fp64 inputs and outputs; M2L (p <= 4), L2P and leaf P2M (p <= 6) and P2P in double-float "
             "arithmetic (fp32 pairs, ~2^-48 relative) on the FP32 pipe, the other stages in fp64")
F64_IEEE_ARITH = "IEEE fp64 in every stage (fmm_plan_set_f64_ieee)"
F64_MUTUAL_ARITH = ("fp64 inputs and outputs; mutual M2L and P2P in IEEE fp64, L2P and leaf P2M (p <= 6) in "
                    "double-float, the other stages in fp64")
P2P_FLOPS_PER_PAIR = 20  # 3 sub, 3 mul + 2 add (r^2), rsqrt (1), 3 mul (m/r, /r^2), 3 FMA (a), 1 add (phi) ~ 19 + 1

# The double-float kernels run on the FP32 pipe, so their roofline is that
# pipe: FP32 FMA-pipe lane operations they issue per pair (an FFMA counted
# once, like the pipe does), times pairs, over time, against
# FP32_LANE_OPS_PEAK. The per-pair counts are ncu's
# sm__thread_inst_executed_pipe_fma_pred_on over the pairs of one launch (Plummer
# 1e5 fp64, p 4), keyed by the hash of the kernel sources they were counted on;
# a changed kernel reports null until it is counted again.
DF_FMA_OPS_PER_PAIR = {
    # k_p2p_df: 9,098,613,344 FMA-pipe thread instructions (all scalar) over the 48,723,340 pairs the
    # roofline counts (the interactions less the 1e5 zero-separation self pairs)
    ("k_p2p_df", "453998eb2c42ecbf"): 186.74,
    # k_m2l_df<4>: 6,072,086,944 over 1,833,964 pairs (the moments' conversion kernel is not counted)
    ("k_m2l_df", "159774f6b7e517df"): 3310.9,
}

# DRAM traffic of the P2P kernel per launch (dram__bytes_read.sum +
# dram__bytes_write.sum, one warm launch of clustered N = 2^20 fp32), keyed by
# the hash of the kernel sources it was taken on; null once they change.
TRAFFIC = {
    # k_p2p<float>: 52,590,336 B read + 4,480,768 B written
    ("clustered_2p20_f32", "25d0a0c48336f2ac"): 57071104,
}


def kernel_source_hash(files=("k_down.cu", "expansions_gen.cuh", "common.cuh")):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "body_forces_morton_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


DF_SOURCES = {"k_p2p_df": ("k_p2p_df.cu", "dfloat.cuh", "common.cuh"),
              "k_m2l_df": ("k_m2l_df.cu", "expansions_df_gen.cuh", "dfloat.cuh", "common.cuh")}


def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            # nvidia-smi's first query stalls the driver for milliseconds: let it happen before timing
            t0 = time.perf_counter()
            while not self.lines and time.perf_counter() - t0 < 3.0 and self.proc.poll() is None:
                time.sleep(0.01)
            self.lines = []
        except (FileNotFoundError, OSError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(w, n_sample, steps=1, nthreads=0):
    """Oracle FMM (as it stands) on the first n_sample particles' recipe; particles/s.
    nthreads 0 takes every host core (OpenMP over receivers), 1 runs single-threaded."""
    import oracle

    g = W.generate(w, n=n_sample)
    oracle.lib()
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        oracle.fmm(g["pos"], g["mass"], w.p, w.theta, w.leaf, nthreads=nthreads)
        ts.append(time.perf_counter() - t0)
    return n_sample / statistics.median(ts), statistics.median(ts)


def time_direct_sums():
    """The oracle's O(N^2) direct sum (Kahan-compensated, fp64, every host core) on the configurations
    where it runs in full: uniform 4096 and Plummer 1e4; particles/s and seconds."""
    import oracle

    out = {}
    for idx in (1, 2):
        wk = W.WORKLOADS[idx]
        g = W.generate(wk)
        t0 = time.perf_counter()
        oracle.direct_sum(g["pos"], g["mass"], nthreads=0)
        t = time.perf_counter() - t0
        out[wk.name] = {"value": wk.n / t, "unit": "particles/s", "s": t}
    return out


def run_reference(args, rank, world):
    if rank != 0:
        return
    w = W.workload(args.workload)
    n_sample = args.cpu_sample
    vals = []
    t_all = time.perf_counter()
    for _ in range(args.warmup):
        time_oracle(w, n_sample)
    for _ in range(args.steps):
        v, _ = time_oracle(w, n_sample)
        vals.append(v)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": "FMM eval particles/s", "value": value, "unit": "particles/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * n_sample / value,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded generator)",
        "config": {"workload": w.name, "n": w.n, "p": w.p, "theta": w.theta, "leaf": w.leaf},
        "cpu_baseline": {"value": value, "unit": "particles/s", "cores": cpu_cores(), "kind": "oracle",
                         "sample": f"full oracle FMM (keys..P2P, fp64 expansions) on N={n_sample} particles of the "
                                   f"{w.name} recipe, median of {args.steps}"},
        "e2e": {"value": value, "unit": "particles/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_all,
    }
    print(json.dumps(line), flush=True)


def flush_l2(buf):
    buf.fill_(1.0)


def aggregate_over_ranks(local_ms: float, n_local: int, world: int, dist=None, device=None):
    """Whole-job throughput of independent replicas: every rank timed its own
    evaluations; the job takes as long as the slowest rank (max over ranks), and
    all ranks' particles count. Returns (value particles/s, max ms)."""
    total = float(local_ms)
    if dist is not None and world > 1:
        import torch

        t = torch.tensor([total], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total = float(t.item())
    return world * n_local / (total / 1e3), total


KDK_WARMUP, KDK_STEPS = 3, 5  # the KDK leg's fixed window (the clustered state evolves from step to step)


def bench_kdk(w, torch, native, stream):
    """Particles/s per kick-drift-kick step (one force evaluation per step, the
    step's first kick reuses the cached acceleration). The state evolves (the
    halos' velocities are not in equilibrium, so their cores collapse and the
    near field grows), so the leg always times the same steps, KDK_WARMUP + 1
    to KDK_WARMUP + KDK_STEPS from the seeded initial state, whatever --steps
    and --warmup say."""
    g = W.generate(w)
    tdt = torch.float32 if w.dtype == "f32" else torch.float64
    pos = torch.from_numpy(g["pos"]).to("cuda", tdt)
    vel = torch.from_numpy(g["vel"]).to("cuda", tdt)
    mass = torch.from_numpy(g["mass"]).to("cuda", tdt)
    with native.Plan(w.n, w.p, w.theta, w.leaf, w.dtype) as plan, torch.cuda.stream(stream):
        for _ in range(KDK_WARMUP):
            plan.kdk_step(pos, vel, mass, 1e-3, stream=stream)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(KDK_STEPS):
            plan.kdk_step(pos, vel, mass, 1e-3, stream=stream)
        e1.record(stream)
        e1.synchronize()
        ms = e0.elapsed_time(e1) / KDK_STEPS
    return {"value": w.n / (ms / 1e3), "unit": "particles/s per KDK step", "ms_per_step": ms, "dtype": w.dtype,
            "p": w.p, "theta": w.theta, "leaf": w.leaf, "n": w.n,
            "window": f"steps {KDK_WARMUP + 1}..{KDK_WARMUP + KDK_STEPS} from the seeded initial state"}


def bench_vjp(w, steps, warmup, torch, native, stream):
    """One fmm_vjp (the forward evaluation it runs first, then the dipole FMM and
    the leaf terms) per step, particles/s; seeded random cotangents."""
    g = W.generate(w)
    tdt = torch.float32 if w.dtype == "f32" else torch.float64
    pos = torch.from_numpy(g["pos"]).to("cuda", tdt)
    mass = torch.from_numpy(g["mass"]).to("cuda", tdt)
    rng = np.random.default_rng(7)
    abar = torch.from_numpy(rng.normal(size=(w.n, 3))).to("cuda", tdt)
    pbar = torch.from_numpy(rng.normal(size=w.n)).to("cuda", tdt)
    xbar = torch.empty_like(pos)
    mbar = torch.empty_like(mass)
    ms = []
    with native.Plan(w.n, w.p, w.theta, w.leaf, w.dtype) as plan, torch.cuda.stream(stream):
        for _ in range(warmup):
            plan.vjp(pos, mass, abar, pbar, xbar, mbar, stream=stream)
        torch.cuda.synchronize()
        for _ in range(steps):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.vjp(pos, mass, abar, pbar, xbar, mbar, stream=stream)
            e1.record(stream)
            e1.synchronize()
            ms.append(e0.elapsed_time(e1))
        launches = plan.stats()["launches"]
    m = float(np.median(ms))
    return {"value": w.n / (m / 1e3), "unit": "particles/s per VJP (forward evaluation included)", "ms_per_step": m,
            "dtype": w.dtype, "p": w.p, "theta": w.theta, "leaf": w.leaf, "n": w.n, "launches": launches}


def bench_reversibility(torch, native, steps=20, dt=1e-3):
    """Config 5's companion: N = 2^18 fp64, `steps` steps forward then back, with the
    plain floating-point step and with the integer-lattice step; the return error
    max_i |x_i^end - x_i^0| / box side (and the plain step's percentiles)."""
    w = W.KDK_REVERSIBILITY
    g = W.generate(w)
    side = float((g["pos"].max(axis=0) - g["pos"].min(axis=0)).max())
    out = {"n": w.n, "dtype": "f64", "steps": steps, "dt": dt, "p": w.p, "theta": w.theta, "leaf": w.leaf}
    with native.Plan(w.n, w.p, w.theta, w.leaf, "f64") as plan:
        for mode in ("plain", "lattice"):
            x0 = g["pos"].copy()
            v0 = g["vel"].copy()
            if mode == "lattice":
                q = 2.0 ** -40
                x0, v0 = np.rint(x0 / q) * q, np.rint(v0 / q) * q
            tp = torch.from_numpy(x0.copy()).cuda()
            tv = torch.from_numpy(v0.copy()).cuda()
            tm = torch.from_numpy(g["mass"]).cuda()
            plan.kdk_reset()
            step = plan.kdk_step if mode == "plain" else plan.kdk_step_lattice
            for sgn in (1.0, -1.0):
                for _ in range(steps):
                    step(tp, tv, tm, sgn * dt)
            err = np.linalg.norm(tp.cpu().numpy() - x0, axis=1) / side
            out[mode] = {"max": float(err.max()), "p99_9": float(np.percentile(err, 99.9)),
                         "median": float(np.median(err)), "bit_exact": bool(np.array_equal(tp.cpu().numpy(), x0))}
    out["note"] = ("the plain fp64 step misses 1e-9 for a few chaotic close pairs (unsoftened); "
                   "the lattice step returns bit for bit")
    return out


def bench_workload(w, steps, warmup, torch, native, stream, flush_buf, n_override=None, dtype=None, f64_ieee=False,
                   m2l_rotation=False, mutual=False):
    """Times `steps` evaluations; returns dict with per-step ms, stage ms, stats."""
    n = n_override or w.n
    dtype = dtype or w.dtype
    g = W.generate(w, n=n, dtype=dtype)
    tdt = torch.float32 if dtype == "f32" else torch.float64
    pos = torch.from_numpy(g["pos"]).to("cuda", tdt)
    mass = torch.from_numpy(g["mass"]).to("cuda", tdt)
    acc = torch.empty_like(pos)
    pot = torch.empty_like(mass)
    plan = native.Plan(n, w.p, w.theta, w.leaf, dtype, f64_ieee=f64_ieee, m2l_rotation=m2l_rotation, mutual=mutual)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            plan.eval(pos, mass, acc, pot, stream=stream)
        torch.cuda.synchronize()
        step_ms, stages, launches = [], [], 0
        stats = None
        gc.collect()
        gc.disable()  # no collector pause inside a timed step (the host launches every kernel)
        for _ in range(steps):
            flush_l2(flush_buf)
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            plan.eval(pos, mass, acc, pot, stream=stream)
            e1.record(stream)
            e1.synchronize()
            step_ms.append(e0.elapsed_time(e1))
            stats = plan.stats()
            stages.append(stats["stage_ms"])
            launches += stats["launches"]
        gc.enable()
        torch.cuda.synchronize()
    stage_avg = {k: float(np.mean([s[k] for s in stages])) for k in stages[0]}
    return {"plan": plan, "pos": pos, "mass": mass, "g": g, "step_ms": step_ms, "stage_ms": stage_avg,
            "stats": stats, "launches": launches, "n": n}


def bench_e2e(plan, g, steps, torch):
    pos_h = torch.from_numpy(g["pos"]).pin_memory()
    mass_h = torch.from_numpy(g["mass"]).pin_memory()
    acc_h = torch.empty_like(pos_h).pin_memory()
    pot_h = torch.empty_like(mass_h).pin_memory()
    plan.eval_host(pos_h, mass_h, acc_h, pot_h)
    ts = []
    for _ in range(steps):
        t0 = time.perf_counter()
        plan.eval_host(pos_h, mass_h, acc_h, pot_h)
        ts.append(time.perf_counter() - t0)
    h2d = pos_h.numel() * pos_h.element_size() + mass_h.numel() * mass_h.element_size()
    d2h = acc_h.numel() * acc_h.element_size() + pot_h.numel() * pot_h.element_size()
    return plan.n / statistics.median(ts), h2d, d2h


def run_ours(args, rank, world, local_rank):
    import torch

    from body_forces_morton_b300 import native

    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    stream = torch.cuda.Stream()
    flush_buf = torch.empty(64 * 1024 * 1024, dtype=torch.float32, device="cuda")  # 256 MiB > 126 MB L2
    w = W.workload(args.workload)

    def barrier():
        torch.cuda.synchronize()
        if dist:
            dist.barrier()

    sampler = ClockSampler(local_rank)
    barrier()
    sampler.start()
    t_wall = time.perf_counter()
    if args.vjp:
        r = bench_vjp(w, args.steps, args.warmup, torch, native, stream)
        clocks = sampler.stop()
        if rank == 0:
            print(json.dumps({"metric": "FMM VJP particles/s", "value": r["value"], "unit": r["unit"],
                              "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": r["ms_per_step"], "higher_is_better": True, "scaling": "weak",
                              "vs_baseline": None, "dtype": w.dtype, "data": "synthetic (seeded generator)",
                              "config": {"workload": w.name, "n": w.n, "p": w.p, "theta": w.theta, "leaf": w.leaf},
                              "gpu_launches": r["launches"] * args.steps, "clocks": clocks}), flush=True)
        return
    res = bench_workload(w, args.steps, args.warmup, torch, native, stream, flush_buf, n_override=args.n,
                         m2l_rotation=args.m2l_rotation, mutual=args.mutual)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    value, total_ms = aggregate_over_ranks(float(np.sum(res["step_ms"])) / args.steps, res["n"], world, dist,
                                           device="cuda")
    ms_per_step = total_ms

    # secondary points: the other configurations and the benchmark spec's exact sizes
    also = {}
    if not args.no_also:
        n_also = max(3, args.steps // 2)

        def leg(w, name, n=None, dtype=None, f64_ieee=False, roofs=False, m2l_rotation=False, mutual=False):
            r = bench_workload(w, n_also, args.warmup, torch, native, stream, flush_buf, n_override=n, dtype=dtype,
                               f64_ieee=f64_ieee, m2l_rotation=m2l_rotation, mutual=mutual)
            ms = float(np.median(r["step_ms"]))  # median: a rare driver stall of ~3 ms would skew a short mean
            dt = dtype or w.dtype
            d = {"value": r["n"] / (ms / 1e3), "unit": "particles/s", "ms_per_step": ms, "n": r["n"], "dtype": dt,
                 "step_ms_spread": {"min": min(r["step_ms"]), "max": max(r["step_ms"]), "steps": len(r["step_ms"])},
                 "p": w.p, "theta": w.theta, "leaf": w.leaf, "stage_ms": r["stage_ms"],
                 "counts": {k: r["stats"][k] for k in ("n_nodes", "n_m2l", "n_p2p_interactions")}}
            if dt == "f64":
                d["arith"] = (F64_IEEE_ARITH if f64_ieee or m2l_rotation else
                              F64_MUTUAL_ARITH if mutual else F64_ARITH)
            d["m2l_operator"] = "rotation (solid harmonics)" if m2l_rotation else "reduced Cartesian"
            if mutual:
                d["mutual"] = True
            if roofs:
                d["roofline"] = p2p_roofline(r, w, dt, f64_ieee)
                d["m2l_roofline"] = m2l_roofline(r, w, dt, f64_ieee)
                d["eval_roofline"] = eval_roofline(r, w, ms, *hbm_peak_gbs(), dtype=dt, f64_ieee=f64_ieee)
            r["plan"].close()
            also[name] = d

        w3 = W.WORKLOADS[3]
        leg(w3, w3.name, roofs=True)
        leg(w3, w3.name + "_ieee", f64_ieee=True, roofs=True)
        leg(W.WORKLOADS[1], W.WORKLOADS[1].name)
        leg(W.WORKLOADS[2], W.WORKLOADS[2].name)
        leg(w, "clustered_1e6_f32", n=1000000, dtype="f32")
        leg(w, "clustered_1e6_f64", n=1000000, dtype="f64")
        # the two M2L operators (same result): p = 4 at the default workload, p = 8 on the Plummer recipe
        leg(w, w.name + "_m2l_rotation", m2l_rotation=True)
        w3p8 = dataclasses.replace(w3, name="plummer_1e5_f32_p8", p=8, dtype="f32")
        leg(w3p8, w3p8.name)
        leg(w3p8, w3p8.name + "_m2l_rotation", m2l_rotation=True)
        # the mutual evaluation (each unordered pair once, both directions; same result)
        leg(w, w.name + "_mutual", mutual=True)
        leg(w3, w3.name + "_mutual", mutual=True)
        w5 = W.WORKLOADS[5]
        also[w5.name] = bench_kdk(w5, torch, native, stream)
        also["kdk_reversibility_2p18_f64"] = bench_reversibility(torch, native)
        also[w.name + "_vjp"] = bench_vjp(w, n_also, args.warmup, torch, native, stream)

    e2e = None
    if not args.no_e2e:
        e2e_val, h2d, d2h = bench_e2e(res["plan"], res["g"], max(3, args.steps // 2), torch)
        e2e = {"value": e2e_val, "unit": "particles/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
    st = res["stats"]
    src_hash = kernel_source_hash()
    roof = p2p_roofline(res, w)
    roof["traffic"] = TRAFFIC.get((w.name, src_hash)) if args.n is None else None  # captured at the recipe's N
    line = {
        "metric": "FMM eval particles/s", "value": value, "unit": "particles/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        **({"arith": F64_ARITH} if w.dtype == "f64" else {}), "data": "synthetic (seeded generator)",
        "config": {"workload": w.name, "n": res["n"], "p": w.p, "theta": w.theta, "leaf": w.leaf,
                   "l2": "flushed between timed steps (256 MiB write, outside the step events)",
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   **({"mutual": True} if args.mutual else {}),
                   **({"m2l_operator": "rotation (solid harmonics)"} if args.m2l_rotation else {})},
        "step_ms_spread": {"min": min(res["step_ms"]), "median": statistics.median(res["step_ms"]),
                           "max": max(res["step_ms"]), "argmax": int(np.argmax(res["step_ms"]))},
        "stage_ms": res["stage_ms"],
        "counts": {k: st[k] for k in ("n_nodes", "n_leaves", "depth", "n_m2l", "n_p2p", "n_p2p_interactions",
                                      "walk_pairs")},
        "roofline": roof,
        "m2l_roofline": m2l_roofline(res, w),
        "eval_roofline": eval_roofline(res, w, ms_per_step, *hbm_peak_gbs()),
        "e2e": e2e,
        "gpu_launches": res["launches"],
        "clocks": clocks,
        "also": also,
        "wall_s": t_wall,
        "kernel_src": src_hash,
    }
    if rank == 0 and not args.no_cpu:
        v, t = time_oracle(w, args.cpu_sample, steps=3)
        n1 = max(1, args.cpu_sample // 16)
        v1, t1 = time_oracle(w, n1, steps=1, nthreads=1)
        line["cpu_baseline"] = {"value": v, "unit": "particles/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": f"full oracle FMM (fp64 expansions, OpenMP) on N={args.cpu_sample} "
                                          f"particles of the {w.name} recipe, median of 3 runs ({t:.1f} s each)",
                                "single_thread": {"value": v1, "unit": "particles/s", "cores": 1,
                                                  "sample": f"the same on N={n1}, one run ({t1:.1f} s)"},
                                "direct_sum": time_direct_sums()}
    res["plan"].close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def df_pipe_roofline(kernel, pairs, ms):
    """Double-float kernel against the FP32 pipe that executes it (see DF_FMA_OPS_PER_PAIR)."""
    src = kernel_source_hash(DF_SOURCES[kernel])
    ops = DF_FMA_OPS_PER_PAIR.get((kernel, src))
    out = {"kernel": kernel, "bound": "alu", "unit": "FP32 lane-ops/s", "peak": FP32_LANE_OPS_PEAK,
           "peak_note": "derived: 148 SM x 128 FP32 lanes x 2.032 GHz", "source_hash": src}
    if ops is None:
        out.update({"achieved": None, "frac": None, "note": "FMA-pipe operations per pair not counted on this source"})
    else:
        achieved = ops * pairs / (ms / 1e3)
        out.update({"achieved": achieved, "frac": achieved / FP32_LANE_OPS_PEAK, "fma_ops_per_pair": ops})
    return out


def p2p_roofline(res, w, dtype=None, f64_ieee=False):
    """P2P kernel (near field, plus adding the far field and the scatter) against the ALU peak.

    fp32: 20 flop per particle pair against the FP32 peak. fp64 IEEE: the same
    against the FP64 peak. fp64 double-float: against the FP32 pipe it runs on
    (df_pipe_roofline), with the fp64-equivalent rate reported beside it."""
    dtype = dtype or w.dtype
    st = res["stats"]
    ms = res["stage_ms"]["p2p"]
    pairs = st["n_p2p_interactions"] - res["n"]  # zero-separation self pairs are skipped
    achieved = P2P_FLOPS_PER_PAIR * pairs / (ms / 1e3) / 1e12
    flops_note = f"{P2P_FLOPS_PER_PAIR} flop per particle pair, {pairs} pairs per launch"
    if dtype == "f32" or f64_ieee:
        peak = FP32_PEAK_TFLOPS if dtype == "f32" else FP64_PEAK_TFLOPS
        return {"kernel": "k_p2p" if dtype == "f32" else "k_p2p<double>", "bound": "alu", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_note": "derived: 148 SM x 128 FP32 lanes x 2 x 2.032 GHz" if dtype == "f32"
                else "derived: 148 SM x 2 FP64 FMA x 2 x 2.032 GHz",
                "flops_note": flops_note, "ms": ms, "traffic": None}
    out = df_pipe_roofline("k_p2p_df", pairs, ms)
    out.update({"ms": ms, "fp64_equivalent_tflops": achieved, "flops_note": flops_note, "traffic": None})
    return out


def hbm_peak_gbs():
    """HBM copy bandwidth from MEASURED_PEAKS.json (driver-written), else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError, TypeError):
        return 6400.0, "fallback"


def hbm_bytes_per_particle(wbytes):
    """Algorithmic bytes per particle of the memory-bound stages (w = element width in bytes)."""
    return {
        "keys": 3 * wbytes + 8,     # positions read, 8-byte key written (the first pass makes the index)
        "sort": 24 * 8,             # 8 passes, each reading and writing key and index (12 + 12 bytes)
        "gather": 8 * wbytes,       # position and mass read, sorted (x, y, z, m) written
        "tree": 16,                 # sorted keys read for the node boundaries, node records amortised
        "p2m": 4 * wbytes,          # sorted particles read once (moments amortised by the leaf size)
        "l2p": 7 * wbytes,          # particle position read, (phi, a) written
        "scatter": 8 * wbytes,      # (phi, a) read, caller-order outputs written
    }


def eval_roofline(res, w, ms_eval, hbm_gbs, hbm_source, dtype=None, f64_ieee=False):
    """Whole-evaluation roofline fraction: the sum over stages of algorithmic work / peak, over
    the measured evaluation time. P2P and M2L count their flops against the ALU peak of the
    pipe they run on (FP32 for fp32 plans and for the double-float stages of fp64 plans, whose
    fp64-equivalent flops are counted against the FP32 peak; FP64 for IEEE fp64 plans); the
    memory-bound stages count hbm_bytes_per_particle against the HBM copy bandwidth. Stages
    with no algorithmic work of their own (walk, lists, M2M, L2L) count zero."""
    dtype = dtype or w.dtype
    n, st = res["n"], res["stats"]
    alu = (FP64_PEAK_TFLOPS if f64_ieee else FP32_PEAK_TFLOPS) * 1e12
    p2p_ms = P2P_FLOPS_PER_PAIR * (st["n_p2p_interactions"] - n) / alu * 1e3
    m2l_ms = m2l_flops_per_pair(w.p) * st["n_m2l"] / alu * 1e3
    per_particle = hbm_bytes_per_particle(4 if dtype == "f32" else 8)
    hbm_ms = sum(per_particle.values()) * n / (hbm_gbs * 1e9) * 1e3
    ideal = p2p_ms + m2l_ms + hbm_ms
    return {"frac": ideal / ms_eval, "ideal_ms": ideal, "ms": ms_eval,
            "terms_ms": {"p2p_alu": p2p_ms, "m2l_alu": m2l_ms, "hbm": hbm_ms},
            "hbm_bytes_per_particle": per_particle,
            "peaks": {"alu_tflops": alu / 1e12, "hbm_gbs": hbm_gbs, "hbm_source": hbm_source}}


def m2l_flops_per_pair(p):
    """Flops of the reduced (trace-free) M2L per pair: 2 per contraction term,
    sum_{lk} (2 lk + 1) (p - lk + 1)^2 terms, ~10 per derivative of the (p + 1)^2
    with D_z-exponent <= 1, one add for each of the p(p - 1)/2 with exponent 2."""
    terms = sum((2 * lk + 1) * (p - lk + 1) ** 2 for lk in range(p + 1))
    return 2 * terms + 10 * (p + 1) ** 2 + p * (p - 1) // 2


def m2l_roofline(res, w, dtype=None, f64_ieee=False):
    """Algorithmic M2L flops per pair (m2l_flops_per_pair: 566 at p = 4) over the M2L stage time,
    against the FP32 peak (fp32), the FP64 peak (IEEE fp64), or, for the double-float kernels of
    fp64 plans with p <= 4, the FP32 pipe they run on (df_pipe_roofline)."""
    dtype = dtype or w.dtype
    per_pair = m2l_flops_per_pair(w.p)
    ms = res["stage_ms"]["m2l"]
    pairs = res["stats"]["n_m2l"]
    achieved = per_pair * pairs / (ms / 1e3) / 1e12
    if dtype == "f32" or f64_ieee or w.p > 4:
        peak = FP64_PEAK_TFLOPS if dtype == "f64" else FP32_PEAK_TFLOPS
        return {"kernel": "k_m2l" if dtype == "f32" else "k_m2l<double>", "bound": "alu", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak, "flops_per_pair": per_pair,
                "pairs": pairs, "ms": ms}
    out = df_pipe_roofline("k_m2l_df", pairs, ms)
    out.update({"ms": ms, "pairs": pairs, "fp64_equivalent_tflops": achieved, "flops_per_pair": per_pair})
    return out


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="clustered_2p20_f32")
    ap.add_argument("--cpu-sample", type=int, default=1 << 20)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--no-also", action="store_true", help="skip the secondary points (other configs, KDK)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--m2l-rotation", action="store_true", help="main leg: the rotation-based M2L")
    ap.add_argument("--mutual", action="store_true", help="main leg: the mutual evaluation (fmm_plan_set_mutual)")
    ap.add_argument("--n", type=int, default=None,
                    help="main leg: this many particles of the workload's recipe (small ncu captures)")
    ap.add_argument("--vjp", action="store_true", help="main leg: fmm_vjp (forward evaluation + adjoint) per step")
    args = ap.parse_args()
    rank, world, local_rank = env_rank()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
