#!/usr/bin/env python
"""Throughput of the fused log-domain Sinkhorn path on one GB300 (or N, weak scaling).

Workload (per GPU): B=1, n=m=70000, d=64, X ~ N(0, I), Y ~ N(mu, I),
mu ~ N(0, 0.25 I), a, b = softmax of N(0,1) logits, eps = 0.1, 100 fixed
iterations, then cost + gradient wrt X.  One step = one pass of the whole
path over that input: preprocessing, 100 iterations (200 fused half-steps),
the marginal error of the result, and plan application (cost, gradient).

Metric: Sinkhorn pair-evaluations per second, 2 B n m iterations / step time
(one pair-evaluation = one score + exp of one (i, j) in one half-step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]

--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload on this machine's host cores (rank 0 only).
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
import shutil
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sinkhorn_point_cloud_gb300 import datagen  # noqa: E402

WORKLOAD_ID = 4
L2_FLUSH_BYTES = 512 << 20  # > 129 MB L2
METRIC = "Sinkhorn pair-evaluations/s (n=m=70000, d=64)"
UNIT = "Gpair-evals/s"


KERNEL_SOURCES = {
    "tc_half_kernel": ["k_tc.cu", "tc_ptx.cuh", "common.cuh", "tc.h", "kernels.h"],
    "tc_screen_kernel": ["k_tc.cu", "tc_ptx.cuh", "common.cuh", "tc.h", "kernels.h"],
    "dense_half_kernel": ["k_dense.cu", "common.cuh", "kernels.h"],
    "point_half_kernel": ["k_point.cu", "common.cuh", "kernels.h"],
    "point_cluster_kernel": ["k_cluster.cu", "common.cuh", "kernels.h"],
}


def kernel_source_hash(kernel: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "sinkhorn_point_cloud_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from profiles/traffic.json,
    or None when no capture exists or the kernel source changed since it was taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        entries = json.load(fh)
    for e in entries:
        if e.get("kernel") == kernel and e.get("workload") == workload and \
                e.get("source_hash") == kernel_source_hash(kernel):
            return e.get("bytes_per_launch")
    return None


def metric_name(wid: int) -> str:
    if wid == WORKLOAD_ID:
        return METRIC
    return f"Sinkhorn pair-evaluations/s ({datagen.WORKLOADS[wid]['name']})"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            return json.load(fh), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "sm_max_mhz": 2070.0}, \
        "fallback"


def alu_rates():
    """Measured per-SM-per-clock rates of MUFU ex2, FFMA lanes and packed f32x2
    FMA lanes (libsotpeaks probes), or None if the probe library is absent."""
    import ctypes as C
    from sinkhorn_point_cloud_gb300 import build
    if not os.path.exists(build.PEAKS_LIB):
        return None
    L = C.CDLL(build.PEAKS_LIB)
    L.sotpeaks_measure.argtypes = [C.c_int, C.POINTER(C.c_double)]
    out = {}
    for kind, name in ((0, "ex2_per_sm_clk"), (1, "ffma_lanes_per_sm_clk"), (2, "ffma2_lanes_per_sm_clk")):
        v = C.c_double(0)
        if L.sotpeaks_measure(kind, C.byref(v)) != 0:
            return None
        out[name] = round(v.value, 2)
    return out


# ---- clocks ---------------------------------------------------------------
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    def __init__(self, index: int, out_path: str | None = None):
        self.index = index
        self.proc = None
        self.path = out_path

    def __enter__(self):
        if shutil.which("nvidia-smi"):
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()
            if self.path:
                with open(self.path, "w") as fh:
                    fh.write(self.text)
        return False

    def summary(self):
        return parse_clocks(getattr(self, "text", ""))


def parse_clocks(text: str):
    sm, mx, reasons = [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for row in csv.reader(io.StringIO(text)):
        if len(row) < 9:
            continue
        try:
            sm.append(float(row[1]))
            mx.append(float(row[2]))
        except ValueError:
            continue
        for nm, v in zip(names, row[5:9]):
            if v.strip().lower() == "active":
                reasons.add(nm)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
            "samples": len(sm)}


# ---- distributed helpers ------------------------------------------------------
def clocks_csv_path():
    """Where to keep the raw nvidia-smi samples of the timed region (the JSON
    line carries their summary either way): $SOT_CLOCKS_CSV, or nowhere."""
    return os.environ.get("SOT_CLOCKS_CSV") or None


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(value: float, ws: int, device=None) -> float:
    if ws <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# ---- reference arm: the fp64 oracle on host cores -------------------------------
def oracle_rate(target_s: float, X, Y, b, eps, cost="sqeuclidean"):
    """Time the oracle's f-half on a sample of rows (all m columns) for about
    target_s seconds; when every row fits in less time, whole f-halves are
    repeated.  Returns (pair-evals/s, sample description, seconds, threads)."""
    from oracle import oracle as O
    orc = O.get()
    with orc.cost(cost):
        return _oracle_rate(orc, target_s, X, Y, b, eps)


def oracle_single_core(target_s: float, X, Y, b, eps, cost="sqeuclidean"):
    """The same oracle sample with one OpenMP thread: {"value" (G pair-evals/s),
    "sample"}.  The oracle's thread count is restored afterwards."""
    from oracle import oracle as O
    orc = O.get()
    threads = orc.num_threads
    orc.set_num_threads(1)
    try:
        with orc.cost(cost):
            r, sample, _, _ = _oracle_rate(orc, target_s, X, Y, b, eps)
    finally:
        orc.set_num_threads(threads)
    return {"value": r / 1e9, "sample": sample}


def _oracle_rate(orc, target_s, X, Y, b, eps):
    m = Y.shape[0]
    g = np.zeros(m)
    rows = min(X.shape[0], 2 * orc.num_threads)
    t0 = time.perf_counter()
    orc.f_half(X[:rows], Y, b, g, eps)
    t = max(time.perf_counter() - t0, 1e-4)
    rows = int(max(min(orc.num_threads, X.shape[0]), min(X.shape[0], rows * target_s / t)))
    reps = 0
    t0 = time.perf_counter()
    while True:  # whole f-halves are repeated when all rows take less than target_s
        orc.f_half(X[:rows], Y, b, g, eps)
        reps += 1
        t = time.perf_counter() - t0
        if rows < X.shape[0] or t >= 0.9 * target_s:
            break
    sample = f"f-half of {rows} rows x {m} columns (d={X.shape[1]})" + (f", {reps} times" if reps > 1 else "") + \
        f", {t:.1f} s"
    return reps * rows * m / t, sample, t, orc.num_threads


def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    w = datagen.WORKLOADS[args.workload]
    X, Y, a, b = datagen.make_batch(args.workload, B=1)
    rates = []
    for _ in range(args.warmup):
        oracle_rate(0.5, X[0], Y[0], b[0], w["eps"], args.cost)
    sample = None
    for _ in range(args.steps):
        r, sample, t, thr = oracle_rate(args.ref_step_s, X[0], Y[0], b[0], w["eps"], args.cost)
        rates.append(r)
    value = float(np.median(rates)) / 1e9
    one = oracle_single_core(args.ref_step_s / 3, X[0], Y[0], b[0], w["eps"], args.cost)
    # one whole step at this rate (the annealed workload: its 67 stages of 20
    # iterations, the least it runs)
    iters = w.get("iters") or 67 * w["iters_per_stage"]
    ms_step = 2.0 * w["B"] * w["n"] * w["m"] * iters / (value * 1e9) * 1e3 if value > 0 else None
    line = {"impl": "reference", "metric": metric_name(args.workload), "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "ms_per_step_basis": "one whole step of the workload at the sampled rate",
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w["name"], "B": w["B"], "n": w["n"], "m": w["m"], "d": w["d"], "eps": w["eps"],
                       "iters": w.get("iters"), **({"cost": "cosine"} if args.cost == "cosine" else {})},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample,
                             "single_core": one},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---- GPU arm -------------------------------------------------------------------
def run_gpu(args, ws, rank, local):
    import torch
    import sinkhorn_point_cloud_gb300 as sot
    from sinkhorn_point_cloud_gb300 import build

    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()
    wid = args.workload
    w = datagen.WORKLOADS[wid]
    B, n, m, d, eps = w["B"], w["n"], w["m"], w["d"], w["eps"]
    iters = w.get("iters", 0)
    if args.n:
        n = m = args.n
    if args.d:
        d = args.d
    if args.iters:
        iters = args.iters
    # weak scaling: every rank solves its own problem(s), seeded by rank
    X, Y, a, b = datagen.make_batch(wid, B=B, n=n, m=m, d=d, clouds=range(rank * B, rank * B + B))
    weighted = w["kind"] == "gauss"  # the other recipes use uniform weights (NULL in the ABI)
    host_in = [torch.from_numpy(v).pin_memory() for v in ((X, Y, a, b) if weighted else (X, Y))]
    dev_in = [v.to(dev) for v in host_in]
    flags = {"auto": sot.SOT_PREC_AUTO, "fp32": sot.SOT_PREC_FP32, "f16x3": sot.SOT_PREC_F16X3}[args.prec]
    if args.no_screen:
        flags |= sot.SOT_TC_NO_SCREEN
    if args.no_cluster:
        flags |= sot.SOT_NO_CLUSTER
    if args.cost == "cosine":
        flags |= sot.SOT_COST_COSINE
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step(ins):
        Xs, Ys = ins[0], ins[1]
        As, Bs = (ins[2], ins[3]) if weighted else (None, None)
        if wid == 3:
            f, g, info = sot.sot_potentials_ex(Xs, Ys, As, Bs, eps=eps, eps_init=w["eps_init"],
                                               eps_factor=w["eps_factor"], iters_per_stage=w["iters_per_stage"],
                                               max_iters=w["max_iters"], tol=w["tol"], flags=flags, stats=True)
            return [f, g], info
        f, g, info = sot.sot_potentials_ex(Xs, Ys, As, Bs, eps=eps, iters_per_stage=iters, max_iters=iters,
                                           flags=flags, stats=True)
        if wid == 5:
            coo = sot.sot_plan_coo(Xs, Ys, As, Bs, f, g, eps, threshold=w["tau"], dirs=3)
            gs = sot.sot_grad_x_coo(Xs, Ys, coo["rows"], coo["cols"], coo["vals"], coo["batch_offsets"])
            info["nnz"] = coo["nnz"]
            return [coo["rows"], coo["cols"], coo["vals"], gs], info
        cost, grad, _ = sot.sot_plan_apply(Xs, Ys, As, Bs, f, g, eps, flags=flags & (3 | sot.SOT_COST_COSINE))
        return [cost, grad], info

    def step_pairs(info):
        return 2.0 * B * n * m * info["iters_done"]

    for _ in range(args.warmup):
        step(dev_in)
    torch.cuda.synchronize()

    # ---- device-resident timing, L2 flushed before every step -------------
    launches0 = sot.sot_kernel_launches()
    sot.sot_profile_read()
    sot.sot_profile_enable(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    clk_path = clocks_csv_path()
    barrier(ws)
    torch.cuda.synchronize()
    info = None
    pairs_total = 0.0
    with ClockSampler(local, clk_path) as cs:
        t_wall0 = time.perf_counter()
        for k in range(args.steps):
            flush_buf.zero_()
            ev[k][0].record(stream)
            outs, info = step(dev_in)
            ev[k][1].record(stream)
            pairs_total += step_pairs(info)
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall0
    barrier(ws)
    sot.sot_profile_enable(False)
    kinds = sot.sot_profile_read_kinds()
    nl = sum(v[0] for v in kinds.values())
    half_ms = sum(v[1] for v in kinds.values())
    launches = sot.sot_kernel_launches() - launches0
    step_ms = [e0.elapsed_time(e1) for e0, e1 in ev]
    t_dev = sum(step_ms) / 1e3
    t_max = max_over_ranks(t_dev, ws, dev)
    clocks = cs.summary()

    # ---- end to end through the public API with host buffers -------------------
    h2d = sum(v.numel() * v.element_size() for v in host_in)
    d2h = 0
    barrier(ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms, e2e_pairs = 0.0, 0.0
    for k in range(0 if args.no_e2e else args.steps):
        flush_buf.zero_()
        e0.record(stream)
        ins = [v.to(dev, non_blocking=True) for v in host_in]
        outs, inf2 = step(ins)
        hosts = [o.to("cpu", non_blocking=True) for o in outs]
        e1.record(stream)
        e1.synchronize()
        d2h = sum(o.numel() * o.element_size() for o in outs)
        e2e_ms += e0.elapsed_time(e1)
        e2e_pairs += step_pairs(inf2)
    e2e_max = max_over_ranks(e2e_ms / 1e3, ws, dev) if not args.no_e2e else None

    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    # the dominant kernel: the kind that took the most time (per half-step averages;
    # a cluster-resident launch counts the half-steps it covers)
    dom = max(kinds, key=lambda k: kinds[k][1])
    nl_dom, ms_dom = kinds[dom]
    per_launch_ms = ms_dom / max(nl_dom, 1)
    per_launch_pairs = B * n * m
    mhz = float(pk.get("sm_max_mhz", 2070.0))
    rates = alu_rates()
    secs = per_launch_ms / 1e3
    mufu = None
    if rates and dom != "screened":  # a screened half-step forms exponentials for the kept pairs only
        mufu_peak = rates["ex2_per_sm_clk"] * sms * mhz * 1e6
        mufu = {"achieved_ex2_per_s": per_launch_pairs / secs, "peak_ex2_per_s": mufu_peak,
                "frac": per_launch_pairs / secs / mufu_peak}
    path = sot.sot_select_path(d, flags)
    if path == 2:
        if dom == "screened":
            flops_pair = 2 * d  # one fp16 product hi*hi per pair, 2 flops per multiply-add
            kname, kern = "tc_screen_kernel", "tc_screen_kernel (tcgen05 kind::f16 hi*hi screen + exact kept pairs)"
        else:
            flops_pair = 3 * 2 * d  # fp16 products hi*hi + hi*lo + lo*hi, 2 flops per multiply-add
            kname, kern = "tc_half_kernel", "tc_half_kernel (tcgen05 kind::f16, 3 products per pair)"
        achieved = flops_pair * per_launch_pairs / secs / 1e12
        peak = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": measured_traffic(kname, w["name"]),
                "peak_source": f"{pk_kind} sustained bf16 dense GEMM (fp16 has the same nominal rate)",
                "kernel": kern}
        dtype = "f16x3"
    else:
        lanes = rates["ffma_lanes_per_sm_clk"] if rates else 128.0
        src = f"{'measured' if rates else 'nominal'} {lanes:.0f} FP32 lanes/SM/clk x {sms} SMs x {mhz:.0f} MHz"
        if path == 1:
            ops_pair, unit, kern = 2 * d, "TFLOP/s", "dense_half_kernel (fp32 FMA, 2 flops per FMA)"
            peak = 2 * lanes * sms * mhz * 1e6 / 1e12
            src += " x 2"
        else:
            # direct form: one FADD for the bias, d x (FADD + FFMA) for the distance, one FADD into the sum
            ops_pair, unit = 2 + 2 * d, "Tops/s"
            if dom == "cluster":
                # the cluster-resident kernel evaluates all three coordinates
                ops_pair = 8
                kern = "point_cluster_kernel (cluster-resident iterations; 8 FP32 lane-ops + 1 MUFU ex2 per pair)"
            else:
                kern = f"point_half_kernel ({2 + 2 * d} FP32 lane-ops + 1 MUFU ex2 per pair)"
            peak = lanes * sms * mhz * 1e6 / 1e12
        achieved = ops_pair * per_launch_pairs / secs / 1e12
        kname = "dense_half_kernel" if path == 1 else ("point_cluster_kernel" if dom == "cluster" else "point_half_kernel")
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": unit, "frac": achieved / peak,
                "traffic": measured_traffic(kname, w["name"]), "peak_source": src, "kernel": kern}
        dtype = "f32"
    roof["mufu"] = mufu
    roof["alu_rates"] = rates
    # CPU baseline: the oracle on a bounded sample of the same workload
    cpu = None
    if not args.no_cpu_baseline and ws == 1:  # rank 0 at N = 1 only
        r, sample, t, thr = oracle_rate(args.cpu_baseline_s, X[0], Y[0], b[0], eps, args.cost)
        cpu = {"value": r / 1e9, "unit": UNIT, "cores": thr, "kind": "oracle", "sample": sample,
               "single_core": oracle_single_core(args.cpu_baseline_s / 5, X[0], Y[0], b[0], eps, args.cost)}
    value = ws * pairs_total / t_max / 1e9
    line = {
        "metric": metric_name(wid), "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": dtype, "data": "synthetic",
        "config": {"workload": w["name"], "B": B, "n": n, "m": m, "d": d, "eps": eps,
                   "iters": info["iters_done"], **({"stages": info["stages_done"]} if wid == 3 else {}),
                   **({"nnz": info.get("nnz")} if wid == 5 else {}),
                   **({"cost": "cosine"} if args.cost == "cosine" else {}),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "flushed (512 MiB write) before every timed step"},
        "iters_per_s": ws * sum([info["iters_done"]]) * args.steps / t_max,
        "half_step": {"count": nl, "avg_ms": half_ms / max(nl, 1), "pairs_per_half_step": per_launch_pairs,
                      **{k: {"count": v[0], "avg_ms": v[1] / max(v[0], 1)} for k, v in kinds.items()}},
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": None if e2e_max is None else {"value": ws * e2e_pairs / e2e_max / 1e9, "unit": UNIT,
                                             "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": int(launches),
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "marginal_err": max(info["err"]) if info else None,
        "wall_s": t_wall,
    }
    print(json.dumps(line), flush=True)
    return 0


def setup_device(ws, local):
    """One GPU per rank (NCCL process group for N > 1), the library built."""
    import torch
    from sinkhorn_point_cloud_gb300 import build

    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    build.build()
    return torch.device("cuda", local)


def time_steps(step, args, ws, local, dev):
    """Warm-up, then args.steps steps bracketed by CUDA events on the current
    stream, L2 flushed before each and clocks sampled meanwhile.  Returns
    (max-over-ranks seconds, clock summary, kernel launches)."""
    import torch
    import sinkhorn_point_cloud_gb300 as sot

    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    launches0 = sot.sot_kernel_launches()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local, clocks_csv_path()) as cs:
        for k in range(args.steps):
            flush_buf.zero_()
            ev[k][0].record(stream)
            step()
            ev[k][1].record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    launches = sot.sot_kernel_launches() - launches0
    t_max = max_over_ranks(sum(e0.elapsed_time(e1) for e0, e1 in ev) / 1e3, ws, dev)
    return t_max, cs.summary(), launches


def run_transport(args, ws, rank, local):
    """Transport-matrix products (sot_transport_apply): one step is P V (V with
    `args.transport` columns) and P^T U on a workload, from potentials solved
    once before the timed region.  Same timing rules as the solver line."""
    import torch
    import sinkhorn_point_cloud_gb300 as sot

    dev = setup_device(ws, local)
    wid = args.workload
    w = datagen.WORKLOADS[wid]
    B, n, m, d, eps = w["B"], w["n"], w["m"], w["d"], w["eps"]
    if args.n:
        n = m = args.n
    c = args.transport
    flags = sot.SOT_COST_COSINE if args.cost == "cosine" else 0
    X, Y, a, b = datagen.make_batch(wid, B=B, n=n, m=m, clouds=range(rank * B, rank * B + B))
    weighted = w["kind"] == "gauss"
    Xd, Yd = torch.from_numpy(X).to(dev), torch.from_numpy(Y).to(dev)
    ad, bd = (torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)) if weighted else (None, None)
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=args.iters or 100,
                                 max_iters=args.iters or 100, flags=flags)
    rng = np.random.default_rng(20260700 + rank)
    host_in = [torch.from_numpy(rng.standard_normal((B, m, c)).astype(np.float32)).pin_memory(),
               torch.from_numpy(rng.standard_normal((B, n, c)).astype(np.float32)).pin_memory()]
    V, U = [v.to(dev) for v in host_in]
    outs = [torch.empty(B, n, c, device=dev), torch.empty(B, m, c, device=dev)]
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    gy = torch.empty(B, m, d, device=dev) if args.grad_y else None

    def step(v, u):
        if args.grad_y:  # the gradient with respect to Y: P^T X and a pointwise step
            return [sot.sot_grad_y(Xd, Yd, ad, bd, f, g, eps, flags=flags, out=gy)]
        o0 = sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, v, side=0, flags=flags, out=outs[0])
        o1 = sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, u, side=1, flags=flags, out=outs[1])
        return [o0, o1]

    t_max, clocks, launches = time_steps(lambda: step(V, U), args, ws, local, dev)
    # end to end: V and U from pinned host memory, both products back to the host
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = 0.0
    for k in range(0 if args.no_e2e else args.steps):
        flush_buf.zero_()
        e0.record(stream)
        v, u = [h.to(dev, non_blocking=True) for h in host_in]
        hosts = [o.to("cpu", non_blocking=True) for o in step(v, u)]
        e1.record(stream)
        e1.synchronize()
        e2e_ms += e0.elapsed_time(e1)
    e2e_max = max_over_ranks(e2e_ms / 1e3, ws, dev) if not args.no_e2e else None
    if rank != 0:
        return 0
    pairs_step = (1.0 if args.grad_y else 2.0) * B * n * m
    pk, pk_kind = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rates = alu_rates()
    lanes = rates["ffma_lanes_per_sm_clk"] if rates else 128.0
    mhz = float(pk.get("sm_max_mhz", 2070.0))
    # the fp32 screen of every pair: a subtraction and an FMA per coordinate, one
    # FMA for the exponent estimate (the exact evaluation of the pairs that
    # matter and the c FMAs of their terms are extra work, not counted)
    ops_pair = 2 * d + 1
    achieved = ops_pair * pairs_step * args.steps / t_max / 1e12
    peak = lanes * sms * mhz * 1e6 / 1e12
    cpu = None
    if not args.no_cpu_baseline and ws == 1:  # rank 0 at N = 1 only
        from oracle import oracle as O
        orc = O.get()
        rows = max(1, min(n, int(64 * orc.num_threads)))
        fh, gh = f[0].double().cpu().numpy(), g[0].double().cpu().numpy()
        t0 = time.perf_counter()
        with orc.cost(args.cost):
            orc.transport(X[0][:rows], Y[0], a[0][:rows] if weighted else None, b[0] if weighted else None,
                          fh[:rows], gh, eps, host_in[0][0].numpy(), side=0)
        tc = time.perf_counter() - t0
        cpu = {"value": rows * m / tc / 1e9, "unit": UNIT, "cores": orc.num_threads, "kind": "oracle",
               "sample": f"P V on {rows} rows x {m} columns, c={c} (d={d}), {tc:.1f} s"}
    line = {
        "metric": (f"gradient with respect to Y pair-evaluations/s ({w['name']})" if args.grad_y else
                   f"transport products P V, P^T U pair-evaluations/s ({w['name']}, c={c})"),
        "value": ws * pairs_step * args.steps / t_max / 1e9, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w["name"], "B": B, "n": n, "m": m, "d": d, "eps": eps, "c": c,
                   **({"cost": "cosine"} if args.cost == "cosine" else {}),
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "flushed (512 MiB write) before every timed step"},
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tops/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"FP32 lanes/SM/clk from the ALU probe x {sms} SMs x {mhz:.0f} MHz",
                     "kernel": f"transport_kernel ({ops_pair} FP32 lane-ops per pair in the screen)"},
        "cpu_baseline": cpu,
        "e2e": None if e2e_max is None else {"value": ws * pairs_step * args.steps / e2e_max / 1e9, "unit": UNIT,
                                             "h2d_bytes_per_step": 0 if args.grad_y else
                                             sum(h.numel() * 4 for h in host_in),
                                             "d2h_bytes_per_step": gy.numel() * 4 if args.grad_y else
                                             sum(o.numel() * 4 for o in outs)},
        "gpu_launches": int(launches),
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_apml(args, ws, rank, local):
    """Sparse APML (sot_apml_coo) on the support sot_plan_coo extracts from a
    solved workload, `args.apml` normalisations, temperature eps; one step is
    one call (softmaxes, symmetrisation, normalisations, loss, support
    gradient).  Same timing rules as the solver line."""
    import torch
    import sinkhorn_point_cloud_gb300 as sot

    dev = setup_device(ws, local)
    wid = args.workload
    w = datagen.WORKLOADS[wid]
    B, n, m, d, eps = w["B"], w["n"], w["m"], w["d"], w["eps"]
    if args.n:
        n = m = args.n
    X, Y, a, b = datagen.make_batch(wid, B=B, n=n, m=m, clouds=range(rank * B, rank * B + B))
    weighted = w["kind"] == "gauss"
    Xd, Yd = torch.from_numpy(X).to(dev), torch.from_numpy(Y).to(dev)
    ad, bd = (torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)) if weighted else (None, None)
    iters = args.iters or w.get("iters", 100)
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters)
    coo = sot.sot_plan_coo(Xd, Yd, ad, bd, f, g, eps, threshold=w.get("tau", 1e-8), dirs=3)
    nnz = int(coo["nnz"])
    K = args.apml
    t_max, clocks, launches = time_steps(lambda: sot.sot_apml_coo(Xd, Yd, ad, bd, coo, eps, K), args, ws, local,
                                         dev)
    if rank != 0:
        return 0
    pk, pk_kind = peaks()
    # algorithmic bytes per stored entry of the factored passes: validation and
    # cost read both indices and write C (12 B); the row softmax statistics read
    # C and the column (8 B); the symmetrisation reads them again and writes S
    # (12 B); each further normalisation reads S and the column (8 B); the last
    # pass reads S, the column and C and writes P (16 B; 12 B without
    # normalisations, P being S).  The support gradient is fused into the last
    # pass for d <= 3; otherwise its own pass reads both indices and P (12 B).
    bytes_entry = 12 + 8 + 12 + (8 * (K - 1) + 16 if K > 0 else 12) + (0 if d <= 3 else 12)
    achieved = bytes_entry * nnz * args.steps / t_max / 1e9
    peak = float(pk.get("hbm_gbs", 6800.0))
    line = {
        "metric": f"sparse APML stored entries/s ({w['name']}, {K} normalisations)",
        "value": ws * nnz * args.steps / t_max / 1e9, "unit": "Gentries/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w["name"], "B": B, "n": n, "m": m, "d": d, "eps": eps, "T": eps, "nnz": nnz,
                   "normalisations": K, "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "flushed (512 MiB write) before every timed step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": None, "peak_source": f"{pk_kind} HBM copy bandwidth",
                     "kernel": f"APML passes ({bytes_entry} algorithmic bytes per stored entry)"},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": int(launches),
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_hvp(args, ws, rank, local):
    """Hessian-vector products (sot_hvp) on a d <= 9 workload, from potentials
    solved once before the timed region: one step is one H V with exactly
    `args.hvp` conjugate-gradient steps (cg_tol = 0), i.e. 3 + 2 K transport
    products of n x m pairs per cloud.  Same timing rules as the solver line."""
    import torch
    import sinkhorn_point_cloud_gb300 as sot

    dev = setup_device(ws, local)
    wid = args.workload
    w = datagen.WORKLOADS[wid]
    B, n, m, d, eps = w["B"], w["n"], w["m"], w["d"], w["eps"]
    if args.n:
        n = m = args.n
    X, Y, a, b = datagen.make_batch(wid, B=B, n=n, m=m, clouds=range(rank * B, rank * B + B))
    weighted = w["kind"] == "gauss"
    Xd, Yd = torch.from_numpy(X).to(dev), torch.from_numpy(Y).to(dev)
    ad, bd = (torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)) if weighted else (None, None)
    iters = args.iters or w.get("iters") or 100
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters)
    rng = np.random.default_rng(20260800 + rank)
    host_v = torch.from_numpy(rng.standard_normal((B, n, d)).astype(np.float32)).pin_memory()
    Vd = host_v.to(dev)
    out = torch.empty(B, n, d, device=dev)
    K = args.hvp
    t_max, clocks, launches = time_steps(
        lambda: sot.sot_hvp(Xd, Yd, ad, bd, f, g, eps, Vd, cg_iters=K, cg_tol=0.0, out=out), args, ws, local, dev)
    if rank != 0:
        return 0
    pairs_step = (3 + 2 * K) * B * n * m
    pk, pk_kind = peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    rates = alu_rates()
    lanes = rates["ffma_lanes_per_sm_clk"] if rates else 128.0
    mhz = float(pk.get("sm_max_mhz", 2070.0))
    ops_pair = 2 * d + 1  # the transport kernel's fp32 screen of every pair
    achieved = ops_pair * pairs_step * args.steps / t_max / 1e12
    peak = lanes * sms * mhz * 1e6 / 1e12
    line = {
        "metric": f"Hessian-vector products/s ({w['name']}, {K} CG steps)",
        "value": ws * B * args.steps / t_max, "unit": "HVP/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": w["name"], "B": B, "n": n, "m": m, "d": d, "eps": eps, "cg_iters": K,
                   "parallelism": f"replicas x{ws}" if ws > 1 else "single GPU",
                   "l2": "flushed (512 MiB write) before every timed step"},
        "pair_evals_per_s": ws * pairs_step * args.steps / t_max / 1e9, "pair_evals_unit": UNIT,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "Tops/s",
                     "frac": achieved / peak, "traffic": None,
                     "peak_source": f"FP32 lanes/SM/clk from the ALU probe x {sms} SMs x {mhz:.0f} MHz",
                     "kernel": f"transport_kernel ({ops_pair} FP32 lane-ops per pair in the screen, "
                               f"{3 + 2 * K} products per step)"},
        "cpu_baseline": None,
        "e2e": None,
        "gpu_launches": int(launches),
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
    }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--prec", choices=["auto", "fp32", "f16x3"], default="auto")
    ap.add_argument("--workload", type=int, choices=sorted(datagen.WORKLOADS), default=WORKLOAD_ID,
                    help="1-5; the default (4: n=m=70000, d=64) is the headline configuration")
    ap.add_argument("--n", type=int, default=0, help="override n = m (testing only)")
    ap.add_argument("--d", type=int, default=0, help="override d (the Gaussian recipe; testing only)")
    ap.add_argument("--iters", type=int, default=0, help="override the iteration count (testing only)")
    ap.add_argument("--ref-step-s", type=float, default=3.0, help="seconds of oracle work per reference step")
    ap.add_argument("--cpu-baseline-s", type=float, default=15.0,
                    help="seconds of oracle work for the cpu_baseline sample of the GPU arm")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg (profiling runs)")
    ap.add_argument("--no-screen", action="store_true", help="tensor path: full half-steps only (comparison runs)")
    ap.add_argument("--no-cluster", action="store_true",
                    help="point path: streaming half-steps only, no cluster-resident iterations (comparison runs)")
    ap.add_argument("--transport", type=int, default=0, metavar="C",
                    help="time the transport products P V and P^T U with C columns instead of the solver")
    ap.add_argument("--grad-y", action="store_true", help="with --transport: time sot_grad_y instead")
    ap.add_argument("--apml", type=int, default=0, metavar="K",
                    help="time sparse APML with K normalisations on the workload's COO support instead")
    ap.add_argument("--hvp", type=int, default=0, metavar="K",
                    help="time Hessian-vector products with K CG steps on a d <= 9 workload instead")
    ap.add_argument("--cost", choices=["sqeuclidean", "cosine"], default="sqeuclidean",
                    help="cost function (cosine: 2 - 2 cos, on the normalised points)")
    args = ap.parse_args(argv)
    if args.cost == "cosine" and args.workload == 5:
        ap.error("the COO workload runs with the squared-Euclidean cost only")
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    if args.transport:
        return run_transport(args, ws, rank, local)
    if args.apml:
        return run_apml(args, ws, rank, local)
    if args.hvp:
        return run_hvp(args, ws, rank, local)
    return run_gpu(args, ws, rank, local)


if __name__ == "__main__":
    sys.exit(main())
