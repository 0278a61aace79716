#!/usr/bin/env python
"""Selective-scan forward bench: HBM GB/s, (b*d*l) elements/s and the fraction
of the GB300 HBM roofline, on seeded synthetic Mamba-layer workloads.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference] [--shard]

One step = one selective-scan forward over the whole workload (all of the
path: softplus, exp, recurrence, C contraction, D skip, silu gate, last_state),
inputs resident in HBM. Each step is preceded (outside its timed interval) by a
write of 2x the L2 size so that no input is served from L2. Kernel time is
measured with CUDA events on the launching stream; the reported time is the
max over ranks.

Without --workload the scan bench times the four full-size workloads one after
the other in the same process and prints one line for the largest
(long_fixed_fp32) with all four under "per_config". Under torchrun every rank
runs its own copy of the workload (independent problems, no data-path
collective: weak scaling); with --shard the ranks split ONE problem over batch
x dim instead (whole groups where the rows allow; strong scaling).

--impl reference times the fp64 CPU oracle (as it stands) on the host cores on
bounded samples of the same workload, in the same metric.
"""
from __future__ import annotations

import argparse
import ctypes
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from state_space_model_03_gb300 import workloads  # noqa: E402

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")
METRIC = "selective-scan fwd HBM GB/s (compulsory bytes / kernel time)"
DEFAULT_WORKLOAD = "mamba130m_bf16"
# FP32 lane-ops per (state, step) pair on the dominant path: exponent product,
# dt*u*B product, state FMA, C contraction FMA (3 for fixed B/C, where the
# state is carried as x / B).
PAIR_FP32_OPS = {"variable": 4, "fixed": 3}


def _env_int(k, d):
    try:
        return int(os.environ.get(k, d))
    except ValueError:
        return d


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# Sources that define each timed kernel (its traffic record stays valid while
# these files are unchanged).
KERNEL_SOURCES = {
    "scan": ("ss_fwd_kernel.cuh", "ss_fwd_instances.cuh", "ss_fwd_f32.cu", "ss_fwd_f16.cu", "ss_fwd_bf16.cu",
             "ss_fwd_lane.cu"),
    "state_update": ("ss_state_update.cu", "ss_fwd_kernel.cuh"),
    "conv1d": ("ss_conv1d.cu", "ss_fwd_kernel.cuh"),
    "bwd": ("ss_bwd.cu", "ss_fwd_kernel.cuh"),
    "complex": ("ss_fwd_complex.cu", "ss_fwd_kernel.cuh"),
}


def _kernel_hash(op="scan"):
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[op]:
        with open(os.path.join(ROOT, "state_space_model_03_gb300", "csrc", name), "rb") as fh:
            h.update(name.encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def _traffic(workload, op="scan"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources and this workload; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != _kernel_hash(op):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons, power, util = [], None, set(), [], []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm_v, mx_v, p_v, u_v = float(f[0]), float(f[1]), float(f[2]), float(f[3])
            except ValueError:
                continue
            sm.append(sm_v)
            mx = mx_v
            power.append(p_v)
            util.append(u_v)
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        loaded = [s for s, u in zip(sm, util) if u >= 50.0] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_under_load": len(loaded),
                "power_w_max": max(power) if power else None}


def max_over_ranks(values, world, device=None):
    """Element-wise max of per-rank timings (one tiny all-reduce of the
    timings themselves; the selective scan has no data-path collective)."""
    import torch
    t = torch.tensor(list(values), dtype=torch.float64, device=device)
    if world > 1:
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(v) for v in t]


def job_rate(units_per_rank, world, ms):
    """Whole-job rate: every rank processes its own copy of the workload
    (weak scaling), in the slowest rank's time."""
    return world * units_per_rank / (ms * 1e-3)


def _oracle_rows_rate(w, x, rows, threads):
    import oracle
    t0 = time.perf_counter()
    oracle.selective_scan_rows(rows, **{k: x[k] for k in NAMES}, delta_softplus=x["delta_softplus"],
                               threads=threads)
    return time.perf_counter() - t0


def _row_bytes(w):
    """Compulsory bytes of one (batch, channel) row, for sampled CPU timing."""
    return workloads.compulsory_bytes(w) / (w.batch * w.dim)


def cpu_baseline(w, x, budget_s=15.0):
    """Oracle timed on a bounded sample of rows (all host cores)."""
    import numpy as np
    threads = os.cpu_count() or 1
    rng = np.random.default_rng(0)
    nrows = w.batch * w.dim
    probe = [(int(r // w.dim), int(r % w.dim)) for r in rng.choice(nrows, size=min(nrows, threads), replace=False)]
    dt = _oracle_rows_rate(w, x, probe, threads)
    per_row = dt / len(probe) * min(threads, len(probe))  # seconds of one row on one core
    want = int(min(nrows, max(threads, budget_s * threads / max(per_row, 1e-9))))
    sel = rng.choice(nrows, size=want, replace=False)
    rows = [(int(r // w.dim), int(r % w.dim)) for r in sel]
    dt = _oracle_rows_rate(w, x, rows, threads)
    gbs = len(rows) * _row_bytes(w) / dt / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "elems_per_s": len(rows) * w.seqlen / dt, "seconds": dt,
            "sample": f"{len(rows)} of {nrows} (batch, channel) rows of {w.name}, full seqlen {w.seqlen}, "
                      f"fp64 C oracle, {threads} host threads"}


# The largest single-GPU workload is the headline line; the default run also
# times the other full-size workloads in the same process (per_config).
HEADLINE_WORKLOAD = "long_fixed_fp32"
PER_CONFIG = ("mamba130m_bf16", "mamba130m_bf16_l2047", "grouped_bf16", "mamba2p8b_fp16", "long_fixed_fp32")
PUBLISHED_NOTE = ("the pages quote no throughput, latency or hardware for this operator (the published "
                  "figures of the baseline are empty), so there is no context line to compare with")


def _config(w, world, shard_mode):
    """The workload as both arms describe it (identical keys and values)."""
    return {"workload": w.name, "batch": w.batch, "dim": w.dim, "seqlen": w.seqlen, "dstate": w.dstate,
            "groups": w.groups, "bc": w.bc, "io_dtype": w.dtype, "z": w.has_z,
            "return_last_state": w.return_last_state,
            "parallelism": (f"partitioned x{world} (batch x dim)" if shard_mode else f"independent x{world}")}


def run_reference(args, rank, world):
    """--impl reference: the fp64 CPU oracle as it stands, on host cores."""
    if rank != 0:
        return
    import numpy as np
    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w)
    threads = os.cpu_count() or 1
    nrows = w.batch * w.dim
    rng = np.random.default_rng(1)
    probe = [(int(r // w.dim), int(r % w.dim)) for r in rng.choice(nrows, size=min(nrows, threads), replace=False)]
    per_row = _oracle_rows_rate(w, x, probe, threads) / len(probe) * min(threads, len(probe))
    budget = min(2.0, 150.0 / max(1, args.steps + args.warmup))  # seconds per step
    R = int(min(nrows, max(1, budget * threads / max(per_row, 1e-9))))
    order = rng.permutation(nrows)
    step_rows = [[(int(order[(i * R + k) % nrows] // w.dim), int(order[(i * R + k) % nrows] % w.dim))
                  for k in range(R)] for i in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        _oracle_rows_rate(w, x, step_rows[i], threads)
    times = [_oracle_rows_rate(w, x, step_rows[args.warmup + i], threads) for i in range(args.steps)]
    t = sum(times)
    gbs = args.steps * R * _row_bytes(w) / t / 1e9
    sample = (f"each step: {R} of {nrows} (batch, channel) rows of {w.name} (a rotating sample), full seqlen, "
              f"fp64 C oracle on {threads} host threads; the rate is the sampled rows' bytes over their time")
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
            "higher_is_better": True, "scaling": "strong" if args.shard else "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, Mamba-layer shapes)",
            "config": _config(w, world, args.shard),
            "method": {"sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": threads, "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "published": None, "published_note": PUBLISHED_NOTE}
    print(json.dumps(line), flush=True)


def _measure(w, x, args, world, rank, dev, shard_mode):
    """Time args.steps forward steps of workload w on this rank (the whole
    problem, or this rank's blocks of the partition when shard_mode), L2
    flushed before each step outside the timed interval. Returns the per-step
    kernel time (max over ranks) and the launch facts."""
    import torch
    from state_space_model_03_gb300 import api, shard
    lib = api.load_library()
    B4 = x["B"].unsqueeze(1) if x["B"].dim() == 3 else x["B"]
    groups = 1 if w.bc == "fixed" else B4.shape[1]
    if shard_mode:
        blocks = shard.plan(w.batch, w.dim, groups, world)[rank]
    else:
        blocks = [shard.Block(0, w.batch, 0, w.dim)]
    xx = dict(x)
    if x["B"].dim() == 3:
        xx["B"], xx["C"] = x["B"].unsqueeze(1), x["C"].unsqueeze(1)
    jobs = []
    for blk in blocks:
        o = shard.block_operands(xx, blk, groups)
        d = {k: (None if o[k] is None else o[k].contiguous().to(dev)) for k in NAMES}
        nu = api.normalise(*(d[k] for k in NAMES))
        out = torch.empty(nu[0].shape, dtype=nu[0].dtype, device=dev)
        last = (torch.empty(nu[0].shape[0], nu[0].shape[1], w.dstate, dtype=torch.float32, device=dev)
                if w.return_last_state else None)
        params = api.make_params(*nu, w.delta_softplus, out, last)
        ws = api.attach_workspace(params, dev)
        jobs.append((params, ws, d, nu, out, last))
    launches_per_step = sum(2 if j[1] is not None else 1 for j in jobs)
    prefs = [ctypes.byref(j[0]) for j in jobs]
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step():
        for pr in prefs:
            st = lib.ss_fwd(pr, sptr)
            if st != 0:
                raise RuntimeError(api.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    region0 = torch.cuda.Event(enable_timing=True)
    region1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank_of(dev)) as clk, torch.cuda.stream(stream):
        region0.record(stream)
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        region1.record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if api.device_error() != 0:
        raise RuntimeError("device error word set during the bench")
    kms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = sum(kms) / len(kms)
    region_ms = region0.elapsed_time(region1) / args.steps
    ms, region_ms = max_over_ranks([ms, region_ms], world, dev)
    del jobs, prefs, flush_buf
    torch.cuda.empty_cache()
    return {"ms": ms, "region_ms": region_ms, "launches_per_step": launches_per_step,
            "segmented": launches_per_step > len(blocks), "blocks": [list(b) for b in blocks],
            "clocks": clk.summary(), "l2_flush_mib": 2 * l2 >> 20}


def local_rank_of(dev):
    return dev.index if dev.index is not None else 0


def _rates(w, ms, world, shard_mode, peak):
    """Whole-job rates of a step of ms milliseconds (slowest rank): N copies of
    the problem (weak scaling) or one problem split over N ranks (strong).
    frac is per GPU: the bytes one rank moved over its time, over its peak."""
    cb = workloads.compulsory_bytes(w)
    units = 1 if shard_mode else world
    gbs = units * cb / (ms * 1e-3) / 1e9
    return {"ms_per_step": ms, "gbs": gbs, "elems_per_s": units * w.elems / (ms * 1e-3),
            "frac": gbs / world / peak}


def run_ours(args, rank, world, local_rank):
    import torch
    from state_space_model_03_gb300 import api

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    peak, peak_src = _peaks()
    names = [args.workload] if args.workload else list(PER_CONFIG)
    head = args.workload or HEADLINE_WORKLOAD
    per_config, measured = {}, {}
    for name in names:
        w = workloads.WORKLOADS[name]
        x = workloads.make_inputs(w)
        m = _measure(w, x, args, world, rank, dev, args.shard)
        measured[name] = (w, x, m)
        r = _rates(w, m["ms"], world, args.shard, peak)
        per_config[name] = {"ms_per_step": r["ms_per_step"], "gbs": r["gbs"], "elems_per_s": r["elems_per_s"],
                            "frac": r["frac"],
                            "launches_per_step": m["launches_per_step"],
                            "sequence_segmented": m["segmented"], "traffic": _traffic(name)}
    w, x, m = measured[head]
    ms = m["ms"]
    cb = workloads.compulsory_bytes(w)
    r = _rates(w, ms, world, args.shard, peak)

    # end to end through the C ABI with host buffers (pinned), copies inside the
    # timed region: this rank's whole problem, or its blocks of the partition
    from state_space_model_03_gb300 import shard
    xx = dict(x)
    if x["B"].dim() == 3:
        xx["B"], xx["C"] = x["B"].unsqueeze(1), x["C"].unsqueeze(1)
    groups = 1 if w.bc == "fixed" else xx["B"].shape[1]
    hosts = []
    for blk in [shard.Block(*b) for b in m["blocks"]]:
        o = shard.block_operands(xx, blk, groups)
        hx = {k: (None if o[k] is None else o[k].contiguous().pin_memory()) for k in NAMES}
        hosts.append((api.HostRunner(**hx, delta_softplus=w.delta_softplus,
                                     return_last_state=w.return_last_state, device=dev), hx))
    e2e_steps = max(3, min(args.steps, 20))
    stream0 = hosts[0][0].stream
    for _ in range(2):
        for runner, hx in hosts:
            runner.run(**hx)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream0)
    for _ in range(e2e_steps):
        for runner, hx in hosts:
            if runner.stream is not stream0:
                runner.stream.wait_stream(stream0)
            runner.enqueue(**hx)
            if runner.stream is not stream0:
                stream0.wait_stream(runner.stream)
    e1.record(stream0)
    stream0.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], world, dev)[0]
    h2d = sum(rn.h2d_bytes for rn, _ in hosts)
    d2h = sum(rn.d2h_bytes for rn, _ in hosts)

    if rank != 0:
        return
    clocks = m["clocks"]
    sm_mhz = clocks.get("sm_mhz") or 1900.0
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    pair_ops = PAIR_FP32_OPS[w.bc]
    alu_floor_s = w.elems * w.dstate * pair_ops / (128.0 * nsm * sm_mhz * 1e6)
    cfg = _config(w, world, args.shard)
    line = {
        "metric": METRIC, "value": r["gbs"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "strong" if args.shard else "weak",
        "vs_baseline": None, "published": None, "published_note": PUBLISHED_NOTE,
        "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16"}[w.dtype],
        "data": "synthetic (seeded, Mamba-layer shapes)",
        "config": cfg,
        "method": {"l2": f"flushed before every step ({m['l2_flush_mib']} MiB write, outside the kernel interval)",
                   "sequence_segmented": m["segmented"], "launches_per_step": m["launches_per_step"],
                   "rank0_blocks": m["blocks"]},
        "elems_per_s": r["elems_per_s"],
        "compulsory_bytes_per_step": cb,
        "region_ms_per_step_incl_flush": m["region_ms"],
        "roofline": {"bound": "hbm", "achieved": r["gbs"] / world, "peak": peak, "unit": "GB/s",
                     "frac": r["frac"], "peak_source": peak_src,
                     "traffic": _traffic(w.name),
                     "note": ("achieved = compulsory bytes of the step over the step's kernel time "
                              f"({m['launches_per_step']} launch(es) per step on the launching stream)")},
        "alu_floor": {"fp32_lane_ops_per_pair": pair_ops, "pairs_per_step": w.elems * w.dstate,
                      "fp32_lanes_per_sm_clk": 128, "sms": nsm, "sm_mhz": sm_mhz,
                      "floor_ms": alu_floor_s * 1e3,
                      "gbs_at_floor": cb / alu_floor_s / 1e9},
        "per_config": per_config,
        "e2e": {"value": _rates(w, e2e_ms, world, args.shard, peak)["gbs"], "unit": "GB/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps},
        "gpu_launches": args.steps * sum(v["launches_per_step"] for v in per_config.values()),
        "clocks": clocks,
        "kernel_hash": _kernel_hash(),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, x, budget_s=args.cpu_budget)
    print(json.dumps(line), flush=True)


DECODE_METRIC = "selective-state-update (decode step) HBM GB/s (compulsory bytes / kernel time)"
DEFAULT_DECODE = "decode130m_bf16"


def _decode_rate_oracle(w, x, budget_s):
    """The numpy fp64 step oracle on whole steps of the workload, repeated
    for about budget_s seconds; returns (GB/s in the bench metric, seconds, steps)."""
    import oracle
    cb = workloads.decode_compulsory_bytes(w)
    args = [x[k] for k in ("state", "u", "delta", "A", "B", "C")]
    t0 = time.perf_counter()
    n = 0
    while True:
        oracle.selective_state_update_ref(*args, D=x["D"], z=x["z"], delta_bias=x["delta_bias"],
                                          delta_softplus=True)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= 1000:
            return cb * n / el / 1e9, el, n


def run_decode(args, rank, world, local_rank):
    """One decode step (ss_state_update) per bench step on a resident state."""
    import torch
    from state_space_model_03_gb300 import api

    name = args.workload if args.workload in workloads.DECODE_WORKLOADS else DEFAULT_DECODE
    w = workloads.DECODE_WORKLOADS[name]
    x = workloads.make_decode_inputs(w)
    cb = workloads.decode_compulsory_bytes(w)
    if args.impl == "reference":
        if rank != 0:
            return
        gbs, el, n = _decode_rate_oracle(w, x, max(1.0, args.cpu_budget))
        cpu = {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": 1,
               "sample": f"{n} whole steps of {w.name}, numpy fp64 step oracle, {el:.1f} s"}
        print(json.dumps({"impl": "reference", "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s",
                          "n_gpus": 1, "steps": n, "warmup": 0, "ms_per_step": el / n * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded, Mamba-layer decode shapes)",
                          "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate},
                          "cpu_baseline": cpu,
                          "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = api.load_library()
    d = {k: v.to(dev) for k, v in x.items()}
    out = torch.empty(w.batch, w.dim, dtype=d["u"].dtype, device=dev)
    params = api.make_state_update_params(d["state"], d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                                          d["delta_bias"], True, out)
    pref = ctypes.byref(params)
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step():
        st = lib.ss_state_update(pref, sptr)
        if st != 0:
            raise RuntimeError(api.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    kms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = max_over_ranks([sum(kms) / len(kms)], world, dev)[0]
    gbs = job_rate(cb, world, ms) / 1e9
    peak, peak_src = _peaks()
    clocks = clk.summary()

    # end to end: each step copies the token's inputs from pinned host memory,
    # runs the step on the resident state and reads out back
    host = {k: x[k].pin_memory() for k in ("u", "delta", "z", "B", "C")}
    h_out = torch.empty(w.batch, w.dim, dtype=d["u"].dtype, pin_memory=True)
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    e2e_steps = max(3, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for k, t in host.items():
                d[k].copy_(t, non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], world, dev)[0]
    if rank != 0:
        return
    line = {
        "metric": DECODE_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16"}[w.dtype],
        "data": "synthetic (seeded, Mamba-layer decode shapes)",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "dstate": w.dstate, "groups": w.groups,
                   "parallelism": f"independent x{world}",
                   "l2": f"flushed before every step ({2 * l2 >> 20} MiB write, outside the kernel interval)"},
        "compulsory_bytes_per_step": cb,
        "roofline": {"bound": "hbm", "achieved": cb / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": cb / (ms * 1e-3) / 1e9 / peak, "peak_source": peak_src,
                     "traffic": _traffic(w.name, "state_update")},
        "e2e": {"value": job_rate(cb, world, e2e_ms) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": h_out.numel() * h_out.element_size(),
                "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "kernel_hash": _kernel_hash("state_update"),
    }
    if world == 1 and not args.no_cpu_baseline:
        gbs_cpu, el, n = _decode_rate_oracle(w, x, min(args.cpu_budget, 10.0))
        line["cpu_baseline"] = {"value": gbs_cpu, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} whole steps of {w.name}, numpy fp64 step oracle, {el:.1f} s"}
    print(json.dumps(line), flush=True)


CONV_METRIC = "causal conv1d fwd HBM GB/s (compulsory bytes / kernel time)"
DEFAULT_CONV = "conv130m_bf16"


def _conv_rate_oracle(w, x, budget_s):
    """The numpy fp64 conv oracle on bounded row samples of the workload, for
    about budget_s seconds; returns (GB/s in the bench metric, seconds, rows)."""
    from oracle import conv1d
    cb = workloads.conv_compulsory_bytes(w)
    rows = w.batch * w.dim
    per_row = cb / rows
    t0 = time.perf_counter()
    n = 0
    while True:
        b = n % w.batch
        conv1d.causal_conv1d_ref(x["x"][b:b + 1, :64], x["weight"][:64], x["bias"][:64], activation="silu")
        n += 64
        el = time.perf_counter() - t0
        if el >= budget_s or n >= rows:
            return per_row * n / el / 1e9, el, n


def run_conv(args, rank, world, local_rank):
    """One causal conv1d forward (silu, bias) per bench step."""
    import torch
    from state_space_model_03_gb300 import api

    name = args.workload if args.workload in workloads.CONV_WORKLOADS else DEFAULT_CONV
    w = workloads.CONV_WORKLOADS[name]
    x = workloads.make_conv_inputs(w)
    cb = workloads.conv_compulsory_bytes(w)
    if args.impl == "reference":
        if rank != 0:
            return
        gbs, el, n = _conv_rate_oracle(w, x, max(1.0, args.cpu_budget))
        cpu = {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": 1,
               "sample": f"{n} of {w.batch * w.dim} rows of {w.name}, numpy fp64 oracle, {el:.1f} s"}
        print(json.dumps({"impl": "reference", "metric": CONV_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
                          "steps": 1, "warmup": 0, "ms_per_step": cb / (gbs * 1e9) * 1e3, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded, Mamba-layer shapes)",
                          "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "seqlen": w.seqlen,
                                     "width": w.width},
                          "cpu_baseline": cpu,
                          "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = api.load_library()
    d = {k: v.to(dev) for k, v in x.items()}
    out = torch.empty(d["x"].shape, dtype=d["x"].dtype, device=dev)
    params = api.make_conv1d_params(d["x"], d["weight"], d["bias"], None, None, None, out, "silu")
    pref = ctypes.byref(params)
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step():
        st = lib.ss_causal_conv1d(pref, sptr)
        if st != 0:
            raise RuntimeError(api.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    kms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = max_over_ranks([sum(kms) / len(kms)], world, dev)[0]
    gbs = job_rate(cb, world, ms) / 1e9
    peak, peak_src = _peaks()
    clocks = clk.summary()
    # end to end: x from pinned host memory, the conv, out back to pinned host memory
    hx = x["x"].pin_memory()
    h_out = torch.empty(hx.shape, dtype=hx.dtype, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            d["x"].copy_(hx, non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], world, dev)[0]
    if rank != 0:
        return
    line = {
        "metric": CONV_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16"}[w.dtype],
        "data": "synthetic (seeded, Mamba-layer shapes)",
        "config": {"workload": w.name, "batch": w.batch, "dim": w.dim, "seqlen": w.seqlen, "width": w.width,
                   "activation": "silu", "bias": True, "parallelism": f"independent x{world}",
                   "l2": f"flushed before every step ({2 * l2 >> 20} MiB write, outside the kernel interval)"},
        "elems_per_s": job_rate(w.elems, world, ms),
        "compulsory_bytes_per_step": cb,
        "roofline": {"bound": "hbm", "achieved": cb / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": cb / (ms * 1e-3) / 1e9 / peak, "peak_source": peak_src,
                     "traffic": _traffic(w.name, "conv1d")},
        "e2e": {"value": job_rate(cb, world, e2e_ms) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": hx.numel() * hx.element_size(),
                "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "kernel_hash": _kernel_hash("conv1d"),
    }
    if world == 1 and not args.no_cpu_baseline:
        gbs_cpu, el, n = _conv_rate_oracle(w, x, min(args.cpu_budget, 10.0))
        line["cpu_baseline"] = {"value": gbs_cpu, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {w.batch * w.dim} rows of {w.name}, numpy fp64 oracle, {el:.1f} s"}
    print(json.dumps(line), flush=True)


BWD_METRIC = "selective-scan bwd HBM GB/s (compulsory bytes / kernel time)"
# Algorithmic fp32 operations of the backward per (batch, channel, state, step):
# state recompute (dt*A, a*h + (dt u)*B: 3), y += C h (1), adjoint
# lam = a*lam' + dy*C (2), du += (lam dt)*B (2), ddt += lam (A (a h_prev) + B u)
# (4), dA += (lam dt)(a h_prev) (1), dB term (1), dC term (1); plus one exp.
BWD_OPS_PER_PAIR = 15
FP32_LANES_PER_SM = 128


def _bwd_rate_oracle(w, x, dout, budget_s):
    """The numpy fp64 backward oracle on sampled (batch, channel) rows for about
    budget_s seconds; returns (GB/s in the bench metric, seconds, rows)."""
    import numpy as np
    from oracle import backward as bwd_oracle
    cb = workloads.backward_compulsory_bytes(w)
    nrows = w.batch * w.dim
    rng = np.random.default_rng(0)
    # the stored inputs widened to fp64 once (the oracle's own first step), outside the timing
    f64 = {k: (None if x[k] is None else x[k].double().numpy()) for k in NAMES}
    g64 = dout.double().numpy()
    t0 = time.perf_counter()
    n = 0
    while True:
        r = int(rng.integers(nrows))
        bwd_oracle.selective_scan_bwd_rows([(r // w.dim, r % w.dim)], g64, **f64,
                                           delta_softplus=x["delta_softplus"])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= nrows:
            return cb / nrows * n / el / 1e9, el, n


def run_bwd(args, rank, world, local_rank):
    """One selective-scan backward (ss_bwd: the zero fill of the reduced
    gradients and the kernel) per bench step."""
    import torch
    from state_space_model_03_gb300 import api

    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w)
    dout_h = workloads.make_dout(w)
    cb = workloads.backward_compulsory_bytes(w)
    pairs = w.elems * w.dstate
    base_cfg = {"workload": w.name, "batch": w.batch, "dim": w.dim, "seqlen": w.seqlen, "dstate": w.dstate,
                "groups": w.groups, "bc": w.bc, "has_z": w.has_z}
    if args.impl == "reference":
        if rank != 0:
            return
        gbs, el, n = _bwd_rate_oracle(w, x, dout_h, max(1.0, args.cpu_budget))
        cpu = {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": 1,
               "sample": f"{n} of {w.batch * w.dim} rows of {w.name}, numpy fp64 backward oracle, {el:.1f} s"}
        print(json.dumps({"impl": "reference", "metric": BWD_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
                          "steps": 1, "warmup": 0, "ms_per_step": cb / (gbs * 1e9) * 1e3, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded, Mamba-layer shapes)", "config": base_cfg,
                          "cpu_baseline": cpu,
                          "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = api.load_library()
    d = {k: (None if x[k] is None else x[k].to(dev)) for k in NAMES}
    u, delta, A, B, C, D, z, bias = api.normalise(*(d[k] for k in NAMES))
    dout = dout_h.to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    du, ddelta = torch.empty_like(u), torch.empty_like(u)
    dz = torch.empty_like(u) if z is not None else None
    dA, dB, dC = torch.empty(A.shape, **f32), torch.empty(B.shape, **f32), torch.empty(C.shape, **f32)
    dD = torch.empty(w.dim, **f32) if D is not None else None
    ddb = torch.empty(w.dim, **f32) if bias is not None else None
    params = api.make_bwd_params(dout, u, delta, A, B, C, D, z, bias, x["delta_softplus"], None,
                                 du, ddelta, dz, dA, dB, dC, dD, ddb, None)
    ws = api.attach_bwd_workspace(params, dev)  # noqa: F841 (kept alive for the calls below)
    pref = ctypes.byref(params)
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step():
        st = lib.ss_bwd(pref, sptr)
        if st != 0:
            raise RuntimeError(api.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    if api.device_error() != 0:
        raise RuntimeError("device-side error word set")
    kms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = max_over_ranks([sum(kms) / len(kms)], world, dev)[0]
    gbs = job_rate(cb, world, ms) / 1e9
    clocks = clk.summary()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = nsm * FP32_LANES_PER_SM * 2070e6 / 1e9  # Gop/s at the maximum SM clock
    achieved = BWD_OPS_PER_PAIR * pairs / (ms * 1e-3) / 1e9
    # end to end: inputs from pinned host memory, every gradient back to pinned host memory
    hin = {k: (None if t is None else t.pin_memory()) for k, t in
           (("u", x["u"]), ("delta", x["delta"]), ("z", x["z"]), ("B", x["B"]), ("C", x["C"]), ("dout", dout_h))}
    dins = {"u": u, "delta": delta, "z": z, "B": B, "C": C, "dout": dout}
    outs = [t for t in (du, ddelta, dz, dA, dB, dC, dD, ddb) if t is not None]
    houts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in hin.values() if t is not None)
    d2h = sum(t.numel() * t.element_size() for t in houts)
    e2e_steps = max(3, min(args.steps, 20))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for k, t in hin.items():
                if t is not None:
                    dins[k].copy_(t.view(dins[k].shape), non_blocking=True)
            step()
            for ho, do in zip(houts, outs):
                ho.copy_(do, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], world, dev)[0]
    if rank != 0:
        return
    line = {
        "metric": BWD_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16"}[w.dtype],
        "data": "synthetic (seeded, Mamba-layer shapes)",
        "config": dict(base_cfg, parallelism=f"independent x{world}",
                       l2=f"flushed before every step ({2 * l2 >> 20} MiB write, outside the kernel interval)"),
        "elems_per_s": job_rate(w.elems, world, ms),
        "compulsory_bytes_per_step": cb,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "Gop/s",
                     "frac": achieved / alu_peak,
                     "peak_source": f"derived: {nsm} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2070 MHz",
                     "ops_per_pair": BWD_OPS_PER_PAIR, "traffic": _traffic(w.name + ":bwd", "bwd")},
        "hbm": {"achieved_gbs": gbs, "peak": _peaks()[0], "frac": gbs / _peaks()[0]},
        "e2e": {"value": job_rate(cb, world, e2e_ms) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps},
        "gpu_launches": args.steps,
        "memsets_per_step": 3 + (D is not None) + (bias is not None),
        "clocks": clocks,
        "kernel_hash": _kernel_hash("bwd"),
    }
    if world == 1 and not args.no_cpu_baseline:
        gbs_cpu, el, n = _bwd_rate_oracle(w, x, dout_h, min(args.cpu_budget, 10.0))
        line["cpu_baseline"] = {"value": gbs_cpu, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {w.batch * w.dim} rows of {w.name}, numpy fp64 backward "
                                          f"oracle, {el:.1f} s"}
    print(json.dumps(line), flush=True)


CX_METRIC = "complex-A selective-scan fwd HBM GB/s (compulsory bytes / kernel time)"
# Algorithmic fp32 operations of the complex-A forward per (batch, channel,
# state, step): dt Re A, dt Im A (2), the decay's two parts e cos, e sin (2),
# x <- a x + (dt u) B (5), y += C Re x (1); plus exp, sin and cos.
CX_OPS_PER_PAIR = 10


def _complex_A(w):
    """An S4D-Lin-like complex A: -1/2 + i pi n for state n, every channel."""
    import torch
    n = torch.arange(w.dstate, dtype=torch.float32)
    return torch.complex(torch.full((w.dim, w.dstate), -0.5), (math.pi * n).expand(w.dim, w.dstate).contiguous())


def _cx_rate_oracle(w, x, budget_s):
    """The complex-A fp64 oracle on sampled (batch, channel) rows for about
    budget_s seconds; returns (GB/s in the bench metric, seconds, rows)."""
    import numpy as np
    from oracle import complex_a
    cb = workloads.compulsory_bytes(w) + w.dim * w.dstate * 4  # A is twice as wide
    nrows = w.batch * w.dim
    rng = np.random.default_rng(0)
    f64 = {k: (None if x[k] is None else (x[k].numpy() if x[k].is_complex() else x[k].double().numpy()))
           for k in NAMES}
    t0 = time.perf_counter()
    n = 0
    while True:
        r = int(rng.integers(nrows))
        b, d = r // w.dim, r % w.dim
        sl = {k: (f64[k][b:b + 1, d:d + 1] if k in ("u", "delta", "z") and f64[k] is not None else f64[k])
              for k in NAMES}
        sl["A"] = f64["A"][d:d + 1]
        sl["D"] = None if f64["D"] is None else f64["D"][d:d + 1]
        sl["delta_bias"] = None if f64["delta_bias"] is None else f64["delta_bias"][d:d + 1]
        if f64["B"].ndim == 2:
            sl["B"], sl["C"] = f64["B"][d:d + 1], f64["C"][d:d + 1]
        elif f64["B"].ndim == 3:
            sl["B"], sl["C"] = f64["B"][b:b + 1], f64["C"][b:b + 1]
        else:
            gi = d // (w.dim // f64["B"].shape[1])
            sl["B"], sl["C"] = f64["B"][b:b + 1, gi:gi + 1], f64["C"][b:b + 1, gi:gi + 1]
        complex_a.selective_scan_complex_ref(**sl, delta_softplus=x["delta_softplus"])
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or n >= nrows:
            return cb / nrows * n / el / 1e9, el, n


def run_complex(args, rank, world, local_rank):
    """One complex-A forward (ss_fwd_complex) per bench step."""
    import torch
    from state_space_model_03_gb300 import api

    w = workloads.WORKLOADS[args.workload]
    x = workloads.make_inputs(w)
    x["A"] = _complex_A(w)
    cb = workloads.compulsory_bytes(w) + w.dim * w.dstate * 4
    pairs = w.elems * w.dstate
    base_cfg = {"workload": w.name + " (complex A = -1/2 + i pi n)", "batch": w.batch, "dim": w.dim,
                "seqlen": w.seqlen, "dstate": w.dstate, "groups": w.groups, "bc": w.bc, "has_z": w.has_z}
    if args.impl == "reference":
        if rank != 0:
            return
        gbs, el, n = _cx_rate_oracle(w, x, max(1.0, args.cpu_budget))
        cpu = {"value": gbs, "unit": "GB/s", "kind": "oracle", "cores": 1,
               "sample": f"{n} of {w.batch * w.dim} rows, numpy fp64 complex-A oracle, {el:.1f} s"}
        print(json.dumps({"impl": "reference", "metric": CX_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": 1,
                          "steps": 1, "warmup": 0, "ms_per_step": cb / (gbs * 1e9) * 1e3, "higher_is_better": True,
                          "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic (seeded, Mamba-layer shapes)", "config": base_cfg,
                          "cpu_baseline": cpu,
                          "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    lib = api.load_library()
    d = {k: (None if x[k] is None else x[k].to(dev)) for k in NAMES}
    u, delta, A, B, C, D, z, bias = api.normalise(*(d[k] for k in NAMES))
    out = torch.empty_like(u)
    params = api.make_complex_params(u, delta, A, B, C, D, z, bias, x["delta_softplus"], out, None)
    pref = ctypes.byref(params)
    stream = torch.cuda.Stream(device=dev)
    sptr = stream.cuda_stream
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=dev)

    def step():
        st = lib.ss_fwd_complex(pref, sptr)
        if st != 0:
            raise RuntimeError(api.status_string(st))

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            flush_buf.fill_(i & 0xFF)
            step()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local_rank) as clk, torch.cuda.stream(stream):
        for i in range(args.steps):
            flush_buf.fill_(i & 0xFF)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        stream.synchronize()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    kms = [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)]
    ms = max_over_ranks([sum(kms) / len(kms)], world, dev)[0]
    gbs = job_rate(cb, world, ms) / 1e9
    clocks = clk.summary()
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    alu_peak = nsm * FP32_LANES_PER_SM * 2070e6 / 1e9
    achieved = CX_OPS_PER_PAIR * pairs / (ms * 1e-3) / 1e9
    # end to end: inputs from pinned host memory, out back to pinned host memory
    hin = {k: t.pin_memory() for k, t in (("u", x["u"]), ("delta", x["delta"]), ("z", x["z"]), ("B", x["B"]),
                                          ("C", x["C"])) if t is not None}
    dins = {"u": u, "delta": delta, "z": z, "B": B, "C": C}
    h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    e2e_steps = max(3, min(args.steps, 50))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            for k, t in hin.items():
                dins[k].copy_(t.view(dins[k].shape), non_blocking=True)
            step()
            h_out.copy_(out, non_blocking=True)
        e1.record(stream)
        stream.synchronize()
    e2e_ms = max_over_ranks([e0.elapsed_time(e1) / e2e_steps], world, dev)[0]
    if rank != 0:
        return
    line = {
        "metric": CX_METRIC, "value": gbs, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"fp32": "f32", "fp16": "f16", "bf16": "bf16"}[w.dtype],
        "data": "synthetic (seeded, Mamba-layer shapes)",
        "config": dict(base_cfg, parallelism=f"independent x{world}",
                       l2=f"flushed before every step ({2 * l2 >> 20} MiB write, outside the kernel interval)"),
        "elems_per_s": job_rate(w.elems, world, ms),
        "compulsory_bytes_per_step": cb,
        "roofline": {"bound": "alu", "achieved": achieved, "peak": alu_peak, "unit": "Gop/s",
                     "frac": achieved / alu_peak,
                     "peak_source": f"derived: {nsm} SMs x {FP32_LANES_PER_SM} fp32 lanes x 2070 MHz",
                     "ops_per_pair": CX_OPS_PER_PAIR, "traffic": _traffic(w.name + ":complex", "complex")},
        "hbm": {"achieved_gbs": gbs, "peak": _peaks()[0], "frac": gbs / _peaks()[0]},
        "e2e": {"value": job_rate(cb, world, e2e_ms) / 1e9, "unit": "GB/s", "ms_per_step": e2e_ms,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hin.values()),
                "d2h_bytes_per_step": h_out.numel() * h_out.element_size(), "steps": e2e_steps},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "kernel_hash": _kernel_hash("complex"),
    }
    if world == 1 and not args.no_cpu_baseline:
        gbs_cpu, el, n = _cx_rate_oracle(w, x, min(args.cpu_budget, 10.0))
        line["cpu_baseline"] = {"value": gbs_cpu, "unit": "GB/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} of {w.batch * w.dim} rows of {w.name}, numpy fp64 complex-A "
                                          f"oracle, {el:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--op", default="scan", choices=["scan", "state_update", "conv1d", "bwd", "complex"],
                    help="scan: the selective-scan forward (the headline); state_update: one decode step; "
                         "conv1d: the causal conv1d forward; bwd: the selective-scan backward; "
                         "complex: the complex-A forward")
    ap.add_argument("--workload", default=None,
                    choices=sorted(workloads.WORKLOADS) + sorted(workloads.DECODE_WORKLOADS)
                    + sorted(workloads.CONV_WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--shard", action="store_true",
                    help="scan only: partition ONE problem over the ranks (batch x dim, whole groups where the "
                         "rows allow; strong scaling) instead of one independent copy per rank")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, world, local_rank = _env_int("RANK", 0), _env_int("WORLD_SIZE", 1), _env_int("LOCAL_RANK", 0)
    if args.op == "conv1d":
        if args.workload is not None and args.workload not in workloads.CONV_WORKLOADS:
            ap.error("--op conv1d takes a conv workload")
        if world > 1 and args.impl == "ours":
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        try:
            run_conv(args, rank, world, local_rank)
        finally:
            if world > 1 and args.impl == "ours":
                import torch
                torch.distributed.destroy_process_group()
        return
    if args.op == "state_update":
        if args.workload is not None and args.workload not in workloads.DECODE_WORKLOADS:
            ap.error("--op state_update takes a decode workload")
        if world > 1 and args.impl == "ours":
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        try:
            run_decode(args, rank, world, local_rank)
        finally:
            if world > 1 and args.impl == "ours":
                import torch
                torch.distributed.destroy_process_group()
        return
    if args.workload is not None and args.workload not in workloads.WORKLOADS:
        ap.error(f"--op {args.op} takes a scan workload")
    if args.workload is None and (args.op != "scan" or args.impl == "reference"):
        args.workload = DEFAULT_WORKLOAD if args.op != "scan" else HEADLINE_WORKLOAD
    if args.op in ("bwd", "complex"):
        if world > 1 and args.impl == "ours":
            import torch
            torch.cuda.set_device(local_rank)
            torch.distributed.init_process_group("nccl")
        try:
            (run_bwd if args.op == "bwd" else run_complex)(args, rank, world, local_rank)
        finally:
            if world > 1 and args.impl == "ours":
                import torch
                torch.distributed.destroy_process_group()
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl")
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
