#!/usr/bin/env python3
"""Benchmark: AG-GEMM / GEMM-RS bf16 TFLOP/s on GB300, and % of dense tensor-core peak.

One step = one pass of the hot path over the largest configuration, the
AllGather->GEMM layer with skewed readiness: R=8 logical ranks, each shard
A_r 4096x8192 bf16, B 8192x8192 bf16, C = concat(A_0..A_7) @ B (32768x8192),
the ranks published in a seeded permutation with seeded 0-50 us start
delays.  Every step is one launch through the C ABI with a fresh epoch.
Inputs (about 1.7 GB per step) are larger than L2, so no flush is needed
between steps.  The tp_layer step (AG-GEMM TP then GEMM-RS TP) and every
other configuration are reported in the per_config section.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With --gpus N > 1 (under torchrun) every rank runs its own replica of the
workload (the path has no cross-GPU exchange on this machine); the time is
the max over ranks and the value counts every rank's work.

--impl reference times the CPU oracle (the slow, obviously correct
definition) on a bounded sample of the same workload, on the host cores.
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "AG-GEMM / GEMM-RS bf16 TFLOP/s on 1 GB300 and % of dense tensor-core peak"
UNIT = "TFLOP/s"
HEADLINE = "ag_skew"
WORKLOAD = ("ag_skew: AG-GEMM R=8 A_r 4096x8192 @ B 8192x8192 -> C 32768x8192 bf16, ranks "
            "published in a seeded permutation with seeded 0-50 us start delays")
TP_WORKLOAD = ("tp_layer: AG-GEMM R=8 A_r 1024x4096 @ B 4096x4096 -> C 8192x4096, then "
               "GEMM-RS R=8 A_r 8192x1792 @ B_r 1792x4096 -> 8 x (1024x4096)")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ------------------------------------------------------------------ helpers

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def flops_ag(cfg):
    return 2.0 * cfg["R"] * cfg["M_r"] * cfg["N"] * cfg["K"]


def flops_rs(cfg):
    return 2.0 * cfg["M"] * cfg["N"] * cfg["R"] * cfg["K_r"]


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the GPU
    works.  Each sample is stamped with the host's monotonic clock when it
    arrives, so a summary can cover one timed window."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, device_index: int, interval_ms: int = 20):
        self.proc = None
        self.dev = device_index
        self.interval_ms = interval_ms
        self.samples = []  # (host time, sm MHz, max MHz, power W, set of reasons)
        self._thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.interval_ms), "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self._thread = threading.Thread(target=self._read, daemon=True)
        self._thread.start()

    def _read(self):
        for line in self.proc.stdout:
            t = time.monotonic()
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm, smax, power = float(parts[1]), float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, v in zip(self.NAMES, parts[5:9]) if v.lower().startswith("active")}
            self.samples.append((t, sm, smax, power, reasons))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.proc.wait()
        if self._thread is not None:
            self._thread.join(timeout=5)

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and power, and the throttle reasons seen,
        over the samples that arrived in [t0, t1] (all samples if None)."""
        sel = [x for x in self.samples
               if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        reasons = set()
        for x in sel:
            reasons |= x[4]
        return {"sm_mhz": statistics.median([x[1] for x in sel]) if sel else None,
                "sm_max_mhz": max(x[2] for x in sel) if sel else None,
                "power_w_max": max(x[3] for x in sel) if sel else None,
                "reasons": sorted(reasons), "samples": len(sel)}


TRAFFIC_SOURCES = ("opw_device.cuh", "opw_kernels.h", "opw_host.cu")


def source_hashes(kernel_source: str) -> dict:
    """sha256[:16] of the kernel's source and of the shared sources that shape
    its launch (device helpers, parameter blocks, host-side tile order)."""
    out = {}
    for f in (kernel_source,) + TRAFFIC_SOURCES:
        path = os.path.join(ROOT, "overlap_producer_warps_gb300", "csrc", f)
        out[f] = hashlib.sha256(open(path, "rb").read()).hexdigest()[:16]
    return out


def kernel_traffic(name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    ent = d.get(name)
    if not ent or "sources" not in ent:
        return None
    try:
        now = source_hashes(ent["source"])
    except OSError:
        return None
    return ent["dram_bytes_per_launch"] if now == ent["sources"] else None


def reduce_max(x: float, dist, device) -> float:
    """Max of a per-rank float over all ranks (identity without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, ms_per_step_max: float) -> float:
    """Weak scaling: every rank does the same work; time is the slowest rank's."""
    return world * flops_per_rank_step / (ms_per_step_max * 1e-3) / 1e12


# ------------------------------------------------------------------ CPU oracle sample

def cpu_model() -> str:
    """The host CPU's model as /proc/cpuinfo states it (on Arm: implementer
    and part numbers)."""
    try:
        lines = open("/proc/cpuinfo").read().splitlines()
    except OSError:
        return "unknown"
    fields = {}
    for ln in lines:
        if ":" in ln:
            k, v = ln.split(":", 1)
            fields.setdefault(k.strip().lower(), v.strip())
    if "model name" in fields:
        return fields["model name"]
    if "cpu part" in fields:
        arm = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1",
               "0xd49": "Arm Neoverse N2", "0xd0c": "Arm Neoverse N1"}
        part = fields["cpu part"].lower()
        name = arm.get(part) if fields.get("cpu implementer", "").lower() == "0x41" else None
        return name or f"implementer {fields.get('cpu implementer', '?')} part {part}"
    return "unknown"


def oracle_rows_step(d, rows):
    """The oracle's rows of C = concat(A_r) @ B for one sample (fp64, all host cores)."""
    import oracle
    oracle.ag_gemm_rows(d["heap"], d["rank_off"], d["R"], d["a_off"], d["M_r"], d["N"], d["K"],
                        d["B"], rows)
    return 2.0 * len(rows) * d["N"] * d["K"]


def oracle_sample(d, min_seconds=10.0, max_seconds=30.0):
    """Time the oracle on random rows of the headline layer's C until
    min_seconds have passed."""
    import oracle
    oracle.build()
    rng = np.random.default_rng(7)
    M = d["R"] * d["M_r"]
    chunk = max(4, oracle.threads())
    flops, rows, t0 = 0.0, 0, time.perf_counter()
    while True:
        flops += oracle_rows_step(d, rng.integers(0, M, size=chunk))
        rows += chunk
        el = time.perf_counter() - t0
        if el >= min_seconds or el >= max_seconds:
            break
    return {"value": flops / el / 1e12, "unit": UNIT, "cores": oracle.threads(), "kind": "oracle",
            "cpu_model": cpu_model(),
            "sample": f"{rows} random rows of the {HEADLINE} layer's C (each {d['N']} columns, "
                      f"K={d['K']}), fp64, {el:.1f} s"}


def oracle_rows_results(seconds=2.0):
    """The oracle timed beside each per-configuration row, on the host cores
    (part of the CPU-baseline leg): random output rows of the GEMM layers for
    about `seconds` each, in TFLOP/s, and one whole call of the ring AllReduce
    and of the all-to-all on the same workloads as their GPU rows, in the same
    GB/s of algorithmic bytes."""
    import oracle
    from overlap_producer_warps_gb300 import inputs
    oracle.build()
    cores = oracle.threads()
    chunk = max(4, cores)
    rng = np.random.default_rng(11)
    out = {"cores": cores, "kind": "oracle"}

    def timed(step, unit_work):
        work, n, t0 = 0.0, 0, time.perf_counter()
        while True:
            step()
            work += unit_work
            n += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return work / el, n, el

    for name in ("ag_tp", "ag_mlp"):
        d = inputs.ag_inputs(inputs.CONFIGS[name], seed=0)
        M = d["R"] * d["M_r"]
        rate, n, el = timed(lambda: oracle.ag_gemm_rows(
            d["heap"], d["rank_off"], d["R"], d["a_off"], d["M_r"], d["N"], d["K"], d["B"],
            rng.integers(0, M, size=chunk)), 2.0 * chunk * d["N"] * d["K"])
        out[name] = {"tflops": rate / 1e12, "sample": f"{n * chunk} random rows of C, {el:.1f} s"}
    d = inputs.rs_inputs(inputs.CONFIGS["rs_tp"], seed=0)
    rate, n, el = timed(lambda: oracle.gemm_rs_rows(
        d["heap"], d["rank_off"], d["R"], d["a_off"], d["b_off"], d["M"], d["N"], d["K_r"],
        rng.integers(0, d["M"], size=chunk)), 2.0 * chunk * d["N"] * d["K_r"] * d["R"])
    out["rs_tp"] = {"tflops": rate / 1e12, "sample": f"{n * chunk} random rows of S, {el:.1f} s"}

    R, n = 8, 8 * (1 << 21)   # the ring row's workload
    d = inputs.ring_inputs(R, n, seed=0)
    chunk_b = (n // R) * 4
    algo = R * chunk_b * (2 + 3 * (R - 2) + 4 + 3 * (R - 2) + 2)
    t0 = time.perf_counter()
    oracle.ring_allreduce(d["heap"], d["rank_off"], R, d["data_off"], d["out_off"], n)
    el = time.perf_counter() - t0
    out["ring_allreduce"] = {"ms": el * 1e3, "hbm_gbs": algo / el / 1e9,
                             "sample": "one whole call (8 ranks x 64 MiB, binary32, one thread)"}
    del d
    B = 8 << 20   # the all-to-all row's workload
    d = inputs.alltoall_inputs(R, B, seed=0)
    t0 = time.perf_counter()
    oracle.alltoall(d["heap"], d["rank_off"], R, d["send_off"], d["recv_off"], B)
    el = time.perf_counter() - t0
    out["alltoall"] = {"ms": el * 1e3, "hbm_gbs": 2 * R * R * B / el / 1e9,
                       "sample": "one whole call (8 ranks x 8 MiB slices, one thread)"}
    return out


# ------------------------------------------------------------------ reference arm

def run_reference(args, rank, world):
    if rank != 0:
        return 0
    from overlap_producer_warps_gb300 import inputs
    import oracle
    oracle.build()
    d = inputs.ag_inputs(inputs.CONFIGS[HEADLINE], seed=0)
    rng = np.random.default_rng(11)
    n_rows = max(4, oracle.threads())
    M = d["R"] * d["M_r"]

    def step():
        return oracle_rows_step(d, rng.integers(0, M, size=n_rows))

    for _ in range(args.warmup):
        step()
    flops = 0.0
    t0 = time.perf_counter()
    for _ in range(args.steps):
        flops += step()
    el = time.perf_counter() - t0
    value = flops / el / 1e12
    sample = (f"per step: {n_rows} random rows of the {HEADLINE} layer's C (each {d['N']} "
              f"columns, K={d['K']}), fp64 CPU oracle")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": WORKLOAD + " (bounded row sample per step)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.threads(),
                             "kind": "oracle", "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ workloads on the device

def skew_opts(api, cfg, **kw):
    """Options of an AG-GEMM layer: its skew schedule (if any) plus kw."""
    from overlap_producer_warps_gb300 import inputs
    if cfg.get("skew"):
        perm, delay = inputs.skew_schedule(0, cfg["R"])
        kw = dict(publish_perm=perm, delay_ns=delay, **kw)
    return api.make_opts(**kw)


class AgLayer:
    """One AllGather->GEMM configuration on the device: `sets` copies of every
    input and output buffer (the end-to-end leg double-buffers them) and one
    signal object, shared by the sets since its launches are serial."""

    def __init__(self, api, torch, name, seed=0, sets=1):
        from overlap_producer_warps_gb300 import inputs
        self.api, self.torch, self.name = api, torch, name
        self.cfg = inputs.CONFIGS[name]
        self.d = inputs.ag_inputs(self.cfg, seed=seed)
        d = self.d
        dev = torch.device("cuda")
        self.M = d["R"] * d["M_r"]
        self.bufs = []
        for _ in range(sets):
            self.bufs.append({
                "heap": torch.from_numpy(d["heap"]).to(dev),
                "B": torch.from_numpy(d["B"].view(np.int16)).to(dev).view(torch.bfloat16),
                "G": torch.empty((self.M, d["K"]), dtype=torch.bfloat16, device=dev),
                "C": torch.empty((self.M, d["N"]), dtype=torch.bfloat16, device=dev),
            })
        self.sig = api.Signal(api.ag_num_flags(d["R"], d["M_r"], d["K"]))
        self.flops = flops_ag(self.cfg)
        self._opts = {}

    def opts(self, **kw):
        """The layer's options (its skew schedule, if any, plus kw), built once."""
        key = tuple(sorted(kw.items()))
        if key not in self._opts:
            self._opts[key] = skew_opts(self.api, self.cfg, **kw)
        return self._opts[key]

    def launch(self, stream=None, b=0, epoch=None, **kw):
        d, x = self.d, self.bufs[b]
        e = self.sig.next_epoch() if epoch is None else epoch
        self.api.ag_gemm(x["heap"], d["rank_off"], d["a_off"], d["M_r"], d["N"], d["K"], x["B"],
                         x["G"], x["C"], self.sig, e, self.opts(**kw), stream)

    def check(self):
        st = self.sig.status()
        if st[0] != self.api.OK:
            raise RuntimeError(f"{self.name}: device error latched during the benchmark: {st}")

    def close(self):
        self.sig.close()
        self.bufs = []


class TpLayer:
    """The tp_layer step on the device: AG-GEMM TP then GEMM-RS TP, each with
    its own signal object."""

    def __init__(self, api, torch, seed=0):
        from overlap_producer_warps_gb300 import inputs
        self.api, self.torch = api, torch
        self.ag = AgLayer(api, torch, "ag_tp", seed=seed)
        self.rs_cfg = inputs.CONFIGS["rs_tp"]
        self.rs_d = inputs.rs_inputs(self.rs_cfg, seed=seed)
        self.rs_heap = torch.from_numpy(self.rs_d["heap"]).cuda()
        r = self.rs_d
        self.sig_rs = api.Signal(api.rs_num_flags(r["R"], r["M"], r["N"]))
        self.flops = self.ag.flops + flops_rs(self.rs_cfg)

    def rs(self, stream=None):
        r = self.rs_d
        self.api.gemm_rs(self.rs_heap, r["rank_off"], r["a_off"], r["b_off"], r["out_off"], r["M"],
                         r["N"], r["K_r"], self.sig_rs, self.sig_rs.next_epoch(), None, stream)

    def step(self):
        self.ag.launch()
        self.rs()

    def check(self):
        self.ag.check()
        st = self.sig_rs.status()
        if st[0] != self.api.OK:
            raise RuntimeError(f"rs_tp: device error latched during the benchmark: {st}")

    def close(self):
        self.ag.close()
        self.sig_rs.close()


def time_launches(torch, fn, n, warm=2):
    """Device time (ms) of each of n back-to-back calls of fn(), from CUDA
    events recorded between them on the current stream: mean, median and
    min.  A short spin kernel ahead of the first event keeps the GPU busy
    while the host enqueues the calls, so neither the first call's host-side
    cost nor its launch latency falls inside an interval."""
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    # about 0.3 ms + 0.1 ms per call at 2 GHz: more than the host needs
    spin = getattr(torch.cuda, "_sleep", None)
    if spin is not None:
        spin(int(2e9 * (3e-4 + 1e-4 * n)))
    ev[0].record(s)
    for i in range(n):
        fn()
        ev[i + 1].record(s)
    ev[n].synchronize()
    t = [ev[i].elapsed_time(ev[i + 1]) for i in range(n)]
    return {"mean": statistics.mean(t), "median": statistics.median(t), "min": min(t), "n": n,
            "all": t}


def time_interleaved(torch, fns, rounds=5, per_round=4):
    """Device times of several variants measured in interleaved rounds (each
    round runs every variant for per_round launches), so that no variant is
    favoured by the clock state (boost versus the power cap) it happens to
    run in.  Returns {name: {mean, median, min, n}} over all rounds."""
    samples = {k: [] for k in fns}
    for _ in range(rounds):
        for k, fn in fns.items():
            t = time_launches(torch, fn, per_round, warm=1)
            samples[k].extend(t["all"])
    return {k: {"mean": statistics.mean(v), "median": statistics.median(v), "min": min(v),
                "n": len(v)} for k, v in samples.items()}


def _summ(t):
    """A time_launches() result without the per-launch list."""
    return {k: v for k, v in t.items() if k != "all"}


def tflops_of(flops, t):
    """TFLOP/s at the median (and best) time of a time_launches() result."""
    return {"tflops": flops / t["median"] / 1e9, "tflops_best": flops / t["min"] / 1e9}


def ring_results(api, torch, reps, R=8, n=8 * (1 << 21)):
    """Ring AllReduce over 8 logical ranks of n fp32 values (64 MiB per rank):
    the HBM bytes its schedule moves per second, against the measured HBM peak."""
    from overlap_producer_warps_gb300 import inputs
    peaks, _ = load_peaks()
    d = inputs.ring_inputs(R, n, seed=0)
    heap = torch.from_numpy(d["heap"]).cuda()
    sig = api.Signal(api.ring_num_flags(R, n))

    def run():
        api.ring_allreduce(heap, d["rank_off"], d["data_off"], d["recv_off"], d["out_off"], n, sig,
                           sig.next_epoch())

    t = time_launches(torch, run, reps)
    st = sig.status()
    if st[0] != api.OK:
        raise RuntimeError(f"ring_allreduce: device error {st}")
    chunk_b = (n // R) * 4
    # per rank: send own chunk (r+w), R-2 forwarding reduce steps (2r+w), the last
    # reduce step (2r+2w), R-2 forwarding gather steps (r+2w), the last gather step (r+w)
    algo_bytes = R * chunk_b * (2 + 3 * (R - 2) + 4 + 3 * (R - 2) + 2)
    gbs = algo_bytes / (t["median"] * 1e-3) / 1e9
    busbw = 2 * (R - 1) / R * n * 4 / (t["median"] * 1e-3) / 1e9
    sig.close()
    return {"ranks": R, "values_per_rank": n, "ms": _summ(t), "hbm_gbs": gbs,
            "hbm_frac": gbs / float(peaks["hbm_gbs"]), "algo_bytes": algo_bytes,
            "busbw_gbs": busbw}


def alltoall_results(api, torch, reps, R=8, B=8 << 20):
    """All-to-all over 8 logical ranks, 8 MiB per (sender, receiver) slice."""
    from overlap_producer_warps_gb300 import inputs
    peaks, _ = load_peaks()
    d = inputs.alltoall_inputs(R, B, seed=0)
    heap = torch.from_numpy(d["heap"]).cuda()
    sig = api.Signal(api.alltoall_num_flags(R, B))

    def run():
        api.alltoall(heap, d["rank_off"], d["send_off"], d["recv_off"], B, sig, sig.next_epoch())

    t = time_launches(torch, run, reps)
    st = sig.status()
    if st[0] != api.OK:
        raise RuntimeError(f"alltoall: device error {st}")
    moved = 2 * R * R * B  # every slice read once and written once
    gbs = moved / (t["median"] * 1e-3) / 1e9
    sig.close()
    return {"ranks": R, "bytes_per_slice": B, "ms": _summ(t), "hbm_gbs": gbs,
            "hbm_frac": gbs / float(peaks["hbm_gbs"])}


def ag_fused_results(api, torch, name, reps, producer_only=False):
    """Fused AG-GEMM launches of one layer alone (its skew schedule included),
    or, with producer_only, its gather leg alone (GB/s of shard read + G write)."""
    w = AgLayer(api, torch, name)
    kw = {"role": api.ROLE_PRODUCER} if producer_only else {}
    t = time_launches(torch, lambda: w.launch(**kw), reps)
    w.check()
    d = w.d
    w.close()
    if producer_only:
        return {"ms": _summ(t), "gather_hbm_gbs": 2.0 * w.M * d["K"] * 2 / (t["median"] * 1e-3) / 1e9}
    return {"ms": _summ(t), **tflops_of(w.flops, t)}


def rs_results(api, torch, reps, scatter_only=False):
    """GEMM-RS TP launches alone, or, with scatter_only, its scatter leg alone
    (GB/s of bf16 output stored into the ranks' blocks)."""
    from overlap_producer_warps_gb300 import inputs
    cfg = inputs.CONFIGS["rs_tp"]
    d = inputs.rs_inputs(cfg, seed=0)
    R, M, K_r, N = cfg["R"], cfg["M"], cfg["K_r"], cfg["N"]
    heap = torch.from_numpy(d["heap"]).cuda()
    sig = api.Signal(api.rs_num_flags(R, M, N))
    role = api.ROLE_CONSUMER if scatter_only else api.ROLE_FUSED
    t = time_launches(torch, lambda: api.gemm_rs(heap, d["rank_off"], d["a_off"], d["b_off"],
                                                 d["out_off"], M, N, K_r, sig, sig.next_epoch(),
                                                 api.make_opts(role=role)), reps)
    st = sig.status()
    if st[0] != api.OK:
        raise RuntimeError(f"rs_tp: device error {st}")
    sig.close()
    if scatter_only:
        return {"ms": _summ(t), "scatter_hbm_gbs": M * N * 2 / (t["median"] * 1e-3) / 1e9}
    return {"ms": _summ(t), **tflops_of(flops_rs(cfg), t)}


def tiny_results(api, torch, reps=50):
    """The tiny AG-GEMM configuration (R=2, 64x128 shards, K=N=128), which is
    bound by latency: the device time per launch back to back, and the time
    from the host call to the completed launch (call, then synchronise)."""
    w = AgLayer(api, torch, "ag_tiny")
    t_dev = time_launches(torch, w.launch, reps)
    for _ in range(3):
        w.launch()
    torch.cuda.synchronize()
    lat = []
    for _ in range(reps):
        t0 = time.perf_counter()
        w.launch()
        torch.cuda.synchronize()
        lat.append(time.perf_counter() - t0)
    w.check()
    # the no-allocation call captured once in a CUDA graph, then replayed:
    # its clear and AG-GEMM kernels launch with one host call
    x, d = w.bufs[0], w.d
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    args = (x["heap"], d["rank_off"], d["a_off"], d["M_r"], d["N"], d["K"], x["B"], x["G"],
            x["C"], status)
    if api.ag_gemm_noalloc_status(*args) != api.OK:   # first call: outside any capture
        raise RuntimeError("ag_tiny: the no-allocation call failed")
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        rc = api.ag_gemm_noalloc_status(*args, stream=side)
    if rc != api.OK:
        raise RuntimeError(f"ag_tiny: capture failed: {api.status_str(rc)}")
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    glat = []
    for _ in range(reps):
        t0 = time.perf_counter()
        graph.replay()
        torch.cuda.synchronize()
        glat.append(time.perf_counter() - t0)
    if int(status[0].item()) != api.OK:
        raise RuntimeError(f"ag_tiny: device error in a graph replay: {status.tolist()}")
    w.close()
    lat.sort()
    glat.sort()
    return {"us_per_launch_back_to_back_median": t_dev["median"] * 1e3,
            "us_per_launch_back_to_back_min": t_dev["min"] * 1e3,
            "us_call_to_done_median": lat[len(lat) // 2] * 1e6,
            "us_call_to_done_min": lat[0] * 1e6,
            "us_graph_replay_to_done_median": glat[len(glat) // 2] * 1e6,
            "us_graph_replay_to_done_min": glat[0] * 1e6}


def mm_f32_out(torch):
    """A bf16 x bf16 -> fp32 product on the GPU, as cuBLAS gives it: torch.mm
    with out_dtype where this PyTorch has it, else the bf16 product widened
    (lower precision; named in the result)."""
    a = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    try:
        torch.mm(a, a, out_dtype=torch.float32)
        return (lambda x, y: torch.mm(x, y, out_dtype=torch.float32)), "torch.mm(out_dtype=float32)"
    except (TypeError, RuntimeError):
        return (lambda x, y: torch.matmul(x, y).float()), "bf16 matmul widened to fp32"


def ag_config_results(api, torch, name, peak_tflops, reps):
    """One AG-GEMM layer: fused (default schedule), the page's static swizzle,
    serial sync, batched row signals, the legs alone, unfused copy-then-GEMM
    and cuBLAS on the pre-gathered G, measured in interleaved rounds."""
    w = AgLayer(api, torch, name)
    d, cfg = w.d, w.cfg
    R, M_r, K, N = d["R"], d["M_r"], d["K"], d["N"]
    x = w.bufs[0]
    sig_add = api.Signal(api.ag_num_row_counters(R, M_r, K))

    def fused_row_add():
        api.ag_gemm(x["heap"], d["rank_off"], d["a_off"], M_r, N, K, x["B"], x["G"], x["C"],
                    sig_add, sig_add.next_epoch(),
                    skew_opts(api, cfg, signal_mode=api.SIGNAL_ROW_ADD))

    shards = [x["heap"][int(d["rank_off"][r]):int(d["rank_off"][r]) + M_r * K * 2]
              .view(torch.bfloat16).view(M_r, K) for r in range(R)]
    G, B, C = x["G"], x["B"], x["C"]

    def unfused():
        for r in range(R):
            G[r * M_r:(r + 1) * M_r].copy_(shards[r])
        torch.matmul(G, B, out=C)

    fns = {"fused": w.launch,
           "swizzle": lambda: w.launch(schedule=api.SCHED_SWIZZLE),
           # every tile, the consumer's own shard's included, read from G after its flag
           "no_local": lambda: w.launch(local_rank=-1),
           # every consumer waits for the whole gather before its first tile
           "serial": lambda: w.launch(sync_mode=api.SYNC_SERIAL),
           "row_add": fused_row_add,
           "producer_only": lambda: w.launch(role=api.ROLE_PRODUCER),
           # flags still hold the epoch the previous launch published
           "consumer_only": lambda: w.launch(epoch=w.sig.next_epoch() - 1,
                                             role=api.ROLE_CONSUMER),
           "unfused": unfused,
           "gemm_only": lambda: torch.matmul(G, B, out=C)}
    if cfg.get("skew"):
        # the publish order without the per-rank delays
        from overlap_producer_warps_gb300 import inputs
        perm, _ = inputs.skew_schedule(0, R)
        no_delay = api.make_opts(publish_perm=perm)
        fns["no_delay"] = lambda: api.ag_gemm(
            x["heap"], d["rank_off"], d["a_off"], M_r, N, K, x["B"], x["G"], x["C"], w.sig,
            w.sig.next_epoch(), no_delay)
    t = time_interleaved(torch, fns, rounds=max(1, reps // 4), per_round=4)
    w.check()
    if sig_add.status()[0] != api.OK:
        raise RuntimeError(f"{name}: device error with row-ADD signals")
    sig_add.close()
    fl = w.flops
    med = {k: v["median"] for k, v in t.items()}
    e = (med["producer_only"] + med["consumer_only"] - med["fused"]) / min(
        med["producer_only"], med["consumer_only"])
    out = {
        "pair_tile": f"256x{api.ag_tile_n(R, M_r, N)}",
        "fused_tflops": fl / med["fused"] / 1e9,
        "fused_tflops_best": fl / t["fused"]["min"] / 1e9,
        "pct_of_peak": fl / med["fused"] / 1e9 / peak_tflops,
        "swizzle_schedule_tflops": fl / med["swizzle"] / 1e9,
        "serial_sync_tflops": fl / med["serial"] / 1e9,
        "row_add_signal_tflops": fl / med["row_add"] / 1e9,
        "no_local_shard_tflops": fl / med["no_local"] / 1e9,
        "unfused_copy_then_gemm_tflops": fl / med["unfused"] / 1e9,
        "cublas_gemm_only_tflops": fl / med["gemm_only"] / 1e9,
        "fused_vs_cublas_gemm_only": med["gemm_only"] / med["fused"],
        "ms": t,
        "overlap_efficiency": max(0.0, min(1.0, e)),
        "gather_hbm_gbs_producer_only": 2.0 * w.M * K * 2 / (med["producer_only"] * 1e-3) / 1e9,
    }
    if "no_delay" in med:
        out["no_delay_fused_tflops"] = fl / med["no_delay"] / 1e9
    del shards, G, B, C, x
    w.close()
    torch.cuda.empty_cache()
    return out


def rs_config_results(api, torch, peak_tflops, reps):
    """GEMM-RS TP: fused, the legs alone, the unfused path (fp32 partials, an
    fp32 sum in rank order, then the row blocks split off) and one cuBLAS GEMM
    with the same FLOPs, measured in interleaved rounds."""
    from overlap_producer_warps_gb300 import inputs
    cfg = inputs.CONFIGS["rs_tp"]
    d = inputs.rs_inputs(cfg, seed=0)
    R, M, K_r, N = cfg["R"], cfg["M"], cfg["K_r"], cfg["N"]
    heap = torch.from_numpy(d["heap"]).cuda()
    sig = api.Signal(api.rs_num_flags(R, M, N))

    def rs(role=api.ROLE_FUSED):
        api.gemm_rs(heap, d["rank_off"], d["a_off"], d["b_off"], d["out_off"], M, N, K_r, sig,
                    sig.next_epoch(), api.make_opts(role=role))

    A = [heap[int(d["rank_off"][r]) + d["a_off"]:int(d["rank_off"][r]) + d["a_off"] + M * K_r * 2]
         .view(torch.bfloat16).view(M, K_r) for r in range(R)]
    Bs = [heap[int(d["rank_off"][r]) + d["b_off"]:int(d["rank_off"][r]) + d["b_off"] + K_r * N * 2]
          .view(torch.bfloat16).view(K_r, N) for r in range(R)]
    outs = [heap[int(d["rank_off"][j]) + d["out_off"]:int(d["rank_off"][j]) + d["out_off"]
                 + (M // R) * N * 2].view(torch.bfloat16).view(M // R, N) for j in range(R)]
    mm32, mm32_name = mm_f32_out(torch)

    def unfused_rs():
        S = mm32(A[0], Bs[0])
        for r in range(1, R):
            S += mm32(A[r], Bs[r])
        for j in range(R):
            outs[j].copy_(S[j * (M // R):(j + 1) * (M // R)])

    # The same FLOPs as one cuBLAS GEMM with the ranks' K slices side by side
    # ([M, R*K_r] @ [R*K_r, N]): no per-rank partials, no reduction, no scatter.
    A_cat = torch.cat(A, dim=1)
    B_cat = torch.cat(Bs, dim=0)
    C_cat = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    recv = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")

    def rs_consume():
        api.gemm_rs_consume(heap, d["rank_off"], d["a_off"], d["b_off"], d["out_off"], M, N, K_r,
                            recv, sig, sig.next_epoch())

    t = time_interleaved(torch, {
        "fused": rs, "with_receiving_side": rs_consume,
        "gemm_leg_only": lambda: rs(api.ROLE_PRODUCER),
        "scatter_leg_only": lambda: rs(api.ROLE_CONSUMER), "unfused": unfused_rs,
        "gemm_only": lambda: torch.matmul(A_cat, B_cat, out=C_cat)},
        rounds=max(1, reps // 4), per_round=4)
    del A_cat, B_cat, C_cat
    st = sig.status()
    if st[0] != api.OK:
        raise RuntimeError(f"rs_tp: device error {st}")
    fl = flops_rs(cfg)
    med = {k: v["median"] for k, v in t.items()}
    e = (med["gemm_leg_only"] + med["scatter_leg_only"] - med["fused"]) / min(
        med["gemm_leg_only"], med["scatter_leg_only"])
    sig.close()
    return {"fused_tflops": fl / med["fused"] / 1e9,
            "fused_tflops_best": fl / t["fused"]["min"] / 1e9,
            "pct_of_peak": fl / med["fused"] / 1e9 / peak_tflops,
            "with_receiving_side_tflops": fl / med["with_receiving_side"] / 1e9,
            "unfused_partials_then_sum_tflops": fl / med["unfused"] / 1e9,
            "unfused_partials": mm32_name,
            "cublas_single_gemm_tflops": fl / med["gemm_only"] / 1e9,
            "ms": t,
            "overlap_efficiency": max(0.0, min(1.0, e)),
            "scatter_hbm_gbs_scatter_only": M * N * 2 / (med["scatter_leg_only"] * 1e-3) / 1e9}


def tp_layer_results(api, torch, peak_tflops, reps):
    """The tp_layer step (AG-GEMM TP then GEMM-RS TP) back to back."""
    w = TpLayer(api, torch)
    t = time_launches(torch, w.step, reps)
    w.check()
    fl = w.flops
    w.close()
    return {"workload": TP_WORKLOAD, "step_tflops": fl / t["median"] / 1e9,
            "step_tflops_best": fl / t["min"] / 1e9,
            "pct_of_peak": fl / t["median"] / 1e9 / peak_tflops, "ms": _summ(t)}


def per_config_results(api, torch, peak_tflops, reps=20):
    """Each of the pages' tensor-parallel configurations on its own, burst
    (short runs against the burst peak): fused TFLOP/s at the median launch,
    the unfused baselines, cuBLAS with the same FLOPs, overlap efficiency."""
    out = {}
    for name in ("ag_tp", "ag_mlp", "ag_skew"):
        out[name] = ag_config_results(api, torch, name, peak_tflops, reps)
    out["rs_tp"] = rs_config_results(api, torch, peak_tflops, reps)
    out["tp_layer"] = tp_layer_results(api, torch, peak_tflops, reps)
    out["ag_tiny"] = tiny_results(api, torch)
    out["ring_allreduce"] = ring_results(api, torch, reps)
    out["alltoall"] = alltoall_results(api, torch, reps)
    return out


def e2e_results(torch, w, args, dist, world):
    """The headline step through the public API with its inputs and result in
    pinned host memory.  Every step copies the shards and B host -> device,
    runs AG-GEMM and reads C back.  The steps are pipelined over two device
    buffer sets and three streams: step i+1's inputs go in and step i-1's
    result comes out while step i computes.  The timed region runs from
    before step 0's first input copy to after the last step's result copy."""
    d = w.d
    h_heap = torch.from_numpy(d["heap"]).pin_memory()
    h_B = torch.from_numpy(d["B"].view(np.int16)).pin_memory()
    nsets = len(w.bufs)
    h_C = [torch.empty(w.bufs[0]["C"].shape, dtype=torch.bfloat16).pin_memory()
           for _ in range(nsets)]
    h2d = h_heap.numel() + h_B.numel() * 2
    d2h = h_C[0].numel() * 2
    stream, s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event(enable_timing=False)
    in_done = [ev() for _ in range(nsets)]
    comp_done = [ev() for _ in range(nsets)]
    out_done = [ev() for _ in range(nsets)]
    used = [False] * nsets

    def e2e_step(i):
        b = i % nsets
        x = w.bufs[b]
        with torch.cuda.stream(s_in):
            if used[b]:
                s_in.wait_event(comp_done[b])  # step i-2 has finished reading set b
            x["heap"].copy_(h_heap, non_blocking=True)
            x["B"].view(torch.int16).copy_(h_B, non_blocking=True)
            in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if used[b]:
            stream.wait_event(out_done[b])  # step i-2's result is on the host
        w.launch(stream, b)
        comp_done[b].record(stream)
        used[b] = True
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[b])
            h_C[b].copy_(x["C"], non_blocking=True)
            out_done[b].record(s_out)

    def run(n, e0=None, e1=None):
        if e0 is not None:
            e0.record(stream)
            s_in.wait_event(e0)
        for i in range(n):
            e2e_step(i)
        for b in range(nsets):
            if used[b]:
                stream.wait_event(out_done[b])
        if e1 is not None:
            e1.record(stream)

    run(max(1, min(args.warmup, 3)))
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    run(args.steps, e0, e1)
    torch.cuda.synchronize()
    w.check()
    t_e2e = reduce_max(e0.elapsed_time(e1) / args.steps, dist, "cuda")
    return {"value": whole_job_tflops(world, w.flops, t_e2e), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": t_e2e,
            "pipelined": f"{nsets} buffer sets, copy-in / compute / copy-out streams"}


def run_ours(args, rank, world, dist):
    import torch
    from overlap_producer_warps_gb300 import api
    from overlap_producer_warps_gb300 import build as _build
    if not os.path.exists(api.LIB_PATH):
        _build.build()
    api.lib()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    peaks, peak_src = load_peaks()
    peak = float(peaks["bf16_tflops"])  # burst: a kernel timed alone
    # The timed steps follow args.prewarm_s of load, where the 1.4 kW power
    # cap holds the clocks down: compare them with the sustained figure.
    sustained = args.prewarm_s >= 1.0 and "bf16_tflops_sustained" in peaks
    step_peak = float(peaks["bf16_tflops_sustained"]) if sustained else peak
    step_peak_name = ("bf16_tflops_sustained (cuBLAS back to back, under the power cap)"
                      if sustained else "bf16_tflops (burst, cuBLAS)")

    w = AgLayer(api, torch, HEADLINE, sets=2)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    t_load0 = time.monotonic()
    # An idle GPU needs seconds of load before its clocks settle: run the
    # step, untimed, for args.prewarm_s before the W counted warm-up steps.
    t_pre = time.perf_counter() + args.prewarm_s
    while time.perf_counter() < t_pre:
        for _ in range(4):
            w.launch()
        torch.cuda.synchronize()
    for _ in range(args.warmup):
        w.launch()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    t_timed0 = time.monotonic()
    ev[0].record(stream)
    for i in range(args.steps):
        w.launch()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    t_timed1 = time.monotonic()
    if dist is not None:
        dist.barrier()
    w.check()
    launch_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
    ms_total = ev[0].elapsed_time(ev[args.steps])
    t_step = reduce_max(ms_total / args.steps, dist, "cuda")
    value = whole_job_tflops(world, w.flops, t_step)

    # ---- end to end through the public API with host buffers
    e2e = e2e_results(torch, w, args, dist, world)
    sampler.stop()
    # the timed window's own samples; the load samples since the pre-warm began
    clocks = sampler.summary(t_timed0, t_timed1)
    clocks["under_load_since_prewarm"] = sampler.summary(t_load0, t_timed1)

    # ---- roofline of the step's one kernel
    mean_ms = statistics.mean(launch_ms)
    achieved = w.flops / (mean_ms * 1e-3) / 1e12
    roofline = {"bound": "tensor", "kernel": "ag_gemm", "achieved": achieved, "peak": step_peak,
                "unit": "TFLOP/s", "frac": achieved / step_peak,
                "peak_source": f"{peak_src} {step_peak_name}",
                "traffic": kernel_traffic("ag_gemm"),
                "ms_per_launch": mean_ms, "ms_per_launch_median": statistics.median(launch_ms),
                "ms_per_launch_min": min(launch_ms)}

    d = w.d
    perm, delay = None, None
    from overlap_producer_warps_gb300 import inputs
    if w.cfg.get("skew"):
        perm, delay = inputs.skew_schedule(0, d["R"])
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "impl": "ours",
            "config": {"workload": WORKLOAD, "R": d["R"], "M_r": d["M_r"], "K": d["K"],
                       "N": d["N"], "schedule": "ready (default)",
                       "pair_tile": f"256x{api.ag_tile_n(d['R'], d['M_r'], d['N'])}",
                       "publish_perm": None if perm is None else [int(v) for v in perm],
                       "delay_us": None if delay is None else [int(v) // 1000 for v in delay],
                       "epochs": "fresh epoch per launch, no reset",
                       "l2": "inputs larger than L2 (1.74 GB of algorithmic traffic per step "
                             "vs 129 MB L2)",
                       "prewarm_s": args.prewarm_s,
                       "parallelism": f"replicas x{world}"},
            "pct_of_peak": value / world / step_peak,
            "roofline": roofline, "e2e": e2e, "gpu_launches": args.steps, "clocks": clocks}
    w.close()
    del w
    torch.cuda.empty_cache()

    if rank == 0 and world == 1 and not args.no_extra:
        sampler2 = ClockSampler(torch.cuda.current_device())
        sampler2.start()
        line["per_config"] = per_config_results(api, torch, peak)
        sampler2.stop()
        line["per_config"]["clocks"] = sampler2.summary()
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_sample(d, min_seconds=args.cpu_seconds)
        if not args.no_extra:
            line["cpu_baseline"]["rows"] = oracle_rows_results()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="skip the per-configuration table")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--prewarm-s", type=float, default=2.0,
                    help="seconds of untimed steps before the warm-up steps (clock ramp)")
    ap.add_argument("--only", choices=["ring_allreduce", "alltoall", "ag_tiny", "ag_tp", "ag_mlp",
                                       "ag_skew", "ag_tp_gather", "ag_mlp_gather",
                                       "ag_skew_gather", "rs_tp", "rs_tp_scatter", "tp_layer",
                                       "ag_tp_all", "ag_mlp_all", "ag_skew_all", "rs_tp_all"],
                    default=None,
                    help="run only this per-configuration measurement (for profiling) and "
                         "print its result as one JSON line")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if args.impl == "reference":
        return run_reference(args, rank, world)
    if args.only is not None:
        import torch
        from overlap_producer_warps_gb300 import api
        api.lib()
        peak = float(load_peaks()[0]["bf16_tflops"])
        o = args.only
        if o == "ring_allreduce":
            res = ring_results(api, torch, args.steps)
        elif o == "alltoall":
            res = alltoall_results(api, torch, args.steps)
        elif o == "ag_tiny":
            res = tiny_results(api, torch)
        elif o == "tp_layer":
            res = tp_layer_results(api, torch, peak, args.steps)
        elif o == "rs_tp_all":
            res = rs_config_results(api, torch, peak, args.steps)
        elif o.endswith("_all"):
            res = ag_config_results(api, torch, o[:-len("_all")], peak, args.steps)
        elif o.startswith("rs_"):
            res = rs_results(api, torch, args.steps, scatter_only=o.endswith("_scatter"))
        elif o.endswith("_gather"):
            res = ag_fused_results(api, torch, o[:-len("_gather")], args.steps,
                                   producer_only=True)
        else:
            res = ag_fused_results(api, torch, o, args.steps)
        print(json.dumps({o: res}), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as _dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        _dist.init_process_group("nccl")
        dist = _dist
    try:
        return run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
