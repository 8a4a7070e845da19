#!/usr/bin/env python3
"""Throughput of lossless BF16 exponent coding on GB300 (one JSON line on stdout).

Workload: the 64M-element gradient-like BF16 tensor (N(0, 1e-3) body, 0.1%
outliers x1000, 0.01% special values), seeded and synthetic.  One step is one
pass of the whole hot path over it:
  sigma -> codebook (host closed form, uploaded), exact histogram -> top-7
  codebook (device), compress with the histogram codebook, compress with the
  sigma codebook, decompress both streams.
value = uncompressed BF16 bytes through the four codec ops (4 x 2n) per second,
the histogram pass included in the time.  Inputs (134 MB) are larger than the
129 MB L2, and each decompress reads a stream written two ops earlier.

--impl reference times the CPU oracle (plain single-threaded C) on a bounded
sample of the same workload, the same way.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "compress/decompress GB/s (uncompressed BF16) and % of HBM roofline; compression ratio"
WORKLOAD = "gradient-like bf16 tensor, 2^26 elements: N(0,1e-3), 0.1% outliers x1000, 0.01% specials"
SIGMA = 1e-3
FALLBACK_HBM_GBS = 6800.0


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--n-log2", type=int, default=26, help="workload size (default 2^26 elements)")
    p.add_argument("--cpu-sample-log2", type=int, default=25, help="elements of the timed oracle sample")
    p.add_argument("--ref-sample-log2", type=int, default=20, help="elements per reference-arm step")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-workloads", action="store_true", help="skip the per-workload section")
    p.add_argument("--sweep-max-log2", type=int, default=29, help="largest reduce-scatter shard (elements)")
    p.add_argument("--profile", action="store_true",
                   help="for profiler runs: no clock sampling, no soak, no e2e, CPU or workload legs")
    p.add_argument("--profile-pipeline", type=int, default=0, metavar="LOG2_CHUNK",
                   help="for profiler runs: only the transfer pipeline plan on 2^26 values in chunks of "
                        "2^LOG2_CHUNK (three streams), replayed 3 times, checked, no JSON line")
    a = p.parse_args(argv)
    if a.profile:
        a.no_e2e = a.no_cpu_baseline = a.no_workloads = True
    return a


# ------------------------------------------------------------------ distributed helpers
def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(
        os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank defines the job's time)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for r in csv.reader(io.StringIO(f.read())):
                if len(r) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(r[0].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    rows.append((ts, float(r[2]), float(r[3]), [x.strip() for x in r[5:10]]))
                except ValueError:
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if self.t0 is not None and self.t0 - 1 <= r[0] <= self.t1 + 1]
        use = inside or rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3][1:]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "window": "timed region" if inside else "whole run"}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# DRAM traffic per launch (dram__bytes_read.sum + dram__bytes_write.sum) of the
# codec kernels on this workload, each from one ncu capture whose summary sits
# in profiles/.  A figure is tied to a hash of the kernel's device sources at
# capture time (their code: line comments and whitespace are left out) and
# reported as null once that code has changed.
KERNEL_SOURCES = {
    "encode_kernel": ["zc_encode.cu", "zc_device.cuh"],
    "decode_kernel": ["zc_decode.cu", "zc_device.cuh"],
}
OP_KERNEL = {"histogram": "hist_kernel", "compress_hist_cb": "encode_kernel", "compress_sigma_cb": "encode_kernel",
             "decompress_hist_cb": "decode_kernel", "decompress_sigma_cb": "decode_kernel"}
MEASURED_TRAFFIC = {  # kernel: (source hash, bytes per launch)
    "encode_kernel": ("5a562adbe27a5016", 184434688),
    "decode_kernel": ("437ef86f13be512b", 167370496),
}


def source_hash(kernel: str) -> str | None:
    files = KERNEL_SOURCES.get(kernel)
    if not files:
        return None
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "lossless_bf16_exponent_zc_gb300", "csrc", f), encoding="utf-8") as fh:
            for line in fh:
                code = " ".join(line.split("//", 1)[0].split())
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def measured_traffic(kernel: str):
    rec = MEASURED_TRAFFIC.get(kernel)
    if rec is None or rec[0] != source_hash(kernel):
        return None
    return rec[1]


# ------------------------------------------------------------------ the oracle arm (CPU)
def oracle_step(x: np.ndarray):
    import oracle
    cb_s = oracle.codebook_from_sigma(SIGMA)
    cb_h, _ = oracle.histogram_topk(x)
    ma, ea = oracle.compress(x, cb_h)
    mb, eb = oracle.compress(x, cb_s)
    ya = oracle.decompress(ma, ea, x.size)
    yb = oracle.decompress(mb, eb, x.size)
    return ya, yb


def host_info() -> dict:
    """The host the CPU legs ran on: logical CPUs, machine type, CPU model (from /proc/cpuinfo when present)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    key, val = (t.strip() for t in line.split(":", 1))
                    fields.setdefault(key.lower(), val)
    except OSError:
        pass
    model = fields.get("model name") or fields.get("cpu model") or ""
    if not model and "cpu part" in fields:  # Arm: implementer and part numbers
        model = f"implementer {fields.get('cpu implementer', '?')} part {fields['cpu part']}"
    return {"nproc": os.cpu_count(), "machine": platform.machine(), "cpu": model or platform.processor()}


def cpu_baseline(x: np.ndarray, sample_log2: int) -> dict:
    m = min(x.size, 1 << sample_log2)
    sample = x[:m]
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle_step(sample)
        reps += 1
        if time.perf_counter() - t0 >= 10.0 or reps >= 8:
            break
    dt = time.perf_counter() - t0
    return {"value": round(4 * 2 * m * reps / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first 2^{int(math.log2(m))} elements of the workload, {reps} full step(s) "
                      f"(sigma and histogram codebooks, 2 compress + 2 decompress), single-threaded C, "
                      f"{dt:.1f} s", "host": host_info()}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    m = 1 << args.ref_sample_log2
    x = workloads.gradient(n=1 << args.n_log2)[:m].copy()
    for _ in range(args.warmup):
        oracle_step(x)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(x)
    dt = time.perf_counter() - t0
    value = 4 * 2 * m * args.steps / dt / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "sample": f"first 2^{args.ref_sample_log2} elements per step",
                   "element_dtype": "bf16, coded losslessly (the codec works on the bit patterns with integer operations on 32-bit words)",
                   "parallelism": "rank 0 only (CPU oracle)"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"first 2^{args.ref_sample_log2} elements of the workload per step",
                         "host": host_info()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ the GPU arm
def run_ours(args):
    import torch
    from lossless_bf16_exponent_zc_gb300 import zc

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    n = 1 << args.n_log2
    x = workloads.gradient(n=n)
    xt = torch.from_numpy(x.view(np.int16)).to(device)
    mb, eb = zc.compressed_size(n)
    main_a = torch.empty(mb, dtype=torch.uint8, device=device)
    main_b = torch.empty(mb, dtype=torch.uint8, device=device)
    esc_a = torch.empty(eb, dtype=torch.uint8, device=device)
    esc_b = torch.empty(eb, dtype=torch.uint8, device=device)
    y = torch.empty(n, dtype=torch.int16, device=device)
    ws = zc.workspace(n, device=device)
    st = zc.new_status(device=device)
    cb_hist = torch.empty(7, dtype=torch.uint8, device=device)
    cb_sig = torch.empty(7, dtype=torch.uint8, device=device)
    cb_pinned = torch.empty(7, dtype=torch.uint8).pin_memory()
    stream = torch.cuda.current_stream(device)

    ops = ["histogram", "compress_hist_cb", "compress_sigma_cb", "decompress_hist_cb", "decompress_sigma_cb"]

    def step(events=None):
        cb_pinned.numpy()[:] = zc.codebook_from_sigma(SIGMA)
        cb_sig.copy_(cb_pinned, non_blocking=True)
        calls = [
            lambda: zc.histogram_topk(xt, ws, st, cb_out=cb_hist),
            lambda: zc.compress(xt, cb_hist, ws, st, main=main_a, esc=esc_a),
            lambda: zc.compress(xt, cb_sig, ws, st, main=main_b, esc=esc_b),
            lambda: zc.decompress(main_a, esc_a, n, st, out=y),
            lambda: zc.decompress(main_b, esc_b, n, st, out=y),
        ]
        for i, c in enumerate(calls):
            if events is not None:
                events[i][0].record(stream)
            c()
            if events is not None:
                events[i][1].record(stream)

    # correctness of this very run: round trip, status
    step()
    torch.cuda.synchronize()
    if zc.status_value(st) != 0:
        raise SystemExit(f"device status {zc.status_string(zc.status_value(st))}")
    if not torch.equal(y, xt):
        raise SystemExit("round trip mismatch")
    n_esc_a, n_esc_b = zc.header_n_esc(main_a), zc.header_n_esc(main_b)

    for _ in range(args.warmup):
        step()
    clocks = ClockSampler(local)
    if not args.profile:
        clocks.start()
        # keep the GPU busy ~1 s so clock samples reflect load
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < 1.0:
            step()
    torch.cuda.synchronize()

    evs = [[[torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)] for _ in ops]
           for _ in range(args.steps)]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark_start()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(args.steps):
        step(evs[k])
    end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    clocks.mark_end()
    clk = clocks.stop()
    local_ms = start.elapsed_time(end)
    ms = max_over_ranks(local_ms, world, device)
    per_op_ms = {op: statistics.mean(evs[k][i][0].elapsed_time(evs[k][i][1]) for k in range(args.steps))
                 for i, op in enumerate(ops)}
    if zc.status_value(st) != 0:
        raise SystemExit(f"device status {zc.status_string(zc.status_value(st))}")

    units_per_step = 4 * 2 * n                        # uncompressed bytes through the codec ops
    value = sum_over_ranks(units_per_step, world, device) * args.steps / (ms / 1e3) / 1e9

    # roofline of the dominant kernel (algorithmic bytes / mean launch time)
    peak, peak_kind = hbm_peak()
    table = 4 * math.ceil(n / 4096)
    alg = {
        "histogram": 2 * n,
        "compress_hist_cb": 2 * n + mb + n_esc_a,
        "compress_sigma_cb": 2 * n + mb + n_esc_b,
        "decompress_hist_cb": mb + n_esc_a + 2 * n,
        "decompress_sigma_cb": mb + n_esc_b + 2 * n,
    }
    dominant = max(ops, key=lambda o: per_op_ms[o])
    achieved = alg[dominant] / (per_op_ms[dominant] / 1e3) / 1e9
    ops_report = {o: {"ms": round(per_op_ms[o], 4), "GB_per_s_uncompressed": round(2 * n / per_op_ms[o] / 1e6, 1),
                      "alg_bytes": alg[o], "alg_GB_per_s": round(alg[o] / per_op_ms[o] / 1e6, 1),
                      "frac_of_hbm": round(alg[o] / per_op_ms[o] / 1e6 / peak, 4)} for o in ops}

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(args, zc, torch, device, x, mb, eb, world)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(x, args.cpu_sample_log2)

    per_workload = None
    if world == 1 and not args.no_workloads:
        del main_a, main_b, esc_a, esc_b, y
        per_workload = run_workloads(args, zc, torch, device, peak)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded)",
            "config": {"workload": WORKLOAD, "elements": n, "codebooks": "exact histogram top-7 and sigma=1e-3",
                       "element_dtype": "bf16, coded losslessly (the codec works on the bit patterns with integer operations on 32-bit words)",
                       "l2": "inputs (134 MB bf16) larger than the 129 MB L2; no flush",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                         "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": measured_traffic(OP_KERNEL[dominant]), "alg_bytes": alg[dominant],
                         "peak_source": peak_kind},
            "compression": {
                "ratio_hist_cb": round(2 * n / (mb + n_esc_a), 4), "escape_rate_hist_cb": round(n_esc_a / n, 5),
                "ratio_sigma_cb": round(2 * n / (mb + n_esc_b), 4), "escape_rate_sigma_cb": round(n_esc_b / n, 5)},
            "ops": ops_report,
            "gpu_launches": 5 * args.steps,
            "clocks": clk,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "workloads": per_workload,
            "cost_model": cost_model_context(zc, ops_report, per_workload, n, 2 * n / (mb + n_esc_b)),
            # last, so that a reader of the line's tail sees every workload: fraction of measured HBM per op
            "summary_frac_of_hbm": workload_summary(ops_report, per_workload),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def workload_summary(ops_report, per_workload):
    """{workload: {op: fraction of the measured HBM peak}} for the step's ops and every workload section."""
    out = {"gradient_2^26_step": {o: v["frac_of_hbm"] for o, v in ops_report.items()}}
    for name, sec in (per_workload or {}).items():
        if isinstance(sec, dict) and "frac_of_hbm" in sec:
            out[name] = sec["frac_of_hbm"]
        elif isinstance(sec, dict):
            ops = {op: v["frac_of_hbm"] for op, v in sec.items() if isinstance(v, dict) and "frac_of_hbm" in v}
            for sub, v in sec.items():  # one level further (raw bypass, QLC)
                if isinstance(v, dict) and not ("frac_of_hbm" in v):
                    ops.update({f"{sub}.{op}": w["frac_of_hbm"] for op, w in v.items()
                                if isinstance(w, dict) and "frac_of_hbm" in w})
            if ops:
                out[name] = ops
    return out


def cost_model_context(zc, ops_report, per_workload, n, ratio):
    """The host cost models fed with this run's measured codec throughput and ratio, for two example links
    (a 400 Gb/s network port, 50 GB/s, 5 us; an NVLink-class link, 900 GB/s, 2 us): does compressing a
    2^26-value tensor pay, and which reduce-scatter would the switcher pick at P = 8 (with the measured
    decode-reduce throughput when the workload section ran).  Context only: no link is measured on one GPU."""
    c = ops_report["compress_sigma_cb"]["GB_per_s_uncompressed"]
    d = ops_report["decompress_sigma_cb"]["GB_per_s_uncompressed"]
    dr = d
    if per_workload and "reduce_scatter_8x2^25" in per_workload:
        dr = per_workload["reduce_scatter_8x2^25"]["GB_per_s_uncompressed"]
    out = {"compress_gbps": c, "decompress_gbps": d, "decompress_reduce_gbps": dr, "ratio": round(ratio, 4),
           "links": {}}
    for name, bw, lat in (("network_50GBps_5us", 50.0, 5.0), ("nvlink_900GBps_2us", 900.0, 2.0)):
        pays, t_raw, t_zip = zc.transfer_pays(2 * n, bw, lat, c, d, ratio)
        use, t_nat, t_rs = zc.reduce_scatter_choose(2 * n, 8, bw, lat, c, dr, ratio)
        out["links"][name] = {"transfer_pays": pays, "t_raw_us": round(t_raw, 1), "t_zipped_us": round(t_zip, 1),
                              "reduce_scatter_zipped": use, "t_native_rs_us": round(t_nat, 1),
                              "t_zipped_rs_us": round(t_rs, 1)}
    return out


def run_e2e(args, zc, torch, device, x, mb, eb, world):
    """The same step through the public API as a full host round trip, all buffers pinned: upload the tensor,
    encode with both codebooks, download each main stream (fixed size) and then each escape stream (its size
    read from the downloaded header), upload both streams again into separate receive buffers, decode from
    those and download both decoded tensors.  The two codebooks' paths run on two streams (each with its own
    workspace), and the host waits for each path's main stream on an event, so one path's copies overlap the
    other's kernels.  Steps are software-pipelined over three buffer sets: step k + 1 uploads, encodes and
    downloads its main streams before step k's receiving side is enqueued, so the link carries both directions
    at once and the download queue never waits for an upload; a set is reused only after its previous step
    has finished."""
    n = x.size
    x_h = torch.from_numpy(x.view(np.int16)).pin_memory()
    cb_pinned = torch.empty(7, dtype=torch.uint8).pin_memory()
    cb_pinned.numpy()[:] = zc.codebook_from_sigma(SIGMA)
    st = zc.new_status(device=device)

    def buffer_set():
        return {
            "y_h": [torch.empty(n, dtype=torch.int16).pin_memory() for _ in range(2)],
            "m_h": [torch.empty(mb, dtype=torch.uint8).pin_memory() for _ in range(2)],
            "e_h": [torch.empty(eb, dtype=torch.uint8).pin_memory() for _ in range(2)],
            "xt": torch.empty(n, dtype=torch.int16, device=device),
            "mains": [torch.empty(mb, dtype=torch.uint8, device=device) for _ in range(2)],
            "escs": [torch.empty(eb, dtype=torch.uint8, device=device) for _ in range(2)],
            "r_mains": [torch.empty(mb, dtype=torch.uint8, device=device) for _ in range(2)],
            "r_escs": [torch.empty(eb, dtype=torch.uint8, device=device) for _ in range(2)],
            "ys": [torch.empty(n, dtype=torch.int16, device=device) for _ in range(2)],
            "wss": [zc.workspace(n, device=device) for _ in range(2)],
            "cbs": [torch.empty(7, dtype=torch.uint8, device=device) for _ in range(2)],
            "streams": [torch.cuda.Stream(device=device) for _ in range(2)],
            "ev_in": torch.cuda.Event(), "ev_main": [torch.cuda.Event() for _ in range(2)],
            "ev_done": torch.cuda.Event(), "used": False}
    sets = [buffer_set() for _ in range(3)]
    moved = [0, 0]

    def begin(k):
        """Step k, first half: upload, codebooks, encode, download the main streams (static part)."""
        S = sets[k % 3]
        if S["used"]:
            S["ev_done"].synchronize()                           # this set's previous step has finished
        S["used"] = True
        s0, s1 = S["streams"]
        xt, cbs, wss = S["xt"], S["cbs"], S["wss"]
        with torch.cuda.stream(s0):
            xt.copy_(x_h, non_blocking=True)
            cbs[1].copy_(cb_pinned, non_blocking=True)
            S["ev_in"].record(s0)
            zc.histogram_topk(xt, wss[0], st, cb_out=cbs[0], stream=s0)
        s1.wait_event(S["ev_in"])
        for i in range(2):
            with torch.cuda.stream(S["streams"][i]):
                zc.compress(xt, cbs[i], wss[i], st, main=S["mains"][i], esc=S["escs"][i], stream=S["streams"][i])
                S["m_h"][i].copy_(S["mains"][i], non_blocking=True)
                S["ev_main"][i].record(S["streams"][i])

    def finish(k):
        """Step k, second half: escapes sized from the downloaded headers, the receiving side's uploads,
        decode, download of the decoded tensors."""
        S = sets[k % 3]
        s0, s1 = S["streams"]
        ks = []
        for i in range(2):
            S["ev_main"][i].synchronize()                        # this path's main stream has arrived
            kk = int.from_bytes(S["m_h"][i][24:32].numpy().tobytes(), "little")
            ks.append(kk)
            with torch.cuda.stream(S["streams"][i]):
                if kk:
                    S["e_h"][i][:kk].copy_(S["escs"][i][:kk], non_blocking=True)  # the dynamic part
                S["r_mains"][i].copy_(S["m_h"][i], non_blocking=True)            # the receiving side uploads it
                if kk:
                    S["r_escs"][i][:kk].copy_(S["e_h"][i][:kk], non_blocking=True)
                zc.decompress(S["r_mains"][i], S["r_escs"][i], n, st, out=S["ys"][i], stream=S["streams"][i])
                S["y_h"][i].copy_(S["ys"][i], non_blocking=True)
        s0.wait_stream(s1)
        S["ev_done"].record(s0)
        streams_b = 2 * mb + sum(ks)
        moved[0] = 2 * n + 7 + streams_b
        moved[1] = streams_b + 2 * 2 * n

    def run(count):
        """count whole steps, software-pipelined: step k + 1 begins before step k finishes."""
        begin(0)
        for k in range(count):
            if k + 1 < count:
                begin(k + 1)
            finish(k)

    run(max(3, args.warmup))
    steps = max(5, args.steps // 10)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    run(steps)
    torch.cuda.synchronize()
    dt = max_over_ranks(time.perf_counter() - t0, world, device)
    if not all(torch.equal(y, x_h) for S in sets for y in S["y_h"]):
        raise SystemExit("end-to-end round trip mismatch")
    value = sum_over_ranks(4 * 2 * n, world, device) * steps / dt / 1e9
    return {"value": round(value, 2), "unit": "GB/s", "h2d_bytes_per_step": moved[0],
            "d2h_bytes_per_step": moved[1], "steps": steps,
            "path": "host tensor -> device -> histogram + 2 compress -> host streams -> device -> "
                    "2 decompress -> host tensors, pinned buffers, one stream per codebook, steps "
                    "software-pipelined over three buffer sets"}


# ------------------------------------------------------------------ per-workload section
def _time_ms(torch, fn, reps, warmup=2):
    for _ in range(warmup):
        fn()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record()
    for _ in range(reps):
        fn()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / reps


def _time_graph_ms(torch, fn, calls=20, replays=10):
    """Per-call device time of fn with the host out of the way: `calls` calls captured in one CUDA graph,
    replayed `replays` times.  Small calls timed back to back on a stream measure how fast the host submits
    them; this measures the GPU.  None if the calls cannot be captured."""
    try:
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                fn()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(calls):
                fn()
        g.replay()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(replays):
            g.replay()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / (calls * replays)
    except Exception:  # capture unsupported here: report the stream timing only
        return None


def run_workloads(args, zc, torch, device, peak):
    """Per-kernel GB/s (uncompressed and algorithmic), HBM fraction, ratio and escape rate for the other
    workloads: the 2^20 Gaussian (L2-resident), the 9-tensor Llama-3-8B bucket (batched), the MoE payload
    (histogram codebook, 8 Zipf chunks batched), the reduce-scatter local stage (P = 8) with its
    shard-size sweep, the raw bypass (adaptive compression of coded and incompressible 2^26 tensors), and the
    zipped transfer pipeline (16 or 4 chunks on three streams against one stream and a plain copy), and
    Quad Length Codes on 2^26 FP8 e4m3 bytes.
    Inputs above L2 size are not flushed between repetitions of the same op."""
    import math as _m
    out = {}
    st = zc.new_status(device=device)
    dev = lambda a: torch.from_numpy(a.view(np.int16)).to(device)

    def entry(ms, n_unc, alg):
        return {"ms": round(ms, 4), "GB_per_s_uncompressed": round(n_unc / ms / 1e6, 1),
                "alg_GB_per_s": round(alg / ms / 1e6, 1), "frac_of_hbm": round(alg / ms / 1e6 / peak, 4)}

    # 0. the histogram on its own: two 2^26 N(0, 1e-3) tensors alternated, so every call reads from HBM and no
    #    decompress output is being written back from L2 meanwhile (inside the gradient step it is)
    ha = [workloads.gaussian_on_device(1 << 26, 1e-3, seed=40 + i, device=device) for i in range(2)]
    hws = zc.workspace(1 << 26, device=device)
    hcb = torch.empty(7, dtype=torch.uint8, device=device)
    calls = [0]

    def hist_alt():
        zc.histogram_topk(ha[calls[0] & 1], hws, st, cb_out=hcb)
        calls[0] += 1
    th_alone = _time_ms(torch, hist_alt, 20)
    out["histogram_2^26_alone"] = entry(th_alone, 2 << 26, 2 << 26)
    del ha, hws

    # 1. gaussian 2^20, sigma codebook
    x = workloads.gaussian()
    n = x.size
    xt = dev(x)
    cb = zc.codebook_to_device(zc.codebook_from_sigma(workloads.GAUSSIAN_SIGMA), device)
    ws = zc.workspace(n, device=device)
    mb, eb = zc.compressed_size(n)
    m_t = torch.empty(mb, dtype=torch.uint8, device=device)
    e_t = torch.empty(eb, dtype=torch.uint8, device=device)
    y = torch.empty(n, dtype=torch.int16, device=device)
    fc = lambda: zc.compress(xt, cb, ws, st, main=m_t, esc=e_t)
    tc = _time_ms(torch, fc, 50)
    k = zc.header_n_esc(m_t)
    fd = lambda: zc.decompress(m_t, e_t, n, st, out=y)
    td = _time_ms(torch, fd, 50)
    gc, gd = _time_graph_ms(torch, fc), _time_graph_ms(torch, fd)
    out["gaussian_2^20_L2_resident"] = {"compress": entry(tc, 2 * n, 2 * n + mb + k),
                                        "decompress": entry(td, 2 * n, 2 * n + mb + k),
                                        "graph_replay_us": {"compress": round(1e3 * gc, 2) if gc else None,
                                                            "decompress": round(1e3 * gd, 2) if gd else None},
                                        "ratio": round(2 * n / (mb + k), 4), "escape_rate": round(k / n, 5)}

    # 2. Llama-3-8B layer bucket, one batched launch each way
    bucket = workloads.llama_bucket()
    items, outs, total_n = [], [], 0
    for name, a, sigma in bucket:
        mb_i, eb_i = zc.compressed_size(a.size)
        items.append(zc.BatchItem(bf16=dev(a), main=torch.empty(mb_i, dtype=torch.uint8, device=device),
                                  esc=torch.empty(eb_i, dtype=torch.uint8, device=device),
                                  cb=zc.codebook_to_device(zc.codebook_from_sigma(sigma), device)))
        total_n += a.size
    del bucket
    ws = zc.workspace([it.bf16.numel() for it in items], device=device)
    tc = _time_ms(torch, lambda: zc.compress_batched(items, ws, st), 10)
    mains = sum(it.main.numel() for it in items)
    escs = sum(zc.header_n_esc(it.main) for it in items)
    outs = [zc.BatchItem(bf16=torch.empty_like(it.bf16), main=it.main, esc=it.esc) for it in items]
    td = _time_ms(torch, lambda: zc.decompress_batched(outs, st), 10)
    ok = all(torch.equal(o.bf16, it.bf16) for o, it in zip(outs, items))
    out["llama3_8b_layer_bucket_9_tensors"] = {
        "elements": total_n, "compress_batched": entry(tc, 2 * total_n, 2 * total_n + mains + escs),
        "decompress_batched": entry(td, 2 * total_n, 2 * total_n + mains + escs),
        "ratio": round(2 * total_n / (mains + escs), 4), "escape_rate": round(escs / total_n, 5), "round_trip_ok": ok}
    del items, outs

    # 3. MoE all-to-all payload: histogram codebook over the payload, 8 destination chunks
    x, counts = workloads.moe_payload()
    n = x.size
    xt = dev(x)
    del x
    ws = zc.workspace([c * 4096 for c in counts], device=device)
    cbh = torch.empty(7, dtype=torch.uint8, device=device)
    th = _time_ms(torch, lambda: zc.histogram_topk(xt, ws, st, cb_out=cbh), 10)
    items, start = [], 0
    for c in counts:
        m_ = c * 4096
        mb_i, eb_i = zc.compressed_size(m_)
        items.append(zc.BatchItem(bf16=xt[start:start + m_], main=torch.empty(mb_i, dtype=torch.uint8, device=device),
                                  esc=torch.empty(eb_i, dtype=torch.uint8, device=device), cb=cbh))
        start += m_
    tc = _time_ms(torch, lambda: zc.compress_batched(items, ws, st), 10)
    mains = sum(it.main.numel() for it in items)
    escs = sum(zc.header_n_esc(it.main) for it in items)
    outs = [zc.BatchItem(bf16=torch.empty_like(it.bf16), main=it.main, esc=it.esc) for it in items]
    td = _time_ms(torch, lambda: zc.decompress_batched(outs, st), 10)
    ok = torch.equal(torch.cat([o.bf16 for o in outs]), xt)
    out["moe_payload_16384x4096_8_chunks"] = {
        "histogram": entry(th, 2 * n, 2 * n), "compress_batched": entry(tc, 2 * n, 2 * n + mains + escs),
        "decompress_batched": entry(td, 2 * n, 2 * n + mains + escs), "ratio": round(2 * n / (mains + escs), 4),
        "escape_rate": round(escs / n, 5), "round_trip_ok": bool(ok)}
    del items, outs, xt

    # 4. reduce-scatter local stage: P = 8 shards of 2^25, sigma codebook in, sigma*sqrt(8) out
    P = 8
    shards = workloads.rs_shards()
    base = [dev(a) for a in shards]
    del shards
    cb_in = zc.codebook_to_device(zc.codebook_from_sigma(workloads.RS_SIGMA), device)
    cb_out = zc.codebook_to_device(zc.codebook_from_sigma(workloads.RS_SIGMA * _m.sqrt(P)), device)

    def reduce_case(m):
        """Compress P shards of m elements (tiling the 2^25 base shards), time decompress_reduce."""
        reps_src = -(-m // base[0].numel())
        src = [b.repeat(reps_src)[:m] if reps_src > 1 else b[:m] for b in base]
        ws_ = zc.workspace(m, device=device)
        mains_, escs_ = [], []
        for s_ in src:
            a_, b_ = zc.compress(s_, cb_in, ws_, st)
            mains_.append(a_)
            escs_.append(b_)
        del src
        mb_, eb_ = zc.compressed_size(m)
        y_ = torch.empty(m, dtype=torch.int16, device=device)
        om_ = torch.empty(mb_, dtype=torch.uint8, device=device)
        oe_ = torch.empty(eb_, dtype=torch.uint8, device=device)
        reps = max(20, min(50, int(2e9 // (P * m * 2))))
        fr = lambda: zc.decompress_reduce(mains_, escs_, m, st, out=y_, out_cb=cb_out, out_main=om_, out_esc=oe_,
                                          ws=ws_)
        t_ = _time_ms(torch, fr, reps)
        g_ = _time_graph_ms(torch, fr) if m <= (1 << 22) else None
        in_bytes = sum(mb_ + zc.header_n_esc(a_) for a_ in mains_)
        k_out = zc.header_n_esc(om_)
        alg = in_bytes + 2 * m + mb_ + k_out
        r = entry(t_, 2 * P * m, alg)
        r.update({"shard_elements": m, "escape_rate_in": round((in_bytes - P * mb_) / (P * m), 5),
                  "escape_rate_out": round(k_out / m, 5)})
        if g_ is not None:
            r["graph_replay_us"] = round(1e3 * g_, 2)
        return r

    out["reduce_scatter_8x2^25"] = reduce_case(1 << 25)
    # the senders' side of the same workload: compress and decompress of 2^25-element shards, cycling
    # through the 8 shards (and 8 output buffers) so that consecutive calls miss L2
    m = 1 << 25
    ws_ = zc.workspace(m, device=device)
    mb_, eb_ = zc.compressed_size(m)
    sm_ = [torch.empty(mb_, dtype=torch.uint8, device=device) for _ in range(P)]
    se_ = [torch.empty(eb_, dtype=torch.uint8, device=device) for _ in range(P)]
    sy_ = [torch.empty(m, dtype=torch.int16, device=device) for _ in range(P)]
    it = [0]

    def shard_compress():
        i = it[0] % P
        it[0] += 1
        zc.compress(base[i], cb_in, ws_, st, main=sm_[i], esc=se_[i])

    def shard_decompress():
        i = it[0] % P
        it[0] += 1
        zc.decompress(sm_[i], se_[i], m, st, out=sy_[i])

    tc_ = _time_ms(torch, shard_compress, 4 * P)
    k_ = sum(zc.header_n_esc(t) for t in sm_) / P
    td_ = _time_ms(torch, shard_decompress, 4 * P)
    out["reduce_scatter_shard_2^25"] = {"compress": entry(tc_, 2 * m, 2 * m + mb_ + k_),
                                        "decompress": entry(td_, 2 * m, 2 * m + mb_ + k_),
                                        "ratio": round(2 * m / (mb_ + k_), 4), "escape_rate": round(k_ / m, 5),
                                        "l2": "8 shards and 8 output sets in rotation (512 MB of inputs)"}
    # a sender compresses its 8 destination shards in one batched launch; a receiver decodes them likewise
    wsb = zc.workspace([m] * P, device=device)
    items = [zc.BatchItem(bf16=base[i], main=sm_[i], esc=se_[i], cb=cb_in) for i in range(P)]
    tcb = _time_ms(torch, lambda: zc.compress_batched(items, wsb, st), 10)
    kb = sum(zc.header_n_esc(t) for t in sm_)
    outs_b = [zc.BatchItem(bf16=sy_[i], main=sm_[i], esc=se_[i]) for i in range(P)]
    tdb = _time_ms(torch, lambda: zc.decompress_batched(outs_b, st), 10)
    okb = all(torch.equal(sy_[i], base[i]) for i in range(P))
    out["reduce_scatter_8_shards_batched"] = {
        "compress_batched": entry(tcb, 2 * m * P, P * (2 * m + mb_) + kb),
        "decompress_batched": entry(tdb, 2 * m * P, P * (2 * m + mb_) + kb), "round_trip_ok": bool(okb)}
    del ws_, sm_, se_, sy_, wsb, items, outs_b
    sweep = []
    for lg in range(15, args.sweep_max_log2 + 1):
        sweep.append(reduce_case(1 << lg))
        torch.cuda.empty_cache()
    out["reduce_scatter_sweep_P8"] = [{"shard_bytes": r["shard_elements"] * 2, "ms": r["ms"],
                                       "GB_per_s_uncompressed": r["GB_per_s_uncompressed"],
                                       "frac_of_hbm": r["frac_of_hbm"],
                                       "graph_replay_us": r.get("graph_replay_us")} for r in sweep]
    del base

    # 5. raw bypass [CCCL §3.3, §5.2]: adaptive compression of a 2^26 N(0, 1e-3) tensor (stays coded: the cost
    #    is the device-side decision) and of 2^26 uniformly random bit patterns (stored RAW; its algorithmic
    #    bytes are those of a copy: read 2n, write the 2n-byte RAW image)
    n = 1 << 26
    mb, _ = zc.compressed_size(n)
    spill = zc.raw_spill(n)
    ws = zc.workspace(n, device=device)
    m_t = torch.empty(mb, dtype=torch.uint8, device=device)
    e_t = torch.empty(n, dtype=torch.uint8, device=device)
    y = torch.empty(n, dtype=torch.int16, device=device)
    xt = dev(workloads.gaussian(n, sigma=workloads.RS_SIGMA, seed=6))
    cbg = zc.codebook_to_device(zc.codebook_from_sigma(workloads.RS_SIGMA), device)
    tp = _time_ms(torch, lambda: zc.compress(xt, cbg, ws, st, main=m_t, esc=e_t), 20)
    ta = _time_ms(torch, lambda: zc.compress_adaptive(xt, cbg, ws, st, main=m_t, esc=e_t), 20)
    k = zc.header_n_esc(m_t)
    coded = {"compress": entry(tp, 2 * n, 2 * n + mb + k), "compress_adaptive": entry(ta, 2 * n, 2 * n + mb + k),
             "stored_raw": zc.header_is_raw(m_t), "decision_cost_us": round(1e3 * (ta - tp), 2)}
    xt = dev(workloads.random_bits(n))
    tp = _time_ms(torch, lambda: zc.compress(xt, cbg, ws, st, main=m_t, esc=e_t), 5)
    k = zc.header_n_esc(m_t)
    ta = _time_ms(torch, lambda: zc.compress_adaptive(xt, cbg, ws, st, main=m_t, esc=e_t), 20)
    is_raw = zc.header_is_raw(m_t)
    td = _time_ms(torch, lambda: zc.decompress(m_t, e_t, n, st, out=y), 20)
    ok = torch.equal(y, xt)
    out["raw_bypass_2^26"] = {
        "coded_gaussian": coded,
        "random_bits": {"compress_coded": entry(tp, 2 * n, 2 * n + mb + k), "coded_escape_rate": round(k / n, 5),
                        "compress_adaptive": entry(ta, 2 * n, 4 * n), "decompress": entry(td, 2 * n, 4 * n),
                        "stored_raw": is_raw, "bytes_sent": mb + spill, "ratio": round(2 * n / (mb + spill), 4),
                        "round_trip_ok": bool(ok)}}
    del xt, m_t, e_t, y

    # 6. zipped transfer pipeline [CCCL §3.2, ZipCCL §2.D]: 2^26 N(0, 1e-3) values in chunks of 2^22 and 2^24,
    #    compress / link (device-to-device copy standing in for the network) / decompress on three streams,
    #    against the same calls on one stream and a plain copy of the uncompressed tensor
    xt = dev(workloads.gaussian(n, sigma=workloads.RS_SIGMA, seed=6))
    y = torch.empty(n, dtype=torch.int16, device=device)
    yc = torch.empty_like(xt)
    tcopy = _time_ms(torch, lambda: yc.copy_(xt), 10)
    cur = torch.cuda.current_stream()
    s3 = (cur, torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    pipe = {"uncompressed_device_copy_ms": round(tcopy, 4)}
    # the same transfer unchunked: compress the whole tensor, copy its main stream and escapes, decompress
    wws = zc.workspace(n, device=device)
    wm, we = torch.empty(mb, dtype=torch.uint8, device=device), torch.empty(n, dtype=torch.uint8, device=device)
    rm, re_ = torch.empty_like(wm), torch.empty_like(we)
    zc.compress(xt, cbg, wws, st, main=wm, esc=we)
    kw = zc.header_n_esc(wm)

    def whole():
        zc.compress(xt, cbg, wws, st, main=wm, esc=we)
        rm.copy_(wm)
        re_[:kw].copy_(we[:kw])
        zc.decompress(rm, re_, n, st, out=y, esc_bytes=kw)
    tw = _time_ms(torch, whole, 10)
    pipe["whole_tensor_compress_copy_decompress_ms"] = round(tw, 4)
    del wws, wm, we, rm, re_
    for lg in (22, 24):
        chunk = 1 << lg
        pws = zc.pipeline_workspace(chunk, device=device)
        t3 = _time_ms(torch, lambda: zc.pipelined_transfer(xt, cbg, chunk, pws, st, out=y, streams=s3), 10)
        ok = torch.equal(y, xt)
        t1 = _time_ms(torch, lambda: zc.pipelined_transfer(xt, cbg, chunk, pws, st, out=y, streams=(cur, cur, cur)),
                      10)
        # the launch sequence captured once as a CUDA graph (zc_pipeline_plan_*) and replayed
        y.zero_()
        p3 = zc.pipeline_plan(xt, cbg, chunk, pws, st, out=y, overlap=True)
        tp3 = _time_ms(torch, p3.launch, 10)
        ok_plan = torch.equal(y, xt)
        p1 = zc.pipeline_plan(xt, cbg, chunk, pws, st, out=y, overlap=False)
        tp1 = _time_ms(torch, p1.launch, 10)
        p3.close()
        p1.close()
        pipe[f"chunks_2^{lg}"] = {
            "chunks": n // chunk,
            "three_streams": {"ms": round(t3, 4), "GB_per_s_uncompressed": round(2 * n / t3 / 1e6, 1)},
            "one_stream": {"ms": round(t1, 4), "GB_per_s_uncompressed": round(2 * n / t1 / 1e6, 1)},
            "overlap_speedup": round(t1 / t3, 3), "round_trip_ok": bool(ok),
            "plan_three_streams": {"ms": round(tp3, 4), "GB_per_s_uncompressed": round(2 * n / tp3 / 1e6, 1)},
            "plan_one_stream": {"ms": round(tp1, 4)}, "plan_overlap_speedup": round(tp1 / tp3, 3),
            "plan_vs_whole_tensor": round(tp3 / tw, 3), "plan_round_trip_ok": bool(ok_plan)}
        del pws
    out["pipelined_transfer_2^26"] = pipe
    del xt, y, yc

    # 7. Quad Length Codes on 2^26 FP8 e4m3 bytes [QLC §3-§4]: FFN1-activation and gradient stand-ins, the
    #    table from each tensor's histogram, static widths; algorithmic bytes = read n + write the stream
    #    (compress) and the reverse (decompress)
    qlc = {}
    wsq = zc.workspace(n, device=device)
    for name, gen in (("fp8_ffn1", workloads.fp8_ffn1), ("fp8_gradient", workloads.fp8_gradient)):
        xb = gen(n)
        table = zc.zq_table_from_histogram(np.bincount(xb, minlength=256))
        xq = torch.from_numpy(xb).to(device)
        del xb
        sq = torch.empty(zc.zq_max_bytes(n), dtype=torch.uint8, device=device)
        yq = torch.empty(n, dtype=torch.uint8, device=device)
        tq = _time_ms(torch, lambda: zc.zq_compress(xq, table, wsq, st, out=sq), 20)
        nbytes = zc.zq_stream_bytes(sq)
        tdq = _time_ms(torch, lambda: zc.zq_decompress(sq, n, st, out=yq, in_bytes=nbytes), 20)
        ok = torch.equal(yq, xq)
        qlc[name] = {"compress": entry(tq, n, n + nbytes), "decompress": entry(tdq, n, n + nbytes),
                     "ratio": round(n / nbytes, 4), "saving": round(1 - nbytes / n, 4), "round_trip_ok": bool(ok)}
        del xq, sq, yq
    out["qlc_fp8_2^26"] = qlc

    if zc.status_value(st) != 0:
        out["status"] = zc.status_string(zc.status_value(st))
    return out


def profile_pipeline(log2_chunk: int) -> int:
    """The transfer pipeline plan alone, for a profiler's launch list: 2^26 N(0, 1e-3) values through compress
    -> link -> decompress in chunks of 2^log2_chunk on three streams, replayed three times, output checked."""
    import torch
    from lossless_bf16_exponent_zc_gb300 import zc
    n, chunk = 1 << 26, 1 << log2_chunk
    xt = torch.from_numpy(workloads.gaussian(n, sigma=workloads.RS_SIGMA, seed=6).view(np.int16)).cuda()
    cb = zc.codebook_to_device(zc.codebook_from_sigma(workloads.RS_SIGMA))
    st = zc.new_status()
    plan = zc.pipeline_plan(xt, cb, chunk, zc.pipeline_workspace(chunk), st)
    for _ in range(3):
        out = plan.launch()
    torch.cuda.synchronize()
    if zc.status_value(st) != 0 or not torch.equal(out, xt):
        raise SystemExit("pipeline round trip failed")
    plan.close()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.profile_pipeline:
        return profile_pipeline(args.profile_pipeline)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
