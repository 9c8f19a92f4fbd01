#!/usr/bin/env python3
"""Benchmark of the SparCML-style sparse-reduction hot path on GB300.

One step = one error-feedback step of the whole path for P emulated nodes:
Top-k with residual (guess, stream and select kernels), packing into
{uint32 index, fp32 value} streams, b-bit stochastic quantisation where the
workload has it, and the sparse sum-reduce with the dense switch. The default
workload is the largest one, LSTM/ASR-like: P=16 nodes of N=67,108,864 fp32
gradients, Top-k 1% per node, 4-bit quantisation in buckets of 512, fused
dequantise + sparse reduce. ``value`` is the gradient input the sparse-reduce
step consumes per second (P * N * 4 bytes per step) with inputs resident in
HBM; the reduce's own input rate (8 B per stream entry, or the quantised
form's bytes) and roofline are reported beside it in ``reduce``; ``e2e`` is
the step with every step's gradients copied in from pinned host memory and
the reduced result copied back.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun each rank runs an independent replica on its own GPU (the
path has no cross-GPU exchange); rank 0 prints one JSON line.
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
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-reduce step input GB/s and elems/s at 1 GB300; % of HBM peak (ncu)"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0  # the part's rated HBM3e bandwidth: context beside the measured peak


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["resnet50", "asr", "sweep", "logreg", "qsgd", "ssar",
                                           "asr_reduce"],
                    default="asr",
                    help="resnet50/asr: the whole EF step; sweep/logreg: the sparse reduce alone "
                         "on given streams (density-sweep cell / Zipf logistic regression); "
                         "qsgd: b-bit quantisation of a dense reduced result; "
                         "ssar: recursive-doubling sparse allreduce of a density-sweep cell")
    ap.add_argument("--overlap", action="store_true",
                    help="EF-step workloads: the quantise and reduce of step t on a second stream, "
                         "overlapping step t+1's Top-k (default: every step on one stream)")
    ap.add_argument("--bits", type=int, default=4, choices=[2, 4, 8],
                    help="asr / qsgd: width of the quantised codes")
    ap.add_argument("--op", default="sum", choices=["sum", "max", "min", "or"],
                    help="sweep / logreg: the reduction (each with its neutral element)")
    ap.add_argument("--sweep-p", type=int, default=64)
    ap.add_argument("--sweep-d", type=float, default=10,
                    help="per-node density in percent: 0.1, 1, 5 or 10")
    ap.add_argument("--e2e-steps", type=int, default=40)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--nodes", type=int, default=0,
                    help="override P (smaller device footprint for profiling captures)")
    ap.add_argument("--cpu-segments", type=int, default=48,
                    help="resnet50: layer segments per node in the bounded CPU-baseline sample")
    ap.add_argument("--cpu-entries", type=int, default=1 << 23,
                    help="asr: entries per node (one segment) in the bounded CPU-baseline sample")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
class Ranks:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = False
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend=backend)
            self.pg = True

    def device(self):
        return torch.device("cuda", self.local) if torch.cuda.is_available() else torch.device("cpu")

    def barrier(self):
        if self.pg:
            import torch.distributed as dist
            dist.barrier()

    def max(self, x: float) -> float:
        return reduce_max(x, self.pg, self.device())

    def close(self):
        if self.pg:
            import torch.distributed as dist
            dist.destroy_process_group()


def gpu_head_start(calls: int, us_per_call: float = 60.0):
    """Hold the GPU in a short spin before a loop of small timed calls, so the
    host queues the calls ahead of the GPU and no timed interval includes host
    launch latency (each call's interval is bracketed by its own events)."""
    torch.cuda._sleep(int(min(calls * us_per_call, 200_000.0) * 2_000))  # ~2 GHz cycles


def job_rate(world: int, units_per_rank: float, seconds: float) -> float:
    """Whole-job throughput: every rank processes the same units (weak
    scaling), and the job takes as long as its slowest rank."""
    return world * units_per_rank / seconds


def reduce_max(x: float, pg: bool, device) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    if not pg:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    """Samples the SM clock, its maximum, the board power and the active
    clock-event reasons of the benchmarked GPU from a background thread,
    every few milliseconds, through NVML (the driver's management library,
    read-only queries), or every 50 ms through nvidia-smi if NVML cannot be
    loaded. summary(t0, t1) reports the samples inside [t0, t1] (host
    time.time()); if none fell there it reports the whole sampling run and
    says so in "window"."""
    REASONS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
               "hw_thermal_slowdown": 0x40, "hw_power_brake_slowdown": 0x80}

    def __init__(self, device, period_s: float = 0.002):
        import ctypes as C
        self.samples = []  # (time, sm_mhz, max_mhz, power_w, reason bits)
        self.stop_flag = threading.Event()
        self.proc = None
        self.source = None
        uuid = None
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            uuid = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            pass
        try:
            nv = C.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                raise OSError("nvmlInit failed")
            h = C.c_void_p()
            if uuid is None or nv.nvmlDeviceGetHandleByUUID(uuid.encode(), C.byref(h)) != 0:
                raise OSError("no NVML handle")
            get_reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                nv.nvmlDeviceGetCurrentClocksThrottleReasons
            self.nv, self.h, self.get_reasons, self.period = nv, h, get_reasons, period_s
            self.source = "nvml"
            self.thread = threading.Thread(target=self._poll_nvml, daemon=True)
            self.thread.start()
        except Exception:
            self._start_smi(uuid if uuid else str(device.index))

    def _poll_nvml(self):
        import ctypes as C
        sm, mx, pw, rs = C.c_uint(), C.c_uint(), C.c_uint(), C.c_ulonglong()
        while not self.stop_flag.is_set():
            ok = (self.nv.nvmlDeviceGetClockInfo(self.h, 1, C.byref(sm)) == 0 and
                  self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, C.byref(mx)) == 0)
            pok = self.nv.nvmlDeviceGetPowerUsage(self.h, C.byref(pw)) == 0
            rok = self.get_reasons(self.h, C.byref(rs)) == 0
            if ok:
                self.samples.append((time.time(), float(sm.value), float(mx.value),
                                     pw.value / 1000.0 if pok else None,
                                     int(rs.value) if rok else 0))
            time.sleep(self.period)

    def _start_smi(self, ident):
        fields = ["clocks.sm", "clocks.max.sm", "power.draw",
                  "clocks_event_reasons.sw_power_cap", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown"]
        bits = [0x4, 0x8, 0x20, 0x40]
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(fields), "--format=csv,noheader,nounits",
                 "-i", ident, "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None
            return
        self.source = "nvidia-smi"

        def read():
            def num(x):
                try:
                    return float(x)
                except ValueError:
                    return None
            for line in self.proc.stdout:
                p = [x.strip() for x in line.split(",")]
                if len(p) != len(fields) or num(p[0]) is None:
                    continue
                r = sum(b for b, x in zip(bits, p[3:]) if x.lower().startswith("active"))
                self.samples.append((time.time(), num(p[0]), num(p[1]), num(p[2]), r))
        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def summary(self, t0, t1):
        w = [x for x in self.samples if t0 <= x[0] <= t1]
        window = "timed region"
        if not w:
            w, window = list(self.samples), "whole run (no sample inside the timed region)"
        if not w:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "source": self.source}
        sm = [x[1] for x in w]
        mx = [x[2] for x in w]
        pw = [x[3] for x in w if x[3] is not None]
        reasons = sorted(n for n, b in self.REASONS.items() if any(x[4] & b for x in w))
        return {"sm_mhz": statistics.median(sm), "sm_min_mhz": min(sm), "sm_max_mhz": max(mx),
                "reasons": reasons, "samples": len(w), "window": window,
                "power_w_max": max(pw) if pw else None, "source": self.source}

    def stop(self):
        self.stop_flag.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
def workload_spec(name):
    from top_gradient_compression_gb300 import workloads as W
    if name == "resnet50":
        c = W.RESNET50
        return dict(name="resnet50", P=c["P"], N=c["N"], seg_len=c["seg_len"], k_num=c["k_num"],
                    k_den=c["k_den"], quant=False,
                    desc=("ResNet-50-sized EF step: P=8 nodes x N=25,557,032 fp32, Top-k 0.1% per "
                          "100,000-entry layer block with error feedback, sparse sum-reduce with "
                          "dense switch at 25%"),
                    gen=lambda t, dev: W.resnet50_grads(t, device=dev),
                    gen_sample=lambda t, n: W.resnet50_grads(t, N=n),
                    data="synthetic: N(0, sigma_b^2), sigma_b log-uniform in [1e-4, 1e-1] per "
                         "100k-entry block (seeded torch generator on device)")
    if name != "asr":
        raise ValueError(f"workload {name!r} has no EF-step spec")
    c = W.ASR
    return dict(name="asr", P=c["P"], N=c["N"], seg_len=c["seg_len"], k_num=c["k_num"],
                k_den=c["k_den"], quant=True, bucket=c["bucket"],
                desc=("LSTM/ASR-like EF step: P=16 x N=67,108,864 fp32, Top-k 1%, 4-bit "
                      "stochastic quantisation in buckets of 512, fused dequantise + sparse reduce"),
                gen=lambda t, dev: W.asr_grads(t, device=dev),
                gen_sample=lambda t, n: W.asr_grads(t, N=n),
                data="synthetic: Laplace(0, 1e-3) (seeded torch generator on device)")


def file_sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


CSRC = os.path.join(ROOT, "top_gradient_compression_gb300", "csrc")


def load_traffic(kernel, workload, src):
    """DRAM bytes per launch of `kernel` on `workload` from a committed ncu
    summary (profiles/traffic.json, keyed "kernel@workload"), if it was taken
    on the current source of the kernel (else None)."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        e = t[f"{kernel}@{workload}"]
        if e.get("source_sha") != file_sha(src):
            return None
        return e
    except Exception:
        return None


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# CPU baseline: the oracle as it stands, on a bounded sample
# ---------------------------------------------------------------------------
def cpu_sample(spec, args, reference=False):
    """The bounded slice of the workload the oracle is timed on: (entries per
    node n, segment table of that slice, description). resnet50: the first
    --cpu-segments layer blocks of every node; asr: the first --cpu-entries
    entries of every node as one segment at the workload's density (half as
    many for the per-step reference arm)."""
    import oracle
    P, N, L = spec["P"], spec["N"], spec["seg_len"]
    if spec["name"] == "resnet50":
        nseg = min(args.cpu_segments if not reference else 8, (N + L - 1) // L)
        n = min(N, nseg * L)
        desc = f"the first {nseg} layer blocks ({n:,} entries) of each of the {P} nodes"
    else:
        n = min(N, args.cpu_entries if not reference else args.cpu_entries // 2)
        desc = f"the first {n:,} entries of each of the {P} nodes as one segment"
    b, k = oracle.uniform_segments(n, min(L, n), spec["k_num"], spec["k_den"])
    return n, (b, k), desc


def cpu_step(spec, g, res, table, step, threads):
    """One oracle EF step on the sample: Top-k + EF, quantise + dequantise
    where the workload has it, and the sparse reduce."""
    import oracle
    from top_gradient_compression_gb300 import workloads as W
    oi, ov, on = oracle.topk_ef_segments(g, res, table[0], table[1], threads=threads)
    if spec["quant"]:
        b = spec.get("bits", 4)
        c, sc = oracle.quantize(ov, spec["bucket"], b, W.quant_seed(step), idx=oi, nnz=on)
        ov = oracle.dequantize(c, sc, oi.shape[1], spec["bucket"], b, nnz=on)
    oracle.sparse_reduce(oi, ov, on, g.shape[1], threads=threads)


def cpu_baseline_run(spec, args, grads_dev):
    """Times the oracle on the bounded sample, on one host core and on every
    host core (the same results either way). Returns the cpu_baseline object."""
    n, table, desc = cpu_sample(spec, args)
    gh = [grads_dev[b][:, :n].cpu().numpy() for b in range(min(2, len(grads_dev)))]
    cores = os.cpu_count() or 1
    out = {}
    for label, threads in (("one_core", 1), ("all_cores", cores)):
        res = np.zeros_like(gh[0])
        t0 = time.perf_counter()
        for st in range(2):
            cpu_step(spec, gh[st % len(gh)], res, table, st, threads)
        dt = time.perf_counter() - t0
        out[label] = {"GBps": spec["P"] * n * 4 * 2 / dt / 1e9, "seconds": dt, "threads": threads}
    return {"value": out["all_cores"]["GBps"], "unit": "GB/s", "cores": cores, "kind": "oracle",
            "cpu_model": cpu_model(), "one_core_value": out["one_core"]["GBps"],
            "sample": (f"{desc}, 2 EF steps of Top-k + EF" +
                       (" + quantise/dequantise" if spec["quant"] else "") +
                       f" + reduce; gradient bytes / time. All {cores} cores: "
                       f"{out['all_cores']['seconds']:.1f} s; one core: "
                       f"{out['one_core']['seconds']:.1f} s")}


def run_reference(args, ranks):
    """--impl reference: the CPU oracle timed on every host core (rank 0 only)."""
    if ranks.rank != 0:
        return
    if args.workload in ("sweep", "logreg", "qsgd", "ssar", "asr_reduce"):
        return run_reference_op(args)
    spec = workload_spec(args.workload)
    spec["bits"] = args.bits
    n, table, desc = cpu_sample(spec, args, reference=True)
    g = spec["gen_sample"](0, n).numpy()
    res = np.zeros_like(g)
    cores = os.cpu_count() or 1
    for st in range(args.warmup):
        cpu_step(spec, g, res, table, st, cores)
    t0 = time.perf_counter()
    for st in range(args.steps):
        cpu_step(spec, g, res, table, st, cores)
    dt = time.perf_counter() - t0
    P = spec["P"]
    v = P * n * 4 * args.steps / dt / 1e9
    sample = f"oracle on {cores} host threads: {desc} per step"
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
            "elems_per_s": P * n * args.steps / dt, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": spec["data"], "config": {"workload": spec["desc"], "sample": sample},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "cpu_model": cpu_model(), "sample": sample},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_reference_op(args):
    """--impl reference for the single-operation workloads: the oracle's reduce
    (sweep, logreg), quantiser (qsgd) or SSAR on the same inputs."""
    import oracle
    from top_gradient_compression_gb300 import workloads as W
    cores = os.cpu_count() or 1
    if args.workload == "logreg":
        idx, val, nnz = W.logreg_streams()
        N = W.LOGREG["N"]
    elif args.workload == "asr_reduce":  # a bounded sample: 1/8 of N at the same density
        N = W.ASR["N"] // 8
        idx, val, nnz = W.uniform_streams(W.ASR["P"], N, N // 100, W.sub_seed(9, N), std=1e-3)
    else:
        P = args.sweep_p if args.workload in ("sweep", "ssar") else 64
        dpct = args.sweep_d if args.workload in ("sweep", "ssar") else 10
        cell = [(a, b) for a, b in W.SWEEP_D if abs(100.0 * a / b - dpct) < 1e-9][0]
        idx, val, nnz = W.sweep_streams(P, *cell)
        N = W.SWEEP_N
    threads = 1
    if args.workload == "ssar":
        op = lambda s: oracle.ssar(idx, val, nnz, N)  # noqa: E731
        units = int(nnz.astype(np.int64).sum())
        nbytes = 8 * units
        desc = f"SSAR recursive doubling of {idx.shape[0]} streams, N={N:,}"
    elif args.workload == "qsgd":
        x = oracle.sparse_reduce(idx, val, nnz, N)["dense"]
        op = lambda s: oracle.quantize(x, 1024, args.bits, W.quant_seed(s))  # noqa: E731
        units, nbytes = N, 4 * N
        desc = f"QSGD {args.bits}-bit on a dense reduced vector, N={N:,}, buckets of 1024"
    elif args.workload == "asr_reduce":
        threads = cores
        kk = idx.shape[1]

        def op(s):  # decode as the fused reduce does, then the reduce
            c, sc = oracle.quantize4(idx, val, nnz, 512, W.quant_seed(s))
            oracle.sparse_reduce(idx, oracle.dequantize4(c, sc, nnz, kk, 512), nnz, N,
                                 threads=cores)
        units = int(nnz.astype(np.int64).sum())
        nbytes = idx.shape[0] * (4 * kk + -(-kk // 2) + 4 * -(-kk // 512))
        desc = (f"4-bit quantise, decode and sparse reduce of {idx.shape[0]} streams of "
                f"{kk:,} entries, N={N:,} (1/8 of the LSTM/ASR-like reduce)")
    else:
        threads = cores
        op = lambda s: oracle.sparse_reduce(idx, val, nnz, N, threads=cores)  # noqa: E731
        units = int(nnz.astype(np.int64).sum())
        nbytes = 8 * units
        desc = f"sparse reduce of {idx.shape[0]} streams, N={N:,} ({args.workload})"
    for s in range(args.warmup):
        op(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        op(s)
    dt = time.perf_counter() - t0
    v = nbytes * args.steps / dt / 1e9
    sample = f"oracle ({threads} host thread(s)): the whole workload, {args.steps} calls"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s",
        "elems_per_s": units * args.steps / dt, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": desc, "sample": sample},
        "cpu_baseline": {"value": v, "unit": "GB/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
        flush=True)


# ---------------------------------------------------------------------------
# reduce-only workloads (streams given): density sweep cell, logreg
# ---------------------------------------------------------------------------
def run_reduce_only(args, ranks):
    """Times the sparse sum-reduce with the dense switch alone on seeded
    streams. value = stream input bytes (8 per entry) per second."""
    from top_gradient_compression_gb300 import api, workloads as W
    dev = ranks.device()
    torch.cuda.set_device(dev)
    if args.workload == "sweep":
        P, N, dpct = args.sweep_p, W.SWEEP_N, args.sweep_d
        cell = [(a, b) for a, b in W.SWEEP_D if abs(100.0 * a / b - dpct) < 1e-9]
        if not cell:
            raise SystemExit(f"--sweep-d must be one of {[100.0 * a / b for a, b in W.SWEEP_D]}")
        idx, val, nnz = W.sweep_streams(P, *cell[0])
        desc = (f"density-sweep cell: P={P} streams of {int(nnz[0]):,} uniform distinct indices "
                f"(d={dpct}%) over N={N:,}, N(0,1) values")
    else:
        idx, val, nnz = W.logreg_streams()
        P, N = idx.shape[0], W.LOGREG["N"]
        desc = (f"logistic-regression gradients: P={P} streams of 40,000 Zipf(1.1) features over "
                f"N={N:,}, N(0,1e-2) values")
    di = torch.from_numpy(idx.view(np.int32)).to(dev)
    dv = torch.from_numpy(val).to(dev)
    dn = torch.from_numpy(nnz.view(np.int32)).to(dev)
    ws = api.workspace(api.reduce_workspace_size(P, N), dev)
    out = api.reduce_out(N, dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MB > L2
    K, Wm = args.steps, args.warmup
    evs = [api.make_events(3) for _ in range(K)]
    def call(i, timed):
        if args.op == "sum":
            api.sparse_reduce(di, dv, dn, N, out=out, ws=ws, events=evs[i] if timed else None)
        else:  # timed as one interval: split + tile + finish
            if timed:
                evs[i][0].record()
            api.sparse_reduce_op(di, dv, dn, N, args.op, out=out, ws=ws)
            if timed:
                evs[i][1].record()
                evs[i][2].record()

    clocks = ClockSampler(dev)
    for i in range(Wm):
        call(i, False)
    torch.cuda.synchronize()
    launches0 = api.launch_count()
    t_host0 = time.time()
    gpu_head_start(K)
    for i in range(K):
        flush.fill_(float(i))  # inputs do not stay in L2 between timed runs
        call(i, True)
    torch.cuda.synchronize()
    t_host1 = time.time()
    launches = api.launch_count() - launches0
    clk = clocks.summary(t_host0, t_host1)
    clocks.stop()
    if api.get_status(ws) != 0:
        raise RuntimeError("device status set after the timed reduces")
    t_tile = float(np.mean([e[0].elapsed_time(e[1]) for e in evs]))
    t_fix = float(np.mean([e[1].elapsed_time(e[2]) for e in evs]))
    ms = ranks.max(t_tile + t_fix)
    sum_nnz = int(nnz.astype(np.int64).sum())
    U, dense = int(out.nnz.item()), bool(out.is_dense.item())
    in_bytes = 8 * sum_nnz
    out_bytes = 4 * N if dense else 8 * U
    peak, peak_kind = hbm_peak()
    achieved = (in_bytes + out_bytes) / (t_tile * 1e-3) / 1e9
    traffic = None
    if args.workload == "sweep":  # counters committed for the largest cell only
        e = load_traffic("reduce", f"sweep_P{P}_d{dpct:g}", os.path.join(CSRC, "reduce.cu"))
        traffic = None if e is None else e["dram_bytes_per_launch"]
    if ranks.rank != 0:
        return
    print(json.dumps({
        "metric": METRIC, "value": job_rate(ranks.world, in_bytes, ms * 1e-3) / 1e9, "unit": "GB/s",
        "elems_per_s": job_rate(ranks.world, sum_nnz, ms * 1e-3), "n_gpus": ranks.world, "steps": K,
        "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy index sets)",
        "config": {"workload": desc, "P": P, "N": N, "sum_nnz": sum_nnz, "op": args.op,
                   "units": "value = 8 B per input entry / (split+tile+fixup time)",
                   "l2": "256 MB buffer written between timed runs (L2 flushed)"},
        "roofline": {"bound": "hbm", "kernel": "reduce split + tile",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": in_bytes + out_bytes,
                     "traffic": traffic, "launch_ms": t_tile},
        "kernels_ms": {"reduce_split_tile": t_tile, "reduce_fixup": t_fix},
        "reduce": {"U": U, "is_dense": dense},
        "gpu_launches": launches, "clocks": clk}), flush=True)


# ---------------------------------------------------------------------------
# our path
# ---------------------------------------------------------------------------
def run_ours(args, ranks):
    from top_gradient_compression_gb300 import api, workloads as W
    dev = ranks.device()
    if dev.type != "cuda":
        raise RuntimeError("bench.py --impl ours needs a CUDA device")
    torch.cuda.set_device(dev)
    spec = workload_spec(args.workload)
    spec["bits"] = args.bits
    if args.nodes:
        spec["P"] = args.nodes
        spec["desc"] += f" [P overridden to {args.nodes}]"
        gen = spec["gen"]
        spec["gen"] = lambda t, d: gen(t, d)[: args.nodes].contiguous()
    P, N, L, kn, kd = spec["P"], spec["N"], spec["seg_len"], spec["k_num"], spec["k_den"]
    NB = 3 if spec["name"] == "resnet50" else 2  # distinct gradient batches, cycled
    grads = [spec["gen"](t, dev) for t in range(NB)]
    res = torch.zeros((P, N), device=dev)
    cap = api.segment_k_total(N, L, kn, kd)
    nbuf = 2 if args.overlap else 1  # Top-k outputs and codes double-buffered when overlapped
    tk_outs = [(torch.empty((P, cap), dtype=torch.int32, device=dev),
                torch.empty((P, cap), dtype=torch.float32, device=dev),
                torch.empty((P,), dtype=torch.int32, device=dev)) for _ in range(nbuf)]
    tk_out = tk_outs[0]
    tk_ws = api.workspace(api.topk_ef_workspace_size(P, N, L, kn, kd), dev)
    rd_ws = api.workspace(api.reduce_workspace_size(P, N), dev)
    rd_out = api.reduce_out(N, dev)
    quant = spec["quant"]
    if quant:
        bucket, qbits = spec["bucket"], args.bits
        codes_b = [torch.zeros((P, (cap + 8 // qbits - 1) // (8 // qbits)), dtype=torch.uint8,
                               device=dev) for _ in range(nbuf)]
        if qbits != 4:
            spec["desc"] = spec["desc"].replace("4-bit", f"{qbits}-bit")
        scales_b = [torch.zeros((P, (cap + bucket - 1) // bucket), device=dev)
                    for _ in range(nbuf)]
        qstat = api.status_word(dev)

    K, Wm = args.steps, args.warmup
    ev_tk = [api.make_events(4) for _ in range(K)]
    ev_rd = [api.make_events(3) for _ in range(K)]  # reduce: before, split+tile | finish, after
    ev_q = [api.make_events(2) for _ in range(K)] if quant else None  # around the quantiser

    def exchange(i, b, timed):
        """Quantise (where the workload has it) and reduce step i's streams,
        buffer b, on the current stream."""
        o = tk_outs[b]
        if quant:
            if timed:
                ev_q[i][0].record()
            api.quantize(o[1], bucket, qbits, W.quant_seed(i), idx=o[0], nnz=o[2],
                         codes=codes_b[b], scales=scales_b[b], status=qstat)
            if timed:
                ev_q[i][1].record()
                ev_rd[i][0].record()
            api.sparse_reduce_qb(o[0], codes_b[b], scales_b[b], o[2], bucket, qbits, N,
                                 out=rd_out, ws=rd_ws)
            if timed:
                ev_rd[i][1].record()
                ev_rd[i][2].record()
        else:
            api.sparse_reduce(o[0], o[1], o[2], N, out=rd_out, ws=rd_ws,
                              events=ev_rd[i] if timed else None)

    def step(i, grad, timed=False):  # one stream: Top-k, then quantise and reduce
        api.topk_ef(grad, res, L, kn, kd, out=tk_out, ws=tk_ws,
                    events=ev_tk[i] if timed else None)
        exchange(i, 0, timed)

    # Overlapped steps (SparCML's non-blocking collectives, §7): step i's
    # quantise and reduce run on a second stream while step i + 1's Top-k
    # runs on the main one. Step i's Top-k output and codes live in buffer
    # i % 2; the Top-k of step i + 2 waits until the reduce of step i is done
    # with that buffer, and the residual chain stays on the main stream.
    main_s = torch.cuda.current_stream()
    side_s = torch.cuda.Stream(device=dev)
    ev_ready = [torch.cuda.Event() for _ in range(2)]
    ev_free = [torch.cuda.Event() for _ in range(2)]
    for e in ev_free:
        e.record(main_s)

    def step_overlapped(i, grad, timed=False):
        b = i % 2
        main_s.wait_event(ev_free[b])
        api.topk_ef(grad, res, L, kn, kd, out=tk_outs[b], ws=tk_ws,
                    events=ev_tk[i] if timed else None)
        ev_ready[b].record(main_s)
        with torch.cuda.stream(side_s):
            side_s.wait_event(ev_ready[b])
            exchange(i, b, timed)
            ev_free[b].record(side_s)

    def drain():  # the main stream waits for every reduce issued so far
        for e in ev_free:
            main_s.wait_event(e)

    run_step = step_overlapped if args.overlap else step

    clocks = ClockSampler(dev)  # samples from before the warm-up to after the timed steps
    for i in range(Wm):
        run_step(i, grads[i % NB])
    drain()
    torch.cuda.synchronize()
    # Two passes over the same K steps. The timed region (value, ms_per_step)
    # runs them as a user would, with no event between the kernels of a step;
    # the second records CUDA events around every phase for the per-kernel
    # breakdown and the roofline (the events cost a little: they stop the
    # next kernel's launch from overlapping the previous one's drain).
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches0 = api.launch_count()
    ranks.barrier()
    torch.cuda.synchronize()
    t_host0 = time.time()
    ev0.record()
    for i in range(K):
        run_step(i, grads[i % NB])
    drain()  # the timed region ends after the last step's reduce
    ev1.record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    ranks.barrier()
    launches = api.launch_count() - launches0
    ms_local = ev0.elapsed_time(ev1) / K
    time.sleep(0.02)
    clk = clocks.summary(t_host0, t_host1)
    # the breakdown pass
    ev2, ev3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev2.record()
    for i in range(K):
        run_step(i, grads[i % NB], timed=True)
    drain()
    ev3.record()
    torch.cuda.synchronize()
    ms_instrumented = ranks.max(ev2.elapsed_time(ev3) / K)
    clocks.stop()
    for word in (tk_ws, rd_ws) + ((qstat,) if quant else ()):
        st = api.get_status(word)
        if st != 0:
            raise RuntimeError(f"device status {api.STATUS.get(st, st)} after the timed steps")
    ms = ranks.max(ms_local)

    def mean_ms(evs, a, b):
        return float(np.mean([e[a].elapsed_time(e[b]) for e in evs]))
    kern = {"topk_guess": mean_ms(ev_tk, 0, 1), "topk_stream": mean_ms(ev_tk, 1, 2),
            "topk_select": mean_ms(ev_tk, 2, 3)}
    if quant:
        kern[f"quantize{qbits}"] = mean_ms(ev_q, 0, 1)
        kern[f"reduce_q{qbits}"] = mean_ms(ev_rd, 0, 2)
    else:
        kern["reduce_split_tile"] = mean_ms(ev_rd, 0, 1)
        kern["reduce_finish"] = mean_ms(ev_rd, 1, 2)
    reduce_ms = mean_ms(ev_rd, 0, 2)

    U = int(rd_out.nnz.item())
    is_dense = bool(rd_out.is_dense.item())
    nnz_h = tk_outs[(K - 1) % nbuf][2].cpu().numpy().astype(np.int64)
    sum_nnz = int(nnz_h.sum())
    in_bytes_step = P * N * 4
    value = job_rate(ranks.world, in_bytes_step, ms * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    stream_bytes = 12 * P * N  # read grad + residual, write residual
    achieved = stream_bytes / (kern["topk_stream"] * 1e-3) / 1e9
    traffic = load_traffic("topk_stream_kernel", spec["name"], os.path.join(CSRC, "topk_ef.cu"))
    # the reduce's input (the metric's unit): 8 B per stream entry, or 4 B of
    # index + b/8 B of code per entry + 4 B per bucket scale when quantised
    if quant:
        reduce_in = (4 * sum_nnz + sum(-(-int(n) * qbits // 8) for n in nnz_h) +
                     4 * sum(-(-int(n) // bucket) for n in nnz_h))
    else:
        reduce_in = 8 * sum_nnz
    reduce_out_bytes = 4 * N if is_dense else 8 * U
    reduce_achieved = (reduce_in + reduce_out_bytes) / (reduce_ms * 1e-3) / 1e9
    rtraffic = load_traffic("reduce", spec["name"], os.path.join(CSRC, "reduce.cu"))

    # ---- end to end: pinned host gradients in, reduced result out, every step.
    # Step i+1's gradients are copied on a second stream into the other device
    # buffer while step i computes; each step's result is read back before the
    # next one is issued.
    e2e = None
    if args.e2e_steps > 0:
        hg = [torch.empty((P, N), dtype=torch.float32, pin_memory=True) for _ in range(2)]
        for b in range(2):
            hg[b].copy_(grads[b])
        dgrad = [torch.empty((P, N), device=dev) for _ in range(2)]
        copy_stream = torch.cuda.Stream(device=dev)
        compute = torch.cuda.current_stream()
        ev_copied = [torch.cuda.Event() for _ in range(2)]
        ev_used = [torch.cuda.Event() for _ in range(2)]
        for e in ev_used:
            e.record(compute)
        cap_out = rd_out.idx.numel()
        h_idx = torch.empty(cap_out, dtype=torch.int32, pin_memory=True)
        h_val = torch.empty(cap_out, dtype=torch.float32, pin_memory=True)
        h_dense = torch.empty(N, dtype=torch.float32, pin_memory=True)
        h_small = torch.empty(2, dtype=torch.int32, pin_memory=True)
        small = torch.empty(2, dtype=torch.int32, device=dev)
        E = args.e2e_steps

        def issue_copy(i):
            b = i % 2
            with torch.cuda.stream(copy_stream):
                copy_stream.wait_event(ev_used[b])
                dgrad[b].copy_(hg[i % 2], non_blocking=True)
                ev_copied[b].record(copy_stream)

        def read_result():
            small[0:1].copy_(rd_out.nnz)
            small[1:2].copy_(rd_out.is_dense)
            h_small.copy_(small, non_blocking=True)
            compute.synchronize()
            u, dn = int(h_small[0]), int(h_small[1])
            if dn:
                h_dense.copy_(rd_out.dense, non_blocking=True)
                nbytes = 8 + 4 * N
            else:
                h_idx[:u].copy_(rd_out.idx[:u], non_blocking=True)
                h_val[:u].copy_(rd_out.val[:u], non_blocking=True)
                nbytes = 8 + 8 * u
            compute.synchronize()
            return nbytes

        for i in range(2):  # warm-up of the copy path
            issue_copy(i)
            compute.wait_event(ev_copied[i % 2])
            step(i, dgrad[i % 2])
            ev_used[i % 2].record(compute)
            read_result()
        torch.cuda.synchronize()
        ranks.barrier()
        d2h = 0
        t0 = time.perf_counter()
        issue_copy(0)
        for i in range(E):
            if i + 1 < E:
                issue_copy(i + 1)
            compute.wait_event(ev_copied[i % 2])
            step(i, dgrad[i % 2])
            ev_used[i % 2].record(compute)
            d2h += read_result()
        torch.cuda.synchronize()
        dt = ranks.max(time.perf_counter() - t0)
        e2e = {"value": job_rate(ranks.world, in_bytes_step * E, dt) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes_step, "d2h_bytes_per_step": d2h // E,
               "ms_per_step": dt / E * 1e3, "steps": E,
               "note": "next step's host->device copy overlaps this step's kernels"}
        del hg, dgrad

    # ---- CPU baseline (rank 0, single GPU only)
    cpu = None
    if not args.no_cpu_baseline and ranks.world == 1:
        cpu = cpu_baseline_run(spec, args, grads)

    if ranks.rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s",
        "elems_per_s": job_rate(ranks.world, P * N, ms * 1e-3),
        "n_gpus": ranks.world, "steps": K, "warmup": Wm, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": spec["data"],
        "config": {"workload": spec["desc"], "P": P, "N": N, "seg_len": L,
                   "k_per_node": cap,
                   "units": ("value = P*N*4 gradient bytes entering the sparse-reduce step per "
                             "second of whole-step time; elems_per_s = gradient entries per "
                             "second; the reduce's own input rate (the stream bytes it reads) is "
                             "reduce.input_GBps"),
                   "l2": (f"inputs larger than L2 ({NB} x {P * N * 4 / 1e6:,.0f} MB gradient "
                          f"batches + the residual), no flush"),
                   "parallelism": f"replicas x{ranks.world} (no cross-GPU exchange)",
                   "pipeline": ("step t's quantise + reduce on a second stream, overlapping "
                                "step t+1's Top-k (every step does all of its work inside the "
                                "timed region; per-phase times then overlap)" if args.overlap
                                else "one stream: Top-k, quantise, reduce per step")},
        "roofline": {"bound": "hbm", "kernel": "topk_stream_kernel",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": stream_bytes,
                     "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                     "launch_ms": kern["topk_stream"]},
        "kernels_ms": kern,
        "kernels_ms_note": ("per-phase CUDA events from a second pass of the same steps; that "
                            "pass took ms_per_step_instrumented per step"),
        "ms_per_step_instrumented": ms_instrumented,
        "reduce": {"input_bytes": reduce_in, "output_bytes": reduce_out_bytes,
                   "sum_nnz": sum_nnz, "U": U, "is_dense": is_dense, "ms": reduce_ms,
                   "input_GBps": reduce_in / (reduce_ms * 1e-3) / 1e9,
                   "elems_per_s": sum_nnz / (reduce_ms * 1e-3),
                   "roofline": {"bound": "hbm",
                                "kernel": ("fused dequantise + sparse reduce" if quant
                                           else "sparse reduce") + " (all its launches)",
                                "achieved": reduce_achieved, "peak": peak, "unit": "GB/s",
                                "frac": reduce_achieved / peak, "peak_kind": peak_kind,
                                "algorithmic_bytes_per_launch": reduce_in + reduce_out_bytes,
                                "traffic": None if rtraffic is None
                                else rtraffic["dram_bytes_per_launch"],
                                "launch_ms": reduce_ms}},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches,
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# QSGD on the dense reduced result (DSAR's quantised second half, §6)
# ---------------------------------------------------------------------------
def run_qsgd(args, ranks):
    """b-bit stochastic quantisation of a dense reduced vector: the dense result
    of the largest density-sweep cell (P=64, d=10%), buckets of 1,024. One step
    = one quantise call. value = 4 B per input entry / time."""
    from top_gradient_compression_gb300 import api, workloads as W
    dev = ranks.device()
    torch.cuda.set_device(dev)
    N, bits_, bucket = W.SWEEP_N, args.bits, 1024
    idx, val, nnz = W.sweep_streams(64, 10, 100)
    di = torch.from_numpy(idx.view(np.int32)).to(dev)
    dv = torch.from_numpy(val).to(dev)
    dn = torch.from_numpy(nnz.view(np.int32)).to(dev)
    out = api.sparse_reduce(di, dv, dn, N)
    if not bool(out.is_dense.item()):
        raise RuntimeError("the sweep cell's reduced result is expected dense")
    x = out.dense.view(1, N)
    del di, dv, dn
    per = 8 // bits_
    codes = torch.zeros((1, (N + per - 1) // per), dtype=torch.uint8, device=dev)
    scales = torch.zeros((1, (N + bucket - 1) // bucket), device=dev)
    status = api.status_word(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)  # 256 MB > L2
    K, Wm = args.steps, args.warmup
    for i in range(Wm):
        api.quantize(x, bucket, bits_, W.quant_seed(i), codes=codes, scales=scales, status=status)
    torch.cuda.synchronize()
    launches0 = api.launch_count()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    clocks = ClockSampler(dev)
    t_host0 = time.time()
    gpu_head_start(K)
    for i in range(K):
        flush.fill_(float(i))  # the 16.8 MB input does not stay in L2 between calls
        evs[i][0].record()
        api.quantize(x, bucket, bits_, W.quant_seed(i), codes=codes, scales=scales, status=status)
        evs[i][1].record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    clk = clocks.summary(t_host0, t_host1)
    clocks.stop()
    launches = api.launch_count() - launches0
    if api.get_status(status) != 0:
        raise RuntimeError("device status set after the timed quantise calls")
    ms = ranks.max(float(np.mean([a.elapsed_time(b) for a, b in evs])))
    in_bytes = 4 * N
    out_bytes = codes.numel() + 4 * scales.numel()
    peak, peak_kind = hbm_peak()
    achieved = (in_bytes + out_bytes) / (ms * 1e-3) / 1e9
    if ranks.rank != 0:
        return
    print(json.dumps({
        "metric": METRIC, "value": job_rate(ranks.world, in_bytes, ms * 1e-3) / 1e9,
        "unit": "GB/s", "elems_per_s": job_rate(ranks.world, N, ms * 1e-3),
        "n_gpus": ranks.world, "steps": K, "warmup": Wm, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (dense result of the P=64, d=10% density-sweep reduce)",
        "config": {"workload": f"QSGD {bits_}-bit on a dense reduced vector, N={N:,}, buckets of "
                               f"{bucket}", "N": N, "bits": bits_, "bucket": bucket,
                   "units": "value = 4 B per input entry / quantise time",
                   "l2": "256 MB buffer written between timed calls (L2 flushed)"},
        "roofline": {"bound": "hbm", "kernel": f"quantize_kernel<{bits_}>", "achieved": achieved,
                     "peak": peak, "unit": "GB/s", "frac": achieved / peak, "peak_kind": peak_kind,
                     "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": in_bytes + out_bytes, "traffic": None,
                     "launch_ms": ms},
        "cpu_baseline": None, "e2e": None, "gpu_launches": launches, "clocks": clk}), flush=True)


# ---------------------------------------------------------------------------
# SSAR recursive doubling, emulated (§5.3.1): fill-in and GB/s per stage
# ---------------------------------------------------------------------------
def run_asr_reduce(args, ranks):
    """The fused 4-bit dequantise + sparse reduce of the LSTM/ASR-like step
    alone, on C4-shaped streams built on the device (P=16, N=2^26, 671,088
    sorted distinct uniform indices per node, Laplace(0, 1e-3) values
    quantised in buckets of 512). value = the reduce's input bytes (4 B index
    + 0.5 B code per entry + 4 B per bucket scale) per second."""
    from top_gradient_compression_gb300 import api, workloads as W
    dev = ranks.device()
    torch.cuda.set_device(dev)
    P, N, bucket = W.ASR["P"], W.ASR["N"], 512
    di, dv, dn = W.asr_reduce_streams(dev)
    k = di.shape[1]
    codes, scales = api.quantize4(di, dv, dn, bucket, W.quant_seed(0))
    ws = api.workspace(api.reduce_workspace_size(P, N), dev)
    out = api.reduce_out(N, dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    K, Wm = args.steps, args.warmup
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    clocks = ClockSampler(dev)
    for _ in range(Wm):
        api.sparse_reduce_q4(di, codes, scales, dn, bucket, N, out=out, ws=ws)
    torch.cuda.synchronize()
    launches0 = api.launch_count()
    t_host0 = time.time()
    gpu_head_start(K, 300.0)
    for i in range(K):
        flush.fill_(float(i))  # the streams do not stay in L2 between timed runs
        evs[i][0].record()
        api.sparse_reduce_q4(di, codes, scales, dn, bucket, N, out=out, ws=ws)
        evs[i][1].record()
    torch.cuda.synchronize()
    t_host1 = time.time()
    launches = api.launch_count() - launches0
    clk = clocks.summary(t_host0, t_host1)
    clocks.stop()
    if api.get_status(ws) != 0:
        raise RuntimeError("device status set after the timed reduces")
    ms = ranks.max(float(np.mean([a.elapsed_time(b) for a, b in evs])))
    U, dense = int(out.nnz.item()), bool(out.is_dense.item())
    nb = -(-k // bucket)
    in_bytes = P * (4 * k + -(-k // 2) + 4 * nb)
    out_bytes = 4 * N if dense else 8 * U
    peak, peak_kind = hbm_peak()
    achieved = (in_bytes + out_bytes) / (ms * 1e-3) / 1e9
    if ranks.rank != 0:
        return
    print(json.dumps({
        "metric": METRIC, "value": job_rate(ranks.world, in_bytes, ms * 1e-3) / 1e9, "unit": "GB/s",
        "elems_per_s": job_rate(ranks.world, P * k, ms * 1e-3), "n_gpus": ranks.world,
        "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 codes, f32 sums",
        "data": "synthetic (seeded torch generator on device)",
        "config": {"workload": "fused 4-bit dequantise + sparse reduce of the LSTM/ASR-like step: "
                               f"P={P} x {k:,} entries over N={N:,}, buckets of {bucket}",
                   "units": "value = 4.5 B per input entry + 4 B per bucket scale / reduce time",
                   "l2": "256 MB buffer written between timed runs (L2 flushed)"},
        "roofline": {"bound": "hbm", "kernel": "fused dequantise + sparse reduce (all its launches)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "peak_kind": peak_kind, "frac_of_nominal": achieved / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": in_bytes + out_bytes, "traffic": None,
                     "launch_ms": ms},
        "reduce": {"U": U, "is_dense": dense},
        "gpu_launches": launches, "clocks": clk}), flush=True)


def run_ssar(args, ranks):
    """The static sparse allreduce by recursive doubling over the streams of a
    density-sweep cell (--sweep-p, --sweep-d). value = stream input bytes (8
    per entry) / time of all stages; per stage: fill-in and GB/s of that
    stage's own input + output bytes."""
    from top_gradient_compression_gb300 import api, workloads as W
    dev = ranks.device()
    torch.cuda.set_device(dev)
    P, N, dpct = args.sweep_p, W.SWEEP_N, args.sweep_d
    cell = [(a, b) for a, b in W.SWEEP_D if abs(100.0 * a / b - dpct) < 1e-9]
    if not cell or P & (P - 1):
        raise SystemExit("--workload ssar needs a power-of-two --sweep-p and a sweep density")
    idx, val, nnz = W.sweep_streams(P, *cell[0])
    di = torch.from_numpy(idx.view(np.int32)).to(dev)
    dv = torch.from_numpy(val).to(dev)
    dn = torch.from_numpy(nnz.view(np.int32)).to(dev)
    cap = idx.shape[1]
    ws = api.workspace(api.ssar_workspace_size(P, cap, N), dev)
    stages = P.bit_length() - 1
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    K, Wm = args.steps, args.warmup
    evs = [api.make_events(stages + 1) for _ in range(K)]
    for i in range(Wm):
        api.ssar_allreduce(di, dv, dn, N, ws=ws)
    torch.cuda.synchronize()
    launches0 = api.launch_count()
    clocks = ClockSampler(dev)
    t_host0 = time.time()
    gpu_head_start(K)
    for i in range(K):
        flush.fill_(float(i))
        _, _, out_nnz, fill = api.ssar_allreduce(di, dv, dn, N, ws=ws, events=evs[i])
    torch.cuda.synchronize()
    t_host1 = time.time()
    clk = clocks.summary(t_host0, t_host1)
    clocks.stop()
    launches = api.launch_count() - launches0
    if api.get_status(ws) != 0:
        raise RuntimeError("device status set after the timed calls")
    st_ms = [float(np.mean([e[s].elapsed_time(e[s + 1]) for e in evs])) for s in range(stages)]
    ms = ranks.max(sum(st_ms))
    fill = [int(x) for x in fill.cpu().numpy()]
    sum_nnz = int(nnz.astype(np.int64).sum())
    ins = [sum_nnz] + fill[:-1]
    per_stage = [{"stage": s, "partial_results": P >> (s + 1), "entries_in": ins[s],
                  "entries_out": fill[s], "fill_in_density": fill[s] / ((P >> (s + 1)) * N),
                  "ms": st_ms[s], "GBps": 8 * (ins[s] + fill[s]) / (st_ms[s] * 1e-3) / 1e9}
                 for s in range(stages)]
    in_bytes = 8 * sum_nnz
    moved = sum(8 * (ins[s] + fill[s]) for s in range(stages))
    peak, peak_kind = hbm_peak()
    if ranks.rank != 0:
        return
    print(json.dumps({
        "metric": METRIC, "value": job_rate(ranks.world, in_bytes, ms * 1e-3) / 1e9, "unit": "GB/s",
        "elems_per_s": job_rate(ranks.world, sum_nnz, ms * 1e-3), "n_gpus": ranks.world,
        "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic (seeded numpy index sets)",
        "config": {"workload": f"SSAR recursive doubling, P={P} streams of {int(nnz[0]):,} "
                               f"uniform indices (d={dpct:g}%) over N={N:,}",
                   "P": P, "N": N, "units": "value = 8 B per input entry / time of all stages",
                   "l2": "256 MB buffer written between timed runs (L2 flushed)"},
        "stages": per_stage, "result_nnz": int(out_nnz.item()),
        "roofline": {"bound": "hbm", "kernel": "ssar stages (partition + merge)",
                     "achieved": moved / (ms * 1e-3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": moved / (ms * 1e-3) / 1e9 / peak, "peak_kind": peak_kind,
                     "frac_of_nominal": moved / (ms * 1e-3) / 1e9 / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": moved, "traffic": None, "launch_ms": ms},
        "cpu_baseline": None, "e2e": None, "gpu_launches": launches, "clocks": clk}), flush=True)


def main():
    args = parse_args()
    ranks = Ranks()
    try:
        if args.impl == "reference":
            run_reference(args, ranks)
        elif args.workload in ("sweep", "logreg"):
            run_reduce_only(args, ranks)
        elif args.workload == "qsgd":
            run_qsgd(args, ranks)
        elif args.workload == "ssar":
            run_ssar(args, ranks)
        elif args.workload == "asr_reduce":
            run_asr_reduce(args, ranks)
        else:
            run_ours(args, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
