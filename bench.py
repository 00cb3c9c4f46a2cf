#!/usr/bin/env python3
"""Benchmark of the fused GEMM + AllReduce hot path on one GB300 (or N independent replicas).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl mk|reference]
                  [--workload NAME] [--split chained|adaptive|static|accumulate|unfused] [--comm-sms n]
  python bench.py --sweep        # SM-split sweep: adaptive vs every static split, per M

A step is one mk_gemm_allreduce (or mk_gemm_reducescatter) call over one batch of seeded
synthetic inputs already resident in HBM.  Prints ONE JSON line (rank 0).  The default split is
the chained one (compute blocks fold each rank's partial tile into the rank-ordered running
sum, the same bits as the reduce role); the line also carries, on the same inputs, the
controller-driven role split, the unfused two-kernel baseline and the accumulate variant.

Default workload: the row-parallel MLP down-projection GEMM + AllReduce, P=8 logical ranks,
M=N=8192, K_per_rank=3584 (the large AllReduce shape the tensor-peak target refers to).  Its
operands (940 MB) exceed the 129 MB L2, so no flush is needed between steps.

--impl reference times the fp64 CPU oracle (the only reference this method has) on a bounded
row sample of the same workload, on this machine's host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import inputgen as ig  # noqa: E402

DEFAULT_WORKLOAD = "ar_mlp_down_p8_m8192_n8192_k3584"
METRIC = "fused GEMM+AllReduce TFLOP/s on 1 GB300 and % of bf16 tensor/HBM roofline"
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
KERNEL_SOURCES = [os.path.join(ROOT, "gemm_tile_level_gb300", "csrc", f)
                  for f in ("mk_kernels.cu", "mk_ptx.cuh", "mk_device.cuh", "mk_internal.h", "mk_abi.cu")]


def workload_by_name(name: str) -> ig.Workload:
    if name in ig.WORKLOADS:
        return ig.WORKLOADS[name]
    for M in ig.SWEEP_M:
        if ig.sweep_workload(M).name == name:
            return ig.sweep_workload(M)
    raise SystemExit(f"unknown workload {name}; choose from {list(ig.WORKLOADS)}")


def algorithmic_bytes(wl: ig.Workload, partial_bytes: int = 4) -> int:
    """A and B once, every rank's partial tile (fp32, or bf16 with --bf16-partials) written and
    read once, the output once."""
    a = wl.P * wl.M * wl.Kr * 2
    b = wl.P * wl.Kr * wl.N * 2
    partial = wl.P * wl.M * wl.N * partial_bytes
    out = wl.M * wl.N * (2 if wl.out_dtype == "bf16" else 4)
    return a + b + 2 * partial + out


def load_peaks():
    if os.path.exists(PEAKS_FILE):
        with open(PEAKS_FILE) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the kernel sources' code: comments and layout whitespace are left out, so that only
    a change to what compiles makes a committed DRAM capture stale."""
    import hashlib
    import re
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, encoding="utf-8") as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current
    kernel sources (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    kv = {}
    for line in open(TRAFFIC_FILE):
        line = line.strip()
        if "=" in line and not line.startswith("#"):
            k, v = line.split("=", 1)
            kv[k.strip()] = v.strip()
    if kv.get("kernel_src_sha") != kernel_source_hash() or kv.get("workload") != workload:
        return None
    try:
        return int(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ------------------------------------------------------------------ clocks during the timed region
_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x2: "applications_clocks_setting",
            0x10: "sync_boost", 0x100: "display_clock_setting"}


class ClockSampler:
    """Reads SM clock, max clock and clock-event reasons through NVML (read-only queries) every
    few milliseconds in a background thread; falls back to `nvidia-smi -lms`."""

    def __init__(self, index: int, period_s: float = 0.005):
        self.index, self.period = index, period_s
        self.samples, self.reasons, self.max_mhz = [], 0, None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() == 0:
                h = ctypes.c_void_p()
                if nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(h)) == 0:
                    self._nvml, self._h = nv, h
                    m = ctypes.c_uint()
                    if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                        self.max_mhz = m.value
        except OSError:
            self._nvml = None

    def _loop(self):
        nv, h = self._nvml, self._h
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        get_r = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop.is_set():
            if nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(c)) == 0:
                self.samples.append(c.value)
            if get_r(h, ctypes.byref(r)) == 0:
                self.reasons |= r.value
            time.sleep(self.period)

    def start(self):
        if self._nvml is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()
        else:
            try:
                self._proc = subprocess.Popen(
                    ["nvidia-smi", "-i", str(self.index), "--query-gpu=clocks.sm,clocks.max.sm,"
                     "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "50"],
                    stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            except OSError:
                self._proc = None

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            for line in out.splitlines():
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append(int(float(parts[0])))
                    self.max_mhz = int(float(parts[1]))
                    self.reasons |= int(parts[2], 16)
                except (ValueError, IndexError):
                    pass

    def summary(self):
        names = sorted(n for bit, n in _REASONS.items() if self.reasons & bit)
        med = statistics.median(self.samples) if self.samples else None
        return {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": names, "samples": len(self.samples)}


# ------------------------------------------------------------------ CPU oracle leg
def time_oracle(wl: ig.Workload, A, B, target_s: float = 12.0):
    """The fp64 oracle as it stands on a bounded row sample: returns (TFLOP/s, rows, seconds)."""
    import oracle
    t0 = time.perf_counter()
    oracle.allreduce_rows(A, B, 0, 8)
    t_cal = max(time.perf_counter() - t0, 1e-3)
    rows = int(max(8, min(wl.M, 8 * target_s / t_cal)))
    t0 = time.perf_counter()
    oracle.allreduce_rows(A, B, 0, rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * rows * wl.N * wl.Kr * wl.P
    return flops / dt / 1e12, rows, dt


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ distributed plumbing (replicas)
class Ranks:
    def __init__(self, gpus: int):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.dist = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if torch.cuda.is_available():
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.dist = dist
        if gpus != self.world:
            print(f"warning: --gpus {gpus} but WORLD_SIZE={self.world}", file=sys.stderr)

    def barrier(self):
        if self.dist is not None:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if self.dist is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.dist is not None:
            self.dist.destroy_process_group()


def workload_config(args, wl, world: int = 1) -> dict:
    """The `config` object of the JSON line: the same keys for the GPU arm and the reference arm."""
    bf16_partials = bool(_EXTRA_FLAGS & BF16_PARTIALS_FLAG) and args.split in ("adaptive", "static", "unfused")
    return {"workload": wl.name, "op": wl.op, "P": wl.P, "M": wl.M, "N": wl.N,
            "K_per_rank": wl.Kr, "out_dtype": wl.out_dtype, "split": args.split,
            "accumulate": "fp32", "seed": wl.seed, "tiles": args.tiles,
            "partial_tiles": "bf16" if bf16_partials else "fp32",
            "b_layout": "N x K_r" if _EXTRA_FLAGS & B_NK_FLAG else "K_r x N",
            "l2": "operands %.0f MB > 129 MB L2, no flush" % ((wl.P * (wl.M + wl.N) * wl.Kr * 2) / 1e6),
            "parallelism": f"{wl.P} logical ranks on one GPU" + (f"; {world} replicas" if world > 1 else "")}


def reference_arm(args, wl, ranks):
    """--impl reference: the fp64 oracle on host cores, rank 0 only."""
    if ranks.rank != 0:
        return
    A, B = ig.make_operands(wl)
    vals = []
    rows = secs = None
    # each step is a bounded row sample, sized so the whole run stays within a few minutes
    per_step = min(args.reference_step_s, 150.0 / (args.warmup + args.steps))
    for i in range(args.warmup + args.steps):
        v, rows, secs = time_oracle(wl, A, B, target_s=per_step)
        if i >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    sample = f"rows 0..{rows - 1} of {wl.M} (all N={wl.N}, all P={wl.P} ranks, K_r={wl.Kr}), fp64"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": secs * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args, wl, ranks.world), "implementation": "fp64 CPU oracle",
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU arm
_EXTRA_FLAGS = 0   # MK_FLAG_SINGLE_SM_TILES (--tiles single), MK_FLAG_NO_COOPERATIVE (--no-cooperative)
_REDUCE_SPLIT = 0  # --reduce-split (0 = chosen by the library)
_RASTER_GROUP = 0  # --raster-group (0 = chosen by the library)


BF16_PARTIALS_FLAG = 128   # MK_FLAG_BF16_PARTIALS (--bf16-partials)
B_NK_FLAG = 256            # MK_FLAG_B_NK (--b-nk)


def split_opts(api, mk, split: str, comm_sms: int):
    kw = dict(flags=_EXTRA_FLAGS, reduce_split=_REDUCE_SPLIT, raster_group=_RASTER_GROUP)
    if split in ("accumulate", "chained"):
        kw["flags"] &= ~BF16_PARTIALS_FLAG    # these splits store no partial tiles
    if split == "adaptive":
        return api.make_opts(mk.MK_SPLIT_ADAPTIVE, comm_sms=comm_sms, **kw)
    if split == "static":
        return api.make_opts(mk.MK_SPLIT_STATIC, comm_sms=comm_sms, **kw)
    if split == "accumulate":
        return api.make_opts(mk.MK_SPLIT_ACCUMULATE, **kw)
    if split == "chained":
        return api.make_opts(mk.MK_SPLIT_CHAINED, **kw)
    return api.make_opts(mk.MK_SPLIT_UNFUSED, **kw)


class Problem:
    """Device-resident operands, outputs and workspace of one workload."""

    def __init__(self, wl, torch, api, mk, host=None):
        self.wl = wl
        A, B = host if host is not None else ig.make_operands(wl)
        self.A_host, self.B_host = A, B
        # the device copies of B: K_r x N, or N x K_r (a linear layer's weight) with --b-nk
        self.B_dev_host = [np.ascontiguousarray(b.T) for b in B] if _EXTRA_FLAGS & B_NK_FLAG else B
        self.Ad = [api.bf16_device(a) for a in A]
        self.Bd = [api.bf16_device(b) for b in self.B_dev_host]
        out_t = torch.bfloat16 if wl.out_dtype == "bf16" else torch.float32
        self.out_code = mk.MK_BF16 if wl.out_dtype == "bf16" else mk.MK_F32
        self.rs = wl.op == "reducescatter"
        if self.rs:
            self.C = [torch.empty((wl.M // wl.P, wl.N), dtype=out_t, device="cuda") for _ in range(wl.P)]
            self.op = mk.MK_OP_REDUCESCATTER
        else:
            self.C = torch.empty((wl.M, wl.N), dtype=out_t, device="cuda")
            self.op = mk.MK_OP_ALLREDUCE
        self.ws = api.workspace(self.op, wl.P, wl.M, wl.N, wl.Kr)
        self.mk = mk
        torch.cuda.synchronize()   # uploads and the zeroed workspace land before calls on other streams

    def call(self, opts, stream):
        mk, wl = self.mk, self.wl
        if self.rs:
            return mk.mk_gemm_reducescatter(wl.P, wl.M, wl.N, wl.Kr, self.Ad, self.Bd, self.C,
                                            self.out_code, self.ws, opts=opts, stream=stream)
        return mk.mk_gemm_allreduce(wl.P, wl.M, wl.N, wl.Kr, self.Ad, self.Bd, [self.C] * wl.P,
                                    self.out_code, self.ws, opts=opts, stream=stream)


def clear_workspace(torch, ws):
    """Zero a workspace between calls issued on another stream: the calls before it have finished
    and the zeros have landed before any call after it starts."""
    torch.cuda.synchronize()
    ws.zero_()
    torch.cuda.synchronize()


def time_launches(torch, prob, opts, steps, warmup, stream):
    """Returns (total ms over `steps`, per-launch ms list)."""
    for _ in range(warmup):
        prob.mk.check(prob.call(opts, stream))
    prob.mk.check(prob.mk.mk_status_check(prob.ws, stream))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    ev[0].record(stream)
    for i in range(steps):
        st = prob.call(opts, stream)
        ev[i + 1].record(stream)
        if st != 0:
            prob.mk.check(st)
    torch.cuda.synchronize()
    prob.mk.check(prob.mk.mk_status_check(prob.ws, stream))
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[steps]), per


def gpu_arm(args, wl, ranks):
    import torch
    from gemm_tile_level_gb300 import api, mk

    dev = ranks.local if ranks.world > 1 else 0
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        prob = Problem(wl, torch, api, mk)
        opts = split_opts(api, mk, args.split, args.comm_sms)
        if args.split == "accumulate":
            clear_workspace(torch, prob.ws)
        for _ in range(args.warmup):
            mk.check(prob.call(opts, stream))
        mk.check(mk.mk_status_check(prob.ws, stream))

        # ---------------- timed region: K steps, inputs resident in HBM
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
        clocks = ClockSampler(dev)
        ranks.barrier()
        torch.cuda.synchronize()
        clocks.start()
        ev[0].record(stream)
        for i in range(args.steps):
            st = prob.call(opts, stream)
            ev[i + 1].record(stream)
            if st != 0:
                mk.check(st)
        torch.cuda.synchronize()
        clocks.stop()
        ranks.barrier()
        mk.check(mk.mk_status_check(prob.ws, stream))
        total_ms = ev[0].elapsed_time(ev[args.steps])
        per_launch = [ev[i].elapsed_time(ev[i + 1]) for i in range(args.steps)]
        ms_per_step = ranks.max(total_ms / args.steps)
        value = ranks.world * wl.flops / (ms_per_step * 1e-3) / 1e12

        # ---------------- end to end through the C ABI with host buffers
        e2e = None
        if not args.no_e2e:
            e2e = e2e_leg(torch, prob, opts, stream, max(2, min(args.steps, 10)), ranks)

        # ---------------- unfused two-kernel baseline on the same inputs (context, not `value`)
        unfused = None
        if args.split != "unfused" and not args.no_baseline:
            tot, _ = time_launches(torch, prob, split_opts(api, mk, "unfused", 0),
                                   max(3, min(args.steps, 20)), 2, stream)
            n = max(3, min(args.steps, 20))
            unfused = {"value": wl.flops / (tot / n * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "ms_per_step": tot / n, "launches_per_step": 2}

        # ---------------- the accumulate variant (no reduce role) on the same inputs (context)
        accumulate = None
        if args.split != "accumulate" and not args.no_baseline:
            clear_workspace(torch, prob.ws)   # the other modes leave partial tiles where its accumulators go
            n = max(3, min(args.steps, 20))
            tot, _ = time_launches(torch, prob, split_opts(api, mk, "accumulate", 0), n, 2, stream)
            accumulate = {"value": wl.flops / (tot / n * 1e-3) / 1e12, "unit": "TFLOP/s",
                          "ms_per_step": tot / n, "launches_per_step": 1,
                          "note": "MK_SPLIT_ACCUMULATE: L2 reductions into fp32 accumulators, order of additions not fixed"}

        # ---------------- the role split with the on-GPU controller (same bits) (context)
        adaptive = None
        if args.split != "adaptive" and not args.no_baseline:
            n = max(3, min(args.steps, 20))
            tot, _ = time_launches(torch, prob, split_opts(api, mk, "adaptive", 0), n, 2, stream)
            adaptive = {"value": wl.flops / (tot / n * 1e-3) / 1e12, "unit": "TFLOP/s",
                        "ms_per_step": tot / n, "launches_per_step": 1,
                        "note": "MK_SPLIT_ADAPTIVE: compute and reduce roles, SM split set by the on-GPU controller"}

        # ---------------- the chained variant (compute blocks fold in rank order; same bits) (context)
        chained = None
        if args.split != "chained" and not args.no_baseline:
            n = max(3, min(args.steps, 20))
            tot, _ = time_launches(torch, prob, split_opts(api, mk, "chained", 0), n, 2, stream)
            chained = {"value": wl.flops / (tot / n * 1e-3) / 1e12, "unit": "TFLOP/s",
                       "ms_per_step": tot / n, "launches_per_step": 1,
                       "note": "MK_SPLIT_CHAINED: each rank's epilogue adds its tile to the running sum of the ranks "
                               "before it, in rank order (the reduce role's additions, same bits)"}

        # ---------------- cuBLAS through torch on the same operands (context: not the method)
        library = None
        if not args.no_baseline and ranks.world == 1:
            library = library_leg(torch, prob, max(3, min(args.steps, 20)), stream, ms_per_step)

        # ---------------- the controller's trace of one adaptive call (Figure 7a of the method)
        if args.trace:
            trace_leg(torch, api, mk, prob, stream, args.trace, "adaptive")

    peaks, peak_src = load_peaks()

    # ---------------- every other configuration, on the same GPU in the same run
    A_host, B_host = prob.A_host, prob.B_host
    configs = None
    if not args.no_configs and not args.shape and args.workload == DEFAULT_WORKLOAD and ranks.world == 1:
        del prob
        torch.cuda.empty_cache()
        with torch.cuda.stream(stream):
            configs = configs_leg(torch, api, mk, stream, peaks, args.config_steps, 3)
    kernel_ms = statistics.mean(per_launch)
    achieved = wl.flops / (kernel_ms * 1e-3) / 1e12
    bf16_partials = bool(_EXTRA_FLAGS & BF16_PARTIALS_FLAG) and args.split in ("adaptive", "static", "unfused")
    bytes_alg = algorithmic_bytes(wl, 2 if bf16_partials else 4)
    t_tensor = wl.flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = bytes_alg / (peaks["hbm_gbs"] * 1e9)
    bound = "tensor" if t_tensor >= t_hbm else "hbm"
    if bound == "tensor":
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                "frac": achieved / peaks["bf16_tflops"]}
    else:
        gbs = bytes_alg / (kernel_ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / peaks["hbm_gbs"]}
    roof["traffic"] = committed_traffic(wl.name)
    roof["peak_source"] = f"{peak_src} (MEASURED_PEAKS.json, burst)" if peak_src == "measured" else "fallback"
    roof["roofline_frac"] = max(t_tensor, t_hbm) / (kernel_ms * 1e-3)
    roof["algorithmic_bytes"] = bytes_alg
    roof["kernel"] = ("mk_persistent_kernel" if _EXTRA_FLAGS & 2 else "mk_pair_kernel") + (
        "<256>" if wl.N > 128 else "<128>")

    if ranks.rank != 0:
        return
    cpu = None
    if not args.no_cpu_baseline and ranks.world == 1:
        v, rows, secs = time_oracle(wl, A_host, B_host, target_s=args.cpu_seconds)
        cpu = {"value": v, "unit": "TFLOP/s", "cores": host_cores(), "kind": "oracle",
               "sample": f"rows 0..{rows - 1} of {wl.M}, all N={wl.N}, all P={wl.P} ranks, "
                         f"K_r={wl.Kr}; {secs:.1f} s fp64"}
    clk = clocks.summary()
    if roof["bound"] == "tensor":
        # the same launch against the sustained peak (cuBLAS back to back under the power cap), the
        # reference for a long run like the 200 timed steps here; and the SM cycles per launch at
        # the median clock sampled during them
        roof["frac_of_sustained_peak"] = achieved / peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])
        if clk.get("sm_mhz"):
            roof["sm_cycles_per_launch"] = kernel_ms * 1e-3 * clk["sm_mhz"] * 1e6
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ranks.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": workload_config(args, wl, ranks.world),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": args.steps * (2 if args.split == "unfused" else 1),
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "unfused_baseline": unfused, "adaptive_split": adaptive, "accumulate_variant": accumulate,
            "chained_variant": chained, "library_context": library,
            "launch_ms": {"mean": kernel_ms, "median": statistics.median(per_launch), "min": min(per_launch),
                          "max": max(per_launch), "launches": len(per_launch)},
            "configs": configs}
    print(json.dumps(line), flush=True)


def library_leg(torch, prob, steps, stream, mk_ms):
    """cuBLAS (torch.matmul / torch.bmm) on the same operands, as context only: one GEMM over the
    concatenated K (A_cat = [A_0 | ... | A_{P-1}], B_cat = [B_0; ...; B_{P-1}]), the cost of the
    product with no reduction between ranks at all; and the P rank GEMMs as one batched GEMM with
    bf16 outputs, then their sum (an unfused form from library kernels, with bf16 partial tiles, so
    other numerics)."""
    wl = prob.wl
    b_kn = [b.t() for b in prob.Bd] if _EXTRA_FLAGS & B_NK_FLAG else prob.Bd
    with torch.cuda.stream(stream):
        A_cat = torch.cat(prob.Ad, dim=1)
        B_cat = torch.cat(b_kn, dim=0)
        A_st = torch.stack(prob.Ad)
        B_st = torch.stack(b_kn)
    torch.cuda.synchronize()

    def per_call(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            torch.cuda.synchronize()
            e0.record(stream)
            for _ in range(steps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    gemm_ms = per_call(lambda: torch.matmul(A_cat, B_cat))
    bmm_ms = per_call(lambda: torch.bmm(A_st, B_st).sum(dim=0))
    del A_cat, B_cat, A_st, B_st
    torch.cuda.empty_cache()
    tf = lambda ms: wl.flops / (ms * 1e-3) / 1e12
    return {"cublas_gemm_concatenated_k": {"ms": gemm_ms, "tflops": tf(gemm_ms),
                                           "note": "one bf16 GEMM M x (P*K_r) x N, fp32 accumulation, bf16 out: "
                                                   "no reduction between ranks (context, not the method)"},
            "cublas_bmm_then_sum": {"ms": bmm_ms, "tflops": tf(bmm_ms),
                                    "note": "torch.bmm over the P ranks (bf16 partial tiles), then sum over ranks"},
            "value_over_cublas_gemm": gemm_ms / mk_ms, "steps": steps}


def roofline_of(flops: float, nbytes: float, ms: float, peaks: dict) -> dict:
    """Bound and achieved fraction of max(FLOPs / tensor peak, bytes / HBM bandwidth) for one call."""
    t_tensor = flops / (peaks["bf16_tflops"] * 1e12)
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    return {"bound": "tensor" if t_tensor >= t_hbm else "hbm", "frac": max(t_tensor, t_hbm) / (ms * 1e-3),
            "roofline_ms": max(t_tensor, t_hbm) * 1e3}


CONFIG_WORKLOADS = ("ar_p2_m128_n128_k256", "ar_p8_m2048_n4096_k512", "rs_p8_m16384_n8192_k1024",
                    "ar_sweep_p8_m256_n8192_k1024", "ar_sweep_p8_m4096_n8192_k1024")
CONFIG_SPLITS = ("chained", "adaptive", "unfused", "accumulate")
AG_SHAPE = (8, 8192, 3584, 4096)
L2_BYTES = 129 << 20          # GB300 L2
FLUSH_BELOW = 2 * L2_BYTES    # configurations whose operands take less are timed call by call with L2 flushed


def time_config(torch, prob, opts, steps, warmup, stream, flush):
    """Device time per call of one configuration (ms).  With `flush` (a device buffer larger than
    L2): each call alone between two events, the buffer rewritten before it so that the call finds
    none of its operands in L2.  Without: the calls back to back between one pair of events, queued
    behind a short device sleep so that the host's issue rate does not set the time."""
    for _ in range(warmup):
        prob.mk.check(prob.call(opts, stream))
    prob.mk.check(prob.mk.mk_status_check(prob.ws, stream))
    torch.cuda.synchronize()
    if flush is not None:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for e0, e1 in ev:
                flush.add_(1)
                e0.record(stream)
                prob.mk.check(prob.call(opts, stream))
                e1.record(stream)
        torch.cuda.synchronize()
        prob.mk.check(prob.mk.mk_status_check(prob.ws, stream))
        return sum(e0.elapsed_time(e1) for e0, e1 in ev) / steps
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sleep = getattr(torch.cuda, "_sleep", None)
    with torch.cuda.stream(stream):
        if sleep is not None:
            sleep(int(2e6))   # about 1 ms: the host queues the calls meanwhile
        e0.record(stream)
        for _ in range(steps):
            prob.mk.check(prob.call(opts, stream))
        e1.record(stream)
    torch.cuda.synchronize()
    prob.mk.check(prob.mk.mk_status_check(prob.ws, stream))
    return e0.elapsed_time(e1) / steps


def configs_leg(torch, api, mk, stream, peaks, steps: int, warmup: int):
    """Every other configuration of the study, timed on the same GPU in the same run: ms per call,
    TFLOP/s and the roofline fraction of each split (the chained default, the controller-driven
    role split, the unfused two-kernel baseline and the accumulate variant), then AllGather + GEMM
    fused against unfused.  About 20 calls per point."""
    out = {}
    flush = torch.zeros(FLUSH_BELOW // 4, dtype=torch.float32, device="cuda")
    for name in CONFIG_WORKLOADS:
        wl = workload_by_name(name)
        prob = Problem(wl, torch, api, mk)
        nbytes = algorithmic_bytes(wl, 4)
        operand_bytes = wl.P * (wl.M + wl.N) * wl.Kr * 2
        small = operand_bytes < FLUSH_BELOW
        rec = {"op": wl.op, "P": wl.P, "M": wl.M, "N": wl.N, "K_per_rank": wl.Kr, "out_dtype": wl.out_dtype,
               "flops": wl.flops, "algorithmic_bytes": nbytes, "steps": steps,
               "l2": ("operands %.1f MB: L2 flushed (%d MB written) before every timed call, each call timed "
                      "alone" % (operand_bytes / 1e6, FLUSH_BELOW >> 20)) if small else
                     ("operands %.0f MB > 2 x 129 MB L2, no flush; calls back to back" % (operand_bytes / 1e6))}
        for split in CONFIG_SPLITS:
            if split == "accumulate":
                clear_workspace(torch, prob.ws)   # the other modes leave partial tiles where its accumulators go
            ms = time_config(torch, prob, split_opts(api, mk, split, 0), steps, warmup, stream,
                             flush if small else None)
            rf = roofline_of(wl.flops, nbytes, ms, peaks)
            rec["bound"] = rf["bound"]
            rec["roofline_ms"] = rf["roofline_ms"]
            rec[split] = {"ms": ms, "us": ms * 1e3, "tflops": wl.flops / (ms * 1e-3) / 1e12,
                          "roofline_frac": rf["frac"],
                          "tensor_frac": wl.flops / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"]}
        rec["roofline_note"] = ("roofline_ms = max(FLOPs / bf16 peak, algorithmic bytes / HBM peak), the "
                                "algorithmic bytes counting every partial tile written and read once; the "
                                "chained and accumulate splits move no partial tiles and may run below it "
                                "(roofline_frac > 1); tensor_frac = FLOPs / bf16 peak / time")
        rec["chained_over_unfused"] = rec["chained"]["ms"] / rec["unfused"]["ms"]
        rec["adaptive_over_unfused"] = rec["adaptive"]["ms"] / rec["unfused"]["ms"]
        out[name] = rec
        del prob
        torch.cuda.empty_cache()
    del flush
    P, M, N, K = AG_SHAPE
    ag = AgProblem(torch, api, mk, P, M, N, K)
    rec = {"op": "allgather_gemm", "P": P, "M": M, "N": N, "K": K, "out_dtype": "bf16", "flops": ag.flops,
           "algorithmic_bytes": ag.nbytes, "steps": steps}
    for split, mode in (("fused", mk.MK_SPLIT_ADAPTIVE), ("unfused", mk.MK_SPLIT_UNFUSED)):
        ms = ag.time(mode, steps, warmup, stream)
        rf = roofline_of(ag.flops, ag.nbytes, ms, peaks)
        rec["bound"] = rf["bound"]
        rec["roofline_ms"] = rf["roofline_ms"]
        rec[split] = {"ms": ms, "us": ms * 1e3, "tflops": ag.flops / (ms * 1e-3) / 1e12, "roofline_frac": rf["frac"]}
    rec["fused_over_unfused"] = rec["fused"]["ms"] / rec["unfused"]["ms"]
    out[f"ag_p{P}_m{M}_n{N}_k{K}"] = rec
    del ag
    torch.cuda.empty_cache()
    out[RING_WORKLOAD] = ring_record(torch, api, mk, stream, peaks, max(3, steps // 4), 2)
    return out


def trace_leg(torch, api, mk, prob, stream, path: str, split: str, comm_sms: int = 0):
    """One call with the controller's trace buffer attached; writes its records (time, published
    reduce-role SMs, compute units and reduce items finished) to `path` as JSON."""
    cap = 1 << 16
    buf = torch.zeros(cap * 32, dtype=torch.uint8, device="cuda")
    opts = split_opts(api, mk, split, comm_sms)
    opts.trace = buf.data_ptr()
    opts.trace_bytes = buf.numel()
    mk.check(prob.call(opts, stream))
    mk.check(mk.mk_status_check(prob.ws, stream))
    hdr = prob.ws[:64].cpu().numpy().view(np.uint32)
    n = int(hdr[9])   # trace_count of the workspace header
    recs = buf[: n * 32].cpu().numpy().view(np.uint64).reshape(-1, 4)
    rows = []
    for r in recs:
        t_ns = int(r[0])
        w1, w2 = int(r[1]), int(r[2])
        rows.append({"t_ns": t_ns, "target_sms": w1 & 0xFFFFFFFF, "units_done": w1 >> 32,
                     "tiles_done": w2 & 0xFFFFFFFF, "num_blocks": w2 >> 32})
    wl = prob.wl
    doc = {"workload": wl.name, "split": split, "comm_sms": comm_sms, "P": wl.P, "M": wl.M, "N": wl.N,
           "K_per_rank": wl.Kr, "records": rows}
    with open(path, "w") as f:
        json.dump(doc, f)
    return len(rows)


def e2e_leg(torch, prob, opts, stream, steps, ranks):
    """Same metric through the C ABI with host buffers: every step copies this step's inputs
    from pinned host memory to the device, runs the call, and copies the result back.

    Two schedules are timed.  `serial`: copy in, call, copy out, one after the other on one
    stream.  `pipelined` (the reported value): two sets of device buffers, host-to-device copies
    on one stream, calls on another and device-to-host copies on a third, so that step i+1's
    inputs and step i-1's result move while step i computes; events order each buffer's reuse."""
    wl = prob.wl
    mk = prob.mk
    A_pin = [torch.from_numpy(a).view(torch.bfloat16).pin_memory() for a in prob.A_host]
    B_pin = [torch.from_numpy(b).view(torch.bfloat16).pin_memory() for b in prob.B_dev_host]
    outs = prob.C if isinstance(prob.C, list) else [prob.C]
    C_pin = [torch.empty(c.shape, dtype=c.dtype, pin_memory=True) for c in outs]
    h2d = sum(t.numel() * 2 for t in A_pin + B_pin)
    d2h = sum(t.numel() * t.element_size() for t in C_pin)

    def call(Ad, Bd, Cs):
        if prob.rs:
            return mk.mk_gemm_reducescatter(wl.P, wl.M, wl.N, wl.Kr, Ad, Bd, Cs, prob.out_code, prob.ws,
                                            opts=opts, stream=stream)
        return mk.mk_gemm_allreduce(wl.P, wl.M, wl.N, wl.Kr, Ad, Bd, [Cs[0]] * wl.P, prob.out_code, prob.ws,
                                    opts=opts, stream=stream)

    # ---- serial
    def step():
        for d, h in zip(prob.Ad + prob.Bd, A_pin + B_pin):
            d.copy_(h, non_blocking=True)
        mk.check(call(prob.Ad, prob.Bd, outs))
        for h, d in zip(C_pin, outs):
            h.copy_(d, non_blocking=True)

    step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    ranks.barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    ranks.barrier()
    mk.check(mk.mk_status_check(prob.ws, stream))
    serial_ms = ranks.max(e0.elapsed_time(e1) / steps)

    # ---- pipelined
    sets = [(prob.Ad, prob.Bd, outs),
            ([torch.empty_like(a) for a in prob.Ad], [torch.empty_like(b) for b in prob.Bd],
             [torch.empty_like(c) for c in outs])]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def issue(i):
        b = i % 2
        Ad, Bd, Cs = sets[b]
        with torch.cuda.stream(s_in):
            if i >= 2:
                s_in.wait_event(ev_comp[b])          # step i-2 has finished reading set b
            for d, h in zip(Ad + Bd, A_pin + B_pin):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(s_in)
        stream.wait_event(ev_in[b])
        if i >= 2:
            stream.wait_event(ev_out[b])             # step i-2's result has left set b
        mk.check(call(Ad, Bd, Cs))
        ev_comp[b].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[b])
            for h, d in zip(C_pin, Cs):
                h.copy_(d, non_blocking=True)
            ev_out[b].record(s_out)

    for i in range(2):
        issue(i)
    torch.cuda.synchronize()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    ranks.barrier()
    torch.cuda.synchronize()
    p0.record(s_in)
    for i in range(steps):
        issue(i)
    p1.record(s_out)
    torch.cuda.synchronize()
    ranks.barrier()
    mk.check(mk.mk_status_check(prob.ws, stream))
    ms = ranks.max(p0.elapsed_time(p1) / steps)
    return {"value": ranks.world * wl.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms, "steps": steps,
            "schedule": "pipelined: step i+1's host-to-device copies and step i-1's device-to-host copies "
                        "overlap step i's call (three streams, two buffer sets)",
            "serial": {"value": ranks.world * wl.flops / (serial_ms * 1e-3) / 1e12, "ms_per_step": serial_ms}}


# ------------------------------------------------------------------ AllGather + GEMM
class AgProblem:
    """Device-resident operands, gathered buffers, outputs and workspace of AllGather + GEMM: P
    row shards of A ((M/P) x K, N(0,1)) and P column shards of B (K x N, N(0,1/K)), seed 0."""

    def __init__(self, torch, api, mk, P, M, N, K):
        self.torch, self.api, self.mk = torch, api, mk
        self.P, self.M, self.N, self.K = P, M, N, K
        A = [np.empty((M // P, K), np.uint16) for _ in range(P)]
        B = [np.empty((K, N), np.uint16) for _ in range(P)]
        for r in range(P):
            ig.fill_bf16(A[r].reshape(-1), ig.normal(1.0), 0, r, ig.TID_A)
            ig.fill_bf16(B[r].reshape(-1), ig.normal(1.0 / K), 0, r, ig.TID_B)
        self.flops = 2.0 * P * M * N * K
        # shards read once, P gathered copies written and read, B once, P outputs written
        self.nbytes = M * K * 2 + 2 * P * M * K * 2 + P * K * N * 2 + P * M * N * 2
        self.Ad = [api.bf16_device(a) for a in A]
        self.Bd = [api.bf16_device(b) for b in B]
        self.C = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        self.G = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        self.ws = api.workspace(mk.MK_OP_ALLGATHER_GEMM, P, M, N, K)
        torch.cuda.synchronize()   # uploads and the zeroed workspace land before calls on other streams

    def call(self, mode, stream):
        o = self.api.make_opts(mode, flags=_EXTRA_FLAGS & ~(BF16_PARTIALS_FLAG | B_NK_FLAG))
        return self.mk.mk_allgather_gemm(self.P, self.M, self.N, self.K, self.Ad, self.Bd, self.G, self.C,
                                         self.mk.MK_BF16, self.ws, opts=o, stream=stream)

    def time(self, mode, steps, warmup, stream) -> float:
        torch, mk = self.torch, self.mk
        for _ in range(warmup):
            mk.check(self.call(mode, stream))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            mk.check(self.call(mode, stream))
        e1.record(stream)
        torch.cuda.synchronize()
        mk.check(mk.mk_status_check(self.ws, stream))
        return e0.elapsed_time(e1) / steps


class RingProblem:
    """Device-resident Q, K, V of every rank, outputs, logsumexp, ring buffers and workspace of one
    Ring Attention workload (inputgen.ATTN_WORKLOADS)."""

    def __init__(self, torch, api, mk, wl):
        self.torch, self.api, self.mk, self.wl = torch, api, mk, wl
        Q, K, V = ig.make_attn_operands(wl)
        P, H, S, d = wl.P, wl.H, wl.S, wl.d
        self.Qd = [api.bf16_device(x) for x in Q]
        self.Kd = [api.bf16_device(x) for x in K]
        self.Vd = [api.bf16_device(x) for x in V]
        self.O = [torch.empty((H, S, d), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
        self.L = [torch.empty((H, S), dtype=torch.float32, device="cuda") for _ in range(P)]
        self.R = [torch.empty((P - 1, 2, H, S, d), dtype=torch.bfloat16, device="cuda") for _ in range(P)] if P > 1 else None
        self.ws = api.ring_attention_workspace(P, H, S, d)
        torch.cuda.synchronize()   # uploads and the zeroed workspace land before calls on other streams
        # Q, K, V read, the KV forwarded P-1 times (read and written), O and lse written
        self.nbytes = 3 * P * H * S * d * 2 + 2 * (P - 1) * P * H * S * d * 2 * 2 + P * H * S * (d * 2 + 4)

    def call(self, form, stream, comm_sms=0):
        mk, wl = self.mk, self.wl
        mode = {"fused": mk.MK_SPLIT_ADAPTIVE, "static": mk.MK_SPLIT_STATIC, "unfused": mk.MK_SPLIT_UNFUSED,
                "inplace": mk.MK_SPLIT_ADAPTIVE}[form]
        o = self.api.make_opts(mode, comm_sms=comm_sms, flags=_EXTRA_FLAGS & 8)   # MK_FLAG_NO_COOPERATIVE
        return mk.mk_ring_attention(wl.P, wl.H, wl.S, wl.d, self.Qd, self.Kd, self.Vd, self.O, self.L,
                                    None if form == "inplace" else self.R, mk.MK_BF16, 0.0, self.ws, opts=o,
                                    stream=stream)

    def time(self, form, steps, warmup, stream, comm_sms=0) -> float:
        torch, mk = self.torch, self.mk
        for _ in range(warmup):
            mk.check(self.call(form, stream, comm_sms))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(steps):
            mk.check(self.call(form, stream, comm_sms))
        e1.record(stream)
        torch.cuda.synchronize()
        mk.check(mk.mk_status_check(self.ws, stream))
        return e0.elapsed_time(e1) / steps


RING_WORKLOAD = "ring_p8_h32_s4096_d128"


def ring_record(torch, api, mk, stream, peaks, steps, warmup, name=RING_WORKLOAD):
    """Ring Attention: the fused kernel (communication blocks forward the KV tiles, compute blocks
    attend), the same attention reading every slice in place (nothing forwarded), and the unfused
    form (a forwarding kernel, then the attention kernel)."""
    wl = ig.ATTN_WORKLOADS[name]
    rp = RingProblem(torch, api, mk, wl)
    rec = {"op": "ring_attention", "P": wl.P, "H": wl.H, "S_per_rank": wl.S, "d": wl.d, "out_dtype": "bf16",
           "flops": wl.flops, "algorithmic_bytes": rp.nbytes, "steps": steps}
    for form in ("fused", "inplace", "unfused"):
        ms = rp.time(form, steps, warmup, stream)
        rf = roofline_of(wl.flops, rp.nbytes, ms, peaks)
        rec["bound"] = rf["bound"]
        rec["roofline_ms"] = rf["roofline_ms"]
        rec[form] = {"ms": ms, "tflops": wl.flops / (ms * 1e-3) / 1e12, "roofline_frac": rf["frac"]}
    rec["fused_over_unfused"] = rec["fused"]["ms"] / rec["unfused"]["ms"]
    rec["fused_over_inplace"] = rec["fused"]["ms"] / rec["inplace"]["ms"]
    del rp
    torch.cuda.empty_cache()
    return rec


def ring_arm(args):
    """`--op ring`: Ring Attention on P logical ranks of one GPU, fused against its unfused form."""
    import torch
    from gemm_tile_level_gb300 import api, mk

    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    peaks, peak_src = load_peaks()
    wl = ig.ATTN_WORKLOADS[args.ring_workload]
    with torch.cuda.stream(stream):
        rp = RingProblem(torch, api, mk, wl)
        clocks = ClockSampler(0)
        for _ in range(args.warmup):
            mk.check(rp.call("fused", stream))
        clocks.start()
        fused_ms = rp.time("fused", args.steps, 0, stream)
        clocks.stop()
        del rp
        torch.cuda.empty_cache()
        rec = ring_record(torch, api, mk, stream, peaks, max(3, min(args.steps, 20)), 2, args.ring_workload)
    value = wl.flops / (fused_ms * 1e-3) / 1e12
    clk = clocks.summary()
    line = {"metric": "fused Ring Attention TFLOP/s on 1 GB300", "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": fused_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": wl.name, "op": "ring_attention", "P": wl.P, "H": wl.H, "S_per_rank": wl.S,
                       "d": wl.d, "out_dtype": "bf16", "causal": False},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": value / peaks["bf16_tflops"], "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json, burst)"},
            "gpu_launches": args.steps,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "forms": rec}
    print(json.dumps(line), flush=True)


def allgather_arm(args):
    """`--op allgather`: the fused AllGather + GEMM (communication pairs gather 128-row chunks of
    the row-sharded A into every rank's buffer, compute pairs multiply as chunks arrive) against
    its unfused form (a gather kernel, then the GEMM kernel), P logical ranks on one GPU.  The
    default shape is a column-parallel MLP up-projection: 8192 tokens, hidden 4096, 3584 output
    columns per rank."""
    import torch
    from gemm_tile_level_gb300 import api, mk

    P, M, N, K = (int(x) for x in args.ag_shape.split(","))
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ag = AgProblem(torch, api, mk, P, M, N, K)
        clocks = ClockSampler(0)
        clocks.start()
        fused_ms = ag.time(mk.MK_SPLIT_ADAPTIVE, args.steps, args.warmup, stream)
        clocks.stop()
        unfused_ms = ag.time(mk.MK_SPLIT_UNFUSED, max(3, min(args.steps, 50)), args.warmup, stream)
    peaks, peak_src = load_peaks()
    flops = ag.flops
    value = flops / (fused_ms * 1e-3) / 1e12
    clk = clocks.summary()
    line = {"metric": "fused AllGather+GEMM TFLOP/s on 1 GB300", "value": value, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": fused_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"ag_p{P}_m{M}_n{N}_k{K}", "op": "allgather_gemm", "P": P, "M": M, "N": N, "K": K,
                       "gathered_copies": True, "out_dtype": "bf16"},
            "roofline": {"bound": "tensor", "achieved": value, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                         "frac": value / peaks["bf16_tflops"], "traffic": None,
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json, burst)"},
            "gpu_launches": args.steps,
            "clocks": {"sm_mhz": clk["sm_mhz"], "sm_max_mhz": clk["sm_max_mhz"], "reasons": clk["reasons"],
                       "samples": clk["samples"]},
            "unfused_baseline": {"value": flops / (unfused_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                                 "ms_per_step": unfused_ms, "launches_per_step": 2}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ SM-split sweep
def sweep(args):
    import torch
    from gemm_tile_level_gb300 import api, mk

    torch.cuda.set_device(0)
    S = torch.cuda.get_device_properties(0).multi_processor_count
    stream = torch.cuda.Stream()
    results = []
    with torch.cuda.stream(stream):
        if args.sweep_workload:
            wls = [workload_by_name(n) for n in args.sweep_workload]
        else:
            wls = [ig.sweep_workload(M) for M in (args.sweep_m or ig.SWEEP_M)]
        for wl in wls:
            M = wl.M
            prob = Problem(wl, torch, api, mk)
            steps, warm = args.sweep_steps, 2

            # enough steps per point for about 20 ms of GPU time, so that short shapes are not noise
            t1, _ = time_launches(torch, prob, split_opts(api, mk, "static", 2), 3, warm, stream)
            steps = max(args.sweep_steps, int(20.0 / max(t1 / 3, 1e-3)))

            def ms(opts):
                tot, _ = time_launches(torch, prob, opts, steps, warm, stream)
                return tot / steps

            adaptive = ms(split_opts(api, mk, "adaptive", 0))
            # SM-pair tiles assign roles per pair: sweep even SM counts 2..S-2
            lo, step = (1, args.sweep_stride) if _EXTRA_FLAGS & 2 else (2, max(2, args.sweep_stride))
            static = {nr: ms(split_opts(api, mk, "static", nr)) for nr in range(lo, S - 1, step)}
            unf = ms(split_opts(api, mk, "unfused", 0))
            clear_workspace(torch, prob.ws)
            acc = ms(split_opts(api, mk, "accumulate", 0))
            chn = ms(split_opts(api, mk, "chained", 0))
            best_nr = min(static, key=static.get)
            if args.sweep_trace_dir:
                os.makedirs(args.sweep_trace_dir, exist_ok=True)
                trace_leg(torch, api, mk, prob, stream, os.path.join(args.sweep_trace_dir, f"{wl.name}_adaptive.json"),
                          "adaptive")
            rec = {"workload": wl.name, "M": M, "adaptive_ms": adaptive, "best_static_ms": static[best_nr],
                   "best_static_comm_sms": best_nr, "adaptive_over_best_static": adaptive / static[best_nr],
                   "unfused_ms": unf, "fused_over_unfused": adaptive / unf,
                   "accumulate_ms": acc, "accumulate_over_unfused": acc / unf,
                   "chained_ms": chn, "chained_over_unfused": chn / unf,
                   "adaptive_tflops": wl.flops / (adaptive * 1e-3) / 1e12,
                   "static_ms": {str(k): v for k, v in static.items()}}
            results.append(rec)
            print(json.dumps({k: v for k, v in rec.items() if k != "static_ms"}), flush=True)
            del prob
            torch.cuda.empty_cache()
    if args.sweep_out:
        with open(args.sweep_out, "w") as f:
            json.dump(results, f)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["mk", "reference"], default="mk")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--split", choices=["adaptive", "static", "unfused", "accumulate", "chained"], default="chained",
                    help="chained (default): compute blocks fold each rank's tile into the rank-ordered running "
                         "sum; adaptive / static: compute and reduce roles with the controller's or a fixed SM "
                         "split (the same bits); accumulate: unordered L2 reductions; unfused: two kernels")
    ap.add_argument("--comm-sms", type=int, default=0)
    ap.add_argument("--tiles", choices=["pair", "single"], default="pair",
                    help="SM-pair 256 x BN compute tiles (default) or one-SM 128 x BN tiles")
    ap.add_argument("--no-cooperative", action="store_true",
                    help="launch without the cooperative attribute (for profilers that cannot replay it)")
    ap.add_argument("--raster-group", type=int, default=0,
                    help="tile rows per band of the compute order (0 = the library's choice)")
    ap.add_argument("--tile-major", action="store_true",
                    help="compute the P ranks of each tile back to back instead of band by band")
    ap.add_argument("--reduce-split", type=int, default=0,
                    help="column slices per output tile's reduction (0 = the library's choice)")
    ap.add_argument("--b-nk", action="store_true",
                    help="give each B_r as N x K_r (K contiguous, the layout of a linear layer's weight)")
    ap.add_argument("--bf16-partials", action="store_true",
                    help="adaptive / static / unfused splits: store partial tiles as bf16 (MK_FLAG_BF16_PARTIALS)")
    ap.add_argument("--shape", default="", help="P,M,N,K_per_rank override (same distributions); "
                    "for small profiling cases")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-baseline", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--reference-step-s", type=float, default=8.0)
    ap.add_argument("--op", choices=["rowparallel", "allgather", "ring"], default="rowparallel",
                    help="allgather: time the fused AllGather + GEMM against its unfused form instead; "
                         "ring: Ring Attention (sequence parallelism)")
    ap.add_argument("--ring-workload", default=RING_WORKLOAD, help="Ring Attention workload of --op ring")
    ap.add_argument("--ag-shape", default="8,8192,3584,4096", help="P,M,N,K of --op allgather")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--sweep-m", type=int, nargs="*")
    ap.add_argument("--sweep-steps", type=int, default=10)
    ap.add_argument("--sweep-stride", type=int, default=1)
    ap.add_argument("--sweep-out", default="")
    ap.add_argument("--sweep-workload", nargs="*", default=[],
                    help="sweep these workloads instead of the M sweep (e.g. the MLP or ReduceScatter shape)")
    ap.add_argument("--sweep-trace-dir", default="",
                    help="also write one adaptive call's controller trace per swept workload into this folder")
    ap.add_argument("--trace", default="",
                    help="write the controller trace of one adaptive call of the workload to this JSON file")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip timing the other configurations (they run by default with the default workload)")
    ap.add_argument("--config-steps", type=int, default=20)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)   # at least three untimed warm-up steps
    global _EXTRA_FLAGS, _REDUCE_SPLIT, _RASTER_GROUP
    _EXTRA_FLAGS = (2 if args.tiles == "single" else 0) | (8 if args.no_cooperative else 0) | \
        (16 if args.tile_major else 0) | (BF16_PARTIALS_FLAG if args.bf16_partials else 0) | \
        (B_NK_FLAG if args.b_nk else 0)
    _REDUCE_SPLIT = args.reduce_split
    _RASTER_GROUP = args.raster_group
    if args.sweep:
        sweep(args)
        return
    if args.op == "allgather":
        allgather_arm(args)
        return
    if args.op == "ring":
        ring_arm(args)
        return
    wl = workload_by_name(args.workload)
    if args.shape:
        P, M, N, Kr = (int(x) for x in args.shape.split(","))
        wl = wl.with_shape(name=f"{wl.name}@P{P}_M{M}_N{N}_K{Kr}", P=P, M=M, N=N, Kr=Kr)
    ranks = Ranks(args.gpus)
    try:
        if args.impl == "reference":
            reference_arm(args, wl, ranks)
        else:
            gpu_arm(args, wl, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
