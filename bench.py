"""Benchmark: schedule op-times resolved per second on the heterogeneous 1F1B
batch (P=8 stages, M=64 microbatches, 65,536 instances; t_f ~ U[80,120],
t_b ~ U[160,240], comm ~ U[2,8]), with the HBM roofline of the evaluator
kernel, the CPU oracle as a baseline, and an end-to-end number through the
public host API.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

One step = one pp_sched_eval over the whole batch (op order from the cached
plan, max-plus times, reductions to makespan / idle / bubble, peak held
activations), inputs already resident in HBM.  The K timed steps are captured
once in a CUDA graph and replayed once between two CUDA events; the same K
steps launched one by one are timed as well and reported beside it.  N > 1 runs one process per GPU
(torchrun); each rank evaluates its own batch (weak scaling, no collective on
the data path); the slowest rank's time is reported.
"""
from __future__ import annotations

import argparse
import math
import ctypes
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

P, M, N_INST = 8, 64, 65536
METRIC = "schedule op-times resolved/sec (1F1B, P=8, M=64 batch); HBM GB/s vs peak"
UNIT = "op-times/s"
L2_BYTES = 129 * 10**6


def algorithmic_bytes(n, P_=P, M_=M):
    """Bytes one evaluation must move: every cost read once, every comm value
    read once, and the summary outputs written once."""
    costs = 2 * P_ * M_ * n * 4
    comm = (P_ - 1) * n * 4
    outs = n * 4 + n * P_ * 4 + 2 * n * 8 + n * 1 + P_ * 4  # makespan, idle, bub pair, status, peak
    return costs + comm + outs


KERNEL_SOURCES = ("pipeline_schedule_simulation_gb300/csrc/eval_reg.cu",
                  "pipeline_schedule_simulation_gb300/csrc/eval_common.cuh",
                  "pipeline_schedule_simulation_gb300/csrc/checks.cuh",
                  "pipeline_schedule_simulation_gb300/csrc/internal.cuh")
PROFILE = os.path.join(ROOT, "profiles", "eval_reg_1f1b_P8_M64_n65536.md")


def kernel_source_sha():
    import hashlib
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profiled_traffic():
    """DRAM bytes (read + write) per launch of the evaluator from the committed
    ncu summary, or None when the kernel sources changed since that capture."""
    try:
        fields = {}
        with open(PROFILE) as f:
            for line in f:
                line = line.strip().lstrip("-* ")
                if line.startswith(("traffic_bytes_per_launch:", "kernel_source_sha256:")):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip().strip("` ")
        if fields.get("kernel_source_sha256") != kernel_source_sha():
            return None
        return int(fields["traffic_bytes_per_launch"])
    except Exception:
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


# ---------------------------------------------------------------------------
# clock sampling during the timed region (NVML through ctypes, read-only)
# ---------------------------------------------------------------------------

class ClockSampler:
    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, device_index):
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            got = False
            try:
                import torch
                uuid = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
                got = nv.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) == 0
            except Exception:
                got = False
            if not got:
                vis = os.environ.get("CUDA_VISIBLE_DEVICES")
                idx = int(vis.split(",")[device_index]) if vis and vis.split(",")[device_index].isdigit() else device_index
                if nv.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(h)) != 0:
                    return
            self.nv, self.h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self._reason_fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.ok = True
        except Exception:
            self.ok = False

    def _run(self):
        c = ctypes.c_uint()
        r = ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(c)) == 0 and \
                    self._reason_fn(self.h, ctypes.byref(r)) == 0:
                self.samples.append((time.perf_counter(), c.value, r.value))
            time.sleep(0.002)

    def loaded(self):
        """Samples taken while the GPU was not idle."""
        return [s for s in self.samples if not s[2] & 0x1]

    def __enter__(self):
        if self.ok:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self.ok:
            self._stop.set()
            self._t.join()

    def summary(self, timed=None):
        """Median SM clock and the active reasons over the samples taken under
        load; `timed` = (t0, t1) host times of the timed region, whose samples
        are also counted."""
        load = self.loaded() if self.ok else []
        if not load:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "source": "nvml unavailable" if not self.ok else "nvml: no sample under load"}
        bits = 0
        for _, _, r in load:
            bits |= r
        out = {"sm_mhz": statistics.median(s[1] for s in load), "sm_max_mhz": self.max_mhz,
               "reasons": [name for b, name in self.REASONS.items() if bits & b],
               "samples": len(load),
               "source": "nvml every 2 ms from the first warm-up step through the timed region and "
                         "a tail of the same step (idle samples dropped)"}
        if timed:
            inside = [s for s in load if timed[0] <= s[0] <= timed[1]]
            out["samples_in_timed_region"] = len(inside)
            if inside:
                out["sm_mhz_timed_region"] = statistics.median(s[1] for s in inside)
        return out


# ---------------------------------------------------------------------------
# the CPU oracle baseline (bounded sample of the same workload)
# ---------------------------------------------------------------------------

def cpu_model():
    """The host CPU's name from /proc/cpuinfo (x86 "model name"; on Arm the
    implementer / part codes), else the platform's processor string."""
    import platform
    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip(), v.strip())
        if fields.get("model name"):
            return fields["model name"]
        if "CPU implementer" in fields:
            return f"arm implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_baseline(batch, target_s=10.0, max_inst=None, threads=None, fixed=False):
    """Time the oracle on the first instances of `batch`: a sample sized for
    about target_s seconds after a short calibration, or (fixed) exactly
    max_inst instances."""
    import oracle
    threads = threads or os.cpu_count() or 1
    # calibrate on a small chunk, then run a sample sized for ~target_s of wall time
    def run(n):
        sub_f = batch.cost_f.reshape(P, M, batch.n)[:, :, :n]
        sub_b = batch.cost_b.reshape(P, M, batch.n)[:, :, :n]
        sub_c = batch.comm.reshape(P - 1, batch.n)[:, :n]
        cf = np.ascontiguousarray(sub_f).reshape(-1)
        cb = np.ascontiguousarray(sub_b).reshape(-1)
        cm = np.ascontiguousarray(sub_c).reshape(-1)
        t0 = time.perf_counter()
        oracle.eval_batch(1, P, M, 1, cf, cb, (1, M * n, n), comm=cm, comm_strides=(1, n), n=n,
                          method=0, nthreads=threads)
        return time.perf_counter() - t0
    if fixed and max_inst:
        n = int(min(batch.n, max_inst))
    else:
        n0 = min(batch.n, 64 * threads)
        t0 = run(n0)
        n = int(min(batch.n, max(n0, n0 * target_s / max(t0, 1e-6))))
        if max_inst:
            n = min(n, max_inst)
    t = run(n)
    ops = 2 * P * M * n
    return {"value": ops / t, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"first {n} of the {batch.n} instances (1F1B P={P} M={M}), event simulation "
                      f"only, {threads} threads, {t:.2f} s wall",
            "seconds": t, "instances": n}


# ---------------------------------------------------------------------------

def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--n", type=int, default=N_INST)
    ap.add_argument("--no-extra", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    return ap.parse_args()


def bench_config(n, world):
    """The workload description shared by both arms."""
    return {"workload": f"1f1b_hetero_P{P}_M{M}_n{n}", "P": P, "M": M,
            "instances_per_gpu": n, "layout": "instance-minor [S][M][n]",
            "l2": f"inputs {2 * P * M * n * 4 / 1e6:.0f} MB > L2 {L2_BYTES / 1e6:.0f} MB, no flush",
            "parallelism": f"instance-sharded x{world}"}


def dist_env():
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local = int(os.environ.get("LOCAL_RANK", 0))
    return rank, world, local


def reference_arm(args, budget_s=90.0):
    """The oracle, as it stands, on this machine's host cores: each step is a
    bounded sample of the same workload, sized once so that all warm-up and
    timed steps together take about `budget_s` seconds of oracle time."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import pipeline_schedule_simulation_gb300.workloads as W
    batch = W.hetero_1f1b(n=args.n)
    threads = os.cpu_count() or 1
    steps = args.warmup + args.steps
    cal = oracle_baseline(batch, target_s=min(2.0, budget_s / 10))
    per_inst = cal["seconds"] / cal["instances"]
    per_step = int(min(batch.n, max(threads, budget_s / max(steps, 1) / per_inst)))
    times = []
    for i in range(steps):
        r = oracle_baseline(batch, max_inst=per_step, fixed=True)
        if i >= args.warmup:
            times.append(r["seconds"])
    total = sum(times)
    ops = 2 * P * M * per_step * len(times)
    value = ops / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64",
        "data": "synthetic",
        "config": bench_config(args.n, world),
        "sample_instances_per_step": per_step,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"first {per_step} of the {batch.n} instances per step, event simulation, "
                                   f"{threads} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return reference_arm(args)

    import torch
    import torch.distributed as dist

    import pipeline_schedule_simulation_gb300.workloads as W
    from pipeline_schedule_simulation_gb300 import binding as B

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if world > 1:
            dist.barrier()

    batch = W.hetero_1f1b(n=args.n, seed=3 + rank)
    n = batch.n
    dev = lambda a: torch.from_numpy(a).cuda()  # noqa: E731
    cf, cb, cm = dev(batch.cost_f), dev(batch.cost_b), dev(batch.comm)
    outs = {"makespan": torch.empty(n, dtype=torch.int32, device="cuda"),
            "idle": torch.empty((n, P), dtype=torch.int32, device="cuda"),
            "bub_num": torch.empty(n, dtype=torch.int64, device="cuda"),
            "bub_den": torch.empty(n, dtype=torch.int64, device="cuda"),
            "peak": torch.empty(P, dtype=torch.int32, device="cuda"),
            "status": torch.empty(n, dtype=torch.int8, device="cuda")}
    stream = torch.cuda.current_stream()

    def step():
        B.evaluate(batch.policy, P, M, 1, cf, cb, batch.strides, n, comm=cm,
                   comm_strides=batch.comm_strides, out=outs, stream=stream)

    sampler = ClockSampler(local)
    sampler.__enter__()
    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    assert int(outs["status"].max()) == 0

    K = args.steps
    t_all0, t_all1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def region(run):
        """Seconds of the GPU time between events around run(), max over ranks."""
        barrier()
        torch.cuda.synchronize()
        t_all0.record(stream)
        run()
        t_all1.record(stream)
        torch.cuda.synchronize()
        barrier()
        return t_all0.elapsed_time(t_all1) / 1e3

    # The timed region: the K evaluations captured once in a CUDA graph (each
    # node one evaluation of the whole batch, in stream order) and replayed
    # once, so consecutive evaluations are not separated by host launch gaps.
    # Where this PyTorch can record timing events inside a captured graph
    # (external events), the graph's first and last nodes are such events and
    # the K evaluations are timed between them on the device; the events on
    # the stream around the replay, which also count the host's graph launch,
    # are reported beside them.  The same K evaluations launched one by one
    # are timed too and reported.
    graph = None
    inner = None
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        try:
            inner = (torch.cuda.Event(enable_timing=True, external=True),
                     torch.cuda.Event(enable_timing=True, external=True))
        except TypeError:
            inner = None
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            if inner:
                inner[0].record(side)
            for _ in range(K):
                B.evaluate(batch.policy, P, M, 1, cf, cb, batch.strides, n, comm=cm,
                           comm_strides=batch.comm_strides, out=outs, stream=side)
            if inner:
                inner[1].record(side)
        graph.replay()
        torch.cuda.synchronize()
    except Exception as e:  # the timed region then launches the evaluations one by one
        graph = None
        inner = None
        graph_error = str(e)[:200]

    def direct():
        for _ in range(K):
            step()

    h0 = time.perf_counter()
    elapsed = region(graph.replay if graph is not None else direct)
    h1 = time.perf_counter()
    outer_s = elapsed
    if inner:
        elapsed = inner[0].elapsed_time(inner[1]) / 1e3
    # A short timed region gives few clock samples: keep running the same step,
    # untimed, until the sampler holds at least 25 samples under load (at
    # least 0.1 s, at most 2 s).
    tail0 = time.perf_counter()
    while sampler.ok and time.perf_counter() - tail0 < 2.0 and \
            (time.perf_counter() - tail0 < 0.1 or len(sampler.loaded()) < 25):
        for _ in range(20):
            step()
        torch.cuda.synchronize()
    sampler.__exit__(None, None, None)
    direct_s = region(direct)
    if world > 1:
        t = torch.tensor([elapsed, direct_s, outer_s], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        elapsed, direct_s, outer_s = float(t[0].item()), float(t[1].item()), float(t[2].item())
    ops_step = 2 * P * M * n
    value = world * ops_step * K / elapsed
    kavg = elapsed / K  # one kernel launch per evaluation
    peak_gbs, peak_src = measured_peaks()
    abytes = algorithmic_bytes(n)
    achieved = abytes / kavg / 1e9

    # ----- end to end through the public host API (pinned host buffers) -----
    host_f = torch.from_numpy(batch.cost_f).pin_memory()
    host_b = torch.from_numpy(batch.cost_b).pin_memory()
    host_c = torch.from_numpy(batch.comm).pin_memory()
    staging = {}
    for _ in range(2):
        B.evaluate_host(batch.policy, P, M, 1, host_f, host_b, n, comm=host_c, stream=stream, staging=staging)
    torch.cuda.synchronize()
    Ke = max(3, min(K, 100))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    e0.record(stream)
    h2d = d2h = 0
    for _ in range(Ke):
        _, h2d, d2h = B.evaluate_host(batch.policy, P, M, 1, host_f, host_b, n, comm=host_c, stream=stream,
                                      staging=staging)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    if world > 1:
        t = torch.tensor([e2e_s], device="cuda", dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_s = float(t.item())
    e2e = {"value": world * ops_step * Ke / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": Ke,
           "api": "pp_sched_eval_host (C ABI, pinned host buffers in, host results out)"}

    extra = {}
    if not args.no_extra and rank == 0:
        extra = secondary(B, W, torch, stream)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": 1e3 * elapsed / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
            "config": bench_config(n, world),
            "gpu_launches": K,
            "roofline": {"bound": "hbm", "kernel": "k_eval_reg<8,1,true,false,true>", "achieved": achieved,
                         "peak": peak_gbs, "unit": "GB/s", "frac": achieved / peak_gbs,
                         "peak_source": peak_src, "traffic": profiled_traffic(),
                         "algorithmic_bytes_per_launch": abytes, "avg_launch_us": kavg * 1e6,
                         "graph_replay_us": outer_s / K * 1e6,
                         "graph_replay_frac": abytes / (outer_s / K) / 1e9 / peak_gbs,
                         "direct_launch_us": direct_s / K * 1e6,
                         "direct_launch_frac": abytes / (direct_s / K) / 1e9 / peak_gbs},
            "timing": (("K evaluations captured in one CUDA graph and replayed once; CUDA events captured as "
                        "the graph's first and last nodes (device time of the K evaluations); average launch "
                        "= elapsed / K; graph_replay_us: events on the stream around the replay, host graph "
                        "launch included" if inner else
                        "K evaluations captured in one CUDA graph and replayed once; CUDA events on the "
                        "launching stream around the replay; average launch = elapsed / K")
                       if graph is not None else f"K direct launches (graph capture failed: {graph_error})"),
            "instances_per_s": world * n * K / elapsed,
            "clocks": sampler.summary(timed=(h0, h1)),
            "e2e": e2e,
        }
        if not args.no_cpu:
            line["cpu_baseline"] = {k: v for k, v in oracle_baseline(batch).items()
                                    if k not in ("seconds", "instances")}
            one = oracle_baseline(batch, target_s=3.0, threads=1)
            line["cpu_baseline"]["single_thread"] = {"value": one["value"], "unit": UNIT, "cores": 1,
                                                     "sample": one["sample"]}
            line["cpu_baseline"]["cpu"] = cpu_model()
        if extra:
            line["secondary"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def secondary(B, W, torch, stream):
    """Short timings of the other workloads (not the headline)."""
    out = {}

    def timed(fn, reps):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / reps

    def timed_eval(fn, reps):
        """An evaluation's seconds per call: `fn(s)` enqueues one call on stream
        s.  The calls are timed launched one by one and, where they can be
        captured, as `reps` calls in one CUDA graph between events captured
        inside it (the device time, without the host's per-call cost, which
        exceeds a short kernel's).  Returns (seconds, direct seconds, how)."""
        direct = timed(lambda: fn(stream), reps)
        try:
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            e0 = torch.cuda.Event(enable_timing=True, external=True)
            e1 = torch.cuda.Event(enable_timing=True, external=True)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=side):
                e0.record(side)
                for _ in range(reps):
                    fn(side)
                e1.record(side)
            for _ in range(2):
                g.replay()
                torch.cuda.synchronize()
            return e0.elapsed_time(e1) / 1e3 / reps, direct, "graph"
        except Exception:  # not capturable (or no external events): the direct launches
            torch.cuda.synchronize()
            return direct, direct, "direct"

    def line(ops, t):
        sec, direct, how = t
        return {"op_times_per_s": ops / sec, "ms": sec * 1e3, "direct_ms": direct * 1e3, "timing": how}

    # per-op start/end stored (instance-minor op layout)
    b3 = W.hetero_1f1b(n=N_INST)
    cf, cb, cm = (torch.from_numpy(x).cuda() for x in (b3.cost_f, b3.cost_b, b3.comm))
    O = 2 * M
    ops_out = {"op_start": torch.empty((P, O, N_INST), dtype=torch.int32, device="cuda"),
               "op_end": torch.empty((P, O, N_INST), dtype=torch.int32, device="cuda")}
    tt = timed_eval(lambda s: B.evaluate(1, P, M, 1, cf, cb, b3.strides, N_INST, comm=cm,
                                         comm_strides=b3.comm_strides, op_times=True, op_strides=(1, N_INST),
                                         out=ops_out, stream=s), 20)
    t = tt[0]
    ob = algorithmic_bytes(N_INST) + 2 * 4 * 2 * P * M * N_INST  # + op_start and op_end, int32 each
    peak_gbs, peak_src = measured_peaks()
    out["1f1b_P8_M64_with_op_times"] = dict(line(2 * P * M * N_INST, tt), algorithmic_bytes=ob, gbs=ob / t / 1e9,
                                            frac_of_hbm_peak=ob / t / 1e9 / peak_gbs, peak_source=peak_src)
    del ops_out, cf, cb, cm
    for v in (2, 4):
        il, base = W.interleaved_vs_1f1b(v)
        for tag, bt in (("interleaved", il), ("1f1b_equal_work", base)):
            f, g, c = (torch.from_numpy(x).cuda() for x in (bt.cost_f, bt.cost_b, bt.comm))
            res_il = B.evaluate(bt.policy, bt.P, bt.M, bt.v, f, g, bt.strides, bt.n, comm=c,
                                comm_strides=bt.comm_strides, stream=stream)
            tt = timed_eval(lambda s: B.evaluate(bt.policy, bt.P, bt.M, bt.v, f, g, bt.strides, bt.n, comm=c,
                                                 comm_strides=bt.comm_strides, out=res_il, stream=s), 20)
            out[f"{tag}_P8_v{v}_M128_n16384"] = line(bt.op_times, tt)
    for pol, name in ((W.ZB1P, "zb1p"), (W.ZB2P, "zb2p")):
        bz = W.hetero_zb(pol, n=N_INST)
        f, g, w, c = (torch.from_numpy(x).cuda() for x in (bz.cost_f, bz.cost_b, bz.cost_w, bz.comm))
        zout = {}
        zout.update(B.evaluate_zb(pol, P, M, f, g, w, bz.strides, N_INST, comm=c, comm_strides=bz.comm_strides,
                                  stream=stream))
        tt = timed_eval(lambda s: B.evaluate_zb(pol, P, M, f, g, w, bz.strides, N_INST, comm=c,
                                                comm_strides=bz.comm_strides, out=zout, stream=s), 10)
        out[f"{name}_P8_M64_n{N_INST}"] = dict(line(bz.op_times, tt),
                                               mean_makespan=float(zout["makespan"].float().mean().item()))
        del f, g, w, c, zout
    bd = W.hetero_dualpipe(n=N_INST)
    m_a = bd.meta["m_a"]
    f, g, c = (torch.from_numpy(x).cuda() for x in (bd.cost_f, bd.cost_b, bd.comm))
    dout = B.evaluate_dualpipe(P, M, m_a, f, g, bd.strides, N_INST, comm=c, comm_strides=bd.comm_strides,
                               stream=stream)
    tt = timed_eval(lambda s: B.evaluate_dualpipe(P, M, m_a, f, g, bd.strides, N_INST, comm=c,
                                                  comm_strides=bd.comm_strides, out=dout, stream=s), 10)
    one = B.evaluate(1, P, M, 1, f, g, bd.strides, N_INST, comm=c, comm_strides=bd.comm_strides, stream=stream)
    out[f"dualpipe_P8_M64_n{N_INST}"] = {
        **line(bd.op_times, tt), "microbatches_per_route": [m_a, M - m_a],
        "mean_makespan": float(dout["makespan"].double().mean().item()),
        "mean_makespan_1f1b_same_costs": float(one["makespan"].double().mean().item()),
        "max_peak": int(dout["peak"].max().item())}
    del f, g, c, dout, one
    out["closed_form_sweep"] = closed_form_sweep(B, W, torch, stream, timed)
    p = W.layer_split()
    lt, lb, la = (torch.from_numpy(x).cuda() for x in (p.layer_tf, p.layer_tb, p.layer_act))
    res = {}
    t = timed(lambda: res.update(B.partition_search(lt, lb, la, p.P, p.M, p.comm, p.cap, p.seed, 0,
                                                    p.n_cand, stream=stream)), 5)
    out["partition_search_L80_P8_M128_1M"] = {
        "candidates_per_s": p.n_cand / t, "ms": t * 1e3,
        "best_idx": int(res["best_idx"].item()), "best_makespan": int(res["best_makespan"].item()),
        "best_cuts": res["best_cuts"].cpu().tolist()}
    total = math.comb(len(p.layer_tf) - 1, p.P - 1)
    ex = {}
    t_ex = timed(lambda: ex.update(B.partition_search_ranks(lt, lb, la, p.P, p.M, p.comm, p.cap, 0, total,
                                                            stream=stream)), 3)
    il = {}
    n_il = 1 << 20
    t = timed(lambda: il.update(B.partition_search_interleaved(lt, lb, la, p.P, 2, p.M, p.comm, p.cap, p.seed, 0,
                                                               n_il, stream=stream)), 3)
    out["partition_search_interleaved_L80_P8_v2_M128_1M"] = {
        "candidates_per_s": n_il / t, "ms": t * 1e3, "op_times_per_candidate": 2 * p.P * p.M * 2,
        "best_idx": int(il["best_idx"].item()), "best_makespan": int(il["best_makespan"].item())}
    out["partition_search_exhaustive_L80_P8_M128"] = {
        "splits": total, "splits_per_s": total / t_ex, "ms": t_ex * 1e3,
        "best_rank": int(ex["best_idx"].item()), "best_makespan": int(ex["best_makespan"].item()),
        "best_cuts": ex["best_cuts"].cpu().tolist()}
    return out


def closed_form_sweep(B, W, torch, stream, timed):
    """The closed-form sweep (GPipe and 1F1B at P 2..16 x M 1..128, interleaved
    v = 2 where P divides M; 16 scalar-cost instances per shape).  Timed as one
    pp_sched_eval per shape -- the first pass from an empty plan cache (every
    shape's plan is built then, one at a time), later passes driven from
    Python, the same calls replayed from a CUDA graph -- and as one prepared
    set of problems (pp_sched_many_*: every plan and table built in one batch,
    then a few fused launches): its preparation from an empty plan cache, its
    evaluation called from Python and replayed from a CUDA graph."""
    calls = []
    op_times = 0
    for pol, P_, M_, v_ in W.sweep_shapes():
        bt = W.sweep_batch(pol, P_, M_, v_)
        f, g, c = (torch.from_numpy(x).cuda() for x in (bt.cost_f, bt.cost_b, bt.comm))
        o = {"makespan": torch.empty(bt.n, dtype=torch.int32, device="cuda"),
             "idle": torch.empty((bt.n, P_), dtype=torch.int32, device="cuda"),
             "bub_num": torch.empty(bt.n, dtype=torch.int64, device="cuda"),
             "bub_den": torch.empty(bt.n, dtype=torch.int64, device="cuda"),
             "peak": torch.empty(P_, dtype=torch.int32, device="cuda"),
             "status": torch.empty(bt.n, dtype=torch.int8, device="cuda")}
        calls.append((bt, f, g, c, o))
        op_times += bt.op_times

    def one_pass(st):
        for bt, f, g, c, o in calls:
            B.evaluate(bt.policy, bt.P, bt.M, bt.v, f, g, bt.strides, bt.n, comm=c,
                       comm_strides=bt.comm_strides, out=o, stream=st)

    # both first passes start from an empty plan cache (as in a fresh process)
    torch.cuda.synchronize()
    B.cache_clear()
    t0 = time.perf_counter()
    one_pass(stream)
    torch.cuda.synchronize()
    first = time.perf_counter() - t0
    problems = [{"policy": bt.policy, "P": bt.P, "M": bt.M, "v": bt.v, "n": bt.n, "strides": bt.strides,
                 "cost_f": f, "cost_b": g, "comm": c, "comm_strides": bt.comm_strides, "out": o}
                for bt, f, g, c, o in calls]
    B.cache_clear()
    t0 = time.perf_counter()
    cold = B.Many(problems, stream=stream)
    torch.cuda.synchronize()
    prepare_cold = time.perf_counter() - t0
    cold.close()
    loop = timed(lambda: one_pass(stream), 3)
    res = {"shapes": len(calls), "instances": 16 * len(calls), "op_times": op_times,
           "first_pass_ms": first * 1e3, "many_prepare_cold_ms": prepare_cold * 1e3,
           "loop_ms": loop * 1e3, "loop_op_times_per_s": op_times / loop}
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            one_pass(side)
        gt = timed(graph.replay, 3)
        res.update(graph_ms=gt * 1e3, graph_op_times_per_s=op_times / gt)
    except Exception as e:  # capture is a measurement aid here, not part of the path
        res.update(graph_ms=None, graph_error=str(e)[:200])
    # the same problems prepared once and evaluated together (pp_sched_many_*)
    many = B.Many(problems, stream=stream)
    mt = timed(lambda: many(stream=stream), 20)
    res.update(many_ms=mt * 1e3, many_op_times_per_s=op_times / mt, many_info=many.info())
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            many(stream=side)
        gt = timed(graph.replay, 20)
        res.update(many_graph_ms=gt * 1e3, many_graph_op_times_per_s=op_times / gt)
    except Exception as e:
        res.update(many_graph_ms=None, many_graph_error=str(e)[:200])
    many.close()
    return res


if __name__ == "__main__":
    sys.exit(main())
