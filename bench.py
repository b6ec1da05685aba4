#!/usr/bin/env python
"""Throughput of the AGoQ element-wise quantization path on GB300.

One step = the DBCA-PP activation workload (LLaMA-7B MLP shapes): the RMSNorm
input BF16 [8192 x 4096] and the SiLU/gate input BF16 [8192 x 11008], Student-t
(nu=4) values, each quantized at 4, 5, 6 and 8 bits and dequantized back: 16
library calls (8 quantize, then 8 dequantize).  The calls run on two streams,
widths {4, 6} on one and {5, 8} on the other (each stream keeps its own
quantize -> dequantize order; the streams join every step), so that one call's
ramp and tail overlap another's streaming; the line also gives the same steps
on one stream.  The metric is algorithmic HBM bytes per second (each call reads
its input and writes its output once: n*(2 + bits/8 + 1/32) bytes) and input
elements per second.

Every width quantizes its own copy of each input tensor, and every dequantize
reads codes written at least 247 MB of HBM traffic earlier; one step moves
2.7 GB, so no call finds its input in the L2 (126 MB) from another call.

The timed region is a window of exactly K steps (barrier and synchronize on
both sides, CUDA events at its ends), repeated until the windows last at least
one second together; value comes from the median window (max over ranks) and
the windows' spread is reported.

Also reported:
  roofline      the dominant kernel's algorithmic GB/s (CUDA events around each
                launch on the launching stream) against the measured HBM copy peak;
  e2e           the same step with inputs copied from pinned host memory and all
                outputs copied back inside the timed region, and the same copies
                alone, one stream per direction (the host link's time for them);
  cpu_baseline  the CPU oracle on the host cores: its all-core (OpenMP) build on
                the full workload where it fits the time budget, and the
                single-threaded build on a bounded sample; `oracle_rows` times
                the all-core oracle on the other workloads (full size or a
                stated sample);
  rows          each other kernel of the path on its own workload, L2 flushed
                before each timed launch (a 256 MB buffer written, then another
                256 MB read, so the launch starts from a cold L2 holding no dirty
                lines): the 2048x4096 4-bit round trip (single launches and a
                100-call CUDA graph), the DBCA-PP tensors' 4-bit calls in 100-call
                graphs and the 16-call step as a graph, QuanGrad accumulation of
                2^30 elements over the 8 micro-batches from a zeroed master, the
                FP8 shard reduce W=8/64 of 2^25 with and without the naive count,
                the INT4-fused weight-gradient GEMM 11008x4096x8192, its fused
                accumulation, the forward GEMM with quantized output and the
                SiLU/RMSNorm backward recompute.

--impl reference times the CPU oracle (the plain restatement the kernels are
checked against), all-core build, on the same workload (all 8192 token rows
when a step fits the time budget, else a bounded sample).
Launch: python bench.py [--gpus N --steps K --warmup W]; for N > 1 under
torch.distributed.run, one rank per GPU, each rank running the workload on its
own GPU (weak scaling, no collective on the data path).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WIDTHS = (4, 5, 6, 8)
METRIC = "HBM GB/s and Gelem/s per quant kernel; fraction of GB300 HBM/tensor peak"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
# Least total length of the timed region: the K-step window is repeated until
# the windows together last at least this long.
MIN_TIMED_S = 1.0


def act_bytes(n, bits):
    """Algorithmic bytes of one quantize or dequantize call on n elements."""
    return n * 2 + n * bits // 8 + (n // 128) * 4


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ----------------------------------------------------------------------- distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend):
    import torch.distributed as dist
    world, rank, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return world, rank


def dist_barrier(device=None):
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(value, device=None):
    """Maximum of a float over all ranks (the value itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ----------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of this GPU's clocks and throttle reasons."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None, period_ms=100):
        self.rows = []
        self.proc = None
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
               "-lms", str(period_ms)]
        if device_uuid:
            cmd[1:1] = ["-i", device_uuid]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        rows = [r for (t, r) in self.rows if t0 <= t <= t1] or [r for (_, r) in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
        sm = [float(r[0]) for r in rows if r[0].replace(".", "").isdigit()]
        smax = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if len(r) > 4 + i and r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------- GPU arm
def gpu_arm(args):
    import torch
    from gradient_quantization_gb300 import agoq, synthetic

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init("nccl")
    hbm_peak, bf16_peak, bf16_sust, peak_kind = measured_peaks()

    # ---- inputs resident in HBM
    x1, x2 = synthetic.dbca_activations_torch(seed=1 + rank, device=device)
    tensors = [("rmsnorm_in", x1), ("silu_in", x2)]
    codes, scales, outs = {}, {}, {}
    # every width quantizes its own copy of each input, so that no call can find
    # its input in L2 from another call's traffic, however the calls are ordered
    # or overlapped
    xin = {}
    for name, x in tensors:
        n = x.numel()
        for b in WIDTHS:
            xin[name, b] = x.clone()
            codes[name, b] = torch.empty(n // 128 * 16 * b, dtype=torch.uint8, device=device)
            scales[name, b] = torch.empty(n // 128, dtype=torch.float32, device=device)
            outs[name, b] = torch.empty(n, dtype=torch.bfloat16, device=device)
    calls = []   # (label, bytes, elems, fn)
    for b in WIDTHS:
        for name, x in tensors:
            n = x.numel()
            calls.append(("quant_b%d_%s" % (b, name), act_bytes(n, b), n,
                          (lambda b=b, name=name: agoq.agoq_quant_act(xin[name, b], b, codes[name, b],
                                                                      scales[name, b]))))
    for b in WIDTHS:
        for name, x in tensors:
            n = x.numel()
            calls.append(("dequant_b%d_%s" % (b, name), act_bytes(n, b), n,
                          (lambda n=n, b=b, name=name: agoq.agoq_dequant_act(codes[name, b], scales[name, b], n, b, outs[name, b]))))
    step_bytes = sum(c[1] for c in calls)
    step_elems = sum(c[2] for c in calls)

    # The step's calls on `args.streams` streams: the widths are split between
    # them ({4, 6} and {5, 8} for two), each stream carrying its own quantize ->
    # dequantize dependencies in the serial order; the streams join at the end
    # of every step.  Widths never share a buffer, so no other ordering is needed.
    main_stream = torch.cuda.current_stream(device)
    groups = ((4, 6), (5, 8)) if args.streams == 2 else (WIDTHS,)
    width_of = {c[0]: int(c[0].split("_")[1][1:]) for c in calls}
    group_calls = [[c for c in calls if width_of[c[0]] in g] for g in groups]
    side = [torch.cuda.Stream(device) for _ in groups]

    def step_serial():
        for c in calls:
            c[3]()

    def step():
        if len(groups) == 1:
            step_serial()
            return
        fork = torch.cuda.Event()
        fork.record(main_stream)
        for st, cl in zip(side, group_calls):
            st.wait_event(fork)
            with torch.cuda.stream(st):
                for c in cl:
                    c[3]()
        for st in side:
            join = torch.cuda.Event()
            join.record(st)
            main_stream.wait_event(join)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)

    # Timed region: windows of exactly K steps, each bracketed by a barrier and
    # a synchronize, with events only at the window's ends (so that consecutive
    # kernels keep their programmatic-dependent-launch overlap).  The window is
    # repeated until the windows last MIN_TIMED_S together; value is the median
    # window (max over ranks), and the spread is reported.
    stream = torch.cuda.current_stream(device)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    windows = []
    t_wall0 = time.time()
    while True:
        dist_barrier(device)
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            step()
        stop.record(stream)
        torch.cuda.synchronize()
        dist_barrier(device)
        windows.append(start.elapsed_time(stop))
        # the same stopping decision on every rank
        if max_over_ranks(sum(windows), device) >= MIN_TIMED_S * 1e3 or len(windows) >= 10000:
            break
    windows = [max_over_ranks(w, device) for w in windows]
    elapsed_ms = statistics.median(windows)
    # the same steps on one stream, for comparison
    one_ms = None
    if len(groups) > 1:
        torch.cuda.synchronize()
        start.record(stream)
        for k in range(args.steps):
            step_serial()
        stop.record(stream)
        torch.cuda.synchronize()
        one_ms = max_over_ranks(start.elapsed_time(stop), device) / args.steps

    # Per-kernel pass: the same steps again with an event after every call
    # (each kernel then runs without overlap with its neighbours: per-kernel
    # durations, for the roofline of the dominant kernel).
    ksteps = min(args.steps, 200)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)] for _ in range(ksteps)]
    torch.cuda.synchronize()
    for k in range(ksteps):
        e = ev[k]
        e[0].record(stream)
        for i, c in enumerate(calls):
            c[3]()
            e[i + 1].record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    per_call = [0.0] * len(calls)
    for k in range(ksteps):
        for i in range(len(calls)):
            per_call[i] += ev[k][i].elapsed_time(ev[k][i + 1])
    per_call = [t / ksteps for t in per_call]
    if sampler:
        time.sleep(0.25)
        sampler.stop()
        clocks = sampler.summary(t_wall0 - 0.05, t_wall1 + 0.3)
    max_ms = elapsed_ms
    total_bytes = sum_over_ranks(step_bytes * args.steps, device)
    total_elems = sum_over_ranks(step_elems * args.steps, device)
    value = total_bytes / (max_ms * 1e-3) / 1e9
    gelem = total_elems / (max_ms * 1e-3) / 1e9

    # ---- dominant kernel and its roofline
    dom = max(range(len(calls)), key=lambda i: per_call[i])
    dom_label, dom_bytes = calls[dom][0], calls[dom][1]
    achieved = dom_bytes / (per_call[dom] * 1e-3) / 1e9
    traffic = None   # DRAM counters come from ncu captures, not from this run
    # the same launch alone, after an L2 flush that leaves no dirty lines (in the
    # step it also writes back what the previous call left dirty in L2)
    flushbuf = torch.zeros(256 << 20 >> 2, dtype=torch.float32, device=device)
    cleanbuf = torch.ones(256 << 20 >> 2, dtype=torch.float32, device=device)
    iso_ms = _time_launch(calls[dom][3], lambda: _flush_l2(flushbuf, cleanbuf), reps=7, warm=2)
    del flushbuf, cleanbuf
    iso_gbs = dom_bytes / (iso_ms * 1e-3) / 1e9
    kernels = {c[0]: {"us": round(per_call[i] * 1e3, 2),
                      "GB/s": round(c[1] / (per_call[i] * 1e-3) / 1e9, 1),
                      "Gelem/s": round(c[2] / (per_call[i] * 1e-3) / 1e9, 2),
                      "frac_of_measured_hbm": round(c[1] / (per_call[i] * 1e-3) / 1e9 / hbm_peak, 4)}
               for i, c in enumerate(calls)}

    # ---- end to end through host buffers
    e2e = e2e_arm(args, tensors, codes, scales, outs, calls, device)

    # ---- the precision-preserved all-reduce across the ranks (N > 1 only)
    allreduce = allreduce_arm(device, world) if world > 1 and not args.no_rows else None

    # ---- other rows of the path
    rows = None
    if rank == 0 and not args.no_rows:
        rows = rows_arm(device, hbm_peak, bf16_peak)

    # ---- CPU oracle baseline
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)
        from oracle import oracle as O
        if O.parallel_available():
            cpu["oracle_rows"] = oracle_rows(device)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "dtypes": {"input": "bf16", "codes": "int4/int5/int6/int8", "scales": "f32",
                       "arithmetic": "f32", "output": "bf16"},
            "windows": {"count": len(windows), "steps_each": args.steps,
                        "timed_region_s": round(sum(windows) / 1e3, 3),
                        "median_ms": round(statistics.median(windows), 4),
                        "min_ms": round(min(windows), 4), "max_ms": round(max(windows), 4),
                        "value_from": "median window"},
            "gelem_per_s": round(gelem, 2),
            "frac_of_measured_hbm": round(value / world / hbm_peak, 4),
            "frac_of_nominal_hbm": round(value / world / NOMINAL_HBM_GBS, 4),
            "streams": {"count": len(groups), "widths": [list(g) for g in groups],
                        "one_stream_ms_per_step": round(one_ms, 4) if one_ms else None},
            "config": {"workload": "DBCA-PP activations: RMSNorm in BF16[8192x4096] + SiLU in "
                                   "BF16[8192x11008], Student-t nu=4, quantize+dequantize at 4/5/6/8 bits",
                       "calls_per_step": len(calls), "bytes_per_step": step_bytes,
                       "elems_per_step": step_elems,
                       "l2": "inputs larger than L2: every call reads its own input (one copy of "
                             "each tensor per width) or codes written >=247 MB of traffic earlier; "
                             "2.7 GB moved per step",
                       "parallelism": "dp%d (independent replicas)" % world},
            "roofline": {"kernel": dom_label, "bound": "hbm", "achieved": round(achieved, 1),
                         "peak": hbm_peak, "unit": "GB/s",
                         "frac": round(achieved / hbm_peak, 4), "peak_kind": peak_kind,
                         "bytes_per_launch": dom_bytes, "us_per_launch": round(per_call[dom] * 1e3, 2),
                         "traffic": traffic,
                         "isolated": {"us_per_launch": round(iso_ms * 1e3, 2),
                                      "achieved": round(iso_gbs, 1),
                                      "frac": round(iso_gbs / hbm_peak, 4),
                                      "timing": "median of 7 launches alone, each after an L2 "
                                                "flush leaving no dirty lines"}},
            "kernels": kernels,
            "kernels_timing": "separate pass of %d steps with an event after every call; the "
                              "timed region (value) has events only at its ends" % ksteps,
            "e2e": e2e,
            "gpu_launches": len(calls) * args.steps * len(windows),
            "gpu_launches_per_step": len(calls),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        if allreduce is not None:
            line["allreduce"] = allreduce
        if rows is not None:
            line["rows"] = rows
            line["rows_timing"] = ("median of 5 launches, each after an L2 flush that writes 256 MB "
                                   "and then reads another 256 MB (cold L2, no dirty lines)")
        print(json.dumps(line), flush=True)
    # every rank leaves together (rank 0 may still have been timing rows)
    dist_barrier(device)
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.destroy_process_group()


def e2e_arm(args, tensors, codes, scales, outs, calls, device):
    """The step with inputs copied from pinned host memory and every output
    copied back to pinned host memory inside the timed region.  Copies in,
    kernels and copies out run on three streams: each call waits only for its
    input's copy, each output's copy waits only for the call that wrote it, the
    next step's input copies wait for this step's quantizers, and each call
    waits for the previous step's copy of the output it overwrites."""
    import torch
    from gradient_quantization_gb300 import agoq
    host_in = {name: x.cpu().pin_memory() for name, x in tensors}
    dev_in = {name: x for name, x in tensors}
    host_out = {}
    for k in codes:
        host_out[k] = (torch.empty(codes[k].shape, dtype=codes[k].dtype).pin_memory(),
                       torch.empty(scales[k].shape, dtype=scales[k].dtype).pin_memory(),
                       torch.empty(outs[k].shape, dtype=outs[k].dtype).pin_memory())
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for v in host_out.values() for t in v)
    step_bytes = sum(c[1] for c in calls)
    steps = max(1, min(args.steps, 20))
    s_in, s_comp = torch.cuda.Stream(device), torch.cuda.Stream(device)
    s_outs = [torch.cuda.Stream(device) for _ in range(4)]     # several copy engines
    ev = lambda: torch.cuda.Event()   # noqa: E731
    names = [name for name, _ in tensors]
    quant_done = {name: None for name in names}
    copied_out = {k: None for k in codes}
    # (kind, name, bits) per call in the step's order
    plan = [("q", name, b) for b in WIDTHS for name in names] + \
           [("d", name, b) for b in WIDTHS for name in names]

    def one(kernels=True):
        in_ready = {}
        with torch.cuda.stream(s_in):
            for name in names:
                if quant_done[name] is not None:
                    s_in.wait_event(quant_done[name])
                dev_in[name].copy_(host_in[name], non_blocking=True)
                in_ready[name] = ev()
                in_ready[name].record(s_in)
        with torch.cuda.stream(s_comp):
            last_quant = {}
            for kind, name, b in plan:
                k = (name, b)
                if kind == "q":
                    s_comp.wait_event(in_ready[name])
                    if copied_out[k] is not None:
                        s_comp.wait_event(copied_out[k])
                    if kernels:
                        agoq.agoq_quant_act(dev_in[name], b, codes[k], scales[k], stream=s_comp)
                    last_quant[name] = ev()
                    last_quant[name].record(s_comp)
                    done = last_quant[name]
                else:
                    if kernels:
                        agoq.agoq_dequant_act(codes[k], scales[k], outs[k].numel(), b, outs[k],
                                              stream=s_comp)
                    done = ev()
                    done.record(s_comp)
                s_out = s_outs[(WIDTHS.index(b) * len(names) + names.index(name)) % len(s_outs)]
                with torch.cuda.stream(s_out):
                    s_out.wait_event(done)
                    hc, hs, ho = host_out[k]
                    if kind == "q":
                        hc.copy_(codes[k], non_blocking=True)
                        hs.copy_(scales[k], non_blocking=True)
                    else:
                        ho.copy_(outs[k], non_blocking=True)
                        copied_out[k] = ev()
                        copied_out[k].record(s_out)
            for name in names:
                quant_done[name] = last_quant[name]

    # The copies alone: each step's input copies on one stream and its output
    # copies, in the step's order, on one other stream (the two directions of
    # the host link overlap), without the kernels: the link's time for the same
    # bytes.  (The e2e plan itself with the kernels left out is not that bound:
    # with nothing to pace them, all of a step's output copies become ready at
    # once on the four output streams and contend, 7.4-10.1 ms per step in
    # different runs against the 7.35 ms e2e step.)
    def copies_alone(kernels=False):
        with torch.cuda.stream(s_in):
            for name in names:
                dev_in[name].copy_(host_in[name], non_blocking=True)
        with torch.cuda.stream(s_outs[0]):
            for kind, name, b in plan:
                hc, hs, ho = host_out[(name, b)]
                if kind == "q":
                    hc.copy_(codes[(name, b)], non_blocking=True)
                    hs.copy_(scales[(name, b)], non_blocking=True)
                else:
                    ho.copy_(outs[(name, b)], non_blocking=True)

    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def window(fn, streams):
        fn()
        torch.cuda.synchronize()
        a.record(s_comp)
        for st in streams:
            st.wait_event(a)
        for _ in range(steps):
            fn()
        for st in streams:
            e = ev()
            e.record(st)
            s_comp.wait_event(e)
        b.record(s_comp)
        torch.cuda.synchronize()
        return max_over_ranks(a.elapsed_time(b), device)

    # The host link's rate drifts between runs, so the two legs alternate
    # (three windows each) and each reports its median window.
    dist_barrier(device)
    e2e_w, copy_w = [], []
    for _ in range(3):
        e2e_w.append(window(one, [s_in] + s_outs))
        copy_w.append(window(copies_alone, [s_in, s_outs[0]]))
    ms = statistics.median(e2e_w)
    copy_ms = statistics.median(copy_w) / steps
    total = sum_over_ranks(step_bytes * steps, device)
    return {"value": round(total / (ms * 1e-3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 3), "steps": steps,
            "copies_only_ms_per_step": round(copy_ms, 3),
            "overlap": "copies in, kernels and copies out (4 streams) overlapped; "
                       "copies_only_ms_per_step: the same copies alone, one stream per "
                       "direction; each the median of 3 alternating windows"}


def allreduce_arm(device, world, reps=10, warm=3):
    """QuanGrad's precision-preserved all-reduce (all-to-all of FP8 shards, the
    library's local reduce, all-gather) over all ranks: every rank holds an FP8
    gradient of world * 2^25 elements, so each local reduce sees world shards of
    2^25 (the shard reduce's configuration at world = 8).  Times with CUDA events
    between barriers, max over ranks."""
    import torch
    from gradient_quantization_gb300 import synthetic
    from gradient_quantization_gb300.allreduce import precision_preserved_allreduce
    try:
        n = world * synthetic.REDUCE_N
        g = torch.Generator(device=device)
        g.manual_seed(7 + dist_env()[1])
        codes = torch.randint(0, 126, (n,), dtype=torch.uint8, device=device, generator=g)
        codes |= torch.randint(0, 2, (n,), dtype=torch.uint8, device=device, generator=g) << 7
        scales = torch.rand(n // 128, device=device, generator=g) * 1e-4
        for _ in range(warm):
            precision_preserved_allreduce(codes, scales)
        torch.cuda.synchronize()
        dist_barrier(device)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            precision_preserved_allreduce(codes, scales)
        b.record()
        torch.cuda.synchronize()
        ms = max_over_ranks(a.elapsed_time(b) / reps, device)
        nbytes = n + (n // 128) * 4
        return {"us": round(ms * 1e3, 1), "elements_per_rank": n, "ranks": world,
                "gradient_GB/s_per_rank": round(nbytes / (ms * 1e-3) / 1e9, 1),
                "steps": "all-to-all (NCCL) -> agoq_reduce_fp8_shards -> all-gather (NCCL)"}
    except Exception as e:   # a failing collective must not lose the bench line
        return {"unavailable": "%s: %s" % (type(e).__name__, str(e)[:200])}


def _flush_l2(buf, clean):
    """Evict the L2: write `buf` (larger than L2), then read `clean` (larger than
    L2) so that the written lines are written back before the timed launch and
    it starts from a cold cache holding no dirty lines."""
    buf.add_(1)
    clean.sum()


def _time_launch(fn, flush, reps=5, warm=2):
    import torch
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def rows_arm(device, hbm_peak, bf16_peak):
    """Each other kernel of the path on its own workload, L2 flushed before each launch."""
    import torch
    from gradient_quantization_gb300 import agoq, synthetic
    rows = {}
    flushbuf = torch.zeros(256 << 20 >> 2, dtype=torch.float32, device=device)
    cleanbuf = torch.ones(256 << 20 >> 2, dtype=torch.float32, device=device)
    flush = lambda: _flush_l2(flushbuf, cleanbuf)   # noqa: E731

    def row(name, nbytes, elems, ms, extra=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        r = {"us": round(ms * 1e3, 2), "GB/s": round(gbs, 1),
             "Gelem/s": round(elems / (ms * 1e-3) / 1e9, 2),
             "frac_of_measured_hbm": round(gbs / hbm_peak, 4),
             "frac_of_nominal_hbm": round(gbs / NOMINAL_HBM_GBS, 4)}
        if extra:
            r.update(extra)
        rows[name] = r

    # 4-bit round trip on the 2048 x 4096 activation
    x = synthetic.laaq_activation_torch(seed=0, device=device)
    n = x.numel()
    c, s = agoq.agoq_quant_act(x, 4)
    y = torch.empty_like(x)
    row("laaq_int4_quant_2048x4096", act_bytes(n, 4), n,
        _time_launch(lambda: agoq.agoq_quant_act(x, 4, c, s), flush))
    row("laaq_int4_dequant_2048x4096", act_bytes(n, 4), n,
        _time_launch(lambda: agoq.agoq_dequant_act(c, s, n, 4, y), flush))
    # 100 back-to-back calls captured in one CUDA graph, rotating over 16 copies
    # of the activation and its outputs (16 x 21 MB of traffic > L2): the
    # per-call rate without launch gaps
    k = 16
    xs_c = [x.clone() for _ in range(k)]
    cs_c = [torch.empty_like(c) for _ in range(k)]
    ss_c = [torch.empty_like(s) for _ in range(k)]
    ys_c = [torch.empty_like(x) for _ in range(k)]
    for name, fn in (("laaq_int4_quant_2048x4096_graph100",
                      lambda i: agoq.agoq_quant_act(xs_c[i % k], 4, cs_c[i % k], ss_c[i % k])),
                     ("laaq_int4_dequant_2048x4096_graph100",
                      lambda i: agoq.agoq_dequant_act(cs_c[i % k], ss_c[i % k], n, 4, ys_c[i % k]))):
        for i in range(k):
            fn(i)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for i in range(100):
                fn(i)
        ms = _time_launch(graph.replay, flush) / 100
        row(name, act_bytes(n, 4), n, ms, {"calls_per_graph": 100, "rotating_copies": k})
        del graph
    del x, c, s, y, xs_c, cs_c, ss_c, ys_c

    # The DBCA-PP activations (8192 x 4096 and 8192 x 11008): 100 back-to-back
    # 4-bit calls in one CUDA graph over 2 rotating copies of each tensor (every
    # copy is larger than L2, or 2 x 67 MB for the smaller tensor), and the
    # 16-call step on one stream captured as a graph (10 steps per replay).
    xa, xb = synthetic.dbca_activations_torch(seed=1, device=device)
    for label, xt in (("rmsnorm_in_8192x4096", xa), ("silu_in_8192x11008", xb)):
        n = xt.numel()
        k = 2
        xs_c = [xt.clone() for _ in range(k)]
        cs_c = [torch.empty(n // 2, dtype=torch.uint8, device=device) for _ in range(k)]
        ss_c = [torch.empty(n // 128, dtype=torch.float32, device=device) for _ in range(k)]
        ys_c = [torch.empty_like(xt) for _ in range(k)]
        for name, fn in (("dbca_int4_quant_%s_graph100" % label,
                          lambda i: agoq.agoq_quant_act(xs_c[i % k], 4, cs_c[i % k], ss_c[i % k])),
                         ("dbca_int4_dequant_%s_graph100" % label,
                          lambda i: agoq.agoq_dequant_act(cs_c[i % k], ss_c[i % k], n, 4,
                                                          ys_c[i % k]))):
            for i in range(k):
                fn(i)
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for i in range(100):
                    fn(i)
            ms = _time_launch(graph.replay, flush, reps=3, warm=1) / 100
            row(name, act_bytes(n, 4), n, ms, {"calls_per_graph": 100, "rotating_copies": k})
            del graph
        del xs_c, cs_c, ss_c, ys_c
    # the 16-call step: quantize both tensors at 4/5/6/8 bits, then dequantize
    xin, cod, sca, out = {}, {}, {}, {}
    for name, xt in (("a", xa), ("b", xb)):
        for bits in WIDTHS:
            xin[name, bits] = xt.clone()
            cod[name, bits] = torch.empty(xt.numel() // 128 * 16 * bits, dtype=torch.uint8,
                                          device=device)
            sca[name, bits] = torch.empty(xt.numel() // 128, dtype=torch.float32, device=device)
            out[name, bits] = torch.empty_like(xt)

    def dbca_step():
        for bits in WIDTHS:
            for name in ("a", "b"):
                agoq.agoq_quant_act(xin[name, bits], bits, cod[name, bits], sca[name, bits])
        for bits in WIDTHS:
            for name in ("a", "b"):
                agoq.agoq_dequant_act(cod[name, bits], sca[name, bits], xin[name, bits].numel(),
                                      bits, out[name, bits])
    dbca_step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(10):
            dbca_step()
    step_bytes = sum(2 * act_bytes(xt.numel(), bits) for xt in (xa, xb) for bits in WIDTHS)
    ms = _time_launch(graph.replay, flush, reps=5, warm=1) / 10
    row("dbca_step_16_calls_graph", step_bytes,
        sum(2 * xt.numel() for xt in (xa, xb) for _ in WIDTHS), ms,
        {"calls_per_step": 16, "steps_per_graph": 10, "stream": "one"})
    del graph, xin, cod, sca, out, xa, xb

    # SiLU backward recomputed from the 4-bit SiLU input (8192 x 11008)
    xs_ = synthetic.dbca_activations_torch(seed=1, device=device)[1]
    n = xs_.numel()
    c, s = agoq.agoq_quant_act(xs_, 4)
    del xs_
    dy = torch.randn(n, device=device).to(torch.bfloat16)
    dx = torch.empty_like(dy)
    y = torch.empty_like(dy)
    base = n * 4 // 8 + (n // 128) * 4 + 2 * n + 2 * n
    row("silu_backward_b4_8192x11008", base, n,
        _time_launch(lambda: agoq.agoq_silu_backward(c, s, dy, n, 4, dx), flush))
    row("silu_backward_b4_with_forward_8192x11008", base + 2 * n, n,
        _time_launch(lambda: agoq.agoq_silu_backward(c, s, dy, n, 4, dx, y), flush))
    del c, s, dy, dx, y

    # RMSNorm backward recomputed from the 4-bit RMSNorm input (8192 x 4096)
    T, H = synthetic.DBCA_RMSNORM_SHAPE
    xr = synthetic.dbca_activations_torch(seed=1, device=device)[0]
    c, s = agoq.agoq_quant_act(xr, 4)
    del xr
    dy = torch.randn(T * H, device=device).to(torch.bfloat16)
    wt = (1 + 0.1 * torch.randn(H, device=device)).to(torch.bfloat16)
    dx = torch.empty((T, H), dtype=torch.bfloat16, device=device)
    rstd = torch.empty(T, dtype=torch.float32, device=device)
    dwt = torch.empty(H, dtype=torch.float32, device=device)
    n = T * H
    base = n * 4 // 8 + (n // 128) * 4 + 2 * n + 2 * n + 2 * H + 4 * T
    row("rmsnorm_backward_dx_b4_8192x4096", base, n,
        _time_launch(lambda: agoq.agoq_rmsnorm_backward(c, s, dy, wt, T, H, 4, 1e-6, dx, rstd,
                                                        want_dw=False), flush))
    row("rmsnorm_backward_dx_dw_b4_8192x4096", base + 4 * H, n,
        _time_launch(lambda: agoq.agoq_rmsnorm_backward(c, s, dy, wt, T, H, 4, 1e-6, dx, rstd,
                                                        dwt), flush),
        {"note": "algorithmic bytes read the input once; dw reads codes and dy a second time"})
    ws = torch.empty(agoq.agoq_rmsnorm_backward_workspace_bytes(H), dtype=torch.uint8,
                     device=device)
    row("rmsnorm_backward_dx_dw_single_read_b4_8192x4096", base + 4 * H, n,
        _time_launch(lambda: agoq.agoq_rmsnorm_backward_ws(c, s, dy, wt, T, H, 4, 1e-6, ws, dx,
                                                           rstd, dwt), flush),
        {"note": "one read of the input; dw from per-CTA partial sums in a workspace",
         "workspace_bytes": ws.numel()})
    del c, s, dy, dx, ws

    # QuanGrad accumulation, 2^30 elements: the 8 micro-batches of the workload
    # into a zeroed master, each step timed after an L2 flush; the chain is run
    # 3 times from zero, and each step's median and the mean over steps reported
    n = synthetic.QUANGRAD_N
    m = torch.zeros(n, dtype=torch.uint8, device=device)
    ms_ = torch.zeros(n // 128, dtype=torch.float32, device=device)
    grads = [synthetic.quangrad_grad_torch(seed=2, step=k, device=device)
             for k in range(synthetic.QUANGRAD_STEPS)]
    nbytes = n * 4 + (n // 128) * 8
    def chain(acc, label, extra_note=""):
        acc(grads[0])   # warm-up
        step_ms = [[] for _ in grads]
        for _ in range(3):
            m.zero_()
            ms_.zero_()
            for k, g in enumerate(grads):
                flush()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                acc(g)
                b.record()
                b.synchronize()
                step_ms[k].append(a.elapsed_time(b))
        med = [statistics.median(t) for t in step_ms]
        row(label, nbytes, n, sum(med) / len(med),
            {"steps": len(med), "per_step_us": [round(t * 1e3, 1) for t in med],
             "timing": "mean over the 8 micro-batches of each step's median of 3 chains from a "
                       "zeroed master" + extra_note})

    chain(lambda g: agoq.agoq_grad_accum_fp8(m, ms_, g), "quangrad_accum_2^30")
    for mid, label in ((agoq.MID_BF16, "bf16"), (agoq.MID_FP16, "fp16")):
        chain(lambda g, mid=mid: agoq.agoq_grad_accum_fp8_mid(m, ms_, g, mid),
              "quangrad_accum_%smid_2^30" % label)
    del m, ms_, grads

    # FP8 shard local reduce, 2^25 elements per shard
    n = synthetic.REDUCE_N
    for W in synthetic.REDUCE_WS:
        sh, ss = reduce_shards_torch(W, n, device)
        out = torch.empty(n, dtype=torch.uint8, device=device)
        outs = torch.empty(n // 128, dtype=torch.float32, device=device)
        cnt = torch.zeros(1, dtype=torch.int64, device=device)
        nbytes = (W + 1) * (n + (n // 128) * 4)
        ms = _time_launch(lambda: agoq.agoq_reduce_fp8_shards(sh, ss, W, n, out, outs, cnt), flush)
        row("reduce_W%d_2^25" % W, nbytes, W * n, ms,
            {"naive_overflow_count": int(cnt.item()),
             "inputs": "shard r ~ N(0, sd 1e-2 j_r), j_r ~ U[0.5,2), seed 3 (torch generator), "
                       "block-quantized to E4M3 by the library (absmax/448)"})
        row("reduce_W%d_2^25_nocount" % W, nbytes, W * n,
            _time_launch(lambda: agoq.agoq_reduce_fp8_shards(sh, ss, W, n, out, outs), flush))
        del sh, ss, out, outs

    # INT4-dequant-fused weight-gradient GEMM
    M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
    dy, xg = synthetic.wgrad_inputs_torch(seed=4, device=device)
    xc, xs = agoq.agoq_quant_act(xg, 4)
    dw = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    try:
        ms = _time_launch(lambda: agoq.agoq_wgrad_gemm_int4(dy, xc, xs, M, N, K, dw), flush)
        agoq.agoq_device_status()
        tflops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        rows["wgrad_gemm_int4_11008x4096x8192"] = {
            "us": round(ms * 1e3, 1), "TFLOP/s": round(tflops, 1),
            "frac_of_measured_bf16": round(tflops / bf16_peak, 4),
            "bytes": 2 * K * M + K * N // 2 + K * (N // 128) * 4 + 2 * M * N}
        xh = agoq.agoq_dequant_act(xc, xs, K * N, 4).view(K, N)
        ref_ms = _time_launch(lambda: torch.matmul(dy.t(), xh, out=dw), flush)
        rows["wgrad_gemm_int4_11008x4096x8192"]["torch_matmul_bf16_predequantized_us"] = round(ref_ms * 1e3, 1)
    except agoq.AgoqError as e:
        rows["wgrad_gemm_int4_11008x4096x8192"] = {"unavailable": str(e)}

    # Forward GEMM (LLaMA-7B gate projection, 8192 x 4096 -> 11008) with the 4-bit
    # LAAQ quantization of its output fused; beside it the unfused sequence
    # (cuBLAS BF16 matmul, then the quantizer) and cuBLAS alone
    Tf, Kf, Nf = 8192, 4096, 11008
    xf = torch.randn(Tf, Kf, device=device).to(torch.bfloat16)
    wf = (torch.randn(Nf, Kf, device=device) * 0.02).to(torch.bfloat16)
    yf = torch.empty(Tf, Nf, dtype=torch.bfloat16, device=device)
    cf = torch.empty(Tf * Nf // 128 * 64, dtype=torch.uint8, device=device)
    sf = torch.empty(Tf * Nf // 128, dtype=torch.float32, device=device)
    name = "fwd_gemm_quant_b4_8192x4096x11008"
    try:
        ms = _time_launch(lambda: agoq.agoq_fwd_gemm_quant(xf, wf, Tf, Nf, Kf, 4, yf, cf, sf), flush)
        agoq.agoq_device_status()
        tflops = 2.0 * Tf * Nf * Kf / (ms * 1e-3) / 1e12
        rows[name] = {"us": round(ms * 1e3, 1), "TFLOP/s": round(tflops, 1),
                      "frac_of_measured_bf16": round(tflops / bf16_peak, 4)}
        rows[name]["cublas_matmul_then_quant_us"] = round(_time_launch(
            lambda: (torch.matmul(xf, wf.t(), out=yf), agoq.agoq_quant_act(yf, 4, cf, sf)),
            flush) * 1e3, 1)
        rows[name]["cublas_matmul_alone_us"] = round(_time_launch(
            lambda: torch.matmul(xf, wf.t(), out=yf), flush) * 1e3, 1)
    except agoq.AgoqError as e:
        rows[name] = {"unavailable": str(e)}
    del xf, wf, yf, cf, sf

    # The same GEMM with the QuanGrad accumulation into an FP8 master as its epilogue
    master = torch.zeros(M * N, dtype=torch.uint8, device=device)
    mscales = torch.zeros(M * N // 128, dtype=torch.float32, device=device)
    agoq.agoq_grad_accum_fp8(master, mscales, dw.view(-1))
    name = "wgrad_gemm_int4_accum_fp8_11008x4096x8192"
    try:
        ms = _time_launch(lambda: agoq.agoq_wgrad_gemm_int4_accum_fp8(dy, xc, xs, M, N, K, master,
                                                                      mscales), flush)
        agoq.agoq_device_status()
        tflops = 2.0 * M * N * K / (ms * 1e-3) / 1e12
        rows[name] = {
            "us": round(ms * 1e3, 1), "TFLOP/s": round(tflops, 1),
            "frac_of_measured_bf16": round(tflops / bf16_peak, 4),
            "bytes": 2 * K * M + K * N // 2 + K * (N // 128) * 4 + 2 * (M * N + M * (N // 128) * 4),
            "vs_gemm_then_accum_us": None}
        # the unfused sequence it replaces: BF16 dW, then the element-wise accumulation
        def unfused():
            agoq.agoq_wgrad_gemm_int4(dy, xc, xs, M, N, K, dw)
            agoq.agoq_grad_accum_fp8(master, mscales, dw.view(-1))
        rows[name]["vs_gemm_then_accum_us"] = round(_time_launch(unfused, flush) * 1e3, 1)
    except agoq.AgoqError as e:
        rows[name] = {"unavailable": str(e)}
    return rows


# ----------------------------------------------------------------------- CPU oracle
def _oracle_step(O, a, b, parallel=False):
    for x in (a, b):
        flat = x.reshape(-1)
        for bits in WIDTHS:
            c, s = O.quant_act(flat, bits, parallel=parallel)
            O.dequant_act(c, s, flat.size, bits, parallel=parallel)


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), or None."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return None


def cpu_sample(target_s, parallel=False):
    """The workload restricted to its first R token rows, R chosen for about
    target_s of oracle work (all 8192 rows if they fit)."""
    from gradient_quantization_gb300 import synthetic
    from oracle import oracle as O
    O.lib(parallel)
    rows = 64 if parallel else 16
    a, b = synthetic.dbca_activations_np(seed=1, tokens=rows)
    t0 = time.perf_counter()
    _oracle_step(O, a, b, parallel)
    dt = time.perf_counter() - t0
    rows = int(max(16, min(8192, rows * target_s / max(dt, 1e-6))))
    a, b = synthetic.dbca_activations_np(seed=1, tokens=rows)
    nbytes = sum(2 * act_bytes(x.size, bits) for x in (a, b) for bits in WIDTHS)
    nelems = sum(2 * x.size for x in (a, b) for _ in WIDTHS)
    return O, a, b, rows, nbytes, nelems


def _cpu_leg(target_s, parallel):
    O, a, b, rows, nbytes, nelems = cpu_sample(target_s, parallel)
    t0 = time.perf_counter()
    _oracle_step(O, a, b, parallel)
    dt = time.perf_counter() - t0
    what = ("all 8192 token rows" if rows == 8192 else "first %d of 8192 token rows" % rows)
    return {"value": round(nbytes / dt / 1e9, 4), "unit": "GB/s", "cores": O.threads(parallel),
            "kind": "oracle", "gelem_per_s": round(nelems / dt / 1e9, 5), "seconds": round(dt, 2),
            "sample": "%s of both tensors, quantize+dequantize at 4/5/6/8 bits (%s C oracle)"
                      % (what, "all-core OpenMP" if parallel else "single-threaded")}


def cpu_baseline(target_s):
    """The oracle on the host cores: the all-core build (the line's value) and the
    single-threaded build, each on a sample sized for about target_s."""
    from oracle import oracle as O
    single = _cpu_leg(target_s / 2, False)
    if O.parallel_available():
        line = _cpu_leg(target_s / 2, True)
        line["single_thread"] = single
    else:
        line = single
    line["cpu_model"] = cpu_model()
    line["host_cores"] = len(os.sched_getaffinity(0))
    return line


def oracle_rows(device):
    """The all-core oracle on the other workloads, each at full size or on a
    stated sample (a reported baseline, like the step's): the 2048x4096 4-bit
    round trip, one QuanGrad step of 2^30 elements, the shard reduce with its
    count (W=8 at 2^25, W=64 on 2^22 elements per shard) and the binary64
    weight-gradient product on the first 16 rows of dW.  The inputs for the
    larger ones are drawn and quantized on the GPU and copied to the host."""
    import numpy as np
    import torch
    from gradient_quantization_gb300 import agoq, synthetic
    from oracle import oracle as O
    par = True
    rows = {}

    def timed(fn):
        t0 = time.perf_counter()
        out = fn()
        return time.perf_counter() - t0, out

    def host_u16(t):
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    x = synthetic.laaq_activation_np(seed=0).reshape(-1)
    n = x.size
    dt, (c, sc) = timed(lambda: O.quant_act(x, 4, parallel=par))
    rows["laaq_int4_quant_2048x4096"] = {"us": round(dt * 1e6, 1),
                                         "GB/s": round(act_bytes(n, 4) / dt / 1e9, 3),
                                         "Gelem/s": round(n / dt / 1e9, 4), "sample": "full size"}
    dt, _ = timed(lambda: O.dequant_act(c, sc, n, 4, parallel=par))
    rows["laaq_int4_dequant_2048x4096"] = {"us": round(dt * 1e6, 1),
                                           "GB/s": round(act_bytes(n, 4) / dt / 1e9, 3),
                                           "Gelem/s": round(n / dt / 1e9, 4), "sample": "full size"}
    del x, c, sc

    nq = synthetic.QUANGRAD_N
    g = host_u16(synthetic.quangrad_grad_torch(seed=2, step=0, device=device))
    m = np.zeros(nq, np.uint8)
    ms = np.zeros(nq // 128, np.float32)
    dt, _ = timed(lambda: O.grad_accum_fp8(m, ms, g, parallel=par, in_place=True))
    nbytes = nq * 4 + (nq // 128) * 8
    rows["quangrad_accum_2^30"] = {"us": round(dt * 1e6, 1), "GB/s": round(nbytes / dt / 1e9, 3),
                                   "Gelem/s": round(nq / dt / 1e9, 4),
                                   "sample": "one step (micro-batch 0 onto a zeroed master), full size"}
    del g, m, ms

    for W, nr in ((8, synthetic.REDUCE_N), (64, 1 << 22)):
        sh, ss = reduce_shards_torch(W, nr, device)
        shh, ssh = sh.cpu().numpy(), ss.cpu().numpy()
        del sh, ss
        dt, _ = timed(lambda: O.reduce_fp8_shards(shh, ssh, W, nr, count_naive=True, parallel=par))
        nbytes = (W + 1) * (nr + (nr // 128) * 4)
        rows["reduce_W%d_count" % W] = {
            "us": round(dt * 1e6, 1), "GB/s": round(nbytes / dt / 1e9, 3),
            "Gelem/s": round(W * nr / dt / 1e9, 4),
            "sample": "full size (2^25 per shard)" if nr == synthetic.REDUCE_N
                      else "2^22 elements per shard (the workload has 2^25)"}
        del shh, ssh

    M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
    dy, xg = synthetic.wgrad_inputs_torch(seed=4, device=device)
    xc, xs = agoq.agoq_quant_act(xg, 4)
    dyh, xch, xsh = host_u16(dy), xc.cpu().numpy(), xs.cpu().numpy()
    del dy, xg, xc, xs
    nr = 16
    r = np.repeat(np.arange(nr, dtype=np.int32), N)
    cc = np.tile(np.arange(N, dtype=np.int32), nr)
    dt, _ = timed(lambda: O.wgrad_gemm_int4_f64_entries(dyh, xch, xsh, M, N, K, r, cc,
                                                         parallel=par))
    rows["wgrad_gemm_int4_f64"] = {"us": round(dt * 1e6, 1),
                                   "GFLOP/s": round(2.0 * nr * N * K / dt / 1e9, 3),
                                   "sample": "the first %d of %d rows of dW (binary64 sums)" % (nr, M)}
    torch.cuda.synchronize()
    return rows


def reference_arm(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from oracle import oracle as O
    parallel = O.parallel_available()
    # keep the whole reference run within about three minutes of host time
    per_step = min(args.ref_step_seconds, 180.0 / (args.steps + args.warmup))
    O, a, b, rows, nbytes, nelems = cpu_sample(per_step, parallel)
    for _ in range(args.warmup):
        _oracle_step(O, a, b, parallel)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(O, a, b, parallel)
    dt = time.perf_counter() - t0
    value = nbytes * args.steps / dt / 1e9
    cores = O.threads(parallel)
    what = ("all 8192 token rows" if rows == 8192 else "first %d of 8192 token rows" % rows)
    sample = ("%s of both tensors per step, quantize+dequantize at 4/5/6/8 bits (%s C oracle)"
              % (what, "all-core OpenMP" if parallel else "single-threaded"))
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "gelem_per_s": round(nelems * args.steps / dt / 1e9, 5),
            "config": {"workload": "DBCA-PP activations: RMSNorm in BF16[8192x4096] + SiLU in "
                                   "BF16[8192x11008], Student-t nu=4, quantize+dequantize at 4/5/6/8 bits",
                       "sample_rows": rows, "parallelism": "%d host threads" % cores},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": sample, "cpu_model": cpu_model()},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def reduce_shards_torch(W, n, device):
    """The FP8 shard workload: shard r holds N(0, sd 1e-2 * j_r) values, j_r ~ U[0.5, 2)
    (seed 3, torch generator), block-quantized to E4M3 by the library's own
    accumulation into a zeroed master (the a4 requantization rule)."""
    import torch
    from gradient_quantization_gb300 import agoq, synthetic
    vals = synthetic.reduce_shard_values_torch(seed=3, W=W, device=device, n=n)
    sh = torch.zeros((W, n), dtype=torch.uint8, device=device)
    ss = torch.zeros((W, n // 128), dtype=torch.float32, device=device)
    for r in range(W):
        agoq.agoq_grad_accum_fp8(sh[r], ss[r], vals[r])
    del vals
    torch.cuda.synchronize()
    return sh, ss


PROFILE_CASES = ("accum", "reduce8", "reduce8_nocount", "reduce64", "gemm", "gemm_accum", "silu",
                 "rmsnorm", "rmsnorm_ws", "fwd_gemm", "laaq4_small", "dequant4_silu",
                 "dequant8_silu", "quant5_dbca")


def profile_case(name, launches=3):
    """Launch one kernel of the path a few times on a mid-size workload (for
    ncu captures: a few hundred MB on the device, no timing output)."""
    import torch
    from gradient_quantization_gb300 import agoq, synthetic
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    if name == "accum":
        n = 1 << 28
        m = torch.zeros(n, dtype=torch.uint8, device=dev)
        ms = torch.zeros(n // 128, dtype=torch.float32, device=dev)
        g = synthetic.quangrad_grad_torch(seed=2, step=0, device=dev, n=n)
        for _ in range(launches):
            agoq.agoq_grad_accum_fp8(m, ms, g)
    elif name.startswith("reduce"):
        W, n = (64, 1 << 22) if name == "reduce64" else (8, 1 << 25)
        sh, ss = reduce_shards_torch(W, n, dev)
        cnt = None if name.endswith("nocount") else torch.zeros(1, dtype=torch.int64, device=dev)
        for _ in range(launches):
            agoq.agoq_reduce_fp8_shards(sh, ss, W, n, naive_overflow_count=cnt)
    elif name in ("gemm", "gemm_accum"):
        M, N, K = synthetic.WGRAD_M, synthetic.WGRAD_N, synthetic.WGRAD_K
        dy, xg = synthetic.wgrad_inputs_torch(seed=4, device=dev)
        xc, xs = agoq.agoq_quant_act(xg, 4)
        master = torch.zeros(M * N, dtype=torch.uint8, device=dev)
        mscales = torch.zeros(M * N // 128, dtype=torch.float32, device=dev)
        for _ in range(launches):
            if name == "gemm":
                agoq.agoq_wgrad_gemm_int4(dy, xc, xs, M, N, K)
            else:
                agoq.agoq_wgrad_gemm_int4_accum_fp8(dy, xc, xs, M, N, K, master, mscales)
        agoq.agoq_device_status()
    elif name == "fwd_gemm":
        T, K, N = 8192, 4096, 11008
        x = torch.randn(T, K, device=dev).to(torch.bfloat16)
        w = (torch.randn(N, K, device=dev) * 0.02).to(torch.bfloat16)
        for _ in range(launches):
            agoq.agoq_fwd_gemm_quant(x, w, T, N, K, 4)
        agoq.agoq_device_status()
    elif name == "silu":
        x = synthetic.dbca_activations_torch(seed=1, device=dev)[1]
        n = x.numel()
        c, s = agoq.agoq_quant_act(x, 4)
        dy = torch.randn(n, device=dev).to(torch.bfloat16)
        for _ in range(launches):
            agoq.agoq_silu_backward(c, s, dy, n, 4)
    elif name in ("rmsnorm", "rmsnorm_ws"):
        x = synthetic.dbca_activations_torch(seed=1, device=dev)[0]
        T, H = x.shape
        c, s = agoq.agoq_quant_act(x, 4)
        dy = torch.randn(T * H, device=dev).to(torch.bfloat16)
        w = torch.ones(H, device=dev).to(torch.bfloat16)
        ws = torch.empty(agoq.agoq_rmsnorm_backward_workspace_bytes(H), dtype=torch.uint8,
                         device=dev)
        for _ in range(launches):
            if name == "rmsnorm":
                agoq.agoq_rmsnorm_backward(c, s, dy, w, T, H, 4, 1e-6)
            else:
                agoq.agoq_rmsnorm_backward_ws(c, s, dy, w, T, H, 4, 1e-6, ws)
    elif name in ("dequant4_silu", "dequant8_silu"):
        # the SiLU/gate input of the DBCA-PP step, quantized once, then dequantized
        bits = 4 if name == "dequant4_silu" else 8
        x = synthetic.dbca_activations_torch(seed=1, device=dev)[1]
        c, s = agoq.agoq_quant_act(x, bits)
        y = torch.empty_like(x)
        for _ in range(launches):
            agoq.agoq_dequant_act(c, s, x.numel(), bits, y)
    elif name == "quant5_dbca":
        # both DBCA-PP tensors quantized at 5 bits (RMSNorm input, then SiLU input)
        for x in synthetic.dbca_activations_torch(seed=1, device=dev):
            for _ in range(launches):
                agoq.agoq_quant_act(x, 5)
    elif name == "laaq4_small":
        # the 2048 x 4096 4-bit round trip (one activation, 21 MB a call)
        x = synthetic.laaq_activation_torch(seed=0, device=dev)
        for _ in range(launches):
            c, s = agoq.agoq_quant_act(x, 4)
            agoq.agoq_dequant_act(c, s, x.numel(), 4)
    else:
        raise SystemExit("unknown profile case %r (choose from %s)" % (name, ", ".join(PROFILE_CASES)))
    torch.cuda.synchronize()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    ap.add_argument("--no-rows", action="store_true", help="skip the other rows of the path")
    ap.add_argument("--streams", type=int, choices=(1, 2), default=2,
                    help="streams the step's calls are spread over (widths split between them)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU seconds of the oracle baseline sample")
    ap.add_argument("--ref-step-seconds", type=float, default=4.0,
                    help="target seconds of one reference-arm step")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="only launch one kernel a few times on a mid-size workload (for ncu)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)     # at least 3 untimed warm-up steps
    args.steps = max(1, args.steps)
    if args.profile_case:
        profile_case(args.profile_case)
    elif args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
