#!/usr/bin/env python
"""Benchmark of the integer-only (NITI) training step on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload INDEX]

Default workload: the large integer MLP (batch 8192, Linear 4096->4096 x4 +
ReLU, Linear 4096->1000), one full forward / delta propagation / weight
gradient / NITI update per step, seeded synthetic int8 data.

Prints one JSON line (rank 0). `value` is training samples/s of the whole job
(every rank runs its own replica: the step has no cross-GPU exchange here).
Device time per step is taken with CUDA events on the step's stream, with L2
flushed (a 256 MB write) before every timed step and the flush left out of the
timing; `ms_per_step` is the median over five loops of K steps. `roofline` is
the tensor-core contraction class timed with events around each of its
launches (the same steps run again), against the measured burst bf16 peak;
`e2e` is the same metric through the host-buffer C-ABI calls (input copy, step,
stats copy); `cpu_baseline` is the CPU oracle on a bounded sample of the same
workload. With one GPU, `workloads` adds the other seeded workloads (default
0, 1, 2 and 4), each timed the same way in the same process, with its
contraction fraction, nonzero weight updates and CPU-oracle rate.

--impl reference runs the CPU oracle (the reference of this build: the pages
publish no implementation) on the same workload, a bounded batch slice per
step, and prints the same line with "impl": "reference".
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "integer training samples/s and INT8 TOPS (% of dense INT8 peak), bit-exact"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

NB_BATCHES = 8   # distinct resident input batches the model workload cycles through

OVERLAP_MODES = {0: "off: every launch on one stream",
                 1: "delta requantisation and updates on a second stream beside the contractions",
                 2: "weight and offset updates on a second stream beside the contractions"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK), "fallback"


TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "k_gemm_tc2__dram_per_launch__ops_8192x4096x4096.md")
GEMM_SOURCES = [os.path.join(ROOT, "integer_only_nn_gb300", "csrc", f) for f in ("ito_gemm.cu", "ito_device.cuh")]


def gemm_traffic_per_launch(w):
    """DRAM bytes per contraction launch from the committed ncu summary, or
    None when the summary is for another workload or the kernel source has
    changed since the counters were taken."""
    import hashlib
    if w.name != "mlp4096x4-1000_b8192":
        return None
    try:
        text = open(TRAFFIC_PROFILE).read()
        h = hashlib.sha256(b"".join(open(f, "rb").read() for f in GEMM_SOURCES)).hexdigest()[:16]
    except OSError:
        return None
    fields = dict(line.split(": ", 1) for line in text.splitlines() if ": " in line and line[:1].isalpha())
    if fields.get("kernel_source_sha256_16", "").strip() != h:
        return None
    try:
        return float(fields["dram_bytes_per_launch_avg"])
    except (KeyError, ValueError):
        return None


def algorithmic_ops(w):
    """Integer ops (2 per multiply-accumulate) of one training step: forward,
    weight gradient and delta propagation (not for the first layer). For the
    DFP16 workload these are int16 multiply-accumulates; its tensor cores
    execute four bf16 limb products for each."""
    B = w.batch
    if w.kind in ("mlp", "dfp16"):
        d = w.dims
        fwd = sum(d[i] * d[i + 1] for i in range(len(d) - 1))
        dgrad = sum(d[i] * d[i + 1] for i in range(1, len(d) - 1))
        return 2.0 * B * (2 * fwd + dgrad)
    H, W, _ = w.image
    fwd = dgrad = 0
    for l, (ic, oc, s) in enumerate(w.convs):
        H, W = (H + 2 - 3) // s + 1, (W + 2 - 3) // s + 1
        macs = B * H * W * oc * 9 * ic
        fwd += macs
        dgrad += macs if l > 0 else 0
    fc = B * w.fc[0] * w.fc[1]
    return 2.0 * (2 * (fwd + fc) + dgrad + fc)


def max_over_ranks(value, dist, device="cuda"):
    """The largest `value` over all ranks (the slowest rank's time); the value
    itself when running alone."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(samples_per_rank, world, slowest_seconds):
    """Whole-job samples/s: every rank's samples over the slowest rank's time."""
    return samples_per_rank * world / slowest_seconds


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "ito_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        with open(self.path) as f:
            for line in f:
                p = [t.strip() for t in line.split(",")]
                if len(p) < 9:
                    continue
                try:
                    sm.append(float(p[1]))
                    smax.append(float(p[2]))
                except ValueError:
                    continue
                for n, v in zip(names, p[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def oracle_step(w, weights, x, labels):
    """One CPU-oracle training step (plain C loops) of workload w."""
    import oracle as O
    if w.kind == "mlp":
        return O.mlp_step(weights, x, labels, route="loops")
    if w.kind == "cnn":
        return O.cnn_step(weights, x, labels, w.convs)
    if w.apt is not None:
        # the first step of an adaptive-precision run: weights at the initial precision
        ws, ew = [], []
        for W in weights:
            Wk, de = O.dfp_set_bits(W, 16, w.apt.k_init)
            ws.append(Wk)
            ew.append(w.exp_w + de)
        return O.dfp16_step(ws, ew, x, w.exp_x, eta=w.eta, route="loops", wbits=[w.apt.k_init] * len(ws))
    return O.dfp16_step(weights, w.exp_w, x, w.exp_x, eta=w.eta, route="loops")


def cpu_baseline(w, sample_batch, min_seconds=10.0, single_seconds=3.0):
    """The CPU oracle (plain C loops, OpenMP over output rows) on training steps of
    `sample_batch` samples of workload w, repeated for about min_seconds with every
    host core, then (unless single_seconds is None) for about single_seconds on one
    thread (a smaller slice)."""
    import numpy as np
    import oracle as O
    import seeded_inputs as si
    O.build()
    weights = si.make_weights(w)
    x, labels = si.make_batch(w, 0)

    def timed(n, seconds):
        xs = np.ascontiguousarray(x[:n])
        ls = None if labels is None else np.ascontiguousarray(labels[:n])
        # the same step repeated (the loops' cost does not depend on the values)
        steps = 0
        t0 = time.perf_counter()
        while True:
            oracle_step(w, weights, xs, ls)
            steps += 1
            dt = time.perf_counter() - t0
            if dt >= seconds:
                return steps * n / dt, dt, steps

    sample_batch = min(sample_batch, w.batch)
    cores = O.max_threads()
    value, dt, steps = timed(sample_batch, min_seconds)
    if single_seconds is None:
        return value, dt, cores, steps, sample_batch, None
    O.set_threads(1)
    try:
        n1 = max(1, min(sample_batch, sample_batch // 8))
        v1, dt1, steps1 = timed(n1, single_seconds)
    finally:
        O.set_threads(cores)
    single = {"value": v1, "cores": 1,
              "sample": "%d steps on %d samples, %.1f s" % (steps1, n1, dt1)}
    return value, dt, cores, steps, sample_batch, single


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    import numpy as np
    import oracle as O
    import seeded_inputs as si
    O.build()
    sample = args.ref_batch
    weights = si.make_weights(w)
    batches = []
    for t in range(2):
        x, labels = si.make_batch(w, t)
        batches.append((np.ascontiguousarray(x[:sample]),
                        None if labels is None else np.ascontiguousarray(labels[:sample])))
    for i in range(args.warmup):
        x, lab = batches[i % 2]
        oracle_step(w, weights, x, lab)
    t0 = time.perf_counter()
    for i in range(args.steps):
        x, lab = batches[i % 2]
        rec = oracle_step(w, weights, x, lab)
        weights = [rec["w%d" % l] for l in range(len(weights))]
    dt = time.perf_counter() - t0
    value = sample * args.steps / dt
    cores = O.max_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dims": list(w.dims),
                   "reference_step_batch": sample},
        "cpu_baseline": {"value": value, "unit": "samples/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: one oracle training step on %d of the %d samples" % (sample, w.batch)},
        "e2e": {"value": value, "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "int_tops": algorithmic_ops(w) * sample / w.batch * args.steps / dt / 1e12,
    }
    print(json.dumps(line), flush=True)
    return 0


REPEATS = 5   # timed loops of K steps; the reported step time is their median


def timed_median(K, repeats, stream, flush, before, step):
    """Device ms per step: the median over `repeats` loops of K steps. Each step
    runs after an untimed L2 flush and `before(k)`, between CUDA events on
    `stream`. Returns (median, per-loop list)."""
    import torch
    per = []
    for _ in range(repeats):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        with torch.cuda.stream(stream):
            for k in range(K):
                flush.fill_(k & 0xFF)
                before(k)
                starts[k].record(stream)
                step(k)
                ends[k].record(stream)
        torch.cuda.synchronize()
        per.append(sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K)
    return statistics.median(per), per


def profiled_steps(model, K, stream, flush, before, step, classes):
    """The same steps again with an event pair around every launch (on the
    launch's own stream): {class: [ms, work, launches]} summed over K steps, and
    the device ms per step with those events."""
    import torch
    model.profile(True)
    for i in range(4):
        with torch.cuda.stream(stream):
            before(i)
        step(i)
    model.profile_read()
    prof = {c: [0.0, 0.0, 0] for c in classes}
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for k in range(K):
            flush.fill_(k & 0xFF)
            before(k)
            starts[k].record(stream)
            step(k)
            ends[k].record(stream)
            for c, (ms, work, n) in model.profile_read().items():
                prof[c][0] += ms
                prof[c][1] += work
                prof[c][2] += n
    torch.cuda.synchronize()
    model.profile(False)
    return prof, sum(s.elapsed_time(e) for s, e in zip(starts, ends)) / K


class ModelRun:
    """An ito_model of an int8 workload with NB_BATCHES seeded batches resident
    in HBM; before each step (untimed) the step's batch is copied into the
    model's fixed input buffers, which the captured step graphs read."""

    def __init__(self, w, graphs=True):
        import torch
        import integer_only_nn_gb300 as ito
        import seeded_inputs as si
        self.w = w
        self.stream = torch.cuda.Stream()   # a side stream, so that steps can replay from graphs
        self.model = ito.Model(ito.layers_for(w), w.batch)
        for l, W in enumerate(si.make_weights(w)):
            self.model.set_weights(l, W, stream=self.stream)
        self.model.use_graphs(graphs)
        self.xs, self.ls = [], []
        for t in range(NB_BATCHES):
            x, labels = si.make_batch(w, t)
            self.xs.append(torch.from_numpy(x).cuda())
            self.ls.append(torch.from_numpy(labels).cuda())
        self.xbuf, self.lbuf = torch.empty_like(self.xs[0]), torch.empty_like(self.ls[0])
        torch.cuda.synchronize()

    def before(self, k):
        self.xbuf.copy_(self.xs[k % NB_BATCHES])
        self.lbuf.copy_(self.ls[k % NB_BATCHES])

    def step(self, k):
        self.model.train_step(self.xbuf, self.lbuf, stream=self.stream)

    def warm(self, n):
        import torch
        for i in range(n):
            with torch.cuda.stream(self.stream):
                self.before(i)
            self.step(i)
        self.stream.synchronize()

    def nonzero_updates(self):
        st = self.model.stats()
        per = [st["nz%d" % l] for l in range(len(self.model_layers()))]
        return sum(per), per

    def model_layers(self):
        l = 0
        while self.model.stat_index("nz%d" % l) >= 0:
            l += 1
        return range(l)


class DfpRun:
    """An ito_dfp16_model with two seeded input batches resident in HBM,
    alternating; with adaptive precision the epoch-end adjustment (a host
    synchronisation) runs inside the step that ends an epoch."""

    def __init__(self, w):
        import torch
        import integer_only_nn_gb300 as ito
        import seeded_inputs as si
        self.w = w
        self.stream = torch.cuda.current_stream()
        self.model = ito.Dfp16Model(list(w.dims), w.batch, w.exp_w, w.eta)
        for l, W in enumerate(si.make_weights(w)):
            self.model.set_weights(l, W)
        self.xs = [torch.from_numpy(si.make_batch(w, t)[0]).cuda() for t in range(2)]
        a = w.apt
        if a is not None:
            self.model.apt_enable(a.k_init, a.k_min, a.k_max, a.t_min, a.t_max, a.eval_every)
        self.step_no = 0
        torch.cuda.synchronize()

    def before(self, k):
        pass

    def _epoch_end(self):
        a = self.w.apt
        if a is not None and self.step_no % a.epoch == a.epoch - 1:
            self.model.apt_epoch_end()
        self.step_no += 1

    def step(self, k):
        self.model.train_step(self.xs[k % 2], self.w.exp_x)
        self._epoch_end()

    def step_host_async(self, xh, st_h):
        self.model.train_step_host_async(xh, self.w.exp_x, st_h)
        self._epoch_end()

    def warm(self, n):
        import torch
        for i in range(n):
            self.step(i)
        torch.cuda.synchronize()

    def nonzero_updates(self):
        st = self.model.stats()
        per = [int(st["nz%d" % l]) for l in range(self.model.n_layers)]
        return sum(per), per


def rate(entry, unit):
    """work / time of a profiled class [ms, work, launches] in `unit` per second
    (None when the class had no launches)."""
    ms, work, _ = entry
    return work / (ms / 1000.0) / unit if ms > 0 else None


def gemm_roofline(prof, pk, pk_src):
    """Contraction rate over the profiled launches against the measured burst
    bf16 peak (the contraction launches are timed inside steps of a few ms, not
    a seconds-long loop); the sustained figure beside it."""
    g_ms, g_work, g_n = prof["gemm"]
    achieved = g_work / (g_ms / 1000.0) / 1e12
    burst, sust = float(pk["bf16_tflops"]), float(pk["bf16_tflops_sustained"])
    return {"bound": "tensor", "achieved": achieved, "peak": burst, "unit": "TFLOP/s", "frac": achieved / burst,
            "peak_source": "bf16_tflops (burst), %s" % pk_src, "peak_sustained": sust,
            "frac_of_sustained": achieved / sust, "launches_timed": g_n}


def workload_entry(w, args, flush, pk, pk_src, cpu):
    """Step time, throughput, contraction roofline fraction and nonzero weight
    updates of one more workload, timed in the same process as the headline."""
    run = DfpRun(w) if w.kind == "dfp16" else ModelRun(w, graphs=not args.no_graphs)
    K = args.steps
    run.warm(args.warmup)
    ms, per = timed_median(K, REPEATS, run.stream, flush, run.before, run.step)
    nz, nz_per = run.nonzero_updates()
    classes = ("gemm", "down", "update", "other") if w.kind == "dfp16" else ("gemm", "requant", "update", "other")
    # per-launch events in a mode where no two contractions share SMs (see run_ours_model)
    mode = run.model.overlap() if w.kind != "dfp16" else None
    if mode == 3:
        run.model.set_overlap(0)
    prof, prof_ms = profiled_steps(run.model, K, run.stream, flush, run.before, run.step, classes)
    if mode == 3:
        run.model.set_overlap(mode)
    ops = algorithmic_ops(w)
    kernels = run.model.kernels_per_step()
    e = {"batch": w.batch, "ms_per_step": ms, "ms_per_step_repeats": per, "samples_per_s": w.batch / (ms / 1e3),
         "gemm_roofline": gemm_roofline(prof, pk, pk_src), "gemm_ms_per_step": prof["gemm"][0] / K,
         "kernels_per_step": kernels,
         "nonzero_updates_per_step": {"last_step": nz, "per_layer": nz_per}}
    if w.kind == "dfp16":
        e["int16_tops"] = ops / (ms / 1e3) / 1e12
        e["executed_limb_tops"] = 4 * ops / (ms / 1e3) / 1e12
        e["gemm_roofline"]["work"] = "executed bf16 operations, 8*M*N*K per contraction"
    else:
        e["int_tops"] = ops / (ms / 1e3) / 1e12
    if cpu is not None:
        e["cpu_baseline"] = cpu
    del run
    return e


def run_ours(args, w):
    import torch
    import integer_only_nn_gb300 as ito
    import seeded_inputs as si

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    # CPU baselines first (rank 0, one GPU), before any GPU work
    cpu = None
    extra = [] if (world > 1 or args.no_workloads) else [int(v) for v in args.workloads.split(",") if v != ""]
    extra = [si.by_name(i) for i in extra if si.by_name(i).name != w.name]
    extra_cpu = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, dt, cores, nsteps, nsamp, single = cpu_baseline(w, args.cpu_batch)
        cpu = {"value": v, "unit": "samples/s", "cores": cores, "kind": "oracle",
               "sample": "%d oracle training steps (C loops, OpenMP over output rows) on %d of the %d samples "
                         "of %s, %.1f s" % (nsteps, nsamp, w.batch, w.name, dt),
               "single_thread": single}
        for x in extra:
            v, dt, cores, nsteps, nsamp, _ = cpu_baseline(x, args.cpu_batch, min_seconds=3.0, single_seconds=None)
            extra_cpu[x.name] = {"value": v, "unit": "samples/s", "cores": cores, "kind": "oracle",
                                 "sample": "%d steps on %d of %d samples, %.1f s" % (nsteps, nsamp, x.batch, dt)}

    pk, pk_src = peaks()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    if w.kind == "dfp16":
        line = run_ours_dfp16(args, w, cpu, barrier, dist, world, rank, local, flush, pk, pk_src)
    else:
        line = run_ours_model(args, w, cpu, barrier, dist, world, rank, local, flush, pk, pk_src)
    if line is not None and extra:
        line["workloads"] = {x.name: workload_entry(x, args, flush, pk, pk_src, extra_cpu.get(x.name))
                             for x in extra}
        if ito.ito_get_error() != 0:
            raise RuntimeError("device error word set after the extra workloads")
    if line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_ours_model(args, w, cpu, barrier, dist, world, rank, local, flush, pk, pk_src):
    import torch
    import integer_only_nn_gb300 as ito
    run = ModelRun(w, graphs=not args.no_graphs)
    model, stream = run.model, run.stream
    overlap_mode = model.overlap()
    speculate = model.speculation()
    K, Wm = args.steps, args.warmup
    run.warm(Wm)
    assert ito.ito_get_error() == 0

    # the timed region: REPEATS loops of K steps, each step after an untimed L2 flush and
    # input copy, bracketed by CUDA events on the step's stream (no per-kernel events inside)
    clocks = Clocks(local)
    barrier()
    torch.cuda.synchronize()
    spec0 = model.tensor("spec_count").cpu().tolist()
    clocks.start()
    ms, per = timed_median(K, REPEATS, stream, flush, run.before, run.step)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    spec1 = model.tensor("spec_count").cpu().tolist()
    err = ito.ito_get_error()
    if err != 0:
        raise RuntimeError("device error word %d after the timed steps" % err)
    nz, nz_per = run.nonzero_updates()
    ms = max_over_ranks(ms, dist)
    launches = model.kernels_per_step()

    # per-kernel timing: the same K steps again with a pair of events around every launch.
    # In overlap mode 3 the weight gradients run beside the delta propagations and share
    # their SMs, so each launch's event time would count the shared time twice: those steps
    # run in mode 0 (one stream; the same kernels and epilogues, speculation as timed)
    prof_mode = 0 if overlap_mode == 3 else overlap_mode
    model.set_overlap(prof_mode)
    prof, prof_ms = profiled_steps(model, K, stream, flush, run.before, run.step,
                                   ("gemm", "requant", "update", "other"))
    model.set_overlap(overlap_mode)
    if ito.ito_get_error() != 0:
        raise RuntimeError("device error word set after the profiled steps")

    # end to end through the host-buffer entry points: each step copies its own input
    # batch (the resident batches' pinned host copies, in turn) in and its stats out.
    # Pipelined (ito_train_step_host_async: the next batch's copy overlaps the step, one
    # wait after the last step) and blocking (ito_train_step_host: a wait every step).
    nb = NB_BATCHES
    xs_h = [x.cpu().pin_memory() for x in run.xs]
    ls_h = [lab.cpu().pin_memory() for lab in run.ls]
    x_h, l_h = xs_h[0], ls_h[0]
    st_h = torch.zeros(model.num_stats(), dtype=torch.int32).pin_memory()
    for i in range(3):
        model.train_step_host_async(xs_h[i % nb], ls_h[i % nb], st_h, stream=stream)
    stream.synchronize()
    barrier()
    t0 = time.perf_counter()
    for k in range(K):
        model.train_step_host_async(xs_h[k % nb], ls_h[k % nb], st_h, stream=stream)
    stream.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist)
    for i in range(3):
        model.train_step_host(xs_h[i % nb], ls_h[i % nb], st_h, stream=stream)
    barrier()
    t0 = time.perf_counter()
    for k in range(K):
        model.train_step_host(xs_h[k % nb], ls_h[k % nb], st_h, stream=stream)
    e2e_sync_s = max_over_ranks(time.perf_counter() - t0, dist)
    if ito.ito_get_error() != 0:
        raise RuntimeError("device error word set after the end-to-end steps")

    # the same kernels measured alone: one stream, so that no bandwidth pass shares the SMs
    # with a contraction (the timed steps above overlap them); per-kernel figures only
    model.set_overlap(0)
    model.set_speculation(False)
    iso_steps = 10
    iso, _ = profiled_steps(model, iso_steps, stream, flush, run.before, run.step,
                            ("gemm", "requant", "update", "other"))
    model.set_overlap(overlap_mode)
    model.set_speculation(speculate)

    spec_hits, spec_misses = spec1[0] - spec0[0], spec1[1] - spec0[1]

    if args.stats_log and rank == 0:
        # per-step NITI statistics (shift of every requantised tensor, weight shift,
        # nonzero weight steps) for a few steps after the timed ones, one JSON line each
        with open(args.stats_log, "w") as f:
            for t in range(10):
                run.warm(1)
                f.write(json.dumps({"step": t, **{k: int(v) for k, v in model.stats().items()}}) + "\n")

    if rank != 0:
        return None
    samples = world * w.batch * K
    value = job_throughput(w.batch, world, ms / 1000.0)
    roof = gemm_roofline(prof, pk, pk_src)
    roof.update({"kernel": "k_gemm_tc2 / k_gemm_tc (bf16-embedded int8 contractions; re-launches after a "
                           "misprediction not counted)",
                 "traffic": gemm_traffic_per_launch(w),
                 "traffic_unit": "bytes per launch (ncu, committed summary: one launch of each 4096-wide contraction "
                                 "kind at the step's shapes, averaged over the step's mix)",
                 "measured_over": "the same %d steps run again with an event pair around every launch "
                                  "(%.4f ms per step with the events)%s" % (
                                      K, prof_ms, "" if prof_mode == overlap_mode else
                                      ", in backward overlap mode %d (the timed steps' mode %d runs weight "
                                      "gradients beside delta propagations on shared SMs)" % (prof_mode, overlap_mode))})
    hbm = float(pk["hbm_gbs"])
    line = {
        "metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "dims": list(w.dims),
                   "l2": "flushed before every step (256 MB write, untimed)",
                   "timing": "median of %d loops of %d steps" % (REPEATS, K),
                   "graphs": not args.no_graphs, "backward_overlap": overlap_mode,
                   "speculation": ("on, %d/%d shift predictions held" % (spec_hits, spec_hits + spec_misses))
                                  if speculate else "off",
                   "inputs": "%d resident batches" % nb,
                   "parallelism": "replicas" if world > 1 else "single"},
        "ms_per_step_repeats": per,
        "int_tops": algorithmic_ops(w) * world / (ms / 1000.0) / 1e12,
        "nonzero_updates_per_step": {"last_step": nz, "per_layer": nz_per,
                                     "note": "weight steps that are nonzero (Step 4's operand is the shifted, "
                                             "saturated gradient: none once the gradient shift reaches 10)"},
        "roofline": roof,
        "passes": {"note": "kernel time per step by class over the profiled steps (overlapped launches include "
                           "their wait for SM resources); per-pass bandwidth is under 'isolated'",
                   "hbm_peak_gbs": hbm, "peak_source": pk_src,
                   "ms_per_step": {k: v[0] / K for k, v in prof.items()}},
        "isolated": {"note": "one stream, no speculation, %d steps: per-kernel rates (null for a class with "
                             "no launches: contractions that requantise or update in their epilogue)" % iso_steps,
                     "gemm_tflops": rate(iso["gemm"], 1e12),
                     "gemm_frac": rate(iso["gemm"], 1e12) / roof["peak"],
                     "requant_gbs": rate(iso["requant"], 1e9),
                     "update_gbs": rate(iso["update"], 1e9),
                     "ms_per_step": {c: v[0] / iso_steps for c, v in iso.items()}},
        "e2e": {"value": samples / e2e_s, "unit": "samples/s",
                "h2d_bytes_per_step": int(x_h.numel() + 4 * l_h.numel()),
                "d2h_bytes_per_step": int(4 * st_h.numel()),
                "call": "ito_train_step_host_async (input copy overlapping the previous step), one wait "
                        "after the last step",
                "blocking_value": samples / e2e_sync_s,
                "blocking_call": "ito_train_step_host (copy, step, stats copy, wait, every step)"},
        "gpu_launches": launches * K,
        "gpu_launches_all_repeats": launches * K * REPEATS,
        "clocks": clk,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def run_op(args):
    """Times one standalone single-layer call (the contraction plus its
    requantisation) at a given shape; prints a JSON line. Used as the small
    case for kernel profiles: python bench.py --op fwd --shape 8192,4096,4096"""
    import numpy as np
    import torch
    import integer_only_nn_gb300 as ito
    B, IC, OC = (int(v) for v in args.shape.split(","))
    rng = np.random.default_rng(5)
    if args.op in ("dfp16_fwd_f32", "bdfp16_fwd_f32"):
        # DFP16 forward with FP32 output, one exponent per tensor or per block of IC
        x = torch.from_numpy(rng.integers(-32767, 32768, (B, IC)).astype(np.int16)).cuda()
        W = torch.from_numpy(rng.integers(-32767, 32768, (OC, IC)).astype(np.int16)).cuda()
        nb = (IC + args.block - 1) // args.block
        ex = torch.from_numpy(rng.integers(-40, 0, (B, nb)).astype(np.int8)).cuda()
        ew = torch.from_numpy(rng.integers(-40, 0, (OC, nb)).astype(np.int8)).cuda()
        exd, ewd = ito._i32dev(-12), ito._i32dev(-17)
        call = {"dfp16_fwd_f32": lambda: ito.ito_dfp16_linear_fwd_f32(x, exd, W, ewd),
                "bdfp16_fwd_f32": lambda: ito.ito_bdfp16_linear_fwd_f32(x, ex, W, ew, args.block)}[args.op]
        ops_per_mac = 8.0      # four bf16 limb products per int16 multiply-accumulate
    else:
        x = torch.from_numpy(rng.integers(-127, 128, (B, IC)).astype(np.int8)).cuda()
        W = torch.from_numpy(rng.integers(-127, 128, (OC, IC)).astype(np.int8)).cuda()
        e = torch.from_numpy(rng.integers(-127, 128, (B, OC)).astype(np.int8)).cuda()
        call = {"fwd": lambda: ito.ito_linear_fwd(x, W, 1),
                "dgrad": lambda: ito.ito_linear_bwd_delta(e, W, x),
                "wgrad": lambda: ito.ito_linear_wgrad(e, x)}[args.op]
        ops_per_mac = 2.0
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record()
    for _ in range(args.steps):
        call()
    s1.record()
    torch.cuda.synchronize()
    ms = s0.elapsed_time(s1) / args.steps
    line = {"op": args.op, "shape": [B, IC, OC], "ms_per_call": ms,
            "tflops_incl_conversions": ops_per_mac * B * IC * OC / (ms / 1000.0) / 1e12}
    if args.op.startswith("bdfp"):
        line["block"] = args.block
    print(json.dumps(line), flush=True)
    return 0


def run_ours_dfp16(args, w, cpu, barrier, dist, world, rank, local, flush, pk, pk_src):
    """Step time of the DFP16 workload (device-timed with CUDA events)."""
    import torch
    import integer_only_nn_gb300 as ito
    run = DfpRun(w)
    model, stream = run.model, run.stream
    K = args.steps
    run.warm(args.warmup)
    clocks = Clocks(local)
    barrier()
    torch.cuda.synchronize()
    clocks.start()
    ms, per = timed_median(K, REPEATS, stream, flush, run.before, run.step)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    if ito.ito_get_error() != 0:
        raise RuntimeError("device error word set after the timed steps")
    nz, nz_per = run.nonzero_updates()
    ms = max_over_ranks(ms, dist)
    launches = model.kernels_per_step()

    # per-kernel timing: the same K steps again with an event pair around every launch
    prof, prof_ms = profiled_steps(model, K, stream, flush, run.before, run.step, ("gemm", "down", "update", "other"))

    # end to end through the public API: each step copies its input mantissas from pinned
    # host memory and its statistics back. Pipelined (ito_dfp16_train_step_host_async: the
    # next batch's copy overlaps the step, one wait after the last step) and blocking (a
    # host-to-device copy, the step and a statistics read with a wait, every step)
    xs_h = [x.cpu().pin_memory() for x in run.xs]
    st_h = torch.zeros(model.num_stats(), dtype=torch.int64).pin_memory()
    for i in range(3):
        run.step_host_async(xs_h[i % 2], st_h)
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    for k in range(K):
        run.step_host_async(xs_h[k % 2], st_h)
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist)
    for i in range(3):
        run.xs[i % 2] = xs_h[i % 2].to("cuda", non_blocking=True)
        run.step(i)
        model.stats()
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(K):
        run.xs[k % 2] = xs_h[k % 2].to("cuda", non_blocking=True)
        run.step(k)
        model.stats()
    e2e_sync_s = max_over_ranks(time.perf_counter() - t0, dist)
    if ito.ito_get_error() != 0:
        raise RuntimeError("device error word set after the end-to-end steps")
    if rank != 0:
        return None
    ops = algorithmic_ops(w)
    roof = gemm_roofline(prof, pk, pk_src)
    roof.update({"kernel": "k_gemm_dfp4 / k_gemm_dfp2 / k_gemm_dfp (int16 limb contractions: four bf16 limb products per "
                           "int16 multiply-add, exact int64 sums)",
                 "work": "executed bf16 operations, 8*M*N*K per contraction", "traffic": None,
                 "measured_over": "the same %d steps run again with an event pair around every launch "
                                  "(%.4f ms per step with the events)" % (K, prof_ms)})
    line = {"metric": METRIC, "value": world * w.batch / (ms / 1000.0), "unit": "samples/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int16 (DFP16)",
            "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "dims": list(w.dims), "eta": w.eta,
                       "l2": "flushed before every step (256 MB write, untimed)",
                       "timing": "median of %d loops of %d steps" % (REPEATS, K),
                       "inputs": "2 resident batches, alternating",
                       "parallelism": "replicas" if world > 1 else "single"},
            "ms_per_step_repeats": per,
            "int16_tops": ops * world / (ms / 1000.0) / 1e12,
            "executed_limb_tops": 4 * ops * world / (ms / 1000.0) / 1e12,
            "nonzero_updates_per_step": {"last_step": nz, "per_layer": nz_per},
            "roofline": roof,
            "passes": {"ms_per_step": {c: v[0] / K for c, v in prof.items()},
                       "down_gbs": rate(prof["down"], 1e9),
                       "update_gbs": rate(prof["update"], 1e9),
                       "note": "down-conversions and updates run on a second stream beside the contractions: "
                               "their times include waits for SM resources"},
            "e2e": {"value": world * w.batch * K / e2e_s, "unit": "samples/s",
                    "h2d_bytes_per_step": int(xs_h[0].numel() * 2), "d2h_bytes_per_step": int(8 * st_h.numel()),
                    "call": "ito_dfp16_train_step_host_async (input copy overlapping the previous step), one "
                            "wait after the last step",
                    "blocking_value": world * w.batch * K / e2e_sync_s,
                    "blocking_call": "host-to-device copy, ito_dfp16_train_step, statistics read, every step"},
            "gpu_launches": launches * K,
            "gpu_launches_all_repeats": launches * K * REPEATS,
            "clocks": clk}
    apt = w.apt
    if apt is not None:
        line["config"]["apt"] = {"k_init": apt.k_init, "k_min": apt.k_min, "k_max": apt.k_max, "t_min": apt.t_min,
                                 "t_max": str(apt.t_max), "epoch_steps": apt.epoch, "eval_every": apt.eval_every}
        line["apt_bits_after"] = [model.precision(l)[0] for l in range(model.n_layers)]
    if cpu is not None:
        line["cpu_baseline"] = cpu
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="3")
    ap.add_argument("--cpu-batch", type=int, default=128, help="samples in the CPU-oracle baseline step")
    ap.add_argument("--ref-batch", type=int, default=16, help="samples per reference-arm oracle step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workloads", default="0,1,2,4",
                    help="more workloads timed after the headline one, reported under 'workloads'")
    ap.add_argument("--no-workloads", action="store_true", help="time the headline workload only")
    ap.add_argument("--no-graphs", action="store_true", help="launch every kernel directly (no CUDA graphs)")
    ap.add_argument("--op", choices=("fwd", "dgrad", "wgrad", "dfp16_fwd_f32", "bdfp16_fwd_f32"),
                    help="time one single-layer call instead")
    ap.add_argument("--block", type=int, default=512, help="Blocked-DFP block length for --op bdfp16_fwd_f32")
    ap.add_argument("--stats-log", default=None,
                    help="write per-step NITI statistics (shifts, nonzero updates) of 10 steps after the timed "
                         "ones to this JSONL file")
    ap.add_argument("--shape", default="8192,4096,4096", help="B,IC,OC for --op")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.op:
        return run_op(args)
    import seeded_inputs as si
    w = si.by_name(int(args.workload) if args.workload.isdigit() else args.workload)
    if args.impl == "reference":
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
