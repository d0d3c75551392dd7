"""Benchmark of the shard-local step (one JSON line on stdout from rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY]
                    [--impl ours|reference]

One step = one rank's fused shard-local step over its whole shard: the N
incoming bf16 gradient slices summed in fp32 and scaled by 1/N, AdamW on the
fp32 master/m/v shard, the bf16 cast written into the rank's slot of the
AllGather buffer. Inputs are synthetic (seeded generator), shaped like the
named model's parameter list, and resident in HBM before the timed region;
each step's working set (tens of GB) is far larger than L2, so no flush is
needed between steps.

With --gpus N > 1 (torchrun, one process per GPU) GPU i runs emulated rank
i mod N_ranks of the same workload: per-GPU work is fixed (weak scaling) and
no collective touches the data path; the timed region is bracketed by a
barrier and a synchronize, and the slowest rank's time is reported.

--impl reference times the CPU oracle (single thread) on a bounded sample of
the same workload, on the host's cores, as the reference arm.

Other measurements (--pipeline; the default is the step above):
    clip        global-norm pass + clip coefficient + clipped step
    accum       G-1 gradient accumulations + the accumulated step
    accum_clip  G-1 accumulations + the accumulated gradient's norm + clip
                coefficient + the clipped accumulated step
    gather      the AllGather's assembly of the other ranks' shards
    unshard     FSDP2 copy-out of every wrap unit's gathered parameters
    checkpoint  save, restore, and restore into world N/2 of one rank's state
    sweep       the step over shard sizes x N x gradient and parameter dtypes
--step-path forces either step kernel (register-streaming or staged); --buckets runs the
step as one call per gradient bucket (GPT-2-small's 25M-element buckets) and --rank picks
the emulated rank GPU 0 runs; --graph times one CUDA-graph replay of the K steps.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "shard-step elements/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "elements/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = [os.path.join(ROOT, "fsdp_sharded_mixed_gb300", "csrc", f)
                  for f in ("shard_step.cu", "step_kernel.cuh", "bulk.cuh", "overlap.cuh")]
TRAFFIC_SUMMARY = os.path.join(ROOT, "profiles", "shard_step_traffic.txt")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ----------------------------------------------------------- host helpers ----
def dist_env():
    """(rank, world_size, local_rank) from torchrun's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def emulated_rank(global_rank, n_ranks, first=0):
    """The data-parallel rank whose shard step GPU `global_rank` runs (GPU 0
    runs rank `first`)."""
    return (global_rank + first) % n_ranks


def max_over_ranks(value, device=None):
    """Max of a float over all processes (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def code_of(text):
    """C++ source without comments and with whitespace runs collapsed: what
    the compiler sees (the sources' string literals hold no comment markers)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_sha():
    """sha256[:16] over the code (comments and layout ignored) of the step
    kernel's sources."""
    h = hashlib.sha256()
    for path in KERNEL_SOURCES:
        with open(path, encoding="utf-8") as f:
            h.update(code_of(f.read()).encode())
    return h.hexdigest()[:16]


def committed_traffic(workload_key):
    """ncu DRAM bytes per shard element for the current kernel source, from the
    committed profile summary, or None when absent or taken on other code."""
    try:
        text = open(TRAFFIC_SUMMARY, encoding="utf-8").read()
    except OSError:
        return None
    sha = kernel_sha()
    for line in text.splitlines():
        m = re.match(r"\s*traffic\s+(\S+)\s+kernel_sha=(\w+)\s+bytes_per_elem=([\d.]+)", line)
        if m and m.group(1) == workload_key and m.group(2) == sha:
            return float(m.group(3))
    return None


def host_cpu():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
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


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            peaks = json.load(f)
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ["index", "clocks.sm", "clocks.max.sm", "power.draw",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, uuid=None):
        self.cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                    "--format=csv,noheader,nounits", "-lms", "100"]
        if uuid:
            self.cmd += ["-i", uuid]
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            cols = [c.strip() for c in line.split(",")]
            if len(cols) != len(self.FIELDS):
                continue
            try:
                sm.append(float(cols[1]))
                smax.append(float(cols[2]))
                power.append(float(cols[3]))
            except ValueError:
                continue
            for name, val in zip(names, cols[4:]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(power), "samples": len(sm), "reasons": sorted(reasons)}


# ------------------------------------------------------------ CPU oracle ----
def oracle_time(w, S, P, rank, n_elems, steps, warmup=0):
    """Time the single-threaded oracle on the first n_elems elements of rank's
    shard (n_elems <= 0 or >= S: the whole shard), `steps` steps after `warmup`
    untimed ones. The inputs (the N bf16 slices, the master) are made first by
    the seeded host generator on every core, untimed; the oracle's steps run
    on one pinned core. Returns (elements/s, timed seconds, cores used,
    elements per step)."""
    import numpy as np

    import oracle
    import synth
    o = oracle.default()
    N = w.world
    n = S if n_elems <= 0 else max(8, min(S, n_elems))
    kw = dict(seed=w.seed, sigma=w.grad_sigma, p_limit=P, outlier_frac=w.outlier_frac,
              outlier_scale=w.outlier_scale, bf16=True)
    grads = [synth.fill(n, index0=rank * S, rank=j, step=1, **kw) for j in range(N)]
    master = synth.fill(n, index0=rank * S, seed=w.seed, stream=synth.STREAM_MASTER,
                        sigma=w.master_sigma, p_limit=P)
    m, v = np.zeros(n, np.float32), np.zeros(n, np.float32)
    slot = np.zeros(n, np.uint16)   # rank 0 of an n-element shard: the slot is [0, n)
    hp = w.hparams
    old_aff = None
    if hasattr(os, "sched_setaffinity"):
        old_aff = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(old_aff)})
    try:
        total = 0.0
        for t in range(1, warmup + steps + 1):
            t0 = time.perf_counter()
            o.shard_step(world=N, rank=0, S=n, lo=0, hi=n, grads=grads, master=master, m=m,
                         v=v, full_flat=slot, lr=hp["lr"], beta1=hp["beta1"],
                         beta2=hp["beta2"], eps=hp["eps"], wd=hp["weight_decay"], t=t)
            if t > warmup:
                total += time.perf_counter() - t0
    finally:
        if old_aff is not None:
            os.sched_setaffinity(0, old_aff)
    return n * steps / total, total, 1, n


# ------------------------------------------------------------------ main ----
def bytes_per_elem(world, grad_bytes=2, param_bytes=2):
    return grad_bytes * world + 24 + param_bytes


def run_config(args, w, S, P, P_pad, gworld, r, n_calls):
    """The `config` of both arms' JSON lines (the same dict for the same run)."""
    cfg = {"workload": f"{w.key}: {w.title}", "emulated_ranks": w.world,
           "shard_elems": S, "flat_params": P, "flat_padded": P_pad,
           "grad_dtype": "bf16", "param_dtype": "bf16", "state_dtype": "fp32",
           "bytes_per_elem": bytes_per_elem(w.world),
           "l2": "no flush: each step streams >> 129 MB L2 (inputs larger than L2)",
           "parallelism": f"replicas{gworld}", "emulated_rank_gpu0": r,
           "pipeline": args.pipeline, "step_path": args.step_path, "bucket_calls": n_calls,
           "launch_overlap": not args.no_overlap}
    if args.pipeline in ("clip", "accum_clip"):
        cfg["clip"] = True
    if args.pipeline in ("accum", "accum_clip"):
        cfg["micro_steps"] = max(1, args.micro_steps)
    return cfg


def run_reference(args, w):
    """The reference arm: the CPU oracle, as it stands, one thread, on a
    bounded sample of each step (the first elements of the rank's shard),
    sized so that the warm-up and timed steps take about a minute. Only the
    oracle and the input generator are loaded (the plan is the oracle's)."""
    rank, world_size, _ = dist_env()
    if rank != 0:
        return
    import oracle
    o = oracle.default()
    bucketed = args.buckets and w.bucket_elems > 0 and args.pipeline == "step"
    op = o.plan(w.numels, w.tied_to, world=w.world, align=w.align,
                bucket_elems=w.bucket_elems if bucketed else 0)
    S, P, P_pad = op["S"], op["P"], op["P_pad"]
    r = emulated_rank(0, w.world, args.rank)
    n_calls = 1
    if bucketed:
        n_calls = sum(1 for lo, hi in (o.shard_range(a, b, r, S) for a, b in op["buckets"])
                      if hi > lo)
    budget_s, est_rate = 60.0, 20e6
    sample = int(budget_s * est_rate / max(1, args.steps + args.warmup))
    sample = max(4096, min(S, sample)) // 8 * 8
    rate, secs, cores, n = oracle_time(w, S, P, r, sample, args.steps, warmup=args.warmup)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": run_config(args, w, S, P, P_pad, world_size, r, n_calls),
        "sample_elems_per_step": n,
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"each step: the first {n:,} elements of rank {r}'s "
                                   f"{S:,}-element shard; ms_per_step and value are of that "
                                   f"measured sample (not scaled to the shard)"},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import torch.distributed as dist

    import fsdp_sharded_mixed_gb300 as zs
    import synth

    grank, gworld, local = dist_env()
    if gworld > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    sptr = stream.cuda_stream
    Ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    bucketed = args.buckets and w.bucket_elems > 0 and args.pipeline == "step"
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align,
                              bucket_elems=w.bucket_elems if bucketed else 0)
    N, S, P = plan.world, plan.S, plan.P
    r = emulated_rank(grank, N, args.rank)
    # --buckets: the step as the configuration's ZeRO-2 job runs it, one call
    # per gradient bucket over this rank's part of it, in bucket order.
    ranges = [(0, S)]
    if bucketed:
        ranges = [b for b in (zs.zs_plan_bucket(plan, k, r) for k in range(plan.n_buckets))
                  if b[1] > b[0]]
    hp = w.hparams
    bpe = bytes_per_elem(N)
    norm_bpe = 2 * N  # the norm pass reads the N bf16 slices once
    accum_clip = args.pipeline == "accum_clip"
    clip = args.pipeline == "clip" or accum_clip
    accum_mode = args.pipeline == "accum" or accum_clip
    G = max(1, args.micro_steps)

    # Inputs resident in HBM: one set of incoming slices, master from the
    # generator, zero moments, the full AllGather buffer (not needed by the
    # copy-out pipeline, which holds its own per-unit buffers).
    grads = master = m = v = full = None
    gather_srcs = None
    if args.pipeline == "gather":
        # The emulated AllGather's inputs: the other ranks' bf16 shards, each
        # its own buffer, and the full flat buffer they are assembled into.
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=dev)
        gather_srcs = []
        for j in range(N):
            if j == r:
                gather_srcs.append(None)
                continue
            g = torch.empty(S, dtype=torch.int16, device=dev)
            synth.fill_device(g.data_ptr(), S, index0=j * S, seed=w.seed, rank=j, step=1,
                              sigma=w.grad_sigma, p_limit=P, bf16=True, cuda_stream=sptr)
            gather_srcs.append(g)
    elif args.pipeline != "unshard":
        grads = [torch.empty(S, dtype=torch.int16, device=dev) for _ in range(N)]
        for j, g in enumerate(grads):
            synth.fill_device(g.data_ptr(), S, index0=r * S, seed=w.seed, rank=j, step=1,
                              sigma=w.grad_sigma, p_limit=P, outlier_frac=w.outlier_frac,
                              outlier_scale=w.outlier_scale, bf16=True, cuda_stream=sptr)
        master = torch.empty(S, dtype=torch.float32, device=dev)
        synth.fill_device(master.data_ptr(), S, index0=r * S, seed=w.seed,
                          stream=synth.STREAM_MASTER, sigma=w.master_sigma, p_limit=P,
                          bf16=False, cuda_stream=sptr)
        m = torch.zeros(S, dtype=torch.float32, device=dev)
        v = torch.zeros(S, dtype=torch.float32, device=dev)
        full = torch.zeros(plan.P_pad, dtype=torch.int16, device=dev)

    # Clipping: this rank's partial sum of squares, the N partials (the other
    # ranks' as if every shard had this one's norm: the scalar AllReduce of a
    # real system), the coefficient and skip flag, all on the device.
    ws = parts = coef = bad = acc_buf = None
    max_norm = 1.0
    if clip:
        ws = torch.empty(zs.zs_grad_norm_workspace_bytes(), dtype=torch.uint8, device=dev)
        parts = torch.zeros(N, dtype=torch.float64, device=dev)
        coef = torch.zeros(1, dtype=torch.float32, device=dev)
        bad = torch.zeros(1, dtype=torch.int32, device=dev)
        zs.zs_grad_sqnorm(plan, r, 0, S, grads, zs.ZS_BF16, ws, parts.narrow(0, r, 1),
                          stream=sptr)
        torch.cuda.synchronize()
        own = float(parts[r].item())
        parts.fill_(own)
        max_norm = 0.5 * (N * own) ** 0.5  # so that the step really clips
    if accum_mode:
        acc_buf = torch.zeros(S, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()

    step_no = [0]

    # The parts of one optimizer step: (name, enqueue(stream), algorithmic bytes/elem).
    def part_step(sp):
        for lo, hi in ranges:
            zs.zs_shard_step(plan, r, lo, hi, grads, zs.ZS_BF16, master, m, v, full, zs.ZS_BF16,
                             hp, step_no[0], stream=sp)

    def part_norm(sp):
        zs.zs_grad_sqnorm(plan, r, 0, S, grads, zs.ZS_BF16, ws, parts.narrow(0, r, 1), stream=sp)
        zs.zs_clip_coefficient(parts, N, max_norm, coef, bad, stream=sp)

    def part_clipped(sp):
        zs.zs_shard_step_clipped(plan, r, 0, S, grads, zs.ZS_BF16, master, m, v, full,
                                 zs.ZS_BF16, hp, step_no[0], coef=coef, skip=bad, stream=sp)

    def part_accumulate(sp):
        for k in range(G - 1):
            zs.zs_grad_accumulate(plan, r, 0, S, grads, zs.ZS_BF16, acc_buf, k == 0, stream=sp)

    def part_accumulated(sp):
        zs.zs_shard_step_accumulated(plan, r, 0, S, grads, zs.ZS_BF16, acc_buf, G, master, m, v,
                                     full, zs.ZS_BF16, hp, step_no[0], stream=sp)

    def part_norm_accumulated(sp):
        zs.zs_grad_sqnorm_accumulated(plan, r, 0, S, grads, zs.ZS_BF16, acc_buf, G, ws,
                                      parts.narrow(0, r, 1), stream=sp)
        zs.zs_clip_coefficient(parts, N, max_norm, coef, bad, stream=sp)

    def part_accumulated_clipped(sp):
        zs.zs_shard_step_accumulated_clipped(plan, r, 0, S, grads, zs.ZS_BF16, acc_buf, G, master,
                                             m, v, full, zs.ZS_BF16, hp, step_no[0], coef=coef,
                                             skip=bad, stream=sp)

    units = []
    up_dims = {}
    unit_params = []
    if args.pipeline == "unshard":
        # FSDP2's gather side over the whole model: per wrap unit a row-sharded
        # plan, the rank-major AllGather buffer (filled once from the
        # generator), and the unit's full parameters, written by the copy-out.
        from synth.workloads import wrap_units
        all_units = wrap_units(w)
        for idx in all_units[:args.units] if args.units else all_units:
            local_of = {g_: k for k, g_ in enumerate(idx)}
            ps = [w.params[i] for i in idx]
            ties_u = [local_of[p.tied_to] if p.tied_to >= 0 else -1 for p in ps]
            up = zs.zs_rows_plan([p.shape[0] for p in ps], [p.numel for p in ps], ties_u, world=N,
                                 align_elems=w.align)
            gbuf = torch.empty(up.P_pad, dtype=torch.int16, device=dev)
            synth.fill_device(gbuf.data_ptr(), up.P_pad, seed=w.seed, rank=len(units), step=1,
                              sigma=w.grad_sigma, bf16=True, cuda_stream=sptr)
            outs = [torch.empty(p.numel, dtype=torch.int16, device=dev) if t < 0 else None
                    for p, t in zip(ps, ties_u)]
            units.append((up, gbuf, outs))
            up_dims[id(up)] = [p.shape[0] for p in ps]
            unit_params.extend(i for i, t in zip(idx, ties_u) if t < 0)
        torch.cuda.synchronize()

    def _segments(up, outs):
        c, _ = zs.zs_plan_rows(up)
        return sum(-(-d // ci) for d, ci, o in zip(up_dims[id(up)], c, outs)
                   if o is not None and d > 0)

    def part_unshard(sp):
        for up, gbuf, outs in units:
            zs.zs_unshard(up, gbuf, zs.ZS_BF16, outs, stream=sp)

    def part_gather(sp):
        zs.zs_gather_assemble(plan, r, gather_srcs, full, zs.ZS_BF16, stream=sp)

    if args.pipeline == "gather":
        # every other rank's shard read once and written once into its slot
        pipeline = [("gather_kernel", part_gather, 4 * (N - 1))]
        launches_per_step = 1
    elif args.pipeline == "unshard":
        # bytes per shard element of the workload's plan: every parameter
        # element read once from the gathered buffer and written once.
        unit_bytes = 4 * sum(w.params[i].numel for i in unit_params)
        pipeline = [("segment_copy_kernel", part_unshard, unit_bytes / S)]
        launches_per_step = 0
        for up, _, outs in units:   # one launch per 256 (parameter, rank) row segments
            launches_per_step += -(-_segments(up, outs) // 256)
    elif accum_clip:
        # micro-steps 1 .. G-1 accumulated; the norm of the accumulated
        # gradient (slices + accumulator) and the coefficient; the clipped
        # accumulated step.
        acc_bytes = (2 * N + 4) + (G - 2) * (2 * N + 8) if G > 1 else 0
        pipeline = ([("accumulate_kernel", part_accumulate, acc_bytes)] if G > 1 else []) + \
                   [("grad_sqnorm_kernel+clip_coef_kernel", part_norm_accumulated, norm_bpe + 4),
                    ("shard_step_kernel", part_accumulated_clipped, bpe + 4)]
        launches_per_step = G + 2
    elif clip:
        pipeline = [("grad_sqnorm_kernel+clip_coef_kernel", part_norm, norm_bpe),
                    ("shard_step_kernel", part_clipped, bpe)]
        launches_per_step = 3
    elif accum_mode:
        acc_bytes = (2 * N + 4) + (G - 2) * (2 * N + 8) if G > 1 else 0
        pipeline = ([("accumulate_kernel", part_accumulate, acc_bytes)] if G > 1 else []) + \
                   [("shard_step_kernel", part_accumulated, bpe + 4)]
        launches_per_step = G
    else:
        pipeline = [("shard_step_kernel", part_step, bpe)]
        launches_per_step = len(ranges)
    pipe_bpe = sum(b for _, _, b in pipeline)

    def step(sp=sptr, marks=None):
        step_no[0] += 1
        cur = torch.cuda.current_stream()
        for k, (_, fn, _) in enumerate(pipeline):
            if marks:
                marks[k].record(cur)
            fn(sp)
        if marks:
            marks[-1].record(cur)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        uuid = None
    sampler = ClockSampler(uuid)
    sampler.start()
    t_end = time.time() + 0.4  # keep the GPU busy while nvidia-smi starts
    while time.time() < t_end:
        step()
        torch.cuda.synchronize()

    # The timed region: K steps back to back between two events on the
    # launching stream (or one replay of a CUDA graph holding the K steps).
    # For the clip pipeline, events also mark each step's kernels so each
    # kernel's own average duration is known.
    graph = None
    if args.graph:
        graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.graph(graph, stream=side, capture_error_mode="relaxed"):
            for _ in range(args.steps):
                step(sp=side.cuda_stream)
        stream.wait_stream(side)
        graph.replay()  # one untimed replay
    multi = len(pipeline) > 1
    nmk = len(pipeline) + 1
    marks = [[Ev() for _ in range(nmk)] for _ in range(args.steps)] if (multi and graph is None) \
        else None
    if gworld > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = Ev(), Ev()
    t0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for k in range(args.steps):
            step(marks=marks[k] if marks else None)
    t1.record(stream)
    torch.cuda.synchronize()
    if gworld > 1:
        dist.barrier()
    clocks = sampler.stop()
    elapsed = t0.elapsed_time(t1) / 1e3
    split = "events around each part of direct launches"
    if multi and graph is not None:
        # Each part in place: CUDA graphs of the K steps' pipeline suffixes
        # (parts k.., k = 1, 2, ...), each replayed and timed; part k's time is
        # the difference between the suffixes from k and from k + 1, so it
        # includes its own launches' gaps and whatever the part before it
        # leaves in flight.
        suffix_s = [elapsed]
        for k in range(1, len(pipeline)):
            g_k = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            with torch.cuda.graph(g_k, stream=side, capture_error_mode="relaxed"):
                for _ in range(args.steps):
                    for _, fn, _ in pipeline[k:]:
                        fn(side.cuda_stream)
            stream.wait_stream(side)
            g_k.replay()
            torch.cuda.synchronize()
            a_ev, b_ev = Ev(), Ev()
            a_ev.record(stream)
            g_k.replay()
            b_ev.record(stream)
            torch.cuda.synchronize()
            suffix_s.append(a_ev.elapsed_time(b_ev) / 1e3)
            del g_k
        suffix_s.append(0.0)
        part_s = [(suffix_s[k] - suffix_s[k + 1]) / args.steps for k in range(len(pipeline))]
        split = "in place: differences of CUDA-graph replays of the pipeline's suffixes"
    elif multi:  # direct launches: the events recorded around each part
        part_s = [sum(mk[k].elapsed_time(mk[k + 1]) for mk in marks) / 1e3 / len(marks)
                  for k in range(len(pipeline))]
    else:
        part_s = [elapsed / args.steps]
    step_s = part_s[-1]
    t_max = max_over_ranks(elapsed, dev)
    elems_all = sum_over_ranks(float(S) * args.steps, dev)
    value = elems_all / t_max

    # Per-step spread, measured after the timed region (events around each step).
    n_spread = min(args.steps, 50)
    events = [(Ev(), Ev()) for _ in range(n_spread)]
    for a_ev, b_ev in events:
        a_ev.record(stream)
        step()
        b_ev.record(stream)
    torch.cuda.synchronize()
    per_step = sorted(a_ev.elapsed_time(b_ev) for a_ev, b_ev in events)

    # End to end through the C ABI from pinned host memory: every step copies
    # the N incoming slices host->device and reads the updated slot back. The
    # shard goes in chunks through the [lo, hi) range of the call, so the copy
    # of chunk c+1, the step on chunk c and the read-back of chunk c-1 overlap
    # (how bucketed ReduceScatter output meets the optimizer in a real job).
    e2e = None
    if not args.no_e2e and args.pipeline == "step":
        h_grads = [torch.empty(S, dtype=torch.int16, pin_memory=True) for _ in range(N)]
        for hg, g in zip(h_grads, grads):
            hg.copy_(g)
        h_out = torch.empty(S, dtype=torch.int16, pin_memory=True)
        slot = full.narrow(0, r * S, S)
        nch = max(1, args.e2e_chunks)
        bounds = [min(S, (S * c // nch) // 16 * 16) for c in range(nch)] + [S]
        s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(nch)]
        ev_cmp = [torch.cuda.Event() for _ in range(nch)]
        ev_out = [torch.cuda.Event() for _ in range(nch)]
        for c in range(nch):  # nothing outstanding yet
            ev_cmp[c].record(stream)
            ev_out[c].record(stream)

        def e2e_step():
            step_no[0] += 1
            for c in range(nch):
                lo, hi = bounds[c], bounds[c + 1]
                if hi <= lo:
                    continue
                s_in.wait_event(ev_cmp[c])      # last step's kernel has read chunk c
                with torch.cuda.stream(s_in):
                    for hg, g in zip(h_grads, grads):
                        g[lo:hi].copy_(hg[lo:hi], non_blocking=True)
                ev_in[c].record(s_in)
                s_cmp.wait_event(ev_in[c])
                s_cmp.wait_event(ev_out[c])     # last step's read-back of chunk c is done
                zs.zs_shard_step(plan, r, lo, hi, grads, zs.ZS_BF16, master, m, v, full,
                                 zs.ZS_BF16, hp, step_no[0], stream=s_cmp.cuda_stream)
                ev_cmp[c].record(s_cmp)
                s_out.wait_event(ev_cmp[c])
                with torch.cuda.stream(s_out):
                    h_out[lo:hi].copy_(slot[lo:hi], non_blocking=True)
                ev_out[c].record(s_out)

        for s_ in (s_in, s_cmp, s_out):
            s_.wait_stream(stream)
        e2e_step()
        torch.cuda.synchronize()
        # The host link as it is right now: the same bytes host->device as one
        # copy per slice, no step, no read-back (the link is shared with other
        # tenants of the machine and dips periodically).
        link = []
        for _ in range(args.e2e_steps):
            a, b = Ev(), Ev()
            a.record(stream)
            for hg, g in zip(h_grads, grads):
                g.copy_(hg, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            link.append(2 * N * S / (a.elapsed_time(b) / 1e3) / 1e9)
        if gworld > 1:
            dist.barrier()
        a, b = Ev(), Ev()
        a.record(stream)
        for s_ in (s_in, s_cmp, s_out):
            s_.wait_stream(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        for s_ in (s_in, s_cmp, s_out):
            stream.wait_stream(s_)
        b.record(stream)
        torch.cuda.synchronize()
        e2e_t = max_over_ranks(a.elapsed_time(b) / 1e3, dev)
        e2e_elems = sum_over_ranks(float(S) * args.e2e_steps, dev)
        # The host link during the leg: after the timed steps, e2e steps and
        # plain host->device copies of the same bytes alternate, each timed
        # alone, so that each step's host bandwidth is compared with the link
        # as it was a moment later (the link is shared and dips periodically).
        pair_frac, pair_e2e, pair_link, t_e2e, t_link = [], [], [], 0.0, 0.0
        for _ in range(args.e2e_steps):
            a, b = Ev(), Ev()
            a.record(stream)
            for s_ in (s_in, s_cmp, s_out):
                s_.wait_stream(stream)
            e2e_step()
            for s_ in (s_in, s_cmp, s_out):
                stream.wait_stream(s_)
            b.record(stream)
            torch.cuda.synchronize()
            t_e2e += a.elapsed_time(b) / 1e3
            ge = 2 * N * S / (a.elapsed_time(b) / 1e3) / 1e9
            a, b = Ev(), Ev()
            a.record(stream)
            for hg, g in zip(h_grads, grads):
                g.copy_(hg, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize()
            t_link += a.elapsed_time(b) / 1e3
            gl = 2 * N * S / (a.elapsed_time(b) / 1e3) / 1e9
            pair_e2e.append(ge)
            pair_link.append(gl)
            pair_frac.append(ge / gl)
        e2e = {"value": e2e_elems / e2e_t, "unit": UNIT, "h2d_bytes_per_step": 2 * N * S,
               "d2h_bytes_per_step": 2 * S, "steps": args.e2e_steps,
               "ms_per_step": 1e3 * e2e_t / args.e2e_steps, "chunks": nch,
               "h2d_gbs": 2 * N * S * args.e2e_steps / e2e_t / 1e9,
               "link_h2d_gbs": {"median": statistics.median(link), "min": min(link),
                                "max": max(link),
                                "note": "plain host->device copies of the same bytes, "
                                        "timed just before; the host link is shared"},
               "frac_of_link": statistics.median(pair_frac),
               "frac_of_link_aggregate": t_link / t_e2e,
               "link_during": {"pairs": len(pair_frac),
                               "e2e_h2d_gbs": 2 * N * S * len(pair_frac) / t_e2e / 1e9,
                               "link_h2d_gbs": 2 * N * S * len(pair_frac) / t_link / 1e9,
                               "pair_frac_median": statistics.median(pair_frac),
                               "pair_frac_min": min(pair_frac), "pair_frac_max": max(pair_frac),
                               "note": "one e2e step then one plain copy of its host->device "
                                       "bytes, alternating, each timed alone; frac_of_link = "
                                       "the median over the pairs of the step's host->device "
                                       "GB/s over the copy's; the aggregate divides the sums "
                                       "(a link dip inside one step weighs on it)"}}
        del h_grads, h_out

    # A practical ceiling beside the measured peak: a device-to-device copy
    # moving the step's own algorithmic byte count (half read, half written;
    # at least 1 GiB, at most what free memory allows), timed with events,
    # median of 5.
    copy_gbs = None
    copy_bytes = 0
    if not args.no_copy_ceiling:
        half = int(pipe_bpe * S) // 2 // 256 * 256
        free = torch.cuda.mem_get_info(dev)[0]
        copy_bytes = max(1 << 30, min(half, int(0.4 * free) // 256 * 256))
        src = torch.empty(copy_bytes, dtype=torch.uint8, device=dev)
        dst = torch.empty_like(src)
        src.fill_(1)
        cts = []
        for i in range(7):
            a, b = Ev(), Ev()
            a.record(stream)
            dst.copy_(src)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 2:
                cts.append(a.elapsed_time(b) / 1e3)
        copy_gbs = 2 * copy_bytes / statistics.median(cts) / 1e9
        del src, dst
    if grank == 0:
        peak, peak_kind = measured_peak()
        step_bpe = pipeline[-1][2]
        achieved = step_bpe * S / step_s / 1e9
        kname = pipeline[-1][0]
        if kname == "shard_step_kernel":
            # the step kernel the last call took (the per-call choice)
            kk, ke = zs.zs_last_step_kernel()
            kname = (f"staged_step_kernel ({ke}-element tiles)" if kk == 2 else
                     f"shard_step_kernel ({ke}-element groups)" if kk == 1 else kname)
        traffic_pe = committed_traffic(w.key)
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                    "frac": achieved / peak, "peak_source": peak_kind,
                    "traffic": None if traffic_pe is None else traffic_pe * S,
                    "algorithmic_bytes": step_bpe * S, "kernel": kname,
                    "kernel_sha": kernel_sha()}
        kernels = {}
        for (name, _, b), t in zip(pipeline, part_s):
            gbs = b * S / t / 1e9
            kernels[name] = {"ms": 1e3 * t, "gbs": gbs, "frac": gbs / peak,
                             "bytes_per_elem": b}
        cpu = None
        if not args.no_cpu_baseline and gworld == 1:
            rate, secs, cores, n = oracle_time(w, S, P, r, args.cpu_sample_elems,
                                               args.cpu_steps)
            what = (f"the full shard ({n:,} elements)" if n == S else
                    f"the first {n:,} elements of the {S:,}-element shard")
            cpu = {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle",
                   "sample": f"rank {r}'s step on {what} x {args.cpu_steps} step(s), "
                             f"{secs:.1f} s on 1 pinned thread; inputs made beforehand, "
                             f"untimed",
                   "full_step": n == S,
                   "ns_per_elem": 1e9 / rate, "algorithmic_gbs": rate * bpe / 1e9,
                   "host": host_cpu(), "nproc": os.cpu_count()}
        if copy_gbs is not None:
            roofline["copy_ceiling_gbs"] = copy_gbs
            roofline["copy_ceiling_bytes"] = 2 * copy_bytes
            roofline["frac_of_copy_ceiling"] = achieved / copy_gbs
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": gworld,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": run_config(args, w, S, P, plan.P_pad, gworld, r, len(ranges)),
            "hbm_gbs": pipe_bpe * value / gworld / 1e9,
            "step_ms": {"median": statistics.median(per_step),
                        "p10": per_step[len(per_step) // 10],
                        "p90": per_step[(9 * len(per_step)) // 10],
                        "note": f"{n_spread} steps with events around each, after the timed region"},
            "timing": "cuda graph replay of the K steps" if graph is not None
                      else "K direct launches between two events",
            "roofline": roofline, "kernels": kernels, "kernels_split": split,
            "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps, "clocks": clocks,
        }
        if clip:
            line["clip_max_norm"] = max_norm
        if args.pipeline == "unshard":
            line["wrap_units"] = len(units)
            line["unit_param_bytes"] = unit_bytes // 2
        print(json.dumps(line), flush=True)
    del grads, master, m, v, full
    plan.free()
    if gworld > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_sweep(args):
    """--pipeline sweep: the shard step over a grid of shard sizes S x emulated
    ranks N x incoming-gradient dtype x parameter dtype (one tensor of N*S
    elements, rank 0's step), 20 steps per point with state carried forward,
    captured in a CUDA graph and timed over 5 replays (CUDA events around each
    replay; the per-step time is a replay's over 20); points whose buffers do
    not fit in free
    device memory are reported as skipped, points whose working set fits in
    L2 are marked cache-resident (not roofline points)."""
    import torch

    import fsdp_sharded_mixed_gb300 as zs
    import synth
    from synth.workloads import (SWEEP_GRAD_BYTES, SWEEP_PARAM_BYTES, SWEEP_SHARD_SIZES,
                                 SWEEP_WORLDS)

    grank, gworld, local = dist_env()
    if grank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sptr = torch.cuda.current_stream().cuda_stream
    peak, peak_kind = measured_peak()
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    pdt_of = {2: zs.ZS_BF16, 3: zs.ZS_FP24, 4: zs.ZS_FP32}
    warm, reps, replays = max(3, min(args.warmup, 5)), 20, 5
    sizes = [S for S in SWEEP_SHARD_SIZES if S <= (1 << args.sweep_max_log2)]
    worlds = [int(x) for x in args.sweep_worlds.split(",")] if args.sweep_worlds \
        else SWEEP_WORLDS
    only = None
    if args.sweep_only:
        # "log2S:N:grad_bytes:param_bytes,..." selects points of the grid
        only = {tuple(int(x) for x in q.split(":")) for q in args.sweep_only.split(",")}
    points, launches = [], 0
    clocks_s = ClockSampler()
    clocks_s.start()
    for S in sizes:
        torch.cuda.empty_cache()
        free = torch.cuda.mem_get_info()[0]
        for N in worlds:
            for gb in SWEEP_GRAD_BYTES:
                for pb in SWEEP_PARAM_BYTES:
                    if only is not None and (S.bit_length() - 1, N, gb, pb) not in only:
                        continue
                    need = N * S * gb + 12 * S + N * S * pb
                    pt = {"S": S, "N": N, "grad": "bf16" if gb == 2 else "fp32",
                          "param_bytes": pb, "bytes_per_elem": gb * N + 24 + pb,
                          "footprint_gb": need / 1e9}
                    if need > 0.85 * free:
                        pt["skipped"] = f"needs {need / 1e9:.1f} GB, {free / 1e9:.1f} GB free"
                        points.append(pt)
                        continue
                    plan = zs.zs_flatten_plan([N * S], world=N, align_elems=128)
                    grads = [torch.empty(S * gb, dtype=torch.uint8, device=dev) for _ in range(N)]
                    for j, g in enumerate(grads):
                        synth.fill_device(g.data_ptr(), S, seed=1, rank=j, step=1, sigma=1e-3,
                                          bf16=gb == 2, cuda_stream=sptr)
                    master = torch.empty(S, dtype=torch.float32, device=dev)
                    synth.fill_device(master.data_ptr(), S, seed=1, stream=synth.STREAM_MASTER,
                                      sigma=0.02, bf16=False, cuda_stream=sptr)
                    m = torch.zeros(S, dtype=torch.float32, device=dev)
                    v = torch.zeros(S, dtype=torch.float32, device=dev)
                    full = torch.zeros(N * S * pb, dtype=torch.uint8, device=dev)
                    gdt = zs.ZS_BF16 if gb == 2 else zs.ZS_FP32
                    # Warm-up launches (they also make the first-call set-up),
                    # then `reps` steps captured in a CUDA graph, replayed
                    # `replays` times: the per-step time is a replay's time /
                    # reps, free of host launch overhead (at 2^22 elements a
                    # step is ~25 us, less than a launch from Python costs).
                    side = torch.cuda.Stream()
                    side.wait_stream(torch.cuda.current_stream())
                    with torch.cuda.stream(side):
                        for t in range(1, warm + 1):
                            zs.zs_shard_step(plan, 0, 0, S, grads, gdt, master, m, v, full,
                                             pdt_of[pb], hp, t, stream=side.cuda_stream)
                    torch.cuda.synchronize()
                    graph = torch.cuda.CUDAGraph()
                    with torch.cuda.graph(graph, stream=side):
                        for t in range(warm + 1, warm + reps + 1):
                            zs.zs_shard_step(plan, 0, 0, S, grads, gdt, master, m, v, full,
                                             pdt_of[pb], hp, t, stream=side.cuda_stream)
                    graph.replay()
                    torch.cuda.synchronize()
                    ts = []
                    for _ in range(replays):
                        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(
                            enable_timing=True)
                        a.record()
                        graph.replay()
                        b.record()
                        torch.cuda.synchronize()
                        ts.append(a.elapsed_time(b) / reps)
                    del graph
                    launches += reps * (replays + 1)
                    ts.sort()
                    med = statistics.median(ts)
                    gbs = pt["bytes_per_elem"] * S / med / 1e6
                    pt.update({"ms_median": med, "ms_min": ts[0], "ms_max": ts[-1],
                               "gbs": gbs, "frac": gbs / peak})
                    if need < 129e6:
                        pt["cache_resident"] = True
                    points.append(pt)
                    del grads, master, m, v, full
                    plan.free()
    clocks = clocks_s.stop()
    roof = [p for p in points if "gbs" in p and not p.get("cache_resident")]
    value = statistics.median(p["gbs"] for p in roof) if roof else None
    line = {
        "metric": "C5 sweep: shard-step achieved HBM GB/s per (S, N, grad dtype, param dtype), "
                  "median over the roofline points, 1 GPU",
        "value": value, "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": warm,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": "sweep: one tensor of N*S elements, rank 0's step",
                   "pipeline": "sweep", "step_path": args.step_path,
                   "launch_overlap": not args.no_overlap, "shard_sizes": sizes,
                   "worlds": worlds,
                   "grad_bytes": SWEEP_GRAD_BYTES, "param_bytes": SWEEP_PARAM_BYTES,
                   "timing": "20 steps in a CUDA graph, 5 timed replays per point",
                   "l2": "points under 129 MB of buffers are cache-resident, not roofline points"},
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s",
                     "frac": None if value is None else value / peak, "peak_source": peak_kind,
                     "traffic": None,
                     "min_frac": min((p["frac"] for p in roof), default=None),
                     "max_frac": max((p["frac"] for p in roof), default=None)},
        "points": points, "gpu_launches": launches, "clocks": clocks, "e2e": None,
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def run_checkpoint(args, w):
    """--pipeline checkpoint: one rank's fp32 master/m/v shard (device-resident)
    saved to a file, restored at the same world size, and restored into a
    world of N/2 (its rank 0 reads old ranks 0 and 1). Wall-clock GB/s of
    state bytes per leg, beside plain multi-threaded file writes/reads of the
    same bytes on the same file system (the I/O bound of a leg). The legs are
    host I/O; rank 0 alone runs them."""
    import shutil
    import tempfile
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np
    import torch

    import fsdp_sharded_mixed_gb300 as zs
    import synth

    grank, gworld, local = dist_env()
    if grank != 0:
        return
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sptr = torch.cuda.current_stream().cuda_stream
    plan = zs.zs_flatten_plan(w.numels, w.tied_to, world=w.world, align_elems=w.align)
    N, S, P = plan.world, plan.S, plan.P
    M = max(1, N // 2)
    planM = zs.zs_flatten_plan(w.numels, w.tied_to, world=M, align_elems=w.align)
    state_bytes = 3 * 4 * S
    d = args.ckpt_dir or os.path.join(tempfile.gettempdir(), "zs_ckpt_bench")
    os.makedirs(d, exist_ok=True)
    need = 3 * state_bytes + (1 << 30)
    free = shutil.disk_usage(d).free
    if free < need:
        print(json.dumps({"metric": "sharded checkpoint GB/s", "unavailable":
                          f"needs {need / 1e9:.1f} GB free in {d}, has {free / 1e9:.1f} GB"}))
        return
    st = [torch.empty(S, device=dev) for _ in range(3)]
    for k, a in enumerate(st):
        synth.fill_device(a.data_ptr(), S, seed=w.seed + k, stream=synth.STREAM_MASTER,
                          sigma=0.02, p_limit=P, bf16=False, cuda_stream=sptr)
    stM = [torch.empty(planM.S, device=dev) for _ in range(3)]
    paths = [os.path.join(d, f"{w.key}.rank{k}") for k in range(N)]
    same = [paths[0]] + [None] * (N - 1)
    resize = [paths[0], paths[1] if N > 1 else None] + [None] * (N - 2)
    def drop_cache(path):
        """Write the file back and drop it from the page cache (a cold read)."""
        fd = os.open(path, os.O_RDONLY)
        try:
            os.fsync(fd)
            os.posix_fadvise(fd, 0, 0, os.POSIX_FADV_DONTNEED)
        finally:
            os.close(fd)

    # (leg, call, bytes of state it moves). A save goes to a new file, as a
    # training job's does: the previous one is removed before the clock starts.
    legs = [
        ("save", lambda: zs.zs_checkpoint_save(plan, 0, *st, 10, paths[0]), state_bytes),
        ("load_same_world", lambda: zs.zs_checkpoint_load(plan, 0, same, *st), state_bytes),
        (f"load_into_world_{M}", lambda: zs.zs_checkpoint_load(planM, 0, resize, *stM),
         3 * 4 * planM.S),
    ]
    if N > 1:
        zs.zs_checkpoint_save(plan, 1, *st, 10, paths[1])
    warm = min(args.warmup, 3)
    reps = args.ckpt_reps
    results = {}
    for name, fn, nbytes in legs:
        ts = []
        for i in range(warm + reps):
            if name == "save" and os.path.exists(paths[0]):
                os.remove(paths[0])
            if args.ckpt_cold and name != "save":
                for p in paths[:2]:
                    if os.path.exists(p):
                        drop_cache(p)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            fn()
            t = time.perf_counter() - t0
            if i >= warm:
                ts.append(t)
        results[name] = {"s_median": statistics.median(ts), "s_min": min(ts), "bytes": nbytes,
                         "gbs": nbytes / statistics.median(ts) / 1e9}
        log(f"checkpoint {name}: {results[name]}")
    # restored state equals the saved state (same world) — a cheap end check
    got = [torch.empty(S, device=dev) for _ in range(3)]
    zs.zs_checkpoint_load(plan, 0, same, *got)
    ok = all(torch.equal(a.view(torch.int32), b.view(torch.int32)) for a, b in zip(got, st))
    del got
    # The I/O bound of a leg on this file system: the same bytes written from
    # host memory into a new, preallocated file by one thread in 64 MiB pwrites
    # (the fastest way found to fill a new file), and read back by 16 threads
    # in 8 MiB preadv calls.
    buf = np.empty(state_bytes, np.uint8)
    buf[::4096] = 1
    plain = os.path.join(d, "plain.bin")
    mv = memoryview(buf)

    def plain_write():
        fd = os.open(plain, os.O_RDWR | os.O_CREAT | os.O_TRUNC, 0o644)
        try:
            os.posix_fallocate(fd, 0, state_bytes)
            for o in range(0, state_bytes, 64 << 20):
                os.pwrite(fd, mv[o:o + (64 << 20)], o)
        finally:
            os.close(fd)

    def plain_read():
        fd = os.open(plain, os.O_RDONLY)
        try:
            with ThreadPoolExecutor(16) as ex:
                list(ex.map(lambda o: os.preadv(fd, [mv[o:o + (8 << 20)]], o),
                            range(0, state_bytes, 8 << 20)))
        finally:
            os.close(fd)

    plain_t = {}
    for kind, fn in (("write", plain_write), ("read", plain_read)):
        ts = []
        for i in range(warm + reps):
            if kind == "write" and os.path.exists(plain):
                os.remove(plain)
            if kind == "read" and args.ckpt_cold:   # the timed loads' cold start
                drop_cache(plain)
            t0 = time.perf_counter()
            fn()
            if i >= warm:
                ts.append(time.perf_counter() - t0)
        plain_t[kind] = statistics.median(ts)
    del buf
    for p in paths[:2] + [plain]:
        if os.path.exists(p):
            os.remove(p)
    w_gbs = state_bytes / plain_t["write"] / 1e9
    r_gbs = state_bytes / plain_t["read"] / 1e9
    for name, r in results.items():
        r["frac_of_plain_io"] = r["gbs"] / (w_gbs if name == "save" else r_gbs)
    value = min(r["gbs"] for r in results.values())
    worst = min(results, key=lambda k: results[k]["gbs"])
    line = {
        "metric": "sharded checkpoint GB/s of fp32 optimizer state (save; restore at the same "
                  f"world; restore into world {M}), 1 GPU",
        "value": value, "unit": "GB/s", "n_gpus": 1, "steps": reps, "warmup": warm,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": f"{w.key}: {w.title}", "pipeline": "checkpoint",
                   "shard_elems": S, "state_bytes": state_bytes, "old_world": N,
                   "new_world": M, "files": "cold (fsync + fadvise DONTNEED before each load)"
                   if args.ckpt_cold else "warm page cache", "dir": d},
        "legs": results, "restored_equal": ok,
        "plain_io_gbs": {"write": w_gbs, "read": r_gbs,
                         "note": "the same bytes from host memory: new preallocated file, one "
                                 "writer, 64 MiB pwrite; read back by 16 threads, 8 MiB preadv"
                                 + (" from a dropped page cache" if args.ckpt_cold else "")},
        "roofline": {"bound": "io", "achieved": results[worst]["gbs"],
                     "peak": w_gbs if worst == "save" else r_gbs, "unit": "GB/s",
                     "frac": results[worst]["frac_of_plain_io"], "kernel": worst,
                     "peak_source": "plain file I/O measured in this run", "traffic": None},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": state_bytes,
                "d2h_bytes_per_step": state_bytes,
                "note": "every leg moves the state between HBM and a file"},
        "gpu_launches": 3 * (warm + reps), "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)
    plan.free()
    planM.free()


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="llama-7b")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--graph", action="store_true",
                    help="time one replay of a CUDA graph holding the K launches")
    ap.add_argument("--rank", type=int, default=0,
                    help="the emulated rank GPU 0 runs (GPU g runs rank + g mod N)")
    ap.add_argument("--buckets", action="store_true",
                    help="step pipeline: one call per gradient bucket of the workload "
                         "(GPT-2-small: 25M-element buckets), as its ZeRO-2 job runs it")
    ap.add_argument("--pipeline",
                    choices=["step", "clip", "accum", "accum_clip", "unshard", "gather",
                             "checkpoint", "sweep"],
                    default="step",
                    help="step: the fused shard step; clip: global-norm pass + clip "
                         "coefficient + clipped step; accum: G-1 accumulations + the "
                         "accumulated step; accum_clip: accum with the norm of the "
                         "accumulated gradient and a clipped accumulated step; gather: the emulated AllGather's assembly of "
                         "the other ranks' shards into the flat buffer; unshard: FSDP2 "
                         "copy-out of every wrap unit's "
                         "gathered parameters; checkpoint: save / restore / resharding "
                         "restore of one rank's optimizer state; sweep: the step over "
                         "shard sizes x N x gradient and parameter dtypes")
    ap.add_argument("--units", type=int, default=0,
                    help="--pipeline unshard: only the first K wrap units (0 = all)")
    ap.add_argument("--micro-steps", type=int, default=4,
                    help="G, micro-batches per optimizer step for --pipeline accum")
    ap.add_argument("--step-path", choices=["auto", "direct", "staged"], default="auto",
                    help="the step's kernel: chosen per call (auto), the register-streaming "
                         "kernel (direct) or the bulk-async staged kernel where it applies")
    ap.add_argument("--sweep-max-log2", type=int, default=30,
                    help="--pipeline sweep: largest shard size 2^k")
    ap.add_argument("--sweep-worlds", default=None,
                    help="--pipeline sweep: emulated world sizes N (comma list; default "
                         "2,4,8,16,64)")
    ap.add_argument("--sweep-only", default=None,
                    help="--pipeline sweep: only these points, 'log2S:N:gbytes:pbytes,...'")
    ap.add_argument("--ckpt-dir", default=None,
                    help="directory for --pipeline checkpoint files (default: a temp dir)")
    ap.add_argument("--ckpt-reps", type=int, default=3)
    ap.add_argument("--ckpt-cold", action="store_true",
                    help="drop the files from the page cache before each timed load")
    ap.add_argument("--no-overlap", action="store_true",
                    help="ordinary kernel launches (no programmatic dependent launch)")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--e2e-chunks", type=int, default=32)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-copy-ceiling", action="store_true",
                    help="skip the device-to-device copy measured beside the roofline")
    ap.add_argument("--cpu-sample-elems", type=int, default=0,
                    help="cpu_baseline: the oracle on the first K elements of the shard "
                         "(0 = the full shard)")
    ap.add_argument("--cpu-steps", type=int, default=1)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from synth.workloads import WORKLOADS
    w = WORKLOADS[args.workload]
    if args.impl != "reference" and args.step_path != "auto":
        import fsdp_sharded_mixed_gb300 as zs
        zs.zs_set_step_path({"direct": 1, "staged": 2}[args.step_path])
    if args.impl != "reference" and args.no_overlap:
        import fsdp_sharded_mixed_gb300 as zs
        zs.zs_set_launch_overlap(0)
    if args.impl == "reference":
        run_reference(args, w)
    elif args.pipeline == "checkpoint":
        run_checkpoint(args, w)
    elif args.pipeline == "sweep":
        run_sweep(args)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
