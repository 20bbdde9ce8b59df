"""Benchmark of the fused ZeRO-1 optimizer step on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-cpu-baseline] [--no-e2e]

A step is one pass of the whole hot path over one batch: the M replicas'
bf16 gradients are reduce-scattered (rank-order fp32 sum, scaled by 1/(B*S)),
the fp32 master/m/v get the AdamW update, the overflow flag is ORed and the
bf16 parameters are written once (all-gather) - one fused kernel launch.  The
default workload is the largest flat buffer that the method is stated on
that fits one GPU: 1.3B parameters (P = 1,300,000,768 after padding to
multiples of 8*128), M = 8 replicas, B = 1024; its 54.6 GB of traffic per step
is far larger than the 129 MB L2, so no flush is needed between steps.

Under torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (weak scaling, no collective on the data path); the
timed region is bracketed by a barrier and a device synchronize on every
rank, and the slowest rank's time counts.

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
METRIC = "params/s and achieved HBM GB/s (% of GB300 peak) per fused ZeRO-1 step"
NOMINAL_HBM_GBS = 7900.0   # GB300 HBM3e, nominal
# The fused kernel's sources, hashed in this order (concatenated) to tell
# whether recorded ncu traffic was taken on the kernel as it stands.
KERNEL_SOURCES = [os.path.join(ROOT, "zero_sharded_mixed_zero1_gb300", "csrc", f)
                  for f in ("zero1_fused.cu", "zero1_device.cuh", "zero1_internal.h")]


# ------------------------------------------------------------ helpers ------

def algorithmic_bytes(n_real: int, n_pad: int, M: int) -> int:
    """Bytes the step must move: per real parameter M bf16 gradient reads,
    fp32 master/m/v read and written and one bf16 parameter write (2M + 26);
    per padding element only the fp32 state (24)."""
    return n_real * (2 * M + 24 + 2) + n_pad * 24


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# ncu DRAM counters of the fused kernel, captured on a small case of the same
# kernel (16,777,216 parameters, M = 8: 705 MB per launch, above L2) and
# scaled to a launch of the timed workload by its algorithmic bytes.
TRAFFIC_PROFILE = os.path.join(ROOT, "profiles", "k_fused_step_dram_prof_16M_M8.md")


def recorded_traffic(M: int, bytes_launch: int):
    """DRAM read+write bytes per launch, scaled from the committed ncu
    summary of the small case, if that was taken on the kernel source as it
    stands now and with the same replica count (else None).  Returns
    (bytes, note)."""
    if not os.path.exists(TRAFFIC_PROFILE):
        return None, None
    text = open(TRAFFIC_PROFILE).read()
    sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    tr = re.search(r"dram_bytes_per_launch:\s*([0-9]+)", text)
    alg = re.search(r"algorithmic_bytes_per_launch:\s*([0-9]+)", text)
    reps = re.search(r"replicas:\s*([0-9]+)", text)
    if not (sha and tr and alg and reps) or int(reps.group(1)) != M:
        return None, None
    cur = hashlib.sha256(b"".join(open(f, "rb").read() for f in KERNEL_SOURCES)).hexdigest()
    if sha.group(1) != cur:
        return None, None
    ratio = int(tr.group(1)) / int(alg.group(1))
    return int(round(ratio * bytes_launch)), (
        f"ncu dram__bytes_read.sum + dram__bytes_write.sum of a steady-state launch on the 16,777,216-parameter "
        f"case ({int(tr.group(1))} B against {int(alg.group(1))} B algorithmic, ratio {ratio:.4f}), scaled to "
        f"this launch's {bytes_launch} algorithmic bytes")


def host_cpu() -> dict:
    """This host's logical CPU count and CPU model."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        m = re.search(r"^Model name:\s*(.+)$", out, re.M)
        model = m.group(1).strip() if m else None
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        m = re.search(r"^model name\s*:\s*(.+)$", open("/proc/cpuinfo").read(), re.M)
        model = m.group(1).strip() if m else None
    import platform
    return {"host_cpu_count": os.cpu_count(), "cpu_model": model or "unknown", "machine": platform.machine()}


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs."""
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 20):
        self.proc = None
        try:
            self.f = tempfile.NamedTemporaryFile("w", prefix="clocks_", suffix=".csv", delete=False)
            self.path = self.f.name
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv",
                 "-lms", str(period_ms)], stdout=self.f, stderr=subprocess.DEVNULL)
            deadline = time.time() + 5
            while time.time() < deadline and os.path.getsize(self.path) < 200:
                time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self, t0: float, t1: float) -> dict:
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = list(csv.reader(open(self.path)))
        if len(rows) < 2:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        head = rows[0]
        # nvidia-smi renames some columns in its header (clocks.sm becomes
        # clocks.current.sm): map by position in the query instead
        col = {name: i for i, name in enumerate(self.FIELDS.split(","))}
        sm, smax, reasons, n = [], [], set(), 0
        for r in rows[1:]:
            if len(r) != len(head):
                continue
            try:
                ts = time.mktime(time.strptime(r[col["timestamp"]].strip().split(".")[0], "%Y/%m/%d %H:%M:%S"))
            except ValueError:
                continue
            if ts < int(t0) or ts > t1 + 1:
                continue
            try:
                sm_now = float(r[col["clocks.sm"]].split()[0])
                sm_max = float(r[col["clocks.max.sm"]].split()[0])
            except (ValueError, IndexError):
                continue
            n += 1
            sm.append(sm_now)
            smax.append(sm_max)
            for key in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"):
                if r[col["clocks_event_reasons." + key]].strip() == "Active":
                    reasons.add(key)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, world: int) -> float:
    """The slowest rank's value (the rank-0 value when world == 1)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------ the oracle leg -----

def oracle_sample_rate(w, elems: int, seconds: float, seed: int = 7):
    """Time the CPU oracle (single-threaded C, as it stands) on a sample of
    `elems` elements of workload w, repeating steps for about `seconds`.
    Returns (elements per second, steps run)."""
    import oracle  # test infrastructure: only this baseline leg uses it
    from zero_sharded_mixed_zero1_gb300 import synth
    grads = [synth.normal_bf16(elems, w.grad_std * w.S, synth.seed_of(seed, r)).view(torch.int16).numpy()
             .view(np.uint16) for r in range(w.M)]
    master = synth.normal_f32(elems, w.master_std, synth.seed_of(seed, 99)).numpy()
    m = np.zeros(elems, np.float32)
    v = np.zeros(elems, np.float32)
    params = np.zeros(elems, np.uint16)
    t, done, t0 = 1, 0, time.perf_counter()
    while True:
        hp = oracle.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                          loss_scale=w.S, global_batch=w.B, step=t)
        oracle.zero1_step(grads, elems, master, m, v, params, hp)
        done += 1
        t += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return elems * done / (time.perf_counter() - t0), done


def run_reference(args, w) -> None:
    """The reference arm: the CPU oracle as it stands, on this host's cores,
    timed on a bounded sample of the workload per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    # size each step's sample so the whole run stays near a minute
    rate, _ = oracle_sample_rate(w, 1 << 16, 0.5)
    total_steps = args.steps + args.warmup
    elems = int(max(4096, min(w.n, rate * 60.0 / max(1, total_steps))))
    import oracle
    from zero_sharded_mixed_zero1_gb300 import synth
    grads = [synth.normal_bf16(elems, w.grad_std * w.S, synth.seed_of(11, r)).view(torch.int16).numpy()
             .view(np.uint16) for r in range(w.M)]
    master = synth.normal_f32(elems, w.master_std, synth.seed_of(11, 99)).numpy()
    m, v = np.zeros(elems, np.float32), np.zeros(elems, np.float32)
    params = np.zeros(elems, np.uint16)

    def step(t):
        hp = oracle.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                          loss_scale=w.S, global_batch=w.B, step=t)
        oracle.zero1_step(grads, elems, master, m, v, params, hp)

    for t in range(1, args.warmup + 1):
        step(t)
    t0 = time.perf_counter()
    for t in range(args.warmup + 1, args.warmup + args.steps + 1):
        step(t)
    dt = time.perf_counter() - t0
    value = elems * args.steps / dt
    sample = f"{elems} of {w.n} elements per step, M={w.M} replicas, single-threaded C oracle"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": config_of(w),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": sample,
                         **host_cpu()},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------- our arm ---------

def host_link_rates(dev, nbytes: int = 1 << 30, reps: int = 4) -> dict:
    """Copy-engine bandwidth of the host link in GB/s, measured with CUDA
    events: pinned host -> HBM on two streams, HBM -> pinned host, and both
    directions at once (the sum of the two)."""
    host_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    host_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    dev_a = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    dev_b = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    host_in.fill_(1)
    main = torch.cuda.current_stream(dev)
    side = [torch.cuda.Stream(device=dev) for _ in range(2)]
    half = nbytes // 2

    def timed(jobs):
        """jobs: one list of (dst, src) copies per side stream; returns seconds."""
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(2):                       # the first round warms up
            start.record(main)
            for st, copies in zip(side, jobs):
                st.wait_stream(main)
                with torch.cuda.stream(st):
                    for _ in range(reps):
                        for dst, src in copies:
                            dst.copy_(src, non_blocking=True)
            for st in side[:len(jobs)]:
                main.wait_stream(st)
            end.record(main)
            torch.cuda.synchronize(dev)
        return start.elapsed_time(end) * 1e-3

    # other work on a shared host only ever lowers these rates: keep the best
    # of three measurements as the link's capacity
    h2d = d2h = both = 0.0
    for _ in range(3):
        h2d = max(h2d, nbytes * reps / timed([[(dev_a[:half], host_in[:half])],
                                               [(dev_a[half:], host_in[half:])]]) / 1e9)
        d2h = max(d2h, nbytes * reps / timed([[(host_out, dev_b)]]) / 1e9)
        both = max(both, 2 * nbytes * reps / timed([[(dev_a, host_in)], [(host_out, dev_b)]]) / 1e9)
    return {"h2d_gbs": h2d, "d2h_gbs": d2h, "both_directions_gbs": both,
            "method": f"cudaMemcpyAsync of {nbytes >> 20} MiB pinned buffers x {reps}, CUDA events, "
                      "best of 3"}


def link_roofline(link: dict, h2d_bytes: int, d2h_bytes: int, seconds_per_step: float) -> dict:
    """The host link's lower bound on an end-to-end step that moves h2d_bytes
    in and d2h_bytes out: max(in / h2d rate, out / d2h rate, both / rate of
    both directions at once), and the measured step against it."""
    bound_s = max(h2d_bytes / (link["h2d_gbs"] * 1e9), d2h_bytes / (link["d2h_gbs"] * 1e9),
                  (h2d_bytes + d2h_bytes) / (link["both_directions_gbs"] * 1e9))
    return {"bound": "host_link", "link_bytes_per_step": h2d_bytes + d2h_bytes,
            "achieved_gbs": (h2d_bytes + d2h_bytes) / seconds_per_step / 1e9,
            "bound_ms": bound_s * 1e3, "ms_per_step": seconds_per_step * 1e3,
            "frac": bound_s / seconds_per_step, **link}


def config_of(w, state_on_host: bool = False, op: str = "step", transfer: str = "zero_copy") -> dict:
    c = {"workload": w.name, "n": w.n, "M": w.M, "align": w.align, "global_batch": w.B,
         "loss_scale": w.S, "shards": list(w.shards), "io": "bf16 grads and params, fp32 master/m/v",
         "l2": "inputs larger than L2 (no flush)", "parallelism": "replicas only"}
    if state_on_host:
        c["state"] = "fp32 master/m/v in pinned host memory (offload)"
        c["offload_transfer"] = {"zero_copy": "the kernel reads and writes the host state over the link",
                                 "copy_engines": "state chunks staged through HBM by the copy engines"}[transfer]
    if op == "dynamic":
        c["loss_scaling"] = "dynamic, device-resident (window 1000, hysteresis 2, factor 2)"
    elif op in ("dynamic_pingpong", "bucketed_pingpong"):
        c["loss_scaling"] = ("dynamic, device-resident (window 1000, hysteresis 2, factor 2), ping-pong state "
                             "(two copies of master/m/v)")
        if op == "bucketed_pingpong":
            c["op"] = "gradient buckets updated as they arrive, skip decided after the last bucket"
    elif op != "step":
        c["op"] = op + " (component measurement, not the step)"
    return c


def run_ours(args, w) -> None:
    import zero_sharded_mixed_zero1_gb300 as z
    from zero_sharded_mixed_zero1_gb300 import build as zbuild
    from zero_sharded_mixed_zero1_gb300 import synth

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)

    # CPU baseline first (rank 0, N = 1 only), before any GPU work
    cpu_baseline = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = 1 << 22
        rate, nsteps = oracle_sample_rate(w, sample, args.cpu_seconds)
        cpu_baseline = {"value": rate, "unit": "params/s", "cores": 1, "kind": "oracle",
                        "sample": f"{nsteps} steps over {sample} of {w.n} elements, M={w.M} replicas, "
                                  f"single-threaded C oracle", **host_cpu()}

    if rank == 0 and zbuild.is_stale():
        zbuild.build()
    barrier(world)
    z.load()

    plan = z.zero1_plan(w.n, w.M, w.align)
    sb, se = w.shards
    base, L, nv = plan.shard_range(sb, se)
    stream = torch.cuda.current_stream(dev)

    # two gradient sets, alternated step to step (fresh draws per replica)
    gsets = [[synth.normal_bf16(nv, w.grad_std * w.S, synth.seed_of(w.seed, k, r, rank), dev)
              for r in range(w.M)] for k in range(2)]
    master = torch.zeros(L, dtype=torch.float32, device=dev)
    master[:nv] = synth.normal_f32(nv, w.master_std, synth.seed_of(w.seed, 1, rank), dev)
    m = torch.zeros(L, dtype=torch.float32, device=dev)
    v = torch.zeros(L, dtype=torch.float32, device=dev)
    if args.state_on_host:        # optimizer-state offload: master/m/v in pinned host memory
        master, m, v = (x.cpu().pin_memory() for x in (master, m, v))
    params = torch.zeros(nv, dtype=torch.bfloat16, device=dev)
    flag = torch.zeros(1, dtype=torch.int32, device=dev)

    def hp(t):
        return z.AdamW(lr=w.lr, beta1=w.beta1, beta2=w.beta2, eps=w.eps, weight_decay=w.weight_decay,
                       loss_scale=w.S, global_batch=w.B, step=t)

    def second_copy(x):
        """The ping-pong state's other copy, where x lives (pinned host or HBM)."""
        return torch.empty(x.shape, dtype=x.dtype, pin_memory=True) if x.device.type == "cpu" else torch.empty_like(x)

    op = args.op if "pingpong" in args.op else ("dynamic" if args.dynamic_loss_scale else args.op)
    if op in ("dynamic", "dynamic_pingpong", "bucketed_pingpong"):
        policy = z.LossScalePolicy(initial_scale=w.S if w.S > 1 else 2.0 ** 12, factor=2.0, window=1000,
                                   hysteresis=2, min_scale=1.0)
        scaler = z.new_scaler(dev)
        z.zero1_scaler_init(scaler, policy, hp(1))
        if op == "dynamic" and args.state_on_host and args.offload_transfer == "copy_engines":
            # the fp16 block with offload_optimizer: state staged through HBM,
            # the skip decided by an overflow pass before any chunk is updated
            staged = {id(gs): z.HostStreamedStep(plan, sb, se, gs, master, m, v, params,
                                                 chunk_elems=args.chunk_elems, stream=stream) for gs in gsets}

            def launch(gr, tt, st=None):
                staged[id(gr)].dynamic(hp(tt), scaler, policy)
            n_chunks = len(staged[id(gsets[0])].pieces)
            op_kernel = (f"staged dynamic step: k_overflow + k_fused_step_scaled per {args.chunk_elems}-element "
                         "chunk (state staged through HBM by the copy engines) + k_scaler_update")
            launches_per_step, op_bytes = n_chunks + 2, algorithmic_bytes(nv, L - nv, w.M) + 2 * w.M * nv
        elif op == "dynamic":
            sums = torch.empty(L, dtype=torch.float32, device=dev)

            def launch(gr, tt, st=None):
                z.zero1_step_dynamic(plan, sb, se, gr, master, m, v, params, hp(tt), scaler, policy, sums,
                                     stream=st)
            op_kernel = "dynamic step: k_reduce_scatter + k_apply_sums + k_scaler_update"
            launches_per_step, op_bytes = 3, algorithmic_bytes(nv, L - nv, w.M) + 8 * L
        elif op == "dynamic_pingpong":
            pairs = [[x, second_copy(x)] for x in (master, m, v)]

            def launch(gr, tt, st=None):
                z.zero1_step_dynamic_pingpong(plan, sb, se, gr, *pairs, params, hp(tt), scaler, policy, stream=st)
            op_kernel = ("dynamic step, ping-pong state: k_fused_step_pingpong + k_restore_params (returns at "
                         "once without overflow) + k_scaler_update")
            launches_per_step, op_bytes = 3, algorithmic_bytes(nv, L - nv, w.M)
        else:
            # gradient buckets of reduce_bucket_size elements updated as they
            # arrive, the skip decided once all have run
            pairs = [[x, second_copy(x)] for x in (master, m, v)]
            buckets = z.PingPongBuckets(plan, sb, se, *pairs, params, scaler, policy, stream=stream)
            bucket = args.bucket_elems
            cuts = list(range(0, L, bucket)) + [L]

            def launch(gr, tt, st=None):
                h = hp(tt)
                for e0, e1 in zip(cuts[:-1], cuts[1:]):
                    k = max(0, min(nv, e1) - e0)
                    buckets.bucket(e0, e1, [g[e0:e0 + k] for g in gr], h)
                buckets.finish(h)
            op_kernel = (f"dynamic step, ping-pong state, buckets of {bucket} elements: k_fused_step_pingpong "
                         "per bucket + k_restore_params + k_scaler_update")
            launches_per_step, op_bytes = len(cuts) + 1, algorithmic_bytes(nv, L - nv, w.M)
        if args.graph:
            # S and t live on the device: one attempt per gradient set is
            # captured once and replayed every step
            for gs in gsets:
                launch(gs, 1)
            torch.cuda.synchronize(dev)
            z.zero1_scaler_init(scaler, policy, hp(1))
            graphs = {}
            for gs in gsets:
                gr_ = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr_):
                    launch(gs, 1)
                graphs[id(gs)] = gr_
            z.zero1_scaler_init(scaler, policy, hp(1))
            torch.cuda.synchronize(dev)

            def launch(gr, tt, st=None):      # noqa: F811 - replay instead of the eager call
                graphs[id(gr)].replay()
            op_kernel += " (replayed from a CUDA graph)"
    elif op == "overflow_check":
        def launch(gr, tt, st=None):
            z.zero1_overflow_check(plan, sb, se, gr, flag, stream=st)
        launches_per_step, op_bytes, op_kernel = 1, 2 * w.M * nv, "k_overflow"
    elif op == "allreduce":
        if (sb, se) != (0, w.M):
            raise SystemExit("--op allreduce needs a workload over all shards")
        outs = [torch.empty(nv, dtype=torch.bfloat16, device=dev) for _ in range(w.M)]

        def launch(gr, tt, st=None):
            z.dp_allreduce(plan, gr, outs, 1.0 / (w.B * w.S), stream=st)
        launches_per_step, op_bytes, op_kernel = 1, 4 * w.M * nv, "k_allreduce (bf16 out)"
    elif op == "unfused":
        gbuf = torch.empty(L, dtype=torch.float32, device=dev)

        def launch(gr, tt, st=None):
            h = hp(tt)
            inv = 1.0 / (w.B * w.S)
            z.zero1_reduce_scatter(plan, sb, se, gr, inv, gbuf, flag, stream=st)
            z.zero1_adamw_update(plan, sb, se, gbuf, master, m, v, h, stream=st)
            z.zero1_all_gather(plan, sb, se, master, params, stream=st)
        launches_per_step = 3
        op_bytes = nv * (2 * w.M + 4) + (L - nv) * 4 + 28 * L + 6 * nv
        op_kernel = "unfused: k_reduce_scatter (fp32) + k_adamw + k_all_gather"
    elif op == "tma":
        def launch(gr, tt, st=None):
            z.zero1_step_tma(plan, sb, se, gr, master, m, v, params, hp(tt), flag, stream=st)
        launches_per_step, op_bytes = 1, algorithmic_bytes(nv, L - nv, w.M)
        op_kernel = "k_fused_step_tma (shared-memory staging by bulk copies)"
    elif op == "bucketed":
        # reduce_bucket_size 5e7 elements, as in the pages' DeepSpeed config
        bucket = args.bucket_elems
        cuts = list(range(0, L, bucket)) + [L]
        base_e = sb * plan.shard

        def launch(gr, tt, st=None):
            h = hp(tt)
            for e0, e1 in zip(cuts[:-1], cuts[1:]):
                k = max(0, min(nv, e1) - e0)
                z.zero1_step_bucket(plan, base_e + e0, base_e + e1, [g[e0:e0 + k] for g in gr], master[e0:],
                                    m[e0:], v[e0:], params[e0:] if e0 < nv else params[:0], h, flag, stream=st)
        launches_per_step, op_bytes = len(cuts) - 1, algorithmic_bytes(nv, L - nv, w.M)
        op_kernel = f"k_fused_step per bucket of {bucket} elements"
    else:
        # one prepared step per gradient set: buffers validated once, then each
        # call passes only the hyperparameters (a few microseconds of host time)
        launches_per_step, op_bytes = 1, algorithmic_bytes(nv, L - nv, w.M)
        if args.state_on_host and args.offload_transfer == "copy_engines":
            prepared = {id(gs): z.HostStreamedStep(plan, sb, se, gs, master, m, v, params,
                                                   chunk_elems=args.chunk_elems, overflow_flag=flag, stream=stream)
                        for gs in gsets}
            launches_per_step = len(prepared[id(gsets[0])].pieces)
            op_kernel = (f"k_fused_step per {args.chunk_elems}-element chunk, state chunks staged through HBM "
                         "by the copy engines")
        else:
            prepared = {id(gs): z.FusedStep(plan, sb, se, gs, master, m, v, params, flag, stream=stream)
                        for gs in gsets}
            op_kernel = f"k_fused_step<M={w.M}>" if w.M <= 8 else "k_fused_step_grouped"
            if args.state_on_host:
                op_kernel = f"k_fused_step_offload<{w.M if w.M <= 8 else 0}>"

        def launch(gr, tt, st=None):
            prepared[id(gr)](hp(tt))

    t = 1
    for _ in range(args.warmup):
        launch(gsets[t % 2], t)
        t += 1
    torch.cuda.synchronize(dev)

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(2 * args.steps)]
    sampler = ClockSampler(dev.index) if rank == 0 else None
    barrier(world)
    torch.cuda.synchronize(dev)
    wall0 = time.time()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(args.steps):
        evs[2 * i].record(stream)
        launch(gsets[t % 2], t, stream)
        evs[2 * i + 1].record(stream)
        t += 1
    end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    wall1 = time.time()
    ms_local = start.elapsed_time(end)
    # the launch shape of the step's last streaming kernel (the fused kernel for the default op)
    try:
        shape = z.debug_last_launch()
        last_launch = {"grid": shape["grid"], "block": shape["block"], "blocks_per_sm": shape["blocks_per_sm"],
                       "fp32_32_byte_accesses": shape["w32"]}
    except z.Zero1Error:
        last_launch = None
    launch_ms = np.array([evs[2 * i].elapsed_time(evs[2 * i + 1]) for i in range(args.steps)])
    kernel_ms = float(launch_ms.mean())
    clocks = sampler.summary(wall0, wall1) if sampler else None
    if sampler:
        sampler.stop()
    ms_total = max_over_ranks(ms_local, world)
    overflow = int(flag.item())
    if args.no_e2e or op != "step":
        del gsets

    # end to end through the public API with host buffers: each step's
    # gradients start in pinned host memory and the step's parameters and
    # flag end in pinned host memory.  `e2e`: the fused kernel reads the
    # pinned gradients and writes the pinned parameters over the host link.
    # `e2e_staged`: the copy engines stage the gradients to HBM chunk by chunk,
    # overlapping the step on the previous chunk (zero1_staged_step).
    e2e = e2e_staged = None
    e2e_note = None
    if not args.no_e2e and op == "step":
        # every rank on this host pins its gradients and parameters: leave the
        # end-to-end leg out rather than exhaust host memory
        need = (w.M + 1) * nv * 2 * int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
        # one decision for all ranks (they meet in barriers inside the leg)
        if max_over_ranks(1.0 if need > 0.6 * avail else 0.0, world) > 0:
            e2e_note = (f"end-to-end leg skipped: {need / 1e9:.1f} GB of pinned host memory needed on this host, "
                        f"{avail / 1e9:.1f} GB available on rank {rank}'s check")
    if not args.no_e2e and op == "step" and e2e_note is None:
        # its own step count: each end-to-end step crosses the host link and
        # takes ~100 ms at 1.3B parameters, and a short run's mean is at the
        # mercy of one slow step on a shared host
        e2e_steps = max(3, args.e2e_steps)
        # the e2e gradients: drawn on the device (fast even at 1.3B x 8), then
        # placed in pinned host memory before anything is timed
        host_g = []
        refused = None
        try:
            for r in range(w.M):
                h = torch.empty(nv, dtype=torch.bfloat16, pin_memory=True)
                h.copy_(synth.normal_bf16(nv, w.grad_std * w.S, synth.seed_of(w.seed, 7, r, rank), dev))
                host_g.append(h)
            host_p = torch.empty(nv, dtype=torch.bfloat16, pin_memory=True)
            host_f = torch.empty(1, dtype=torch.int32, pin_memory=True)
        except RuntimeError as e:          # the host refused to pin this much memory
            refused = str(e).splitlines()[0] if str(e) else type(e).__name__
        # one decision for all ranks (they meet in barriers inside the leg)
        if max_over_ranks(1.0 if refused else 0.0, world) > 0:
            host_g = host_p = host_f = None
            e2e_note = f"end-to-end leg skipped: pinning the host buffers failed ({refused or 'on another rank'})"
    if not args.no_e2e and op == "step" and e2e_note is None:
        del gsets
        streamed = z.HostStreamedStep(plan, sb, se, host_g, master, m, v, params, chunk_elems=args.chunk_elems,
                                      params_host=host_p, overflow_flag=flag, stream=stream)

        def copy_step(tt):
            streamed(hp(tt))
            host_f.copy_(flag, non_blocking=True)
            stream.synchronize()

        def zero_copy_step(tt):
            z.zero1_reduce_scatter_adamw_allgather(plan, sb, se, host_g, master, m, v, host_p, hp(tt), flag,
                                                   stream=stream)
            host_f.copy_(flag, non_blocking=True)
            stream.synchronize()

        def timed(fn):
            """Whole-loop seconds (slowest rank) and each step's seconds:
            every step ends with a stream synchronize, so the wall-clock
            delta of one step is that step's end-to-end time."""
            nonlocal t
            fn(t)
            t += 1
            barrier(world)
            w0 = time.perf_counter()
            per_step = []
            for _ in range(e2e_steps):
                s0 = time.perf_counter()
                fn(t)
                per_step.append(time.perf_counter() - s0)
                t += 1
            barrier(world)
            return max_over_ranks(time.perf_counter() - w0, world), np.array(per_step)

        copy_s, copy_steps = timed(copy_step)
        zero_s, zero_steps = timed(zero_copy_step)
        del streamed
        link = host_link_rates(dev)
        bi, bo = w.M * nv * 2, nv * 2 + 4

        def step_stats(steps_s):
            return {"ms_per_step_median": float(np.median(steps_s)) * 1e3, "ms_per_step_min": float(steps_s.min()) * 1e3,
                    "ms_per_step_max": float(steps_s.max()) * 1e3}

        def roof(total_s, steps_s):
            r = link_roofline(link, bi, bo, total_s / e2e_steps)
            r["frac_median_step"] = r["bound_ms"] / (float(np.median(steps_s)) * 1e3)
            return r

        e2e_staged = {"value": world * nv * e2e_steps / copy_s, "unit": "params/s",
                      "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
                      **step_stats(copy_steps),
                      "transfer": f"the gradients staged to HBM in {args.chunk_elems}-element chunks by the copy "
                                  "engines (zero1_staged_step), overlapping the step on the previous chunk; params "
                                  "and flag copied back",
                      "roofline": roof(copy_s, copy_steps)}
        e2e = {"value": world * nv * e2e_steps / zero_s, "unit": "params/s",
               "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo, "steps": e2e_steps,
               **step_stats(zero_steps),
               "transfer": "every step the fused kernel reads the M gradient buffers from pinned host memory and "
                           "writes the bf16 params to pinned host memory over NVLink-C2C (no staging copy); "
                           "the flag is copied back and the stream synchronised",
               "roofline": roof(zero_s, zero_steps)}
        del host_g

    # with the state in host memory the step is bound by the host link: 12 B
    # of master/m/v in and 12 B out per element, measured against the link
    offload_link = None
    if args.state_on_host and op in ("step", "dynamic", "dynamic_pingpong", "bucketed_pingpong"):
        offload_link = link_roofline(host_link_rates(dev), 12 * L, 12 * L, ms_total * 1e-3 / args.steps)
        # host-link steps see occasional stalls from other work on the shared
        # host: the median step against the same bound
        offload_link["frac_median_step"] = offload_link["bound_ms"] / float(np.median(launch_ms))
        offload_link["ms_per_step_median"] = float(np.median(launch_ms))
        offload_link["ms_per_step_min"] = float(launch_ms.min())

    if rank != 0:
        return
    peaks = measured_peaks()
    bytes_launch = op_bytes
    achieved = bytes_launch / (kernel_ms * 1e-3) / 1e9
    traffic, traffic_note = (recorded_traffic(w.M, bytes_launch)
                             if op == "step" and not args.state_on_host else (None, None))
    line = {
        "metric": METRIC,
        "value": world * nv * args.steps / (ms_total * 1e-3),
        "unit": "params/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms_total / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": config_of(w, args.state_on_host, op, args.offload_transfer),
        "hbm_gbs": bytes_launch * args.steps / (ms_total * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "peak_source": peaks["source"],
                     "traffic": traffic, "traffic_source": traffic_note,
                     "kernel": op_kernel,
                     "bytes_per_launch": bytes_launch, "kernel_ms": kernel_ms,
                     "kernel_ms_median": float(np.median(launch_ms)), "kernel_ms_min": float(launch_ms.min()),
                     # context: the part's nominal HBM3e bandwidth (7.9 TB/s), not the roofline
                     "nominal_gbs": NOMINAL_HBM_GBS, "frac_of_nominal": achieved / NOMINAL_HBM_GBS},
        "cpu_baseline": cpu_baseline,
        "offload_link_roofline": offload_link,
        "e2e": e2e if e2e is not None else ({"skipped": e2e_note} if e2e_note else None),
        "e2e_staged": e2e_staged,
        "gpu_launches": args.steps * launches_per_step,
        "last_launch_shape": last_launch,
        "clocks": clocks,
        "overflow_flag": overflow,
    }
    print(json.dumps(line), flush=True)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="flat_1.3B_M8")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=40,
                    help="timed end-to-end steps per host-buffer path (independent of --steps)")
    ap.add_argument("--op", default="step",
                    choices=["step", "dynamic", "dynamic_pingpong", "bucketed_pingpong", "overflow_check",
                             "allreduce", "unfused", "bucketed", "tma"],
                    help="what one timed step runs: the fused ZeRO-1 step (default) or one of the other "
                         "entry points, for component measurements")
    ap.add_argument("--replicas", type=int, default=0, help="override the workload's M (measurement sweeps)")
    ap.add_argument("--params", type=int, default=0, help="override the workload's n (measurement sweeps)")
    ap.add_argument("--graph", action="store_true",
                    help="with --op dynamic: capture one attempt in a CUDA graph and replay it each step")
    ap.add_argument("--bucket-elems", type=int, default=50_000_000,
                    help="bucket size for --op bucketed (the pages' reduce_bucket_size: 5e7)")
    ap.add_argument("--dynamic-loss-scale", action="store_true",
                    help="time the dynamically scaled step (reduce-scatter to fp32 sums, update, scaler) "
                         "with the fp16 block's policy instead of the fused step")
    ap.add_argument("--state-on-host", action="store_true",
                    help="keep fp32 master/m/v in pinned host memory (optimizer-state offload)")
    ap.add_argument("--offload-transfer", choices=["zero_copy", "copy_engines"], default="zero_copy",
                    help="with --state-on-host: the kernel reads and writes the host state over the link "
                         "(zero_copy, the faster one), or chunks are staged through HBM by the copy engines "
                         "(copy_engines)")
    ap.add_argument("--chunk-elems", type=int, default=1 << 23,
                    help="chunk size of the staged (copy-engine) paths")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    sys.path.insert(0, ROOT)
    from zero_sharded_mixed_zero1_gb300 import workloads as W
    if args.workload not in W.BY_NAME:
        ap.error(f"unknown workload {args.workload}; choose from {sorted(W.BY_NAME)}")
    w = W.BY_NAME[args.workload]
    if args.replicas or args.params:          # size overrides for measurement sweeps
        import dataclasses
        w = dataclasses.replace(w, M=args.replicas or w.M, n=args.params or w.n,
                                B=max(w.B, args.replicas or 0), shard_begin=0, shard_end=None,
                                name=f"{w.name}[M={args.replicas or w.M},n={args.params or w.n}]")
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)
    return 0


if __name__ == "__main__":
    sys.exit(main())
