#!/usr/bin/env python
"""Benchmark of the sharded mixed-precision AdamW step over a flat, padded buffer.

One step = one pass of the hot path over one batch of synthetic gradients:
reduce-scatter with averaging over N_d simulated ranks, AdamW on every rank's
shard, all-gather of the bf16 parameters into every rank's replica - one
zs_fused_step call over the whole flat space, which the library walks in
overlapping launches of the fused kernel (each byte crosses HBM once).
--step-mode per-bucket steps the same buckets one by one instead, last first,
as backward makes them ready.

Default workload: Llama-style 1.3B flat buffer (24 layers, d 2048, SwiGLU
5504, vocab 32000, untied), N_d = 8 simulated ranks, ZeRO-2, 25 MiB buckets,
bf16 grads N(0, 5e-4) with 0.1% entries x100, fp32 master/m/v.  Inputs are
59 GB, far larger than the 129 MB L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--profile-case [--profile-elems N]] [--no-e2e]
                  [--no-cpu-baseline] [--step-mode whole|per-bucket|per-bucket-2s]
                  [--bucket-bytes B]

With --gpus N > 1 (launched by torchrun) every rank runs an independent
replica of the workload on its own GPU (the simulated ranks live inside one
GPU, so there is no exchange between GPUs); value = all ranks' parameters
updated / the slowest rank's time.  --impl reference times the CPU oracle on
the host cores on a bounded sample of the same workload.
"""

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sharded AdamW step params/sec and achieved HBM GB/s vs 8 TB/s (1 GB300)"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ------------------------------------------------------------------ distributed plumbing

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def maybe_init_dist(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist

    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def max_over_ranks(dist, value, device):
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ peaks, clocks, profiles

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the files that define each profiled kernel: its code, its argument structs and its launch shape
KERNEL_SOURCES = {
    "k_fused_tma": ("device.cuh", "launch.h", "kernels_tma.cu"),
    "k_fused_tma_dyn": ("device.cuh", "launch.h", "kernels_tma.cu"),
    "k_gather_bulk": ("device.cuh", "launch.h", "kernels_tma.cu"),
    "k_fused": ("device.cuh", "launch.h", "kernels.cu"),
}


def source_digest(kernel_key):
    """Digest of the code of the files that define a kernel (a profile of it is valid only for this
    code); line comments and blank lines are left out, so editing a comment keeps a profile valid."""
    import re

    csrc = os.path.join(ROOT, "fsdp_sharded_optimizer_flatparameter_gb300", "csrc")
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel_key]:
        with open(os.path.join(csrc, name)) as f:
            code = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in f.read().splitlines()]
        h.update(name.encode() + b"\0" + "\n".join(ln for ln in code if ln).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload, kernel_key):
    """DRAM bytes per step from the committed ncu summary (every launch of a step, steady state), if it
    was taken on the current sources."""
    path = os.path.join(ROOT, "profiles", "%s_%s.md" % (kernel_key, workload))
    try:
        fields = {}
        with open(path) as f:
            for line in f:
                if line.startswith("- ") and ":" in line:
                    k, v = line[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("source_digest") != source_digest(kernel_key):
            return None
        return float(fields["traffic_bytes_per_step"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi samples of the benchmarked GPU during the timed region."""

    FIELDS = ("index,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.bus = None
        try:
            import torch

            p = torch.cuda.get_device_properties(device_index)
            self.bus = "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
        except Exception:
            pass
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.thread.join(timeout=5)
        rows = []
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            if self.bus and parts[1].upper() != self.bus.upper():
                continue
            rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i].lower().startswith("active")})
        power = [float(r[4]) for r in rows if r[4].replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


# ------------------------------------------------------------------ device status

class DeviceStatusError(RuntimeError):
    """A kernel recorded a device status code during a timed region: its time is not a valid number."""


def check_device_status(read_status, where, ok_code=0):
    """Reads (and clears) the library's device status word after a timed region.  A staged kernel
    whose bounded wait runs out records a code there and returns early without finishing its
    work, so the region's time would be too short: raise instead of reporting it."""
    code = int(read_status())
    if code != ok_code:
        raise DeviceStatusError("device status %d after %s: a kernel gave up waiting, so no value is "
                                "reported" % (code, where))
    return code


def library_mapped(name="libzs.so"):
    """True when this process has the library mapped (Linux /proc maps)."""
    try:
        with open("/proc/self/maps") as f:
            return any(line.rstrip().endswith("/" + name) for line in f)
    except OSError:
        return False


# ------------------------------------------------------------------ workloads

# The launches of a walked fused step (the rule of launch_fused_walk in csrc/kernels.cu): ranges longer
# than the chunk are cut at multiples of it, none closer than a quarter chunk to a range end; each
# piece is one launch of the staged kernel (plus one per fringe off the 8-element grid), or one
# streaming launch when its body is below the walk's staged threshold.
WALK_CHUNK = 1 << 22           # kFusedWalkChunk
WALK_MIN_STAGED = 1 << 16      # kTmaWalkMinElems
WALK_SHAPE_ND = (2, 4, 8, 16, 32)  # rank counts with a walk shape (fused_walk_shape)
STAGED_ND = (2, 4, 8, 16, 32)


def walk_pieces(ranges, n_d, staged_ok=True):
    out, C = [], WALK_CHUNK
    for lo, hi in ranges:
        while lo < hi:
            end = hi
            if n_d in WALK_SHAPE_ND and staged_ok:
                cut = (lo + C // 4 + C) // C * C
                if cut < hi - C // 4:
                    end = cut
            out.append((lo, end))
            lo = end
    return out


DYN_ND = (2, 4, 8, 16, 32)       # rank counts with a dynamic-order shape (fused_dyn_shape)
DYN_MIN = 1 << 24                # kDynMinElems


def dyn_range(ranges, n_d, staged_ok=True):
    """True when a fused call over these ranges is one dynamic-order launch (one range whose 8-aligned
    body has at least 2^24 elements, a rank count with a dynamic-order shape, device buffers)."""
    if not staged_ok or n_d not in DYN_ND or len(ranges) != 1:
        return False
    lo, hi = ranges[0]
    return hi // 8 * 8 - (lo + 7) // 8 * 8 >= DYN_MIN


def walk_launches(ranges, n_d, staged_ok=True):
    if dyn_range(ranges, n_d, staged_ok):
        lo, hi = ranges[0]
        return 1 + ((lo + 7) // 8 * 8 > lo) + (hi > hi // 8 * 8)
    n = 0
    for lo, hi in walk_pieces(ranges, n_d, staged_ok):
        vlo, vhi = (lo + 7) // 8 * 8, hi // 8 * 8
        if staged_ok and n_d in STAGED_ND and vhi - vlo >= WALK_MIN_STAGED:
            n += 1 + (vlo > lo) + (hi > vhi)
        else:
            n += 1
    return n


def staged_walk_launches(ranges):
    """Launches of a call that gives each range's 8-aligned body of at least 2^24 elements one
    dynamic-order launch, walks a body of at least 2^20 elements with a staged kernel in pieces (cut like
    the fused walk), adds one streaming launch per ragged end, and gives a shorter range one streaming
    launch: zs_adamw_shard_step on one-array buffers (per unit range), and zs_all_reduce_mean and
    zs_dp_step on device buffers at N_d = 4, 8 or 16 (rank counts with both forms)."""
    n, C = 0, WALK_CHUNK
    for lo, hi in ranges:
        vlo, vhi = (lo + 7) // 8 * 8, hi // 8 * 8
        if vhi - vlo < (1 << 20):
            n += 1 if hi > lo else 0
            continue
        n += (vlo > lo) + (hi > vhi)
        if vhi - vlo >= DYN_MIN:
            n += 1
            continue
        while vlo < vhi:
            end = vhi
            cut = (vlo + C // 4 + C) // C * C
            if cut < vhi - C // 4:
                end = cut
            n += 1
            vlo = end
    return n


ZERO3_WALK_CHUNK = 1 << 23     # the ZeRO-3 step's walk chunk (zero3.cu)


def zero3_launches(plan, n_d, reshard=True):
    """Launches of one zs_zero3_step on device buffers: a unit of at least 2^24 elements at N_d <= 16 takes
    one dynamic-order launch per gather and for its reduce-scatter + update; other units' gathers and
    update are walks cut like the fused walk (8 Mi-element chunk).  A piece takes the staged kernel
    (bulk-store gather for bodies of at least 2^20 elements; single-output update for rank counts with
    a staged shape, bodies of at least 2^16) plus one streaming launch per ragged end, else one
    streaming launch; a unit whose base is off the 8-element grid streams every piece."""
    n, C = 0, ZERO3_WALK_CHUNK
    for u in range(plan.n_units):
        base, padded = plan.unit(u)["base"], plan.unit(u)["padded"]
        lo, hi = base, base + padded
        while lo < hi:
            end = hi
            cut = (lo + C // 4 + C) // C * C
            if cut < hi - C // 4 and (padded < DYN_MIN or n_d > 16):   # a long unit at N_d <= 16: one dynamic-order launch per phase
                end = cut
            vlo, vhi = (lo + 7) // 8 * 8, end // 8 * 8
            fringes = (vlo > lo) + (end > vhi)
            vec = base % 8 == 0
            g = 1 + fringes if vec and vhi - vlo >= (1 << 20) else 1
            upd = 1 + fringes if vec and n_d in STAGED_ND and vhi - vlo >= WALK_MIN_STAGED else 1
            n += (2 if reshard else 1) * g + upd
            lo = end
    return n


def bytes_per_padded_element(n_d, kernel):
    """Algorithmic HBM bytes per padded element of one launch (each byte crosses HBM once)."""
    if kernel == "fused":          # read N_d bf16 grads + master/m/v; write master/m/v + N_d bf16 replicas
        return 2 * n_d + 12 + 12 + 2 * n_d
    if kernel == "fused_accumulate":   # the fused step forming each gradient from acc + micro: N_d more reads,
        return 2 * n_d + 2 * n_d + 12 + 12 + 2 * n_d    # no gradient written
    if kernel == "unfused":        # RS (N_d reads, 1 write) + AdamW (2 + 12 read, 12 + 2 write) + AG (2 read, N_d writes)
        return (2 * n_d + 2) + (14 + 14) + (2 + 2 * n_d)
    raise ValueError(kernel)


def oracle_sample(n_d, sample_elems, sigma, outlier_p, seed):
    """Inputs for the oracle's ZeRO step on a bounded sample of the flat buffer."""
    import numpy as np
    import torch

    import synth

    grads, _ = synth.rank_grads(n_d, sample_elems, [], seed=seed, step=1, sigma=sigma, outlier_p=outlier_p)
    g_np = [g.contiguous().view(torch.int16).numpy().view(np.uint16).copy() for g in grads]
    master = synth.master_init(sample_elems, [], seed).numpy().copy()
    return g_np, master


def time_oracle(n_d, sample_elems, sigma, outlier_p, seed, min_seconds, max_reps=1000, reps=None):
    """Runs the oracle's ZeRO step (reduce-scatter with averaging, AdamW per rank, all-gather)
    on a flat buffer of sample_elems elements; returns (seconds per step, steps)."""
    import numpy as np

    from oracle import layout, steps

    import synth

    plan = layout.make_plan([(sample_elems,)], n_d, bucket_bytes=25 << 20)
    g_np, master = oracle_sample(n_d, plan.padded, sigma, outlier_p, seed)
    om = [steps.shard_of(plan, r, master) for r in range(n_d)]
    omm = [np.zeros(plan.shard_total, np.float32) for _ in range(n_d)]
    ov = [np.zeros(plan.shard_total, np.float32) for _ in range(n_d)]
    done, t0 = 0, time.perf_counter()
    while True:
        _, om, omm, ov = steps.zero_step(plan, g_np, om, omm, ov, synth.HPARAMS, done + 1)
        done += 1
        el = time.perf_counter() - t0
        if reps is not None and done >= reps:
            break
        if reps is None and (el >= min_seconds or done >= max_reps):
            break
    return el / done, done, plan.padded


def time_oracle_rows(seconds=1.5):
    """The oracle beside each widening row, each on a bounded sample (params or elements per second,
    one host thread): naive-DP step, ZeRO-3 unit step, FSDP2 chunk-cat + copy-out, checkpoint save +
    resharded load (in memory)."""
    import numpy as np

    from oracle import checkpoint as ock
    from oracle import fsdp2 as ofs
    from oracle import layout, steps

    import synth

    def rate(fn, elems):
        done, t0 = 0, time.perf_counter()
        while True:
            fn(done + 1)
            done += 1
            el = time.perf_counter() - t0
            if el >= seconds:
                return elems * done / el, done

    n_d, E = 8, 1 << 18
    out = {}
    g_np, master = oracle_sample(n_d, E, 1e-3, 0.0, 1)
    st = {"p": master.copy(), "m": np.zeros(E, np.float32), "v": np.zeros(E, np.float32)}

    def dp(t):
        _, st["p"], st["m"], st["v"] = steps.dp_step(g_np, st["p"], st["m"], st["v"], synth.HPARAMS, t)
    r, k = rate(dp, E)
    out["naive_dp"] = {"params_per_s": r, "sample": "oracle naive-DP step, %d elements, N_d=%d, %d steps" % (E, n_d, k)}

    plan = layout.make_plan([(E,)], n_d, unit_of_param=[0])
    sh = [np.zeros(plan.shard_total, np.uint16) for _ in range(n_d)]
    z = {"m": [steps.shard_of(plan, q, master) for q in range(n_d)],
         "mm": [np.zeros(plan.shard_total, np.float32) for _ in range(n_d)],
         "v": [np.zeros(plan.shard_total, np.float32) for _ in range(n_d)]}

    def z3(t):
        _, _, _, z["m"], z["mm"], z["v"] = steps.zero3_unit_step(plan, 0, sh, g_np, z["m"], z["mm"], z["v"],
                                                                  synth.HPARAMS, t)
    r, k = rate(z3, E)
    out["zero3"] = {"params_per_s": r, "sample": "oracle ZeRO-3 unit step (2 gathers + RS + AdamW), %d elements, "
                    "N_d=%d, %d steps" % (E, n_d, k)}

    shapes = [(512, 256)] * 2 + [(256,)]
    p2 = ofs.make_plan(shapes, n_d)
    vals = [np.arange(int(np.prod(sh_)), dtype=np.uint16) for sh_ in shapes]
    n2 = sum(int(np.prod(sh_)) for sh_ in shapes)

    def f2(_):
        ofs.copy_out(p2, 0, ofs.chunk_cat(p2, 0, vals))
    r, k = rate(f2, n2)
    out["fsdp2_copy"] = {"elements_per_s": r, "sample": "oracle chunk-cat + copy-out of %d elements, N_d=%d, %d rounds"
                         % (n2, n_d, k)}

    p8, p4 = layout.make_plan([(E,)], 8), layout.make_plan([(E,)], 4)
    ranks = [{"params": np.zeros(p8.shard_total, np.uint16), "master": np.zeros(p8.shard_total, np.float32),
              "m": np.zeros(p8.shard_total, np.float32), "v": np.zeros(p8.shard_total, np.float32)}
             for _ in range(8)]

    def ck(_):
        saved = ock.save(p8, ranks)
        for name in ("params", "master", "m", "v"):
            ock.load(p4, saved, name)
    r, k = rate(ck, E)
    out["checkpoint"] = {"params_per_s": r, "sample": "oracle save at N_d=8 + load at N_d=4 (in memory), %d elements, "
                         "%d rounds" % (E, k)}
    return out


def _oracle_worker(job):
    """One host process of the all-cores oracle timing (module level, so a spawned process can run it)."""
    n_d, sample, sigma, outlier_p, seed, seconds = job
    per_step, done, padded = time_oracle(n_d, sample, sigma, outlier_p, seed, seconds)
    return padded * done, per_step * done


def time_oracle_all_cores(n_d, sample, sigma, outlier_p, seed, seconds, procs=None):
    """The oracle's ZeRO step on every host core at once: the step is element-wise, so disjoint
    samples in separate processes are the whole step's work split over cores.  Processes are
    spawned (never forked from a process that has touched the GPU)."""
    import multiprocessing as mp

    procs = procs or max(1, os.cpu_count() or 1)
    jobs = [(n_d, sample, sigma, outlier_p, seed + 7919 * k, seconds) for k in range(procs)]
    t0 = time.perf_counter()
    with mp.get_context("spawn").Pool(procs) as pool:          # leaving the block terminates the workers
        results = pool.map_async(_oracle_worker, jobs).get(timeout=4 * seconds + 120)
    wall = time.perf_counter() - t0
    elems = sum(e for e, _ in results)
    busy = max(t for _, t in results)
    return elems / busy, procs, elems, busy, wall


def cpu_threads_used():
    # numpy element-wise ufuncs run on one thread
    return 1


# ------------------------------------------------------------------ reference arm: the CPU oracle

def run_reference(args, ws, rank):
    if rank != 0:
        return 0
    import synth

    wl = synth.WORKLOADS[args.workload]
    n_d = wl["n_d"]
    sample = 1 << 20
    for _ in range(args.warmup):
        time_oracle(n_d, sample, wl["sigma"], wl["outlier_p"], wl["seed"], 0, reps=1)
    per_step, done, padded = time_oracle(n_d, sample, wl["sigma"], wl["outlier_p"], wl["seed"], 0, reps=args.steps)
    value = padded / per_step
    desc = ("oracle ZeRO step (numpy fp32, reduce-scatter-mean + AdamW + all-gather) on a %d-element sample "
            "of the %s flat buffer, N_d=%d, one sample per step" % (padded, wl["model"], n_d))
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "sample_elems": padded, "n_d": n_d},
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": cpu_threads_used(), "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    # the oracle arm must not have the library it judges in its address space
    if library_mapped():
        log("bench.py --impl reference: libzs.so is mapped in the oracle process")
        return 4
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

class Workload:
    """Device buffers and the timed step of one benchmarked workload."""

    def __init__(self, args, dev, stream):
        import torch

        import fsdp_sharded_optimizer_flatparameter_gb300 as zs
        import synth

        self.zs, self.torch = zs, torch
        self.args, self.dev, self.stream = args, dev, stream
        wl = self.wl = dict(synth.WORKLOADS[args.workload])
        shapes, units = synth.workload_params(wl["model"])
        if args.profile_case:
            # the same kernels on a smaller flat buffer (by default 32 Mi elements, 1.9 GB at N_d = 8): for
            # ncu captures
            shapes, units = [(args.profile_elems,)], None
        self.n_d = n_d = wl["n_d"]
        if args.bucket_bytes is not None:
            wl["bucket_bytes"] = args.bucket_bytes
        self.plan = plan = zs.Plan(shapes, n_d, stage=wl["stage"], bucket_bytes=wl["bucket_bytes"],
                                   unit_of_param=units)
        self.order = list(reversed(range(plan.n_buckets)))     # bucket-wise modes: last bucket first
        P, pads = plan.padded, plan.pad_ranges()
        self.P, self.pads = P, pads
        self.hp = synth.HPARAMS
        self.t = 0
        self.master = synth.master_init(P, pads, wl["seed"], device=dev)
        self.m, self.v = torch.zeros_like(self.master), torch.zeros_like(self.master)
        self.kind = "zero3" if wl["stage"] == 3 else ("accumulate+fused" if wl["micro"] > 1 else "fused")
        bf16 = torch.bfloat16
        if self.kind == "zero3":
            U = plan.n_units
            biggest = max(plan.unit(u)["padded"] for u in range(U))
            self.shards = self.master.to(bf16)
            # one set of per-rank gradient buffers, read as every unit's backward gradients
            self.ugrads, self._gb = synth.rank_buffers(n_d, biggest, bf16, dev)
            synth.fill_grads(self.ugrads, [], wl["seed"], 1, wl["sigma"], wl["outlier_p"])
            self.pool = [synth.rank_buffers(n_d, biggest, bf16, dev)[0] for _ in range(2)]
            self.side = torch.cuda.Stream(dev)
            self.resident = (12 + 2) * P + 3 * n_d * biggest * 2
        else:
            self.grads, self._gb = synth.rank_buffers(n_d, P, bf16, dev)
            synth.fill_grads(self.grads, pads, wl["seed"], 1, wl["sigma"], wl["outlier_p"])
            self.reps, self._rb = synth.rank_buffers(n_d, P, bf16, dev)
            self.side = torch.cuda.Stream(dev) if args.step_mode == "per-bucket-2s" else None
            self.resident = 12 * P + 2 * 2 * n_d * P
            if self.kind == "accumulate+fused":
                self.acc, self._ab = synth.rank_buffers(n_d, P, bf16, dev)
                self.resident += 2 * n_d * P

    # algorithmic HBM bytes of one step and the kernel launches it makes
    def step_bytes(self):
        n_d, P = self.n_d, self.P
        walk = walk_launches([(0, P)], n_d, self.staged())
        if self.kind == "fused" and self.args.step_mode != "whole":
            br = [self.plan.bucket(b)[1:] for b in self.order]
            if self.args.step_mode == "per-bucket-2s":
                walk = walk_launches(br[0::2], n_d, self.staged()) + walk_launches(br[1::2], n_d, self.staged())
            else:
                walk = walk_launches(br, n_d, self.staged())
        if self.kind == "fused":
            return bytes_per_padded_element(n_d, "fused") * P, walk
        if self.kind == "accumulate+fused":
            micro = self.wl["micro"]
            if self.args.accumulate_mode == "separate":
                acc = n_d * P * (4 + 6 * (micro - 1))   # first: read micro, write acc; then read both, write acc
                return acc + bytes_per_padded_element(n_d, "fused") * P, micro + walk
            # the last micro-batch inside the step: it reads acc and micro, writes no gradient
            acc = n_d * P * (4 + 6 * (micro - 2))
            return acc + bytes_per_padded_element(n_d, "fused_accumulate") * P, micro - 1 + walk
        # zero3: per unit two gathers (read shard, write N_d copies) + reduce-scatter with update
        return P * (2 * (2 + 2 * n_d) + (2 * n_d + 12 + 12 + 2)), zero3_launches(self.plan, n_d)

    def staged(self):
        zs = self.zs
        v = zs.fused_variant_setting
        big = (self.P >= WALK_MIN_STAGED) if self.kind != "zero3" else True
        return self.n_d in (2, 4, 8, 16, 32) and (v == zs.ZS_FUSED_TMA or (v == zs.ZS_FUSED_AUTO and big))

    def dynamic_order(self):
        """The fused step (plain or with the last micro-batch inside) runs as one dynamic-order launch
        over the whole flat space."""
        return (self.kind in ("fused", "accumulate+fused") and self.args.step_mode == "whole"
                and dyn_range([(0, self.P)], self.n_d, self.staged()))

    def kernel_label(self):
        fused = ("k_fused_tma<%d>" if self.staged() else "k_fused<%d>") % self.n_d
        pieces = len(walk_pieces([(0, self.P)], self.n_d, self.staged())) if self.kind != "zero3" else 1
        dyn = " (one launch, tiles taken in dynamic order)"
        if self.dynamic_order():
            fused = "k_fused_tma_dyn<%d>" % self.n_d + dyn
        elif pieces > 1:
            fused += " walked in %d overlapping launches" % pieces
        if self.kind == "fused":
            return fused
        if self.kind == "accumulate+fused":
            if self.args.accumulate_mode == "separate":
                return "%d x k_accumulate + %s" % (self.wl["micro"], fused)
            return "%d x k_accumulate + %s" % (self.wl["micro"] - 1, fused.replace("k_fused_tma_dyn<", "k_fused_tma_acc_dyn<")
                                                .replace("k_fused_tma<", "k_fused_tma_acc<")
                                                .replace("k_fused<", "k_fused<acc "))
        if self.n_d <= 16:
            return ("2 x k_gather_bulk_dyn + k_fused_tma_single_dyn<%d> per unit, one dynamic-order launch each "
                    "(%d launches per step)" % (self.n_d, zero3_launches(self.plan, self.n_d)))
        return ("2 x k_gather_bulk + k_fused_tma<%d> single output per unit, each walked in launches of 8 Mi elements "
                "(%d launches per step)" % (self.n_d, zero3_launches(self.plan, self.n_d)))

    def step(self):
        zs, plan, hp = self.zs, self.plan, self.hp
        self.t += 1
        t, st = self.t, self.stream
        if self.kind == "fused" and self.args.step_mode != "whole":
            # the step as backward makes buckets ready: every bucket, last first, bucket by bucket
            zs.zs_fused_step_buckets(plan, self.order, self.grads, self.master, self.m, self.v, self.reps, hp, t,
                                     launch_mode=zs.ZS_BUCKETS_PER_BUCKET, stream=st,
                                     side_stream=self.side if self.args.step_mode == "per-bucket-2s" else None)
        elif self.kind == "fused":
            zs.zs_fused_step(plan, -1, self.grads, zs.ZS_RANK_FULL, self.master, self.m, self.v, self.reps, hp, t,
                             stream=st)
        elif self.kind == "accumulate+fused":
            self.accumulate_step(t, st, self.args.accumulate_mode)
        else:
            ug = [self.ugrads] * plan.n_units
            zs.zs_zero3_step(plan, self.shards, self.master, self.m, self.v, ug, self.pool, True, hp, t,
                             main_stream=st, side_stream=self.side)


    def accumulate_step(self, t, st, mode, events=None):
        """The micro-batches accumulated and the step (config with micro > 1).  mode "fused-last": the
        last micro-batch's accumulation inside the step (zs_fused_step_accumulate); "separate": every
        micro-batch accumulated, then zs_fused_step.  events: recorded after every launch call."""
        zs, plan, hp = self.zs, self.plan, self.hp
        micro = self.wl["micro"]
        n_acc = micro if mode == "separate" else micro - 1
        for j in range(n_acc):
            zs.zs_accumulate_grad(plan, self.acc, self.grads, 1.0 / micro, first=(j == 0), stream=st)
            if events:
                events[j].record(st)
        if mode == "separate":
            zs.zs_fused_step(plan, -1, self.acc, zs.ZS_RANK_FULL, self.master, self.m, self.v, self.reps, hp, t,
                             stream=st)
        else:
            zs.zs_fused_step_accumulate(plan, -1, self.acc, self.grads, zs.ZS_RANK_FULL, 1.0 / micro, self.master,
                                        self.m, self.v, self.reps, hp, t, stream=st)
        if events:
            events[n_acc].record(st)


def timed_on_stream(torch, fn, steps, warmup, stream, dev, dist, status=None, where="a timed region"):
    """Mean ms per call over `steps` calls after `warmup`, CUDA events on `stream`, max over ranks;
    status(where), when given, checks the device status word after the region."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(dev)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize(dev)
    if status is not None:
        status(where)
    return max_over_ranks(dist, a.elapsed_time(b) / steps, dev)


def run_sweep(args, ws, rank, local):
    """The 2^28+7-element flat buffer: the fused ZeRO-1/2 step and the ZeRO-3 step for every N_d of
    the sweep, and the bucket-wise ZeRO-2 step (every bucket, descending: as one merged walk, as two
    walks of every other bucket, bucket by bucket on one stream and on two) for every bucket size
    at N_d = 8."""
    import torch

    import fsdp_sharded_optimizer_flatparameter_gb300 as zs
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = maybe_init_dist(ws, "nccl")
    stream = torch.cuda.current_stream(dev)
    wl = synth.WORKLOADS["flat-sweep"]
    shapes, _ = synth.workload_params(wl["model"])
    hp = synth.HPARAMS
    peak, peak_kind = hbm_peak()
    steps = max(3, args.steps)

    def status(where):
        return check_device_status(lambda: zs.zs_device_status(clear=True), where)

    status("setup")

    def timed(fn, n):
        return timed_on_stream(torch, fn, n, args.warmup, stream, dev, dist, status, "a flat-sweep point")

    points, launches = [], 0
    side_bw = torch.cuda.Stream(dev)
    sampler = ClockSampler(local)
    sampler.start()
    for n_d in wl["sweep_n_d"]:
        plan = zs.Plan(shapes, n_d, stage=2, bucket_bytes=wl["bucket_bytes"])
        P, pads = plan.padded, plan.pad_ranges()
        master = synth.master_init(P, pads, wl["seed"], device=dev)
        m, v = torch.zeros_like(master), torch.zeros_like(master)
        grads, _ = synth.rank_buffers(n_d, P, torch.bfloat16, dev)
        synth.fill_grads(grads, pads, wl["seed"], 1, wl["sigma"])
        reps, _ = synth.rank_buffers(n_d, P, torch.bfloat16, dev)
        t = [0]

        def fused():
            t[0] += 1
            zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, hp, t[0], stream=stream)

        ms = timed(fused, steps)
        launches += steps * walk_launches([(0, P)], n_d)
        gbs = bytes_per_padded_element(n_d, "fused") * P / (ms / 1e3) / 1e9
        points.append({"n_d": n_d, "padding": P - plan.numel, "step": "fused, whole buffer", "ms": ms,
                       "params_per_s": plan.numel / (ms / 1e3), "gbs": gbs, "frac": gbs / peak})
        # ZeRO-3 on the same buffer (one unit): forward gather, backward gather, reduce-scatter + update
        p3 = zs.Plan(shapes, n_d, stage=3, bucket_bytes=wl["bucket_bytes"])
        shards = master.to(torch.bfloat16)
        extra, _ = synth.rank_buffers(n_d, P, torch.bfloat16, dev)
        side = torch.cuda.Stream(dev)

        def zero3():
            t[0] += 1
            zs.zs_zero3_step(p3, shards, master, m, v, [grads], [reps, extra], True, hp, t[0],
                             main_stream=stream, side_stream=side)

        ms = timed(zero3, steps)
        launches += zero3_launches(p3, n_d) * steps
        gbs = P * (2 * (2 + 2 * n_d) + (2 * n_d + 26)) / (ms / 1e3) / 1e9
        points.append({"n_d": n_d, "stage": 3, "step": "ZeRO-3: 2 gathers + reduce-scatter/update (one unit)",
                       "ms": ms, "params_per_s": plan.numel / (ms / 1e3), "gbs": gbs, "frac": gbs / peak})
        del shards, extra
        if n_d == 8:
            for mib in wl["sweep_bucket_mib"]:
                bp = zs.Plan(shapes, n_d, stage=2, bucket_bytes=mib << 20)

                order = list(reversed(range(bp.n_buckets)))
                br = [bp.bucket(b)[1:] for b in order]
                modes = (("one walk over the list (neighbours merge into one range)", zs.ZS_BUCKETS_ONE_WALK, None,
                          walk_launches([(0, P)], n_d)),
                         ("two walks: every other bucket, then the rest (disjoint ranges)",
                          "alternate", None, walk_launches(sorted(br[0::2]), n_d) + walk_launches(sorted(br[1::2]), n_d)),
                         ("bucket by bucket (no launch spans two buckets)", zs.ZS_BUCKETS_PER_BUCKET, None,
                          walk_launches(br, n_d)),
                         ("bucket by bucket, odd positions on a side stream", zs.ZS_BUCKETS_PER_BUCKET,
                          side_bw, walk_launches(br[0::2], n_d) + walk_launches(br[1::2], n_d)))
                for label, lm, side, n_launch in modes:

                    def bucketwise(bp=bp, order=order, lm=lm, side=side):
                        t[0] += 1
                        if lm == "alternate":
                            for part in (order[0::2], order[1::2]):
                                zs.zs_fused_step_buckets(bp, part, grads, master, m, v, reps, hp, t[0],
                                                         launch_mode=zs.ZS_BUCKETS_ONE_WALK, stream=stream)
                        else:
                            zs.zs_fused_step_buckets(bp, order, grads, master, m, v, reps, hp, t[0], launch_mode=lm,
                                                     stream=stream, side_stream=side)

                    ms = timed(bucketwise, steps)
                    launches += steps * n_launch
                    gbs = bytes_per_padded_element(n_d, "fused") * P / (ms / 1e3) / 1e9
                    points.append({"n_d": n_d, "bucket_mib": mib, "buckets": bp.n_buckets, "mode": label,
                                   "step": "fused over every bucket (descending), zs_fused_step_buckets", "ms": ms,
                                   "params_per_s": plan.numel / (ms / 1e3), "gbs": gbs, "frac": gbs / peak})
        del master, m, v, grads, reps
        torch.cuda.empty_cache()
    clocks = sampler.stop()
    head = next(p for p in points if p["n_d"] == 8 and p["step"] == "fused, whole buffer")
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        # the oracle beside each point: its ZeRO step and its ZeRO-3 unit step, per N_d, one thread
        import numpy as np

        from oracle import layout as olayout
        from oracle import steps as osteps

        for n_d in wl["sweep_n_d"]:
            sec, k, padded = time_oracle(n_d, 1 << 18, wl["sigma"], 0.0, wl["seed"], min_seconds=1.0)
            for p in points:
                if p["n_d"] == n_d and p.get("stage") is None:
                    p["cpu_oracle"] = {"params_per_s": padded / sec, "sample": "oracle ZeRO step, %d elements, "
                                       "N_d=%d, %d steps" % (padded, n_d, k)}
            oplan = olayout.make_plan([(1 << 18,)], n_d, unit_of_param=[0])
            g_np, master = oracle_sample(n_d, oplan.padded, wl["sigma"], 0.0, wl["seed"])
            sh = [np.zeros(oplan.shard_total, np.uint16) for _ in range(n_d)]
            st = [[osteps.shard_of(oplan, q, master) for q in range(n_d)],
                  [np.zeros(oplan.shard_total, np.float32) for _ in range(n_d)],
                  [np.zeros(oplan.shard_total, np.float32) for _ in range(n_d)]]
            done, t0 = 0, time.perf_counter()
            while time.perf_counter() - t0 < 1.0:
                done += 1
                _, _, _, st[0], st[1], st[2] = osteps.zero3_unit_step(oplan, 0, sh, g_np, st[0], st[1], st[2],
                                                                     synth.HPARAMS, done)
            rate = oplan.padded * done / (time.perf_counter() - t0)
            for p in points:
                if p["n_d"] == n_d and p.get("stage") == 3:
                    p["cpu_oracle"] = {"params_per_s": rate, "sample": "oracle ZeRO-3 unit step, %d elements, "
                                       "N_d=%d, %d steps" % (oplan.padded, n_d, done)}
        ref = next(p for p in points if p["n_d"] == 8 and p.get("stage") is None)["cpu_oracle"]
        cpu = {"value": ref["params_per_s"], "unit": "params/s", "cores": cpu_threads_used(), "kind": "oracle",
               "sample": ref["sample"]}
    if rank == 0:
        line = {
            "metric": METRIC, "value": ws * head["params_per_s"], "unit": "params/s", "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": head["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "flat-sweep", "params": 2 ** 28 + 7, "n_d": 8,
                       "l2": "every step moves >= 10 GB >> 129 MB L2, no flush"},
            "roofline": {"bound": "hbm", "achieved": head["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": head["gbs"] / peak, "peak_kind": peak_kind, "traffic": None},
            "sweep": points, "gpu_launches": launches, "clocks": clocks, "device_status": status("the sweep"),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_next(args, ws, rank, local):
    """The widening rows on their own shapes, each against its algorithmic bytes:
    naive DP (all-reduce-mean, replicated update) on GPT-2-small at N_d = 8; ZeRO-3 with and
    without reshard_after_forward on Llama-1.3B (one unit per layer + root) at N_d = 8; the FSDP2
    Shard(0) layout on the same grouping (gradient chunk-cat, fused step, copy-out); and a sharded
    checkpoint of GPT-2-small saved at N_d = 8 and reloaded at N_d = 8 and N_d = 4."""
    import shutil
    import tempfile

    import torch

    import fsdp_sharded_optimizer_flatparameter_gb300 as zs
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = maybe_init_dist(ws, "nccl")
    stream = torch.cuda.current_stream(dev)
    hp = synth.HPARAMS
    peak, peak_kind = hbm_peak()
    steps = max(3, args.steps)
    bf16 = torch.bfloat16
    rows, launches = [], 0

    def status(where):
        return check_device_status(lambda: zs.zs_device_status(clear=True), where)

    status("setup")

    def timed(fn):
        return timed_on_stream(torch, fn, steps, args.warmup, stream, dev, dist, status, "a widening row")

    def row(name, ms, numel, nbytes, n_launch, **extra):
        gbs = nbytes / (ms / 1e3) / 1e9
        rows.append(dict(row=name, ms=ms, params_per_s=numel / (ms / 1e3), algorithmic_bytes=nbytes, gbs=gbs,
                         frac=gbs / peak, launches_per_step=n_launch, **extra))

    sampler = ClockSampler(local)
    sampler.start()

    # --profile-case: the same kernels on small shapes (a few GB on the device) for ncu captures
    small = args.profile_case
    unit_model = "llama-small-units" if small else "llama-1.3b-units"
    unit_label = "Llama-small (profile case)" if small else "Llama-1.3B"
    dp_label = "flat 2^24 (profile case)" if small else "GPT-2-small"

    # naive DP on GPT-2-small, N_d = 8: every rank holds and updates the whole fp32 state
    n_d = 8
    shapes, _ = synth.workload_params("gpt2-small")
    if small:
        shapes = [(1 << 24,)]
    plan = zs.Plan(shapes, n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    grads, _ = synth.rank_buffers(n_d, P, bf16, dev)
    synth.fill_grads(grads, pads, 1, 1, 1e-3)
    reps, _ = synth.rank_buffers(n_d, P, bf16, dev)
    master0 = synth.master_init(P, pads, 1, device=dev)
    master = [master0.clone() for _ in range(n_d)]
    mm = [torch.zeros_like(master0) for _ in range(n_d)]
    vv = [torch.zeros_like(master0) for _ in range(n_d)]
    t = [0]

    def dp():
        t[0] += 1
        zs.zs_dp_step(plan, grads, master, mm, vv, reps, hp, t[0], stream=stream)

    n_dp = staged_walk_launches([(0, P)])          # one dynamic-order launch (walked below 2^24 elements)
    row("naive DP step (k_dp_tma_dyn, one dynamic-order launch: all-reduce-mean + replicated AdamW), %s, N_d=8"
        % dp_label, timed(dp),
        plan.numel, 28 * n_d * P, n_dp)
    launches += steps * n_dp
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        row("naive DP step, register-streaming kernel (k_dp_step), for comparison", timed(dp), plan.numel,
            28 * n_d * P, 1)
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    launches += steps

    def ar():
        zs.zs_all_reduce_mean(plan, -1, grads, stream=stream)

    n_ar = staged_walk_launches([(0, P)])
    row("naive DP all-reduce-mean alone (k_ar_tma_dyn, one dynamic-order launch), %s, N_d=8" % dp_label, timed(ar),
        plan.numel,
        4 * n_d * P, n_ar)
    launches += steps * n_ar
    z_master, z_m, z_v = master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)

    def zero():
        t[0] += 1
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, z_master, z_m, z_v, reps, hp, t[0], stream=stream)

    row("ZeRO-1/2 fused step on the same buffers, for comparison", timed(zero), plan.numel,
        bytes_per_padded_element(n_d, "fused") * P, walk_launches([(0, P)], n_d))
    launches += steps * walk_launches([(0, P)], n_d)
    state_dp, state_zero = plan.memory_bytes(0), plan.memory_bytes(2)
    del grads, reps, master, mm, vv, z_master, z_m, z_v

    # sharded checkpoint of GPT-2-small: save at N_d = 8, reload at N_d = 8 and (resharded) N_d = 4
    # (host I/O, so not part of the small case)
    if not small:
        plan8, plan4 = zs.Plan(shapes, 8, stage=1), zs.Plan(shapes, 4, stage=1)
        sh = master0.to(bf16)
        cm, cv = torch.zeros_like(master0), torch.zeros_like(master0)
        P4 = plan4.padded
        sh4 = torch.empty(P4, dtype=bf16, device=dev)
        m4, c4m, c4v = (torch.empty(P4, dtype=torch.float32, device=dev) for _ in range(3))
        ckpt_bytes = 14 * plan8.numel
        tmp = tempfile.mkdtemp(prefix="zs_ckpt_")

        def wall(fn):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            return (time.perf_counter() - t0) * 1e3

        try:
            ms = min(wall(lambda: zs.zs_checkpoint_save(plan8, tmp, sh, master0, cm, cv, 7, stream=stream))
                     for _ in range(3))
            row("checkpoint save (N_d=8 shards -> files), GPT-2-small", ms, plan8.numel, ckpt_bytes, 0,
                timing="wall clock")
            ms = min(wall(lambda: zs.zs_checkpoint_load(plan8, tmp, sh, master0, cm, cv, stream=stream))
                     for _ in range(3))
            row("checkpoint load, same N_d=8", ms, plan8.numel, ckpt_bytes, 0, timing="wall clock")
            ms = min(wall(lambda: zs.zs_checkpoint_load(plan4, tmp, sh4, m4, c4m, c4v, stream=stream))
                     for _ in range(3))
            row("checkpoint load resharded to N_d=4", ms, plan4.numel, ckpt_bytes, 0, timing="wall clock")
        finally:
            shutil.rmtree(tmp, ignore_errors=True)
        del sh, cm, cv, sh4, m4, c4m, c4v
    del master0

    # ZeRO-3 on Llama-1.3B (24 layer units + root), N_d = 8, with and without resharding after forward
    shapes, units = synth.workload_params(unit_model)
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, U = plan.padded, plan.n_units
    biggest = max(plan.unit(u)["padded"] for u in range(U))
    master = synth.master_init(P, plan.pad_ranges(), 2, device=dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = master.to(bf16)
    ugrads, _ = synth.rank_buffers(n_d, biggest, bf16, dev)
    synth.fill_grads(ugrads, [], 2, 1, 5e-4)
    side = torch.cuda.Stream(dev)
    pool = [synth.rank_buffers(n_d, biggest, bf16, dev)[0] for _ in range(U)]
    for reshard in (True, False):
        slots = pool[:2] if reshard else pool

        def z3(slots=slots, reshard=reshard):
            t[0] += 1
            zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * U, slots, reshard, hp, t[0],
                             main_stream=stream, side_stream=side)

        gathers = 2 if reshard else 1
        z3n = zero3_launches(plan, n_d, reshard)
        row("ZeRO-3 step, %s, N_d=8, reshard_after_forward=%s" % (unit_label, reshard), timed(z3), plan.numel,
            P * (gathers * (2 + 2 * n_d) + (2 * n_d + 26)), z3n,
            comm_bytes_per_rank=plan.comm_bytes(3, reshard))
        launches += steps * z3n

        # the same step on one stream (side_stream = main_stream: stream order, no events)
        def z3_one(slots=slots, reshard=reshard):
            t[0] += 1
            zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * U, slots, reshard, hp, t[0],
                             main_stream=stream, side_stream=stream)

        row("ZeRO-3 step, reshard_after_forward=%s, one stream (no events)" % reshard, timed(z3_one), plan.numel,
            P * (gathers * (2 + 2 * n_d) + (2 * n_d + 26)), z3n)
        launches += steps * z3n
        # the same step captured once (both streams) and replayed; the replay repeats its step number
        g3, cs = torch.cuda.CUDAGraph(), torch.cuda.Stream(dev)
        with torch.cuda.graph(g3, stream=cs):
            zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * U, slots, reshard, hp, t[0] + 1,
                             main_stream=cs, side_stream=side)
        torch.cuda.synchronize(dev)
        row("ZeRO-3 step, reshard_after_forward=%s, replayed from a CUDA graph" % reshard, timed(g3.replay),
            plan.numel, P * (gathers * (2 + 2 * n_d) + (2 * n_d + 26)), z3n)
        launches += steps * z3n
        del g3
    del master, m, v, shards, ugrads, pool

    # FSDP2 Shard(0) layout on the same grouping: per rank gradient chunk-cat, fused step, copy-out
    plan = zs.Plan(shapes, n_d, stage=2, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    P, pads = plan.padded, plan.pad_ranges()
    master = synth.master_init(P, pads, 2, device=dev)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grads, _ = synth.rank_buffers(n_d, P, bf16, dev)
    reps, _ = synth.rank_buffers(n_d, P, bf16, dev)
    params = [torch.empty(s, dtype=bf16, device=dev).normal_(0, 1e-3) for s in shapes]
    members = [[k for k in range(len(shapes)) if units[k] == u] for u in range(plan.n_units)]
    unit_base = [plan.unit(u)["base"] for u in range(plan.n_units)]
    unit_pad = [plan.unit(u)["padded"] for u in range(plan.n_units)]

    def chunk_cat(q=0, st=None):
        for u in range(plan.n_units):
            zs.zs_fsdp2_chunk_cat(plan, u, [params[k] for k in members[u]],
                                  grads[q][unit_base[u]:unit_base[u] + unit_pad[u]], stream=st or stream)

    def copy_out(q=0, st=None):
        for u in range(plan.n_units):
            zs.zs_fsdp2_copy_out(plan, u, reps[q][unit_base[u]:unit_base[u] + unit_pad[u]],
                                 [params[k] for k in members[u]], stream=st or stream)

    def graphed(body):
        # the per-group calls of one step captured once and replayed: one launch per group as before,
        # without the host's ~30 us per call between them (the library's calls are capturable: no
        # synchronisation, no allocation)
        g, cs = torch.cuda.CUDAGraph(), torch.cuda.Stream(dev)
        with torch.cuda.graph(g, stream=cs):
            body(st=cs)
        torch.cuda.synchronize(dev)
        return g

    for q in range(n_d):
        chunk_cat(q)
    layout_launches = sum((len(mem) + 63) // 64 for mem in members)
    row("FSDP2 gradient chunk-cat, one rank's full gradient -> group buffers (k_fsdp2_copy), %s units" % unit_label,
        timed(chunk_cat), plan.numel, 2 * plan.numel + 2 * P, layout_launches)
    launches += steps * layout_launches
    g_cc = graphed(chunk_cat)
    row("FSDP2 gradient chunk-cat, the same calls replayed from a CUDA graph (k_fsdp2_copy)", timed(g_cc.replay),
        plan.numel, 2 * plan.numel + 2 * P, layout_launches)
    launches += steps * layout_launches
    del g_cc

    def f2():
        t[0] += 1
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, hp, t[0], stream=stream)

    row("FSDP2 layout fused step, %s units, N_d=8" % unit_label, timed(f2), plan.numel,
        bytes_per_padded_element(n_d, "fused") * P, walk_launches([(0, P)], n_d), padding=P - plan.numel)
    launches += steps * walk_launches([(0, P)], n_d)
    row("FSDP2 copy-out, group buffers -> one rank's parameters (k_fsdp2_copy)", timed(copy_out), plan.numel,
        2 * plan.numel * 2, layout_launches)
    launches += steps * layout_launches
    g_co = graphed(copy_out)
    row("FSDP2 copy-out, the same calls replayed from a CUDA graph (k_fsdp2_copy)", timed(g_co.replay), plan.numel,
        2 * plan.numel * 2, layout_launches)
    launches += steps * layout_launches
    del g_co
    del master, m, v, grads, reps, params
    torch.cuda.empty_cache()
    clocks = sampler.stop()

    head = next(r for r in rows if r["row"].startswith("FSDP2 layout fused step"))
    cpu = None
    if rank == 0 and not small and not args.no_cpu_baseline:
        orc = time_oracle_rows()
        for r in rows:
            key = ("naive_dp" if r["row"].startswith("naive DP") else "zero3" if r["row"].startswith("ZeRO-3")
                   else "fsdp2_copy" if "k_fsdp2_copy" in r["row"] else "checkpoint" if r["row"].startswith("checkpoint")
                   else None)
            if key:
                r["cpu_oracle"] = orc[key]
        sec, k, padded = time_oracle(n_d, 1 << 20, 5e-4, 1e-3, 2, min_seconds=5.0)
        cpu = {"value": padded / sec, "unit": "params/s", "cores": cpu_threads_used(), "kind": "oracle",
               "sample": "oracle ZeRO step (numpy fp32) on a %d-element flat sample, N_d=%d, %d steps in %.1f s"
                         % (padded, n_d, k, sec * k)}
        for r in rows:
            if r["row"].startswith("FSDP2 layout fused step") or r["row"].startswith("ZeRO-1/2 fused step"):
                r["cpu_oracle"] = {"params_per_s": cpu["value"], "sample": cpu["sample"]}
    if rank == 0:
        line = {
            "metric": METRIC, "value": ws * head["params_per_s"], "unit": "params/s", "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": head["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "next-rows" + ("-profile-case" if small else ""), "head": head["row"], "n_d": n_d,
                       "l2": "every timed call moves >= 1 GB >> 129 MB L2, no flush",
                       "naive_dp_state_bytes_per_rank": state_dp, "zero2_state_bytes_per_rank": state_zero},
            "roofline": {"bound": "hbm", "achieved": head["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": head["gbs"] / peak, "peak_kind": peak_kind, "traffic": None},
            "rows": rows, "gpu_launches": launches, "clocks": clocks, "device_status": status("the widening rows"),
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def run_ours(args, ws, rank, local):
    import torch

    import fsdp_sharded_optimizer_flatparameter_gb300 as zs

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = maybe_init_dist(ws, "nccl")
    variant = {"auto": zs.ZS_FUSED_AUTO, "ldg": zs.ZS_FUSED_LDG, "tma": zs.ZS_FUSED_TMA}[args.fused_variant]
    zs.zs_set_fused_variant(variant)
    zs.fused_variant_setting = variant

    stream = torch.cuda.current_stream(dev)

    def status(where):
        return check_device_status(lambda: zs.zs_device_status(clear=True), where)

    status("start")
    t_setup = time.perf_counter()
    W = Workload(args, dev, stream)
    plan, n_d, P = W.plan, W.n_d, W.P
    torch.cuda.synchronize(dev)
    log("setup %.1fs: %s, %d params (padded %d), N_d=%d, %.1f GB resident" % (
        time.perf_counter() - t_setup, args.workload, plan.numel, P, n_d, W.resident / 1e9))

    for _ in range(args.warmup):
        W.step()
    torch.cuda.synchronize(dev)
    status("the warm-up steps")

    steps = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    sampler = ClockSampler(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    sampler.start()
    time.sleep(0.3)                              # let the sampler see the start of the region
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        ev[k][0].record(stream)
        W.step()
        ev[k][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    status("the timed steps")
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(dist, t0.elapsed_time(t1), dev)
    step_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)

    value = ws * plan.numel * steps / (total_ms / 1e3)
    algo_bytes, launches = W.step_bytes()
    achieved = algo_bytes / (step_ms / 1e3) / 1e9
    peak, peak_kind = hbm_peak()

    # the accumulate + fused step's launches timed one by one (not part of value)
    breakdown = None
    if W.kind == "accumulate+fused" and rank == 0:
        # both forms of the step, alternately, each launch call timed (events after every call)
        micro = W.wl["micro"]
        # per form: one list per launch call (index j), the whole step at index micro + 1
        ms = {mode: [[] for _ in range(micro + 2)] for mode in ("fused-last", "separate")}
        for k in range(12):
            for mode in ("fused-last", "separate"):
                W.t += 1
                n_calls = micro if mode == "fused-last" else micro + 1
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(n_calls + 1)]
                evs[0].record(stream)
                W.accumulate_step(W.t, stream, mode, events=evs[1:])
                torch.cuda.synchronize(dev)
                if k >= 2:
                    for j in range(n_calls):
                        ms[mode][j].append(evs[j].elapsed_time(evs[j + 1]))
                    ms[mode][micro + 1].append(evs[0].elapsed_time(evs[n_calls]))

        def entry(t_ms, nbytes):
            gbs = nbytes / (t_ms / 1e3) / 1e9
            return {"ms": t_ms, "algorithmic_bytes": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak}

        status("the per-launch breakdown")
        fl, sp = ms["fused-last"], ms["separate"]
        mean = statistics.mean
        breakdown = {"accumulate_first": entry(mean(fl[0] + sp[0]), 4 * n_d * P),
                     "accumulate": entry(mean([x for a in fl[1:micro - 1] + sp[1:micro] for x in a]), 6 * n_d * P),
                     "fused_accumulate": entry(mean(fl[micro - 1]),
                                               bytes_per_padded_element(n_d, "fused_accumulate") * P),
                     "fused": entry(mean(sp[micro]), bytes_per_padded_element(n_d, "fused") * P),
                     "step_fused_last_ms": mean(fl[micro + 1]),
                     "step_separate_ms": mean(sp[micro + 1]),
                     "timing": "launch calls timed one by one with events between them, after 2 untimed rounds; "
                               "both forms alternate"}

    # the unfused path on the same buffers, for comparison (not part of value)
    unfused = None
    if W.kind == "fused" and rank == 0 and args.unfused_steps > 0:
        # the unfused ZeRO-2 step on the same buffers, each kernel timed on its own (not part of value)
        ghat = torch.empty(P, dtype=torch.bfloat16, device=dev)
        shards = torch.empty(P, dtype=torch.bfloat16, device=dev)
        names = ("reduce_scatter_mean", "adamw_shard_step", "all_gather")
        per = {k: [] for k in names}
        total = []
        for k in range(args.unfused_steps + 2):
            W.t += 1
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
            evs[0].record(stream)
            zs.zs_reduce_scatter_mean(plan, -1, W.grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED, stream=stream)
            evs[1].record(stream)
            zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, W.master, W.m, W.v, [shards], zs.ZS_SHARDED,
                                   W.hp, W.t, stream=stream)
            evs[2].record(stream)
            zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, W.reps, stream=stream)
            evs[3].record(stream)
            torch.cuda.synchronize(dev)
            if k >= 2:
                for j, name in enumerate(names):
                    per[name].append(evs[j].elapsed_time(evs[j + 1]))
                total.append(evs[0].elapsed_time(evs[3]))
        status("the unfused steps")
        ums = statistics.mean(total)
        kb = {"reduce_scatter_mean": 2 * n_d + 2, "adamw_shard_step": 28, "all_gather": 2 + 2 * n_d}
        unfused = {"ms_per_step": ums, "params_per_s": plan.numel / (ums / 1e3),
                   "algorithmic_gbs": bytes_per_padded_element(n_d, "unfused") * P / (ums / 1e3) / 1e9,
                   "launches_per_step": 2 + staged_walk_launches([(plan.unit(u)["base"], plan.unit(u)["base"]
                                                                 + plan.unit(u)["padded"])
                                                                for u in range(plan.n_units)]),
                   "kernels": {name: {"ms": statistics.mean(per[name]), "bytes_per_element": kb[name],
                                      "gbs": kb[name] * P / (statistics.mean(per[name]) / 1e3) / 1e9,
                                      "frac_of_peak": kb[name] * P / (statistics.mean(per[name]) / 1e3) / 1e9 / peak}
                               for name in names}}
        del ghat, shards

    # ZeRO-2 as the buckets become ready (config 2's bucket-wise flow): every bucket of the plan, last
    # first, stepped bucket by bucket (no launch spans two buckets), on one stream and with the odd
    # positions on a side stream; and the same list as one walk (touching buckets merge).  Not part of
    # value.
    bucketwise = None
    if W.kind == "fused" and rank == 0 and not args.profile_case and args.bucketwise_steps > 0:
        order = list(reversed(range(plan.n_buckets)))
        branges = [plan.bucket(b)[1:] for b in order]
        side_bw = torch.cuda.Stream(dev)
        recs = []
        for label, lm, sd, nl in (
                ("bucket by bucket, one stream", zs.ZS_BUCKETS_PER_BUCKET, None,
                 walk_launches(branges, n_d, W.staged())),
                ("bucket by bucket, odd positions on a side stream", zs.ZS_BUCKETS_PER_BUCKET, side_bw,
                 walk_launches(branges[0::2], n_d, W.staged()) + walk_launches(branges[1::2], n_d, W.staged())),
                ("one walk over the list (touching buckets merge)", zs.ZS_BUCKETS_ONE_WALK, None,
                 walk_launches([(0, P)], n_d, W.staged()))):

            def bw(lm=lm, sd=sd):
                W.t += 1
                zs.zs_fused_step_buckets(plan, order, W.grads, W.master, W.m, W.v, W.reps, W.hp, W.t, launch_mode=lm,
                                         stream=stream, side_stream=sd)

            ms = timed_on_stream(torch, bw, args.bucketwise_steps, 3, stream, dev, None, status,
                                 "the bucket-wise steps")
            gbs = algo_bytes / (ms / 1e3) / 1e9
            recs.append({"mode": label, "ms_per_step": ms, "params_per_s": plan.numel / (ms / 1e3), "gbs": gbs,
                         "frac": gbs / peak, "launches_per_step": nl})
        bucketwise = {"buckets": plan.n_buckets, "bucket_bytes": W.wl["bucket_bytes"],
                      "order": "descending (the last bucket first, as backward makes them ready)",
                      "step": "zs_fused_step_buckets: reduce-scatter-mean + AdamW + all-gather per bucket",
                      "modes": recs}

    # end to end through the C ABI with host buffers, all inside the timed region, two ways:
    #  (a) zero-copy: zs_fused_step reads every rank's gradients from pinned host memory and writes
    #      rank 0's updated replica to pinned host memory over the host link, in the kernel itself;
    #  (b) staged: zs_zero2_step_host copies the gradients bucket by bucket through a two-slot device
    #      staging ring (copy stream) overlapped with the per-bucket update, and copies rank 0's
    #      replica back on a third stream.
    # e2e reports the faster; the other is kept under e2e_alt.
    e2e = e2e_alt = None
    if W.kind == "fused" and not args.no_e2e and not args.profile_case:
        try:
            e2e, e2e_alt = measure_e2e(torch, zs, W, plan, n_d, P, steps, stream, dev, dist, ws, status)
        except DeviceStatusError:
            raise
        except (RuntimeError, MemoryError) as exc:        # e.g. pinned host memory exhausted
            e2e = {"value": None, "unit": "params/s", "error": str(exc)[:200]}
            torch.cuda.synchronize(dev)

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline and not args.profile_case:
        per_step, done, padded = time_oracle(n_d, 1 << 20, W.wl["sigma"], W.wl["outlier_p"], W.wl["seed"], 10.0)
        cpu = {"value": padded / per_step, "unit": "params/s", "cores": cpu_threads_used(), "kind": "oracle",
               "sample": "oracle ZeRO step (numpy fp32) on a %d-element sample of the %s flat buffer, N_d=%d, "
                         "%d steps in %.1f s" % (padded, W.wl["model"], n_d, done, per_step * done)}
        try:
            rate, procs, elems, busy, _ = time_oracle_all_cores(n_d, 1 << 20, W.wl["sigma"], W.wl["outlier_p"],
                                                                W.wl["seed"], 5.0)
            cpu_all = {"value": rate, "unit": "params/s", "cores": procs, "kind": "oracle",
                       "sample": "the same oracle step in %d spawned processes on disjoint %d-element samples "
                                 "(element-wise, so this is the step split over cores), %d elements in %.1f s"
                                 % (procs, 1 << 20, elems, busy)}
        except Exception as exc:                          # no process pool on this host: say so
            cpu_all = {"value": None, "error": str(exc)[:200]}

    if rank == 0:
        staged = W.staged()
        traffic = None
        if W.kind == "fused" and not args.profile_case:
            traffic = profiled_traffic(args.workload, "k_fused_tma_dyn" if W.dynamic_order()
                                       else ("k_fused_tma" if staged else "k_fused"))
        line = {
            "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": ws, "steps": steps,
            "warmup": args.warmup, "ms_per_step": total_ms / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": args.workload + ("-profile-case" if args.profile_case else ""),
                       "fused_variant": args.fused_variant, "params": plan.numel,
                       "padded": P, "n_d": n_d, "stage": "zero%d" % W.wl["stage"],
                       "bucket_bytes": W.wl["bucket_bytes"], "step": W.kind, "step_mode": args.step_mode,
                       **({"micro_batches": W.wl["micro"], "accumulate_mode": args.accumulate_mode}
                          if W.kind == "accumulate+fused" else {}),
                       "storage": "bf16 params/grads, fp32 master/m/v",
                       "l2": "step moves %.0f GB >> 129 MB L2, no flush" % (algo_bytes / 1e9),
                       "parallelism": "replicas" if ws > 1 else "1 GPU, %d simulated ranks" % n_d},
            "hbm_gbs": achieved,
            "frac_of_8tbs": achieved / NOMINAL_HBM_GBS,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "peak_kind": peak_kind, "traffic": traffic,
                         "traffic_unit": "bytes per step (every launch of a step, ncu, steady state)",
                         "traffic_vs_algorithmic": (traffic / algo_bytes) if traffic else None,
                         "algorithmic_bytes_per_launch": algo_bytes if launches == 1 else None,
                         "algorithmic_bytes_per_step": algo_bytes, "kernel": W.kernel_label(),
                         "launches_per_step": launches, "kernel_ms": step_ms,
                         "timing": ("CUDA events around each step on the launching stream; the step's "
                                    "launches overlap (each starts while the previous drains), so "
                                    "achieved = algorithmic bytes per step / step span")},
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all if cpu is not None else None,
            "e2e": e2e,
            "e2e_alt": e2e_alt,
            "gpu_launches": launches * steps,
            "clocks": clocks,
            "unfused": unfused,
            "bucketwise": bucketwise,
            "kernels": breakdown,
            "device_status": status("the benchmark"),
        }
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()
    return 0


def all_ranks_ok(dist, ok, device):
    """True when every rank reports ok (so no rank enters a collective the others skip)."""
    if dist is None:
        return ok
    import torch

    t = torch.tensor([1.0 if ok else 0.0], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MIN)
    return t.item() > 0.5


def measure_e2e(torch, zs, W, plan, n_d, P, steps, stream, dev, dist, ws, status):
    """Both host-fed paths; returns (faster, other)."""
    try:
        host_g = torch.empty((n_d, P), dtype=torch.bfloat16, pin_memory=True)
        host_out = torch.empty(P, dtype=torch.bfloat16, pin_memory=True)
        ok, why = True, ""
    except (RuntimeError, MemoryError) as exc:          # e.g. pinned host memory exhausted
        host_g = host_out = None
        ok, why = False, str(exc)[:200]
    if not all_ranks_ok(dist, ok, dev):
        raise RuntimeError("pinned host buffers unavailable on some rank" + (": " + why if why else ""))
    for q in range(n_d):
        host_g[q].copy_(W.grads[q])
    hrows = [host_g[q] for q in range(n_d)]
    n_e2e = max(2, min(steps, 5))

    def timed(fn):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for k in range(n_e2e + 1):
            if k == 1:
                a.record(stream)
            W.t += 1
            fn()
        b.record(stream)
        torch.cuda.synchronize(dev)
        status("an end-to-end leg")
        return max_over_ranks(dist, a.elapsed_time(b) / n_e2e, dev)

    zc_ms = timed(lambda: zs.zs_fused_step(plan, -1, hrows, zs.ZS_RANK_FULL, W.master, W.m, W.v,
                                           [host_out] + W.reps[1:], W.hp, W.t, stream=stream))
    biggest = max(hi - lo for _, lo, hi in (plan.bucket(b) for b in range(plan.n_buckets)))
    staging = [zs_synth_buffers(n_d, biggest, dev) for _ in range(2)]
    copy_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    st_ms = timed(lambda: zs.zs_zero2_step_host(plan, hrows, staging, W.master, W.m, W.v, W.reps, W.hp, W.t,
                                                host_replica0=host_out, stream=stream, copy_stream=copy_s,
                                                d2h_stream=d2h_s))
    e2e = e2e_alt = None
    paths = {
        "zero-copy": (zc_ms, "zs_fused_step on pinned host gradients, rank 0's replica written to pinned "
                             "host memory by the kernel over the host link"),
        "staged": (st_ms, "zs_zero2_step_host: bucket-wise H2D through a 2-slot device staging ring on a "
                          "copy stream, fused update per bucket, D2H of rank 0's replica on a third stream"),
    }
    order = sorted(paths, key=lambda k: paths[k][0])
    for i, key in enumerate(order):
        ms_, desc = paths[key]
        rec = {"value": ws * plan.numel / (ms_ / 1e3), "unit": "params/s", "ms_per_step": ms_,
               "h2d_bytes_per_step": n_d * P * 2, "d2h_bytes_per_step": P * 2, "path": desc}
        if i == 0:
            e2e = rec
        else:
            e2e_alt = rec
    del host_g, host_out, hrows, staging
    return e2e, e2e_alt


def zs_synth_buffers(n_d, n, dev):
    import torch

    import synth

    return synth.rank_buffers(n_d, n, torch.bfloat16, dev)[0]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default 200; 20 for the ZeRO-3 workload)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama-1.3b-zero2")
    ap.add_argument("--profile-case", action="store_true")
    ap.add_argument("--profile-elems", type=int, default=32 << 20,
                    help="elements of the --profile-case flat buffer")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--unfused-steps", type=int, default=10)
    ap.add_argument("--bucketwise-steps", type=int, default=10)
    ap.add_argument("--step-mode", choices=["whole", "per-bucket", "per-bucket-2s"], default="whole",
                    help="fused workloads: one call over the whole flat space (default), or every bucket stepped "
                         "bucket by bucket, last first (one stream / two streams)")
    ap.add_argument("--bucket-bytes", type=int, default=None, help="override the workload's bucket size")
    ap.add_argument("--accumulate-mode", choices=["fused-last", "separate"], default="fused-last",
                    help="workloads with micro-batches: the last micro-batch's accumulation inside the step, or "
                         "every micro-batch accumulated before it")
    ap.add_argument("--fused-variant", choices=["auto", "ldg", "tma"], default="auto",
                    help="kernel behind the fused step (all variants compute identical results)")
    args = ap.parse_args()
    if args.impl == "reference":
        import synth

        if args.workload not in synth.WORKLOADS:
            ap.error("--impl reference times the oracle on one of the workloads %s" % sorted(synth.WORKLOADS))
    if args.step_mode != "whole" and args.impl == "ours":
        import synth

        wl = synth.WORKLOADS.get(args.workload, {})
        if wl.get("stage") == 3 or wl.get("micro", 1) > 1 or args.workload in ("flat-sweep", "next-rows"):
            ap.error("--step-mode applies to the fused ZeRO-1/2 workloads without accumulation")
    if args.warmup < 3 and args.impl == "ours" and not args.profile_case:
        log("note: fewer than 3 warm-up steps")
    if args.steps is None:
        args.steps = 20 if "zero3" in args.workload else (10 if args.workload in ("flat-sweep", "next-rows") else 200)
    ws, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, ws, rank)
    try:
        if args.workload == "flat-sweep":
            return run_sweep(args, ws, rank, local)
        if args.workload == "next-rows":
            return run_next(args, ws, rank, local)
        return run_ours(args, ws, rank, local)
    except DeviceStatusError as exc:
        log("bench.py: %s" % exc)
        return 3


if __name__ == "__main__":
    sys.exit(main())
