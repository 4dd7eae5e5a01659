"""Every-element oracle parity at the benchmarked sizes (GPU).

The sampled full-size tests check chunks of the flat space; a race that hits
one element in 10^5 would slip through them.  Here the benchmarked call runs
once on the full workload, then the whole flat space is walked in chunks and
every element of every output is compared with the oracle, bit for bit:

* the Llama-1.3B ZeRO-2 step at N_d = 8 (1,345,423,360 elements), exactly
  the call the benchmark times (zs_fused_step over the whole flat space, the
  whole range in one launch that takes its tiles in dynamic order), at step 2 so the moments going
  in are not zero;
* the whole Llama-7B ZeRO-3 step at N_d = 16 (zs_zero3_step, both streams,
  the 2-slot pool), at step 2, on its largest unit (the root unit: embedding,
  final norm and output, 262,148,096 elements) with the parameter shards;
* the GPT-2-small step with four micro-batches at N_d = 8, the last one
  accumulated inside the step (as benchmarked) and all four before it (every
  stored accumulated gradient too);
* the 2^28+7-element flat buffer at N_d = 32 (padding, the widest rank count);
* a flat buffer past 2^32 elements at N_d = 2 (element offsets, tile counts
  and tile indices that overflow 32-bit integers): the fused step (one
  dynamic-order launch) against the oracle, then the bucket-by-bucket walk and the unfused calls
  against that result on the device.

Every step is element-wise, so the oracle on a chunk needs only that chunk's
inputs.  Chunks are checked by a pool of host threads (numpy releases the GIL
in its array operations), each copying its chunk from the device, running
the oracle's reduce-mean and AdamW on it and comparing.
"""

import concurrent.futures as cf
import gc
import os
import time

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth
from oracle import steps

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16
CHUNK = 1 << 23
THREADS = max(2, min(16, os.cpu_count() or 2))


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _bits16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _f32(t):
    return t.detach().cpu().contiguous().numpy()


def _first_diff(got, want):
    bad = np.flatnonzero(got != want)
    return None if bad.size == 0 else (int(bad.size), int(bad[0]))


def _verify(n, job, label):
    """Runs job(lo, hi) -> list of (name, count, first index) over [0, n) in chunks on a thread pool."""
    t0 = time.perf_counter()
    spans = [(lo, min(n, lo + CHUNK)) for lo in range(0, n, CHUNK)]
    bad = []
    with cf.ThreadPoolExecutor(THREADS) as ex:
        for (lo, hi), res in zip(spans, ex.map(lambda s: job(*s), spans)):
            bad += ["%s [%d,%d): %d values differ, first at %d" % (name, lo, hi, cnt, lo + first)
                    for name, cnt, first in res]
    print("%s: %d elements checked in %d chunks on %d threads, %.1f s"
          % (label, n, len(spans), THREADS, time.perf_counter() - t0))
    assert not bad, "\n".join(bad[:20])


def test_llama13b_zero2_step_every_element():
    wl = synth.WORKLOADS["llama-1.3b-zero2"]
    shapes, _ = synth.workload_params(wl["model"])
    n_d = wl["n_d"]
    plan = zs.Plan(shapes, n_d, stage=wl["stage"], bucket_bytes=wl["bucket_bytes"])
    P, pads = plan.padded, plan.pad_ranges()
    assert plan.numel == 1_345_423_360
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, wl["seed"], 1, wl["sigma"], wl["outlier_p"])
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    synth.fill_grads(grads, pads, wl["seed"], 2, wl["sigma"], wl["outlier_p"])
    torch.cuda.synchronize()
    p0, m0, v0 = _f32(master), _f32(m), _f32(v)           # the state going into step 2
    zs.zs_device_status(clear=True)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 2)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE

    def job(lo, hi):
        g = [_bits16(grads[q][lo:hi]) for q in range(n_d)]
        ghat = steps.reduce_mean(g)
        p, m1, v1, bits = steps.adamw(p0[lo:hi], m0[lo:hi], v0[lo:hi], ghat, HP, 2)
        out = []
        for name, dev_t, want in (("master", master, p), ("m", m, m1), ("v", v, v1)):
            d = _first_diff(_f32(dev_t[lo:hi]).view(np.uint32), want.view(np.uint32))
            if d:
                out.append((name,) + d)
        d = _first_diff(_bits16(reps[0][lo:hi]), bits)
        if d:
            out.append(("replica 0",) + d)
        for q in range(1, n_d):
            if not torch.equal(reps[q][lo:hi], reps[0][lo:hi]):
                out.append(("replica %d vs replica 0" % q, -1, 0))
        return out

    _verify(P, job, "Llama-1.3B ZeRO-2 step, N_d=8")


def test_llama7b_zero3_step_root_unit_every_element():
    wl = synth.WORKLOADS["llama-7b-zero3"]
    shapes, units = synth.workload_params(wl["model"])
    n_d = wl["n_d"]
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, pads = plan.padded, plan.pad_ranges()
    sizes = [plan.unit(u)["padded"] for u in range(plan.n_units)]
    root = int(np.argmax(sizes))
    ud = plan.unit(root)
    base, up = ud["base"], ud["padded"]
    assert up == 262_148_096 and up == ud["numel"]                # no padding in this unit
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = master.to(BF16)
    biggest = max(sizes)
    ugrads, _ = synth.rank_buffers(n_d, biggest, BF16, DEV)
    synth.fill_grads(ugrads, [], wl["seed"], 1, wl["sigma"])
    pool = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(2)]
    side = torch.cuda.Stream()
    zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * plan.n_units, pool, True, HP, 1, side_stream=side)
    synth.fill_grads(ugrads, [], wl["seed"], 2, wl["sigma"])
    torch.cuda.synchronize()
    p0, m0, v0 = (_f32(x[base:base + up]) for x in (master, m, v))
    zs.zs_device_status(clear=True)
    zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * plan.n_units, pool, True, HP, 2, side_stream=side)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE

    def job(lo, hi):
        g = [_bits16(ugrads[q][lo:hi]) for q in range(n_d)]
        ghat = steps.reduce_mean(g)
        p, m1, v1, bits = steps.adamw(p0[lo:hi], m0[lo:hi], v0[lo:hi], ghat, HP, 2)
        out = []
        for name, dev_t, want in (("master", master, p), ("m", m, m1), ("v", v, v1)):
            d = _first_diff(_f32(dev_t[base + lo:base + hi]).view(np.uint32), want.view(np.uint32))
            if d:
                out.append((name,) + d)
        d = _first_diff(_bits16(shards[base + lo:base + hi]), bits)
        if d:
            out.append(("shards",) + d)
        return out

    _verify(up, job, "Llama-7B ZeRO-3 step, N_d=16, root unit")


@pytest.mark.parametrize("mode", ["fused-last", "separate"])
def test_gpt2_small_accumulate_and_step_every_element(mode):
    """GPT-2-small, N_d = 8, four micro-batches with the 1/4 loss scale, as the benchmark steps them:
    "fused-last" accumulates three with zs_accumulate_grad and hands the fourth to
    zs_fused_step_accumulate (the benchmark's default); "separate" accumulates all four, then the
    walked zs_fused_step.  Every stored accumulated gradient and every output element against the
    oracle."""
    wl = synth.WORKLOADS["gpt2-small-zero1"]
    shapes, _ = synth.workload_params(wl["model"])
    n_d, micro_n = wl["n_d"], wl["micro"]
    plan = zs.Plan(shapes, n_d, stage=wl["stage"], bucket_bytes=wl["bucket_bytes"])
    P, pads = plan.padded, plan.pad_ranges()
    acc, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    micro = [synth.rank_buffers(n_d, P, BF16, DEV)[0] for _ in range(micro_n)]
    stored = micro_n if mode == "separate" else micro_n - 1        # micro-batches accumulated into acc
    for j in range(micro_n):
        synth.fill_grads(micro[j], pads, wl["seed"], 100 + j, wl["sigma"])
        if j < stored:
            zs.zs_accumulate_grad(plan, acc, micro[j], 1.0 / micro_n, first=(j == 0))
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    torch.cuda.synchronize()
    p0 = _f32(master)
    zs.zs_device_status(clear=True)
    if mode == "separate":
        zs.zs_fused_step(plan, -1, acc, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    else:
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_FULL, 1.0 / micro_n, master, m, v, reps,
                                    HP, 1)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE

    def job(lo, hi):
        out = []
        accs = []
        for q in range(n_d):
            a = None
            for j in range(micro_n):
                a = steps.accumulate(a, _bits16(micro[j][q][lo:hi]), 1.0 / micro_n, first=(j == 0))
                if j == stored - 1:
                    d = _first_diff(_bits16(acc[q][lo:hi]), a)
                    if d:
                        out.append(("accumulated gradient of rank %d" % q,) + d)
            accs.append(a)
        ghat = steps.reduce_mean(accs)
        z = np.zeros(hi - lo, np.float32)
        p, m1, v1, bits = steps.adamw(p0[lo:hi], z, z, ghat, HP, 1)
        for name, dev_t, want in (("master", master, p), ("m", m, m1), ("v", v, v1)):
            d = _first_diff(_f32(dev_t[lo:hi]).view(np.uint32), want.view(np.uint32))
            if d:
                out.append((name,) + d)
        for q in range(n_d):
            d = _first_diff(_bits16(reps[q][lo:hi]), bits)
            if d:
                out.append(("replica %d" % q,) + d)
        return out

    _verify(P, job, "GPT-2-small 4 micro-batches + ZeRO-1 step (%s), N_d=8" % mode)


def test_flat_sweep_n32_step_every_element():
    """The 2^28+7-element flat buffer at N_d = 32 (25 padding elements, the widest walk shape's rank
    count): the fused step (one dynamic-order launch), every element of every output against the oracle."""
    n_d = 32
    plan = zs.Plan([(2 ** 28 + 7,)], n_d, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    assert P - plan.numel == 25
    master = synth.master_init(P, pads, 4, device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, 4, 1, 1e-3)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    p0 = _f32(master)
    zs.zs_device_status(clear=True)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE

    def job(lo, hi):
        g = [_bits16(grads[q][lo:hi]) for q in range(n_d)]
        ghat = steps.reduce_mean(g)
        z = np.zeros(hi - lo, np.float32)
        p, m1, v1, bits = steps.adamw(p0[lo:hi], z, z, ghat, HP, 1)
        out = []
        for name, dev_t, want in (("master", master, p), ("m", m, m1), ("v", v, v1)):
            d = _first_diff(_f32(dev_t[lo:hi]).view(np.uint32), want.view(np.uint32))
            if d:
                out.append((name,) + d)
        d = _first_diff(_bits16(reps[0][lo:hi]), bits)
        if d:
            out.append(("replica 0",) + d)
        for q in range(1, n_d):
            if not torch.equal(reps[q][lo:hi], reps[0][lo:hi]):
                out.append(("replica %d vs replica 0" % q, -1, 0))
        return out

    _verify(P, job, "flat 2^28+7 fused step, N_d=32")


def test_flat_buffer_past_2p32_elements():
    """One flat tensor of 2^32 + 2^22 + 3 elements at N_d = 2 (one padding element): every offset
    past 2^31 and 2^32 that a 32-bit index would wrap.  The fused step (one dynamic-order launch) is checked against the
    oracle on every element; the same step bucket by bucket (25 MiB buckets, last first) and the
    unfused ZeRO-2 calls (reduce-scatter into a sharded staging buffer, update, all-gather) run on
    copies of the initial state and must reproduce it bit for bit."""
    n_d = 2
    numel = 2 ** 32 + 2 ** 22 + 3
    plan = zs.Plan([(numel,)], n_d, stage=2, bucket_bytes=25 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    assert P == numel + 1 and plan.n_buckets > 300
    free, _ = torch.cuda.mem_get_info()
    # at the peak: grads, replicas and fp32 state twice over (2 n_d + 2 n_d + 12 + 12 + 2 n_d B per
    # element) plus the initial master (4 B), later the staging and shard buffers (2 + 2 B)
    need = P * (6 * n_d + 24 + 4) + (4 << 30)
    if free < need:
        pytest.skip("needs %.0f GB of free device memory, %.0f GB free" % (need / 1e9, free / 1e9))
    master = synth.master_init(P, pads, 4, device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, 4, 1, 1e-3)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    p0 = _f32(master)
    master2 = master.clone()
    m2, v2 = torch.zeros_like(master), torch.zeros_like(master)
    reps2, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    zs.zs_device_status(clear=True)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE

    def job(lo, hi):
        g = [_bits16(grads[q][lo:hi]) for q in range(n_d)]
        ghat = steps.reduce_mean(g)
        z = np.zeros(hi - lo, np.float32)
        p, m1, v1, bits = steps.adamw(p0[lo:hi], z, z, ghat, HP, 1)
        out = []
        for name, dev_t, want in (("master", master, p), ("m", m, m1), ("v", v, v1)):
            d = _first_diff(_f32(dev_t[lo:hi]).view(np.uint32), want.view(np.uint32))
            if d:
                out.append((name,) + d)
        d = _first_diff(_bits16(reps[0][lo:hi]), bits)
        if d:
            out.append(("replica 0",) + d)
        if not torch.equal(reps[1][lo:hi], reps[0][lo:hi]):
            out.append(("replica 1 vs replica 0", -1, 0))
        return out

    _verify(P, job, "flat 2^32+2^22+3 fused step, N_d=2")
    del p0
    gc.collect()

    def same_as_fused(label):
        for name, got, want in (("master", master2, master), ("m", m2, m), ("v", v2, v),
                                ("replica 0", reps2[0], reps[0]), ("replica 1", reps2[1], reps[1])):
            for lo in range(0, P, 1 << 30):
                hi = min(P, lo + (1 << 30))
                assert torch.equal(got[lo:hi], want[lo:hi]), "%s: %s differs in [%d, %d)" % (label, name, lo, hi)

    def reset_state(init):
        master2.copy_(init)
        m2.zero_()
        v2.zero_()
        for r in reps2:
            r.zero_()

    init = master2.clone()
    zs.zs_fused_step_buckets(plan, list(reversed(range(plan.n_buckets))), grads, master2, m2, v2, reps2, HP, 1,
                             launch_mode=zs.ZS_BUCKETS_PER_BUCKET)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    same_as_fused("bucket by bucket")

    reset_state(init)
    del init
    ghat = torch.zeros(P, dtype=BF16, device=DEV)
    shards = torch.zeros(P, dtype=BF16, device=DEV)
    for b in reversed(range(plan.n_buckets)):
        zs.zs_reduce_scatter_mean(plan, b, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
    zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, master2, m2, v2, [shards], zs.ZS_SHARDED, HP, 1)
    zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, reps2)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    same_as_fused("unfused reduce-scatter, update, all-gather")
