"""Full-size parity on the benchmarked model shapes, sampled.

The device runs the whole flat buffer in the launch configuration the
benchmark times; the oracle recomputes chosen chunks of the flat space (both
ends, every bucket or unit boundary probed, random chunks) from the same
inputs.  This is exact, not statistical: every step is element-wise, so a
chunk's result depends on that chunk's inputs only.
"""

import gc

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
W = 4096


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    gc.collect()
    torch.cuda.empty_cache()


def _chunks(P, boundaries, seed, n_random=8, width=W):
    rng = np.random.default_rng(seed)
    out = [(0, min(P, width)), (max(0, P - width), P)]
    for b in boundaries:
        out.append((max(0, b - width // 2), min(P, b + width // 2)))
    for _ in range(n_random):
        s = int(rng.integers(0, max(1, P - width)))
        out.append((s, min(P, s + width)))
    return sorted(set(out))


def _snap(t, lo, hi):
    return t[lo:hi].detach().cpu().clone()


def _np(t):
    return H.to_np_bf16(t) if t.dtype == BF16 else H.to_np_f32(t)


def _fused_sampled(plan, grads, master, m, v, reps, t, chunks, launch):
    before = [([_np(_snap(g, lo, hi)) for g in grads], _np(_snap(master, lo, hi)), _np(_snap(m, lo, hi)),
               _np(_snap(v, lo, hi))) for lo, hi in chunks]
    launch()
    torch.cuda.synchronize()
    for (lo, hi), (gc_, p0, m0, v0) in zip(chunks, before):
        _, p, m1, v1, bits = H.chunk_oracle(gc_, p0, m0, v0, HP, t)
        what = "[%d,%d) t=%d" % (lo, hi, t)
        H.check_f32(_np(_snap(master, lo, hi)), p, "master " + what)
        H.check_f32(_np(_snap(m, lo, hi)), m1, "m " + what)
        H.check_f32(_np(_snap(v, lo, hi)), v1, "v " + what)
        for q, r in enumerate(reps):
            H.check_bf16(_np(_snap(r, lo, hi)), bits, "replica %d %s" % (q, what))


def test_llama13b_zero2_fused_full_size():
    """Llama-style 1.3B flat buffer, N_d = 8, grads N(0, 5e-4) with 0.1% entries x100:
    the single fused launch over the whole flat space, two steps."""
    wl = synth.WORKLOADS["llama-1.3b-zero2"]
    shapes, _ = synth.workload_params(wl["model"])
    plan = zs.Plan(shapes, wl["n_d"], stage=wl["stage"], bucket_bytes=wl["bucket_bytes"])
    P, pads = plan.padded, plan.pad_ranges()
    assert plan.numel == 1_345_423_360
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps, _ = synth.rank_buffers(wl["n_d"], P, BF16, DEV)
    grads, _ = synth.rank_buffers(wl["n_d"], P, BF16, DEV)
    bounds = [plan.bucket(b)[1] for b in range(1, plan.n_buckets)]
    chunks = _chunks(P, bounds[:4] + bounds[-4:], seed=2)
    for t in (1, 2):
        synth.fill_grads(grads, pads, wl["seed"], t, wl["sigma"], wl["outlier_p"])
        _fused_sampled(plan, grads, master, m, v, reps, t, chunks,
                       lambda: zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, t))


def test_gpt2_small_zero1_accumulate_then_fused_full_size():
    """GPT-2-small flat buffer, N_d = 8, 4 micro-batches each x1/4 accumulated, then the fused step."""
    wl = synth.WORKLOADS["gpt2-small-zero1"]
    shapes, _ = synth.workload_params(wl["model"])
    plan = zs.Plan(shapes, wl["n_d"], stage=wl["stage"], bucket_bytes=wl["bucket_bytes"])
    P, pads = plan.padded, plan.pad_ranges()
    assert plan.numel == 124_439_808 and plan.n_buckets == 10
    bounds = [plan.bucket(b)[1] for b in range(1, plan.n_buckets)]
    chunks = _chunks(P, bounds, seed=1)
    acc, _ = synth.rank_buffers(wl["n_d"], P, BF16, DEV)
    micro, _ = synth.rank_buffers(wl["n_d"], P, BF16, DEV)
    ref_acc = {c: [None] * wl["n_d"] for c in chunks}
    for j in range(wl["micro"]):
        synth.fill_grads(micro, pads, wl["seed"], 100 + j, wl["sigma"])
        zs.zs_accumulate_grad(plan, acc, micro, 1.0 / wl["micro"], first=(j == 0))
        for (lo, hi) in chunks:
            for q in range(wl["n_d"]):
                ref_acc[(lo, hi)][q] = steps.accumulate(ref_acc[(lo, hi)][q], _np(_snap(micro[q], lo, hi)),
                                                        1.0 / wl["micro"], first=(j == 0))
    torch.cuda.synchronize()
    for (lo, hi) in chunks:
        for q in range(wl["n_d"]):
            H.check_bf16(_np(_snap(acc[q], lo, hi)), ref_acc[(lo, hi)][q], "acc q=%d [%d,%d)" % (q, lo, hi))
    del micro
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps, _ = synth.rank_buffers(wl["n_d"], P, BF16, DEV)
    _fused_sampled(plan, acc, master, m, v, reps, 1, chunks,
                   lambda: zs.zs_fused_step(plan, -1, acc, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1))


def test_llama7b_zero3_units_full_size():
    """Llama-7B shapes, N_d = 16, one unit per layer plus the root unit: gather,
    reduce-scatter + AdamW per unit on the first layer, the last layer and the root."""
    wl = synth.WORKLOADS["llama-7b-zero3"]
    shapes, units = synth.workload_params(wl["model"])
    n_d = wl["n_d"]
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    assert plan.numel == 6_738_415_616 and plan.n_units == 33
    P, pads = plan.padded, plan.pad_ranges()
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = master.to(BF16)
    for u in (0, 31, 32):
        ud = plan.unit(u)
        base, up = ud["base"], ud["padded"]
        full, _ = synth.rank_buffers(n_d, up, BF16, DEV)
        zs.zs_zero3_gather_unit(plan, u, shards, full)
        torch.cuda.synchronize()
        local = _chunks(up, [r * ud["shard"] for r in range(1, n_d)], seed=u, n_random=4)
        for lo, hi in local:
            want = _np(_snap(shards, base + lo, base + hi))
            for q in range(n_d):
                H.check_bf16(_np(_snap(full[q], lo, hi)), want, "gather u=%d q=%d" % (u, q))
        del full
        grads, _ = synth.rank_buffers(n_d, up, BF16, DEV)
        upads = [(ud["numel"], up)] if up > ud["numel"] else []
        synth.fill_grads(grads, upads, wl["seed"], u, wl["sigma"])
        snaps = [([_np(_snap(g, lo, hi)) for g in grads], _np(_snap(master, base + lo, base + hi)),
                  _np(_snap(m, base + lo, base + hi)), _np(_snap(v, base + lo, base + hi))) for lo, hi in local]
        zs.zs_zero3_rs_step_unit(plan, u, grads, master, m, v, shards, HP, 1)
        torch.cuda.synchronize()
        for (lo, hi), (gc_, p0, m0, v0) in zip(local, snaps):
            _, p, m1, v1, bits = H.chunk_oracle(gc_, p0, m0, v0, HP, 1)
            what = "u=%d [%d,%d)" % (u, lo, hi)
            H.check_f32(_np(_snap(master, base + lo, base + hi)), p, "master " + what)
            H.check_f32(_np(_snap(m, base + lo, base + hi)), m1, "m " + what)
            H.check_f32(_np(_snap(v, base + lo, base + hi)), v1, "v " + what)
            H.check_bf16(_np(_snap(shards, base + lo, base + hi)), bits, "shards " + what)
        del grads


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_flat_2p28_plus_7_sweep(n_d):
    """One flat tensor of 2^28 + 7 elements (padding 1..25): the fused step; bucket-wise
    reduce-scatter at 1 MiB, 64 MiB and 1 GiB buckets; ZeRO-1 in place (odd shard
    sizes take the element-wise path); ZeRO-3 gather and reduce-scatter + update."""
    plan = zs.Plan([(2 ** 28 + 7,)], n_d, stage=1, bucket_bytes=1 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    S = plan.shard_per_rank
    chunks = _chunks(P, [r * S for r in range(1, n_d)][:6] + [P - 13], seed=n_d, n_random=4)
    master = synth.master_init(P, pads, 4, device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, 4, 1, 1e-3)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    _fused_sampled(plan, grads, master, m, v, reps, 1, chunks,
                   lambda: zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1))
    for lo, hi in pads:
        assert not master[lo:hi].any() and not reps[-1][lo:hi].float().any()

    # bucket-wise reduce-scatter into the sharded reduced gradient (ZeRO-2), several bucket sizes
    g_before = {c: [_np(_snap(g, *c)) for g in grads] for c in chunks}
    for mib in (1, 64, 1024):
        bp = zs.Plan([(2 ** 28 + 7,)], n_d, stage=2, bucket_bytes=mib << 20)
        ghat = torch.zeros(P, dtype=BF16, device=DEV)
        for b in reversed(range(bp.n_buckets)):
            zs.zs_reduce_scatter_mean(bp, b, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
        torch.cuda.synchronize()
        for c in chunks:
            H.check_bf16(_np(_snap(ghat, *c)), steps.reduce_mean(g_before[c]), "ghat %d MiB %s" % (mib, c))
        del ghat

    # ZeRO-1 in place: reduce-scatter into the full gradient buffers, update, in-place all-gather
    master2 = synth.master_init(P, pads, 4, device=DEV)
    m2, v2 = torch.zeros_like(master2), torch.zeros_like(master2)
    p_before = {c: _np(_snap(master2, *c)) for c in chunks}
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, grads, zs.ZS_RANK_FULL)
    zs.zs_adamw_shard_step(plan, -1, grads, zs.ZS_RANK_FULL, master2, m2, v2, reps, zs.ZS_RANK_FULL, HP, 1)
    zs.zs_all_gather(plan, reps, zs.ZS_RANK_FULL, reps)
    torch.cuda.synchronize()
    for c in chunks:
        z = np.zeros(c[1] - c[0], np.float32)
        _, p, m1, v1, bits = H.chunk_oracle(g_before[c], p_before[c], z, z, HP, 1)
        H.check_f32(_np(_snap(master2, *c)), p, "zero1 master %s" % (c,))
        H.check_f32(_np(_snap(v2, *c)), v1, "zero1 v %s" % (c,))
        for q in range(n_d):
            H.check_bf16(_np(_snap(reps[q], *c)), bits, "zero1 replica %d %s" % (q, c))
    del reps, grads
    gc.collect()
    torch.cuda.empty_cache()

    # ZeRO-3 with the whole buffer as one unit
    shards = master.to(BF16)
    full, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    zs.zs_zero3_gather_unit(plan, 0, shards, full)
    torch.cuda.synchronize()
    for c in chunks:
        want = _np(_snap(shards, *c))
        for q in (0, n_d - 1):
            H.check_bf16(_np(_snap(full[q], *c)), want, "zero3 gather q=%d %s" % (q, c))
    synth.fill_grads(full, pads, 4, 2, 1e-3)            # reuse the gathered buffers as the unit's gradients
    snaps = {c: ([_np(_snap(g, *c)) for g in full], _np(_snap(master, *c)), _np(_snap(m, *c)), _np(_snap(v, *c)))
             for c in chunks}
    zs.zs_zero3_rs_step_unit(plan, 0, full, master, m, v, shards, HP, 2)
    torch.cuda.synchronize()
    for c in chunks:
        gc_, p0, m0, v0 = snaps[c]
        _, p, m1, v1, bits = H.chunk_oracle(gc_, p0, m0, v0, HP, 2)
        H.check_f32(_np(_snap(master, *c)), p, "zero3 master %s" % (c,))
        H.check_f32(_np(_snap(m, *c)), m1, "zero3 m %s" % (c,))
        H.check_bf16(_np(_snap(shards, *c)), bits, "zero3 shards %s" % (c,))


def test_llama7b_zero3_step_two_streams_full_size():
    """The whole ZeRO-3 step exactly as the benchmark runs it (all 33 units, side stream, 2-slot
    pool, one set of per-rank gradient buffers read as every unit's gradients), sampled chunks of
    three units against the oracle."""
    wl = synth.WORKLOADS["llama-7b-zero3"]
    shapes, units = synth.workload_params(wl["model"])
    n_d = wl["n_d"]
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, pads = plan.padded, plan.pad_ranges()
    master = synth.master_init(P, pads, wl["seed"], device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    shards = master.to(BF16)
    biggest = max(plan.unit(u)["padded"] for u in range(plan.n_units))
    ugrads, _ = synth.rank_buffers(n_d, biggest, BF16, DEV)
    synth.fill_grads(ugrads, [], wl["seed"], 1, wl["sigma"])
    pool = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(2)]
    side = torch.cuda.Stream()
    probe = {}
    for u in (0, 17, 32):
        ud = plan.unit(u)
        for lo, hi in _chunks(ud["padded"], [r * ud["shard"] for r in (1, n_d - 1)], seed=70 + u, n_random=2):
            gb = ud["base"]
            probe[(u, lo, hi)] = ([_np(_snap(g, lo, hi)) for g in ugrads], _np(_snap(master, gb + lo, gb + hi)))
    zs.zs_zero3_step(plan, shards, master, m, v, [ugrads] * plan.n_units, pool, True, HP, 1, side_stream=side)
    torch.cuda.synchronize()
    for (u, lo, hi), (gc_, p0) in probe.items():
        gb = plan.unit(u)["base"]
        z = np.zeros(hi - lo, np.float32)
        _, p, m1, v1, bits = H.chunk_oracle(gc_, p0, z, z, HP, 1)
        # units whose padding falls in the chunk: pad gradients are whatever the buffer holds beyond the
        # unit's real elements, but pad master/m/v are 0 and stay 0 only if the gradient there is 0
        real = min(hi, plan.unit(u)["numel"]) - lo
        what = "u=%d [%d,%d)" % (u, lo, hi)
        H.check_f32(_np(_snap(master, gb + lo, gb + lo + real)), p[:real], "master " + what)
        H.check_f32(_np(_snap(v, gb + lo, gb + lo + real)), v1[:real], "v " + what)
        H.check_bf16(_np(_snap(shards, gb + lo, gb + lo + real)), bits[:real], "shards " + what)
    # after backward, slot u & 1 holds unit 1 and unit 0 gathered before their update
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
