"""Naive data parallelism on the GPU: all-reduce with averaging and the replicated update.

Against the oracle's naive-DP step, and the method's central identity: the
sharded ZeRO step gives every rank the same parameters as naive DP, bit for bit.
"""

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth
from oracle import layout, steps

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.mark.parametrize("n_d,numel,bucket_bytes", [(1, 1000, 0), (3, 70_001, 0), (4, 262_912, 4096), (8, 500_007, 0)])
def test_all_reduce_mean(n_d, numel, bucket_bytes):
    plan = zs.Plan([(numel,)], n_d, stage=0, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    grads, _ = synth.rank_grads(n_d, P, pads, seed=50, step=1, sigma=1e-3, outlier_p=0.01, device=DEV)
    want = steps.reduce_mean([H.to_np_bf16(g) for g in grads])
    if plan.n_buckets > 1:
        for b in range(plan.n_buckets):
            zs.zs_all_reduce_mean(plan, b, grads)
    else:
        zs.zs_all_reduce_mean(plan, -1, grads)
    torch.cuda.synchronize()
    for q in range(n_d):
        H.check_bf16(H.to_np_bf16(grads[q]), want, "rank %d" % q)


@pytest.mark.parametrize("variant", ["auto", "ldg"])
@pytest.mark.parametrize("n_d,numel", [(2, 1_100_003), (4, 1_100_003), (8, 1_100_003), (16, 1_100_003),
                                       (32, 1_100_003), (8, 3 * (1 << 22) + 5), (2, 3 * (1 << 22) + 5)])
def test_all_reduce_mean_every_rank_count(n_d, numel, variant):
    """The in-place all-reduce on buffers of a million elements and more with a ragged tail: the
    bulk-copy staged kernel (3 x 2^22 + 5 elements: walked in three overlapping launches, the ragged
    end streamed) and the register-streaming kernel (ldg) leave the oracle's mean in every rank's
    buffer, bit for bit."""
    plan = zs.Plan([(numel,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    grads, _ = synth.rank_grads(n_d, P, pads, seed=53, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)
    want = steps.reduce_mean([H.to_np_bf16(g) for g in grads])
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG if variant == "ldg" else zs.ZS_FUSED_AUTO)
    try:
        zs.zs_device_status(clear=True)
        zs.zs_all_reduce_mean(plan, -1, grads)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for q in range(n_d):
        H.check_bf16(H.to_np_bf16(grads[q]), want, "rank %d" % q)


@pytest.mark.parametrize("variant", ["tma", "ldg"])
@pytest.mark.parametrize("n_d,numel", [(2, 600_003), (4, 600_003), (8, 600_003), (16, 600_003), (32, 600_003),
                                       (8, 3 * (1 << 22) + 5), (16, (1 << 22) + (1 << 20) + 3), (32, 3_000_005)])
def test_dp_step_every_rank_count(n_d, numel, variant):
    """The naive-DP step on buffers with a ragged tail, every power-of-two rank count, with the staged
    kernel (grads of a tile, then one rank's state after another through the ring; walked in
    overlapping 4 Mi-element launches where the rank count has a walk shape: 3 x 2^22 + 5 elements
    at N_d = 8 are three launches; the tail's few elements by the streaming kernel) and with the
    streaming kernel alone, two steps: every rank's state and replica equal the oracle's, bit for bit."""
    plan = zs.Plan([(numel,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=54, device=DEV)
    dm = [master0.clone() for _ in range(n_d)]
    dmm = [torch.zeros_like(master0) for _ in range(n_d)]
    dv = [torch.zeros_like(master0) for _ in range(n_d)]
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    om, omm, ov = H.to_np_f32(master0), np.zeros(P, np.float32), np.zeros(P, np.float32)
    zs.zs_set_fused_variant(zs.ZS_FUSED_TMA if variant == "tma" else zs.ZS_FUSED_LDG)
    try:
        for t in (1, 2):
            grads, _ = synth.rank_grads(n_d, P, pads, seed=54, step=t, sigma=1e-3, outlier_p=0.001, device=DEV)
            reps_ref, om, omm, ov = steps.dp_step([H.to_np_bf16(g) for g in grads], om, omm, ov, HP, t)
            zs.zs_dp_step(plan, grads, dm, dmm, dv, reps, HP, t)
            torch.cuda.synchronize()
            assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
            for q in range(n_d):
                H.check_f32(H.to_np_f32(dm[q]), om, "master rank %d t=%d" % (q, t))
                H.check_f32(H.to_np_f32(dmm[q]), omm, "m rank %d t=%d" % (q, t))
                H.check_f32(H.to_np_f32(dv[q]), ov, "v rank %d t=%d" % (q, t))
                H.check_bf16(H.to_np_bf16(reps[q]), reps_ref[q], "replica %d t=%d" % (q, t))
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


@pytest.mark.parametrize("n_d", [1, 3, 4, 8])
def test_dp_step_matches_oracle_and_zero(n_d):
    shapes = [(300, 96), (96,), (257, 96), (5,)]
    plan = zs.Plan(shapes, n_d, stage=0)
    ref = layout.make_plan(shapes, n_d)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=51, device=DEV)
    dp_master = [master0.clone() for _ in range(n_d)]
    dp_m = [torch.zeros_like(master0) for _ in range(n_d)]
    dp_v = [torch.zeros_like(master0) for _ in range(n_d)]
    dp_reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    z_master, z_m, z_v = master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)
    z_reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    om, omm, ov = H.to_np_f32(master0), np.zeros(P, np.float32), np.zeros(P, np.float32)
    for t in (1, 2, 3):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=52, step=t, sigma=1e-3, device=DEV)
        reps_ref, om, omm, ov = steps.dp_step([H.to_np_bf16(g) for g in grads], om, omm, ov, HP, t)
        zs.zs_dp_step(plan, grads, dp_master, dp_m, dp_v, dp_reps, HP, t)
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, z_master, z_m, z_v, z_reps, HP, t)
        torch.cuda.synchronize()
        for q in range(n_d):
            H.check_f32(H.to_np_f32(dp_master[q]), om, "dp master rank %d t=%d" % (q, t))
            H.check_f32(H.to_np_f32(dp_v[q]), ov, "dp v rank %d t=%d" % (q, t))
            H.check_bf16(H.to_np_bf16(dp_reps[q]), reps_ref[q], "dp replica %d t=%d" % (q, t))
            # sharded ZeRO == naive DP
            assert torch.equal(z_reps[q], dp_reps[q])
        assert torch.equal(z_master, dp_master[0]) and torch.equal(z_m, dp_m[0]) and torch.equal(z_v, dp_v[0])
    assert plan.memory_bytes(0) == 16 * plan.numel
