"""The fused step with the last micro-batch's accumulation inside it (zs_fused_step_accumulate), on
the GPU, against the oracle: "Infra: Data Parallel", section "Naive Data Parallelism" (gradient
accumulation: each micro-batch's gradient scaled and summed in the bf16 gradient buffer) followed by
the ZeRO step (ZeRO section: reduce-scatter with averaging, AdamW on the shard, all-gather).

The oracle accumulates every micro-batch (steps.accumulate) and then steps on the accumulated
gradients; the library accumulates the first micro-batches with zs_accumulate_grad and hands the
last one to zs_fused_step_accumulate, which forms each rank's gradient in the kernel and never
stores it.  Every element is compared, bit for bit, on sizes that span several tiles, several
launches of a walk and a ragged tail.
"""

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
N_MICRO = 4


@pytest.fixture(autouse=True)
def _status_and_variant():
    zs.zs_device_status(clear=True)
    yield
    zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    torch.cuda.synchronize()
    assert zs.zs_device_status(clear=True) == zs.ZS_DEVERR_NONE


def _setup(n_d, shapes, seed, stage=1, bucket_bytes=0):
    plan = zs.Plan(shapes, n_d, stage=stage, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    micro = [synth.rank_grads(n_d, P, pads, seed=seed, step=j, sigma=1e-3, device=DEV)[0] for j in range(N_MICRO)]
    acc, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    for j in range(N_MICRO - 1):
        zs.zs_accumulate_grad(plan, acc, micro[j], 1.0 / N_MICRO, first=(j == 0))
    master = synth.master_init(P, pads, seed, device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    return plan, micro, acc, master, m, v, reps


def _accumulated(n_d, micro):
    """Oracle: every rank's micro-batches accumulated (the bf16 gradient each rank reduces)."""
    accs = []
    for q in range(n_d):
        a = None
        for j in range(N_MICRO):
            a = steps.accumulate(a, H.to_np_bf16(micro[j][q]), 1.0 / N_MICRO, first=(j == 0))
        accs.append(a)
    return accs


def _oracle_step(accs, p0, m0, v0, t):
    """Oracle: the ZeRO step (mean over ranks, AdamW) on the accumulated gradients."""
    return steps.adamw(p0, m0, v0, steps.reduce_mean(accs), HP, t)


@pytest.mark.parametrize("variant", ["auto", "ldg"])
@pytest.mark.parametrize("n_d,numel", [(1, 4099), (2, 3 * (1 << 22) + 13), (3, 100_003), (4, 5_000_011),
                                       (8, 2 * (1 << 22) + 4099), (8, 1001), (16, 1_048_583), (32, 600_007),
                                       (8, (1 << 24) + 4099), (2, (1 << 24) + 11)])
def test_fused_step_accumulate_matches_oracle(variant, n_d, numel):
    """Two steps (the second with non-zero moments): every element of master, m, v and of every
    replica against the oracle; the accumulators and micro-batch buffers are left as they were.
    Buffers of 2^24 elements and more run as one dynamic-order launch (plus the ragged end)."""
    if variant == "ldg":
        zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    plan, micro, acc, master, m, v, reps = _setup(n_d, [(numel,)], seed=30 + n_d)
    P = plan.padded
    acc_before = [a.clone() for a in acc]
    last_before = [g.clone() for g in micro[-1]]
    p, m1, v1 = H.to_np_f32(master), H.to_np_f32(m), H.to_np_f32(v)
    accs = _accumulated(n_d, micro)
    for t in (1, 2):
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_FULL, 1.0 / N_MICRO, master, m, v, reps,
                                    HP, t)
        torch.cuda.synchronize()
        p, m1, v1, bits = _oracle_step(accs, p, m1, v1, t)
        H.check_f32(H.to_np_f32(master), p, "master t=%d" % t)
        H.check_f32(H.to_np_f32(m), m1, "m t=%d" % t)
        H.check_f32(H.to_np_f32(v), v1, "v t=%d" % t)
        for q in range(n_d):
            H.check_bf16(H.to_np_bf16(reps[q]), bits, "replica %d t=%d" % (q, t))
    for q in range(n_d):
        assert torch.equal(acc[q], acc_before[q]) and torch.equal(micro[-1][q], last_before[q])
    assert P == plan.padded


@pytest.mark.parametrize("n_d", [2, 8, 32])
def test_fused_step_accumulate_equals_accumulate_then_fused_step(n_d):
    """The same two steps through zs_accumulate_grad + zs_fused_step on a copy of the state: identical
    results on a multi-launch walk (4 Mi-element pieces and a ragged end)."""
    numel = 9 * (1 << 20) + 7
    plan, micro, acc, master, m, v, reps = _setup(n_d, [(numel,)], seed=40 + n_d)
    master2, m2, v2 = master.clone(), m.clone(), v.clone()
    reps2, _ = synth.rank_buffers(n_d, plan.padded, BF16, DEV)
    acc2 = [a.clone() for a in acc]
    for t in (1, 2):
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_FULL, 0.25, master, m, v, reps, HP, t)
        full = [a.clone() for a in acc2]
        zs.zs_accumulate_grad(plan, full, micro[-1], 0.25, first=False)
        zs.zs_fused_step(plan, -1, full, zs.ZS_RANK_FULL, master2, m2, v2, reps2, HP, t)
        torch.cuda.synchronize()
        for name, a, b in (("master", master, master2), ("m", m, m2), ("v", v, v2)):
            assert torch.equal(a, b), "%s differs at t=%d" % (name, t)
        for q in range(n_d):
            assert torch.equal(reps[q], reps2[q]), "replica %d differs at t=%d" % (q, t)


@pytest.mark.parametrize("kind", ["full", "bucket"])
def test_fused_step_accumulate_bucket_by_bucket(kind):
    """Every bucket stepped on its own, last first (RANK_FULL buffers, or each bucket's own staging
    buffers with RANK_BUCKET): the whole-buffer oracle result."""
    n_d = 4
    plan, micro, acc, master, m, v, reps = _setup(n_d, [(3000, 7), (77,), (65_536 * 3 + 5,)], seed=51, stage=2,
                                                 bucket_bytes=2 * 70_000)
    assert plan.n_buckets >= 4
    p0 = H.to_np_f32(master)
    for b in reversed(range(plan.n_buckets)):
        _, lo, hi = plan.bucket(b)
        if kind == "full":
            a_b, g_b = acc, micro[-1]
        else:
            a_b = [a[lo:hi].clone() for a in acc]
            g_b = [g[lo:hi].clone() for g in micro[-1]]
        zs.zs_fused_step_accumulate(plan, b, a_b, g_b, zs.ZS_RANK_FULL if kind == "full" else zs.ZS_RANK_BUCKET,
                                    0.25, master, m, v, reps, HP, 1)
    torch.cuda.synchronize()
    z = np.zeros(plan.padded, np.float32)
    p, m1, v1, bits = _oracle_step(_accumulated(n_d, micro), p0, z, z, 1)
    H.check_f32(H.to_np_f32(master), p, "master")
    H.check_f32(H.to_np_f32(v), v1, "v")
    for q in range(n_d):
        H.check_bf16(H.to_np_bf16(reps[q]), bits, "replica %d" % q)


def test_fused_step_accumulate_pinned_host_micro_batch():
    """The last micro-batch and rank 0's replica in pinned host memory (the streaming kernel reads
    and writes them over the host link): the oracle result."""
    n_d = 8
    plan, micro, acc, master, m, v, reps = _setup(n_d, [(2_000_003,)], seed=61)
    host_micro = [g.cpu().pin_memory() for g in micro[-1]]
    host_rep0 = torch.zeros(plan.padded, dtype=BF16).pin_memory()
    reps = [host_rep0] + reps[1:]
    p0 = H.to_np_f32(master)
    zs.zs_fused_step_accumulate(plan, -1, acc, host_micro, zs.ZS_RANK_FULL, 0.25, master, m, v, reps, HP, 1)
    torch.cuda.synchronize()
    z = np.zeros(plan.padded, np.float32)
    p, _, v1, bits = _oracle_step(_accumulated(n_d, micro), p0, z, z, 1)
    H.check_f32(H.to_np_f32(master), p, "master")
    H.check_f32(H.to_np_f32(v), v1, "v")
    H.check_bf16(H.to_np_bf16(host_rep0), bits, "host replica 0")
    H.check_bf16(H.to_np_bf16(reps[n_d - 1]), bits, "replica %d" % (n_d - 1))


def test_fused_step_accumulate_rejects_bad_calls_and_writes_nothing():
    n_d = 2
    plan, micro, acc, master, m, v, reps = _setup(n_d, [(4096,)], seed=71)
    before = master.clone()
    with pytest.raises(zs.ZsError, match="replicas must not be"):
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_FULL, 0.25, master, m, v,
                                    [acc[0], reps[1]], HP, 1)
    with pytest.raises(zs.ZsError, match="scale must be finite"):
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_FULL, float("inf"), master, m, v, reps,
                                    HP, 1)
    with pytest.raises(zs.ZsError, match="bucket"):                 # refused by the binding's size check first
        zs.zs_fused_step_accumulate(plan, -1, acc, micro[-1], zs.ZS_RANK_BUCKET, 0.25, master, m, v, reps, HP, 1)
    torch.cuda.synchronize()
    assert torch.equal(master, before)
