"""zs_rank_shard_step against the oracle (GPU): the local part of a rank's step when every rank is its
own process.

The ranks are simulated in one process (no rank waits on another): for each rank r the slices an
all-to-all would deliver are cut from every rank's gradient buffer with torch, and the call updates
rank r's own shard state (local layout) from them.  The results must equal the oracle's simulated
step (steps.zero_step) bit for bit, bucket by bucket and for the whole shard at once, on plans whose
local offsets keep 16-byte alignment (the staged kernel for parts of 2^20 elements and more) and on
plans whose offsets do not (the streaming kernel element by element).
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

CASES = {
    # S = 2 Mi elements per rank: most bucket parts take the staged kernel
    "aligned-n8": dict(shapes=[(1 << 24,)], units=None, n_d=8, bucket_bytes=25 << 20),
    # ragged: 1,000,003 elements padded to N_d = 8, 128 Ki-element buckets
    "ragged-n8": dict(shapes=[(1_000_003,)], units=None, n_d=8, bucket_bytes=1 << 18),
    # several units, N_d = 3: odd local offsets, element by element
    "units-n3": dict(shapes=[(64, 48), (48,), (100, 30), (30,), (7, 5)], units=[0, 0, 1, 1, 2], n_d=3,
                     bucket_bytes=2_000),
    # more ranks than elements, one-element buckets: most parts empty
    "tiny-n8": dict(shapes=[(3,), (4,)], units=None, n_d=8, bucket_bytes=2),
    # one rank: the rank's part is the whole bucket
    "one-rank": dict(shapes=[(1,), (70_001,)], units=[0, 1], n_d=1, bucket_bytes=1 << 12),
}


def _part_slices(grads, lo, hi):
    """What an all-to-all delivers to the owner of [lo, hi): every rank's gradients there, each in a
    buffer of its own (16-byte aligned, as the call requires)."""
    return [g[lo:hi].clone() for g in grads]


@pytest.mark.parametrize("whole", [False, True])
@pytest.mark.parametrize("case", sorted(CASES))
def test_rank_shard_step_matches_the_oracle(case, whole):
    cfg = CASES[case]
    n_d = cfg["n_d"]
    plan = zs.Plan(cfg["shapes"], n_d, stage=2, bucket_bytes=cfg["bucket_bytes"], unit_of_param=cfg["units"])
    oplan = layout.make_plan(cfg["shapes"], n_d, unit_of_param=cfg["units"], bucket_bytes=cfg["bucket_bytes"])
    P, pads, S = plan.padded, plan.pad_ranges(), plan.shard_per_rank
    master_full = synth.master_init(P, pads, seed=51, device=DEV)
    mf = H.to_np_f32(master_full)
    state = [[torch.from_numpy(steps.shard_of(oplan, r, mf).copy()).to(DEV), torch.zeros(S, device=DEV),
              torch.zeros(S, device=DEV)] for r in range(n_d)]
    shards = [torch.zeros(S, dtype=BF16, device=DEV) for _ in range(n_d)]
    o_m = [steps.shard_of(oplan, r, mf) for r in range(n_d)]
    o_mm = [np.zeros(S, np.float32) for _ in range(n_d)]
    o_v = [np.zeros(S, np.float32) for _ in range(n_d)]
    zs.zs_device_status(clear=True)
    for t in (1, 2):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=52, step=t, sigma=1e-3, outlier_p=0.001, device=DEV)
        for r in range(n_d):
            if whole:
                # the rank's pieces of every unit, back to back in unit order
                pieces = []
                for u in range(plan.n_units):
                    ud = plan.unit(u)
                    lo = ud["base"] + r * ud["shard"]
                    pieces.append(_part_slices(grads, lo, lo + ud["shard"]))
                slices = [torch.cat([p[q] for p in pieces]) for q in range(n_d)]
                zs.zs_rank_shard_step(plan, r, -1, slices, *state[r], shards[r], HP, t)
            else:
                for b in reversed(range(plan.n_buckets)):
                    lo, hi, _ = plan.rank_bucket_part(r, b)
                    if hi > lo:
                        zs.zs_rank_shard_step(plan, r, b, _part_slices(grads, lo, hi), *state[r], shards[r], HP, t)
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        reps, o_m, o_mm, o_v = steps.zero_step(oplan, [H.to_np_bf16(g) for g in grads], o_m, o_mm, o_v, HP, t)
        for r in range(n_d):
            what = "%s rank %d t=%d" % (case, r, t)
            H.check_f32(H.to_np_f32(state[r][0]), o_m[r], "master " + what)
            H.check_f32(H.to_np_f32(state[r][1]), o_mm[r], "m " + what)
            H.check_f32(H.to_np_f32(state[r][2]), o_v[r], "v " + what)
            H.check_bf16(H.to_np_bf16(shards[r]), steps.shard_of(oplan, r, reps[r]), "shard " + what)


def test_rank_shard_step_rejects_bad_arguments():
    plan = zs.Plan([(1 << 12,)], 4, stage=2, bucket_bytes=1 << 10)
    S = plan.shard_per_rank
    st = [torch.zeros(S, device=DEV) for _ in range(3)]
    sh = torch.zeros(S, dtype=BF16, device=DEV)
    lo, hi, _ = plan.rank_bucket_part(0, 0)
    sl = [torch.zeros(max(1, hi - lo), dtype=BF16, device=DEV) for _ in range(4)]
    for rank, bucket in ((4, 0), (-1, 0), (0, plan.n_buckets)):
        with pytest.raises(zs.ZsError):
            zs.zs_rank_shard_step(plan, rank, bucket, sl, *st, sh, HP, 1)
    with pytest.raises(zs.ZsError):
        zs.zs_rank_shard_step(plan, 0, 0, sl, *st, sh, HP, 0)             # 0-based step
    with pytest.raises(ValueError):
        zs.zs_rank_shard_step(plan, 0, 0, sl[:3], *st, sh, HP, 1)         # a missing rank


def test_zero_rank_over_nccl_with_one_rank():
    """ZeroRank end to end on the GPU: an NCCL group of one process (the all-to-all, the all-gather
    and the library's local update on device buffers), two ZeRO-2 steps against the oracle."""
    import socket

    import torch.distributed as dist

    from fsdp_sharded_optimizer_flatparameter_gb300.zero_rank import ZeroRank

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % port, rank=0, world_size=1)
    try:
        shapes = [(300, 96), (96,), (257, 96)]
        plan = zs.Plan(shapes, 1, stage=2, bucket_bytes=10_000)
        oplan = layout.make_plan(shapes, 1, bucket_bytes=10_000)
        P, pads = plan.padded, plan.pad_ranges()
        master0 = synth.master_init(P, pads, seed=53, device=DEV)
        master, m, v = master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)
        shard = torch.zeros(P, dtype=BF16, device=DEV)
        replica = torch.zeros(P, dtype=BF16, device=DEV)
        zr = ZeroRank(plan)
        o = [[H.to_np_f32(master0)], [np.zeros(P, np.float32)], [np.zeros(P, np.float32)]]
        for t in (1, 2):
            grads, _ = synth.rank_grads(1, P, pads, seed=54, step=t, sigma=1e-3, device=DEV)
            zr.step(grads[0], master, m, v, shard, replica, HP, t)
            torch.cuda.synchronize()
            reps, o[0], o[1], o[2] = steps.zero_step(oplan, [H.to_np_bf16(grads[0])], o[0], o[1], o[2], HP, t)
            H.check_f32(H.to_np_f32(master), o[0][0], "master t=%d" % t)
            H.check_f32(H.to_np_f32(v), o[2][0], "v t=%d" % t)
            H.check_bf16(H.to_np_bf16(replica), reps[0], "replica t=%d" % t)
        assert zr.bytes_sent == 0                     # one rank sends nothing
    finally:
        dist.destroy_process_group()
