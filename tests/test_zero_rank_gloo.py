"""One data-parallel rank per process: the exchanges of ZeroRank on CPU gloo groups (world size 2 and 3).

Each process is one rank: it holds only its own gradients, its own shard of the fp32 state and of the
bf16 parameters, and a full replica.  The all-to-all of every bucket, the all-gather of the shards
and the ZeRO-3 unit gathers run over torch.distributed (gloo here, NCCL between GPUs).  The library's
kernels cannot run on a CPU group, so each rank's local update (ZeroRank.local_update, overridden
here) is the oracle's reduce-mean and AdamW on the slices the exchange delivered; the GPU test of zs_rank_shard_step checks the kernel side of
the same update.  Every rank's results must equal the oracle's simulated step (steps.zero_step,
steps.zero3_unit_step) bit for bit, and the bytes each rank sent must equal the plan's
communication count.
"""

import os
import socket
import sys
import traceback

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = {
    "flat": dict(shapes=[(300, 96), (96,), (257, 96)], units=None, bucket_bytes=10_000),
    "units": dict(shapes=[(64, 48), (48,), (100, 30), (30,), (7, 5)], units=[0, 0, 1, 1, 2], bucket_bytes=2_000),
    # fewer elements than ranks have room for: one-element buckets, most parts empty
    "tiny": dict(shapes=[(3,), (2,)], units=None, bucket_bytes=2),
}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def _from_bits(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def _oracle_rank_class(ZeroRank, steps):
    """ZeroRank whose local update is the oracle's, on the exchanged slices (CPU groups, where the
    library's kernels cannot run); the exchanges and gathers are ZeroRank's own."""

    class OracleRank(ZeroRank):
        def local_update(self, bucket, slices, master, m, v, param_shard, hp, t):
            _oracle_update(self.plan, self.rank, steps, bucket, slices, master, m, v, param_shard, hp, t)

    return OracleRank


def _oracle_update(plan, rank, steps, bucket, slices, master, m, v, param_shard, hp, t):
    lo, hi, local = plan.rank_bucket_part(rank, bucket)
    n = hi - lo
    ghat = steps.reduce_mean([_bits(s) for s in slices])
    p, m1, v1, bits = steps.adamw(master[local:local + n].numpy(), m[local:local + n].numpy(),
                                  v[local:local + n].numpy(), ghat, hp, t)
    master[local:local + n] = torch.from_numpy(p)
    m[local:local + n] = torch.from_numpy(m1)
    v[local:local + n] = torch.from_numpy(v1)
    param_shard[local:local + n] = _from_bits(bits)


def _worker(rank, world, port, case, stage, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import fsdp_sharded_optimizer_flatparameter_gb300 as zs
        import synth
        from fsdp_sharded_optimizer_flatparameter_gb300.zero_rank import ZeroRank
        from oracle import layout, steps

        cfg = CASES[case]
        hp = synth.HPARAMS
        plan = zs.Plan(cfg["shapes"], world, stage=stage, bucket_bytes=cfg["bucket_bytes"],
                       unit_of_param=cfg["units"])
        oplan = layout.make_plan(cfg["shapes"], world, unit_of_param=cfg["units"],
                                 bucket_bytes=cfg["bucket_bytes"])
        P, pads, S = plan.padded, plan.pad_ranges(), plan.shard_per_rank
        master_full = synth.master_init(P, pads, seed=41)
        # this rank's own state: its shard of every unit, in its local layout
        mine = steps.shard_of(oplan, rank, master_full.numpy())
        master, m, v = torch.from_numpy(mine.copy()), torch.zeros(S), torch.zeros(S)
        param_shard = _from_bits(np.zeros(S, np.uint16))
        zr = _oracle_rank_class(ZeroRank, steps)(plan)
        o_m = [steps.shard_of(oplan, r, master_full.numpy()) for r in range(world)]
        o_mm = [np.zeros(oplan.shard_total, np.float32) for _ in range(world)]
        o_v = [np.zeros(oplan.shard_total, np.float32) for _ in range(world)]
        o_sh = [np.zeros(oplan.shard_total, np.uint16) for _ in range(world)]
        bad = []
        for t in (1, 2):
            grads, _ = synth.rank_grads(world, P, pads, seed=42, step=t, sigma=1e-3, outlier_p=0.01)
            g_np = [_bits(g) for g in grads]
            if stage == 3:
                for u in range(plan.n_units):
                    ud = plan.unit(u)
                    want = steps.all_gather_unit(oplan, u, o_sh)[rank]
                    for phase in ("forward", "backward"):        # gathered, freed, gathered again
                        full = _from_bits(np.zeros(ud["padded"], np.uint16))
                        zr.gather_unit(u, param_shard, full)
                        if not np.array_equal(_bits(full), want):
                            bad.append("%s gather of unit %d at t=%d" % (phase, u, t))
                    unit_g = [g[ud["base"]:ud["base"] + ud["padded"]] for g in g_np]
                    zr.unit_step(u, grads[rank][ud["base"]:ud["base"] + ud["padded"]].clone(), master, m, v,
                                 param_shard, hp, t)
                    _, _, o_sh, o_m, o_mm, o_v = steps.zero3_unit_step(oplan, u, o_sh, unit_g, o_m, o_mm, o_v,
                                                                      hp, t)
            else:
                replica = _from_bits(np.zeros(P, np.uint16))
                zr.step(grads[rank], master, m, v, param_shard, replica, hp, t)
                reps, o_m, o_mm, o_v = steps.zero_step(oplan, g_np, o_m, o_mm, o_v, hp, t)
                if not np.array_equal(_bits(replica), reps[rank]):
                    bad.append("replica at t=%d" % t)
                o_sh = [steps.shard_of(oplan, r, reps[r]) for r in range(world)]
            for name, got, want in (("master", master.numpy(), o_m[rank]), ("m", m.numpy(), o_mm[rank]),
                                    ("v", v.numpy(), o_v[rank])):
                if not np.array_equal(got.view(np.uint32), want.view(np.uint32)):
                    bad.append("%s at t=%d" % (name, t))
            if not np.array_equal(_bits(param_shard), o_sh[rank]):
                bad.append("parameter shard at t=%d" % t)
        sent_per_step = zr.bytes_sent / 2
        want_sent = plan.comm_bytes(stage)
        out[rank] = (bad, sent_per_step, want_sent)
    except Exception:
        out[rank] = (["exception: " + traceback.format_exc()[-2000:]], 0, 0)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("case,stage", [("flat", 2), ("units", 2), ("units", 3), ("tiny", 2)])
def test_zero_rank_exchanges_match_the_oracle(world, case, stage):
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_worker, args=(world, port, case, stage, out), nprocs=world, join=True,
                       start_method="spawn")
    assert sorted(out.keys()) == list(range(world))
    for r in range(world):
        bad, sent, want = out[r]
        assert not bad, "rank %d: %s" % (r, bad)
        assert sent == want, "rank %d sent %d bytes per step, the plan counts %d" % (r, sent, want)
