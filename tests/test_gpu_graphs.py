"""The step calls under CUDA-graph capture.

Every device call of the C ABI only enqueues work on the streams it is given (no synchronisation,
no allocation), so a sequence of calls can be captured once into a CUDA graph and replayed: a
launch-bound loop of short calls (per-group FSDP2 conversions, per-unit ZeRO-3 work) then runs
without the host's per-call overhead between kernels.  Each test runs the same calls directly and
from a captured graph, from identical states, and requires bit-identical results.  The step
number is a kernel argument, so a replayed graph repeats the step number it was captured with.
The last test runs a chain of dependent launches with programmatic dependent launch on and off.
"""

import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import synth

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


def _run_both(make_state, body, replays=2):
    """body(state, stream) enqueues the calls; returns (direct state, graph state) after `replays` runs."""
    direct, graphed = make_state(), make_state()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(replays):
            body(direct, s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cs):
        body(graphed, cs)
    torch.cuda.synchronize()
    for _ in range(replays):
        g.replay()
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    return direct, graphed


def _assert_same(a, b):
    assert a.keys() == b.keys()
    for k in a:
        xs, ys = (a[k], b[k]) if isinstance(a[k], list) else ([a[k]], [b[k]])
        for i, (x, y) in enumerate(zip(xs, ys)):
            assert torch.equal(x, y), "%s[%d] differs between the two runs" % (k, i)


@pytest.mark.parametrize("n_d,numel", [(8, 1_500_007), (3, 70_001), (8, 10_000_007)])
def test_accumulate_and_fused_step_replay(n_d, numel):
    """ZeRO-1 with four micro-batches: four accumulations then the fused step (staged at the larger
    sizes, streaming at the smallest; at 10 M elements the step is walked in three overlapping
    launches, captured as programmatic edges), captured and replayed twice."""
    plan = zs.Plan([(numel,)], n_d, stage=1)
    P, pads = plan.padded, plan.pad_ranges()
    micro = [synth.rank_grads(n_d, P, pads, seed=70, step=j + 1, sigma=1e-3, device=DEV)[0] for j in range(4)]
    master0 = synth.master_init(P, pads, seed=71, device=DEV)

    def make_state():
        return {"acc": synth.rank_buffers(n_d, P, BF16, DEV)[0], "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0],
                "master": master0.clone(), "m": torch.zeros_like(master0), "v": torch.zeros_like(master0)}

    def body(st, s):
        for j in range(4):
            zs.zs_accumulate_grad(plan, st["acc"], micro[j], 0.25, j == 0, stream=s)
        zs.zs_fused_step(plan, -1, st["acc"], zs.ZS_RANK_FULL, st["master"], st["m"], st["v"], st["reps"], HP, 1,
                         stream=s)

    _assert_same(*_run_both(make_state, body))


def test_bucket_walks_replay():
    """Bucket-wise stepping: a scattered list (list kernel) and one launch per bucket alternating
    over two streams (forked and joined with events inside the call), captured together."""
    n_d = 8
    plan = zs.Plan([(2_500_003,)], n_d, stage=2, bucket_bytes=1 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    assert plan.n_buckets >= 4
    grads = synth.rank_grads(n_d, P, pads, seed=72, step=1, sigma=1e-3, device=DEV)[0]
    master0 = synth.master_init(P, pads, seed=73, device=DEV)
    even = list(range(0, plan.n_buckets, 2))
    odd = list(range(1, plan.n_buckets, 2))

    def make_state():
        return {"reps": synth.rank_buffers(n_d, P, BF16, DEV)[0], "master": master0.clone(),
                "m": torch.zeros_like(master0), "v": torch.zeros_like(master0), "side": torch.cuda.Stream()}

    def body(st, s):
        args = (grads, st["master"], st["m"], st["v"], st["reps"], HP, 1)
        zs.zs_fused_step_buckets(plan, even, *args, launch_mode=zs.ZS_BUCKETS_ONE_WALK, stream=s)
        zs.zs_fused_step_buckets(plan, list(reversed(odd)), *args, launch_mode=zs.ZS_BUCKETS_PER_BUCKET, stream=s,
                                 side_stream=st["side"])

    a, b = _run_both(make_state, body)
    for st in (a, b):
        del st["side"]
    _assert_same(a, b)


def test_zero3_step_two_streams_replay():
    """The whole ZeRO-3 step (per unit: forward gather, backward gather, reduce-scatter + update),
    gathers on a side stream, captured and replayed."""
    n_d, d, ffn, vocab, n_layers = 4, 512, 1408, 2000, 3
    shapes, units = [(vocab, d)], [n_layers]
    for layer in range(n_layers):
        ls = [(d,), (d, d), (d, d), (d, d), (d, d), (d,), (ffn, d), (ffn, d), (d, ffn)]
        shapes += ls
        units += [layer] * len(ls)
    shapes += [(d,), (vocab, d)]
    units += [n_layers, n_layers]
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, pads = plan.padded, plan.pad_ranges()
    U = plan.n_units
    biggest = max(plan.unit(u)["padded"] for u in range(U))
    master0 = synth.master_init(P, pads, seed=74, device=DEV)
    ugrads = []
    for u in range(U):
        ud = plan.unit(u)
        upads = [(ud["numel"], ud["padded"])] if ud["padded"] > ud["numel"] else []
        ugrads.append(synth.rank_grads(n_d, ud["padded"], upads, seed=75 + u, step=1, sigma=5e-4, device=DEV)[0])

    def make_state():
        return {"shards": master0.to(BF16), "master": master0.clone(), "m": torch.zeros_like(master0),
                "v": torch.zeros_like(master0), "pool": [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(2)],
                "side": torch.cuda.Stream()}

    def body(st, s):
        zs.zs_zero3_step(plan, st["shards"], st["master"], st["m"], st["v"], ugrads, st["pool"], True, HP, 1,
                         main_stream=s, side_stream=st["side"])

    a, b = _run_both(make_state, body)
    for st in (a, b):
        del st["side"]
        st["pool"] = [x for slot in st["pool"] for x in slot]
    _assert_same(a, b)


def test_naive_dp_and_fsdp2_conversions_replay():
    """The naive-DP step (staged) and the per-group FSDP2 chunk-cat / copy-out calls of a plan,
    captured and replayed."""
    n_d = 8
    plan = zs.Plan([(1_200_001,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=76, step=1, sigma=1e-3, device=DEV)[0]
    master0 = synth.master_init(P, pads, seed=77, device=DEV)
    shapes = [(1000, 1024), (1024,), (3000, 512), (7,)]
    units = [0, 0, 1, 1]
    p2 = zs.Plan(shapes, n_d, stage=2, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    params = [torch.empty(sh, dtype=BF16, device=DEV).normal_(0, 1e-3) for sh in shapes]
    members = [[k for k in range(len(shapes)) if units[k] == u] for u in range(p2.n_units)]

    def make_state():
        return {"master": [master0.clone() for _ in range(n_d)], "m": [torch.zeros_like(master0) for _ in range(n_d)],
                "v": [torch.zeros_like(master0) for _ in range(n_d)], "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0],
                "flat": torch.zeros(p2.padded, dtype=BF16, device=DEV),
                "back": [torch.zeros(sh, dtype=BF16, device=DEV) for sh in shapes]}

    def body(st, s):
        zs.zs_dp_step(plan, grads, st["master"], st["m"], st["v"], st["reps"], HP, 1, stream=s)
        for u in range(p2.n_units):
            ud = p2.unit(u)
            view = st["flat"][ud["base"]:ud["base"] + ud["padded"]]
            zs.zs_fsdp2_chunk_cat(p2, u, [params[k] for k in members[u]], view, stream=s)
            zs.zs_fsdp2_copy_out(p2, u, view, [st["back"][k] for k in members[u]], stream=s)

    a, b = _run_both(make_state, body)
    _assert_same(a, b)
    for k in range(len(shapes)):
        assert torch.equal(a["back"][k], params[k])


def test_dependent_launch_on_and_off_agree():
    """A chain of back-to-back launches in which each reads what the previous wrote (accumulations,
    bucket-by-bucket fused steps, the in-place all-reduce of their replicas, a naive-DP step on the
    result, a gather from the shards), run with programmatic dependent launch on and off: every
    buffer ends bit-identical."""
    n_d = 8
    plan = zs.Plan([(2_100_003,)], n_d, stage=2, bucket_bytes=1 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    micro = [synth.rank_grads(n_d, P, pads, seed=80, step=j + 1, sigma=1e-3, device=DEV)[0] for j in range(4)]
    master0 = synth.master_init(P, pads, seed=81, device=DEV)
    dp = zs.Plan([(2_100_003,)], n_d, stage=0)
    assert dp.padded == P

    def run(enable):
        zs.zs_set_dependent_launch(enable)
        try:
            st = {"acc": synth.rank_buffers(n_d, P, BF16, DEV)[0], "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0],
                  "master": master0.clone(), "m": torch.zeros_like(master0), "v": torch.zeros_like(master0),
                  "dm": [master0.clone() for _ in range(n_d)], "dmm": [torch.zeros_like(master0) for _ in range(n_d)],
                  "dv": [torch.zeros_like(master0) for _ in range(n_d)], "out": synth.rank_buffers(n_d, P, BF16, DEV)[0]}
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for t in (1, 2):
                    for j in range(4):
                        zs.zs_accumulate_grad(plan, st["acc"], micro[j], 0.25, j == 0, stream=s)
                    zs.zs_fused_step_buckets(plan, list(reversed(range(plan.n_buckets))), st["acc"], st["master"],
                                             st["m"], st["v"], st["reps"], HP, t, launch_mode=zs.ZS_BUCKETS_PER_BUCKET,
                                             stream=s)
                    zs.zs_all_reduce_mean(dp, -1, st["reps"], stream=s)
                    zs.zs_dp_step(dp, st["reps"], st["dm"], st["dmm"], st["dv"], st["out"], HP, t, stream=s)
                    zs.zs_all_gather(plan, [st["out"][0]], zs.ZS_SHARDED, st["acc"], stream=s)
            torch.cuda.synchronize()
            assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
            return st
        finally:
            zs.zs_set_dependent_launch(True)

    _assert_same(run(False), run(True))


def test_overlapping_walks_repeat_the_serialised_result():
    """Race check of the overlapping launches: the bucket-by-bucket step over 128 buckets of
    1 MiB (every later launch starts before its predecessor ends), on one stream and on two, and the
    whole-range step (one dynamic-order launch), repeated 20 times each from the same state, must
    equal bit for bit the same step run with programmatic dependent launch off (every launch waiting
    for the previous one)."""
    n_d = 8
    plan = zs.Plan([(1 << 26,)], n_d, stage=2, bucket_bytes=1 << 20)
    assert plan.n_buckets == 128
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=90, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)[0]
    master0 = synth.master_init(P, pads, seed=91, device=DEV)
    m0 = torch.rand_like(master0) * 1e-3                 # moments going in are not zero
    v0 = torch.rand_like(master0) * 1e-6
    order = list(reversed(range(plan.n_buckets)))
    side = torch.cuda.Stream()

    def fresh():
        return [master0.clone(), m0.clone(), v0.clone()], synth.rank_buffers(n_d, P, BF16, DEV)[0]

    def run(mode, st, reps):
        if mode == "whole":
            zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *st, reps, HP, 3)
        else:
            zs.zs_fused_step_buckets(plan, order, grads, *st, reps, HP, 3, launch_mode=zs.ZS_BUCKETS_PER_BUCKET,
                                     side_stream=side if mode == "two_streams" else None)

    zs.zs_set_dependent_launch(False)
    try:
        ref_st, ref_reps = fresh()
        run("per_bucket", ref_st, ref_reps)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_dependent_launch(True)
    zs.zs_device_status(clear=True)
    for mode in ("per_bucket", "two_streams", "whole"):
        for k in range(20):
            st, reps = fresh()
            run(mode, st, reps)
            torch.cuda.synchronize()
            assert all(torch.equal(x, y) for x, y in zip(st, ref_st)), "%s run %d: state differs" % (mode, k)
            assert all(torch.equal(x, y) for x, y in zip(reps, ref_reps)), "%s run %d: replicas differ" % (mode, k)
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
