"""The fused step over one long range in one dynamic-order launch (GPU).

A broadcast fused step over one range of at least 2^24 elements (the whole flat space, or touching
buckets merged) runs as one persistent launch whose CTAs take their tiles from a counter pair in
module memory: the tile counter hands out tiles front to back, the last CTA to finish sets both
counters back to zero, and launches draw the pairs in turn (1024 of them), so launches in flight on
several streams use different pairs.  These tests check that path against the oracle and the
register-streaming kernel, with ragged ends, on two concurrent streams, after the pairs have all
been used (the counters came back to zero), from a CUDA graph, and inside guard zones.  The
naive-DP all-reduce and step, the update alone, and the unfused reduce-scatter and all-gather take
the same order on such buffers.
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


def _setup(n_d, numel, seed):
    plan = zs.Plan([(numel,)], n_d, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=seed, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)[0]
    master = synth.master_init(P, pads, seed=seed + 1, device=DEV)
    state = [master, torch.rand_like(master) * 1e-3, torch.rand_like(master) * 1e-6]
    return plan, P, grads, state


def _fresh(state, n_d, P):
    return [x.clone() for x in state], synth.rank_buffers(n_d, P, BF16, DEV)[0]


@pytest.mark.parametrize("n_d,numel", [(8, (1 << 24) + 13), (2, (1 << 24) + (1 << 20) + 1), (32, (1 << 24) + 5)])
def test_dynamic_order_step_matches_the_oracle_and_streaming(n_d, numel):
    """Every element of master, m, v and every replica: the one-launch dynamic-order step (with the
    streaming kernel for the ragged end) equals the oracle's ZeRO step and the register-streaming
    kernel, bit for bit."""
    plan, P, grads, state = _setup(n_d, numel, 70)
    ref = layout.make_plan([(numel,)], n_d)
    st, reps = _fresh(state, n_d, P)
    zs.zs_device_status(clear=True)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *st, reps, HP, 3)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        st2, reps2 = _fresh(state, n_d, P)
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *st2, reps2, HP, 3)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    assert all(torch.equal(x, y) for x, y in zip(st, st2))
    assert all(torch.equal(x, y) for x, y in zip(reps, reps2))
    g_np = [H.to_np_bf16(g) for g in grads]
    om, omm, ov = (H.reshard(ref, H.to_np_f32(x)) for x in state)
    want_reps, om, omm, ov = steps.zero_step(ref, g_np, om, omm, ov, HP, 3)
    H.check_f32(H.to_np_f32(st[0]), H.unshard(ref, om), "master")
    H.check_f32(H.to_np_f32(st[1]), H.unshard(ref, omm), "m")
    H.check_f32(H.to_np_f32(st[2]), H.unshard(ref, ov), "v")
    for q in range(n_d):
        H.check_bf16(H.to_np_bf16(reps[q]), want_reps[q], "replica %d" % q)


def test_concurrent_launches_on_two_streams_and_every_counter_pair():
    """Two dynamic-order steps on disjoint buffers run at once on two streams, 600 steps each (1,200
    launches: every counter pair is drawn at least once, and the first 176 twice, so they must have
    come back to zero), and the final states equal the same 600 steps run by the register-streaming
    kernel, bit for bit."""
    n_d, numel = 8, (1 << 24) + 8
    runs = [_setup(n_d, numel, 80 + 10 * k) for k in range(2)]
    plan, P = runs[0][0], runs[0][1]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    for (_, _, grads, state), s in zip(runs, streams):
        outs.append(_fresh(state, n_d, P))
    torch.cuda.synchronize()
    zs.zs_device_status(clear=True)
    for t in range(1, 601):
        for k in range(2):
            st, reps = outs[k]
            zs.zs_fused_step(plan, -1, runs[k][2], zs.ZS_RANK_FULL, *st, reps, HP, t, stream=streams[k])
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        for k in range(2):
            st, reps = outs[k]
            want = _fresh(runs[k][3], n_d, P)
            for t in range(1, 601):
                zs.zs_fused_step(plan, -1, runs[k][2], zs.ZS_RANK_FULL, *want[0], want[1], HP, t)
            torch.cuda.synchronize()
            assert all(torch.equal(x, y) for x, y in zip(st, want[0])), "stream %d: state differs" % k
            assert all(torch.equal(x, y) for x, y in zip(reps, want[1])), "stream %d: replicas differ" % k
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


def test_dynamic_order_step_replays_from_a_graph():
    n_d, numel = 4, (1 << 24) + 3
    plan, P, grads, state = _setup(n_d, numel, 90)
    direct, graphed = _fresh(state, n_d, P), _fresh(state, n_d, P)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *direct[0], direct[1], HP, 2, stream=s)
    torch.cuda.synchronize()
    g, cs = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(g, stream=cs):
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *graphed[0], graphed[1], HP, 2, stream=cs)
    torch.cuda.synchronize()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    assert all(torch.equal(x, y) for x, y in zip(direct[0], graphed[0]))
    assert all(torch.equal(x, y) for x, y in zip(direct[1], graphed[1]))


def test_dynamic_order_step_stays_inside_its_buffers():
    """Sentinel bytes around every buffer of the dynamic-order launches (the fused step, the naive-DP
    all-reduce and step, the update alone) survive them."""
    n_d, numel = 8, (1 << 24) + 21
    plan = zs.Plan([(numel,)], n_d, stage=2)
    P = plan.padded
    guard, fill = 2048, 0x5A
    raws = []

    def mk(n, dtype):
        esz = torch.tensor([], dtype=dtype).element_size()
        raw = torch.full(((n + 2 * guard) * esz,), fill, dtype=torch.uint8, device=DEV)
        raws.append((raw, guard * esz))
        t = raw.view(dtype)[guard:guard + n]
        t.zero_()
        return t

    grads = [mk(P, BF16) for _ in range(n_d)]
    for g in grads:
        g.normal_(0, 1e-3)
    reps = [mk(P, BF16) for _ in range(n_d)]
    master, m, v = mk(P, torch.float32), mk(P, torch.float32), mk(P, torch.float32)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    dm = [mk(P, torch.float32) for _ in range(n_d)]
    dmm = [mk(P, torch.float32) for _ in range(n_d)]
    dv = [mk(P, torch.float32) for _ in range(n_d)]
    zs.zs_dp_step(plan, grads, dm, dmm, dv, reps, HP, 1)
    zs.zs_all_reduce_mean(plan, -1, grads)
    zs.zs_adamw_shard_step(plan, -1, [grads[0]], zs.ZS_SHARDED, master, m, v, [reps[0]], zs.ZS_SHARDED, HP, 2)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for raw, gb in raws:
        head, tail = raw[:gb].cpu().numpy(), raw[raw.numel() - gb:].cpu().numpy()
        assert np.all(head == fill) and np.all(tail == fill)


@pytest.mark.parametrize("n_d,numel", [(8, (1 << 24) + 13), (2, (1 << 24) + (1 << 20) + 1), (32, (1 << 24) + 5)])
def test_dynamic_order_all_reduce_and_dp_step_match_the_oracle(n_d, numel):
    """Naive DP on a buffer of 2^24 elements and more: the in-place all-reduce with averaging (N_d = 4 to
    32) and the replicated step (N_d = 2 to 16) each run as one dynamic-order launch, the ragged end
    streamed; at N_d = 2 the all-reduce is walked and at N_d = 32 the step is one statically ordered
    launch.  Rank 0's mean, state and replica equal the oracle's bit for bit, and every other rank's
    equal rank 0's."""
    plan = zs.Plan([(numel,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=95, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)[0]
    g_np = [H.to_np_bf16(g) for g in grads]
    zs.zs_device_status(clear=True)

    reduced = [g.clone() for g in grads]
    zs.zs_all_reduce_mean(plan, -1, reduced)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    H.check_bf16(H.to_np_bf16(reduced[0]), steps.reduce_mean(g_np), "all-reduce rank 0")
    assert all(torch.equal(r, reduced[0]) for r in reduced[1:]), "the ranks' means differ"
    del reduced

    master0 = synth.master_init(P, pads, seed=96, device=DEV)
    m0, v0 = torch.rand_like(master0) * 1e-3, torch.rand_like(master0) * 1e-6
    dm = [master0.clone() for _ in range(n_d)]
    dmm = [m0.clone() for _ in range(n_d)]
    dv = [v0.clone() for _ in range(n_d)]
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    zs.zs_dp_step(plan, grads, dm, dmm, dv, reps, HP, 3)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    want_reps, om, omm, ov = steps.dp_step(g_np, H.to_np_f32(master0), H.to_np_f32(m0), H.to_np_f32(v0), HP, 3)
    H.check_f32(H.to_np_f32(dm[0]), om, "master rank 0")
    H.check_f32(H.to_np_f32(dmm[0]), omm, "m rank 0")
    H.check_f32(H.to_np_f32(dv[0]), ov, "v rank 0")
    H.check_bf16(H.to_np_bf16(reps[0]), want_reps[0], "replica 0")
    for q in range(1, n_d):
        assert torch.equal(dm[q], dm[0]) and torch.equal(dmm[q], dmm[0]) and torch.equal(dv[q], dv[0]), q
        assert torch.equal(reps[q], reps[0]), q


def test_different_dynamic_order_kernels_share_the_counter_pairs():
    """Dynamic-order launches of different kernels draw from the same 1024 counter pairs: the naive-DP
    step on one stream, the in-place all-reduce and the update alone on another, 400 rounds each
    (1,200 launches, so every pair is drawn by more than one kernel), equal the same rounds run by the
    register-streaming kernels one stream at a time, bit for bit."""
    n_d, numel = 4, (1 << 24) + 3
    plan = zs.Plan([(numel,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=97, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)[0]
    master0 = synth.master_init(P, pads, seed=98, device=DEV)

    def fresh():
        dp = ([master0.clone() for _ in range(n_d)], [torch.zeros_like(master0) for _ in range(n_d)],
              [torch.zeros_like(master0) for _ in range(n_d)], synth.rank_buffers(n_d, P, BF16, DEV)[0])
        ar = [g.clone() for g in grads]
        up = (master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0),
              torch.zeros(P, dtype=BF16, device=DEV))
        return dp, ar, up

    def run(bufs, streams):
        dp, ar, up = bufs
        for t in range(1, 401):
            zs.zs_dp_step(plan, grads, *dp, HP, t, stream=streams[0])
            zs.zs_all_reduce_mean(plan, -1, ar, stream=streams[1])
            zs.zs_adamw_shard_step(plan, -1, [ar[0]], zs.ZS_SHARDED, *up[:3], [up[3]], zs.ZS_SHARDED, HP, t,
                                   stream=streams[1])
        torch.cuda.synchronize()

    got = fresh()
    zs.zs_device_status(clear=True)
    run(got, [torch.cuda.Stream(), torch.cuda.Stream()])
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    want = fresh()
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        s = torch.cuda.current_stream()
        run(want, [s, s])
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    for a, b in zip(got[0], want[0]):
        assert all(torch.equal(x, y) for x, y in zip(a, b)), "naive-DP step differs"
    assert all(torch.equal(x, y) for x, y in zip(got[1], want[1])), "all-reduce differs"
    assert all(torch.equal(x, y) for x, y in zip(got[2], want[2])), "update differs"


@pytest.mark.parametrize("n_d,numel", [(8, (1 << 24) + 13), (2, (1 << 24) + (1 << 20) + 1), (32, (1 << 24) + 5)])
def test_dynamic_order_reduce_scatter_and_all_gather_match_the_oracle(n_d, numel):
    """The unfused ZeRO-2 reduce-scatter with averaging into the sharded array and the all-gather from
    it, each one dynamic-order launch over a unit of 2^24 elements and more (the ragged end
    streamed): the reduced gradient equals the oracle's mean bit for bit, every replica equals the
    sharded source."""
    plan = zs.Plan([(numel,)], n_d, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=99, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)[0]
    ghat = torch.zeros(P, dtype=BF16, device=DEV)
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    zs.zs_device_status(clear=True)
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
    zs.zs_all_gather(plan, [ghat], zs.ZS_SHARDED, reps)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    H.check_bf16(H.to_np_bf16(ghat), steps.reduce_mean([H.to_np_bf16(g) for g in grads]), "reduced gradient")
    for q in range(n_d):
        assert torch.equal(reps[q], ghat), "replica %d" % q
