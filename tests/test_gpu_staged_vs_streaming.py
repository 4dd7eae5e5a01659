"""Every staged (bulk-copy) kernel against its register-streaming twin, every element compared.

The staged kernels keep a ring of shared-memory stages per CTA and write master, m and v back to
the addresses they read them from; the streaming kernels touch each element from one thread.  On
buffers of tens of millions of elements (tens of thousands of tiles per launch, many tiles per
CTA and stage), two steps of each staged kernel must give bit-identical results to the streaming
kernel - not just on sampled chunks.  This is the guard against ordering faults in the rings,
which show up as a few wrong elements in 10^5 rather than as wrong sampled chunks.
"""

import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import synth

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


def _run_both(make_state, body):
    out = {}
    for variant in (zs.ZS_FUSED_LDG, zs.ZS_FUSED_TMA):
        st = make_state()
        torch.cuda.synchronize()
        zs.zs_set_fused_variant(variant)
        try:
            body(st)
            torch.cuda.synchronize()
        finally:
            zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
        out[variant] = st
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    a, b = out[zs.ZS_FUSED_LDG], out[zs.ZS_FUSED_TMA]
    for k in a:
        xs, ys = (a[k], b[k]) if isinstance(a[k], list) else ([a[k]], [b[k]])
        for i, (x, y) in enumerate(zip(xs, ys)):
            bad = int((x != y).sum())
            assert bad == 0, "%s[%d]: %d elements differ between the staged and streaming kernels" % (k, i, bad)


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_fused_step(n_d):
    plan = zs.Plan([((1 << 25) + 7,)], n_d, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    m0 = synth.master_init(P, pads, seed=90, device=DEV)
    grads = [synth.rank_grads(n_d, P, pads, seed=91, step=t, sigma=1e-3, device=DEV)[0] for t in (1, 2)]

    def make_state():
        return {"master": m0.clone(), "m": torch.zeros_like(m0), "v": torch.zeros_like(m0),
                "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0]}

    def body(st):
        for t in (1, 2):
            zs.zs_fused_step(plan, -1, grads[t - 1], zs.ZS_RANK_FULL, st["master"], st["m"], st["v"], st["reps"],
                             HP, t)

    _run_both(make_state, body)


@pytest.mark.parametrize("n_d", [1, 2, 4, 8, 16, 32])
def test_zero3_reduce_scatter_update(n_d):
    plan = zs.Plan([((1 << 25) + 5,)], n_d, stage=3, unit_of_param=[0])
    P, pads = plan.padded, plan.pad_ranges()
    m0 = synth.master_init(P, pads, seed=92, device=DEV)
    grads = [synth.rank_grads(n_d, P, pads, seed=93, step=t, sigma=1e-3, device=DEV)[0] for t in (1, 2)]

    def make_state():
        return {"master": m0.clone(), "m": torch.zeros_like(m0), "v": torch.zeros_like(m0),
                "shards": torch.zeros(P, dtype=BF16, device=DEV)}

    def body(st):
        for t in (1, 2):
            zs.zs_zero3_rs_step_unit(plan, 0, grads[t - 1], st["master"], st["m"], st["v"], st["shards"], HP, t)

    _run_both(make_state, body)


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_naive_dp_step(n_d):
    plan = zs.Plan([((1 << 23) + 3,)], n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    m0 = synth.master_init(P, pads, seed=94, device=DEV)
    grads = [synth.rank_grads(n_d, P, pads, seed=95, step=t, sigma=1e-3, device=DEV)[0] for t in (1, 2)]

    def make_state():
        return {"master": [m0.clone() for _ in range(n_d)], "m": [torch.zeros_like(m0) for _ in range(n_d)],
                "v": [torch.zeros_like(m0) for _ in range(n_d)], "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0]}

    def body(st):
        for t in (1, 2):
            zs.zs_dp_step(plan, grads[t - 1], st["master"], st["m"], st["v"], st["reps"], HP, t)

    _run_both(make_state, body)


def test_bucket_list_and_sharded_adamw():
    """The list kernel (every other 1 MiB bucket: 33 scattered bodies) and the staged AdamW on
    sharded buffers (the single-output kernel with one rank)."""
    n_d = 8
    plan = zs.Plan([((1 << 25) + 7,)], n_d, stage=2, bucket_bytes=1 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    m0 = synth.master_init(P, pads, seed=96, device=DEV)
    grads = synth.rank_grads(n_d, P, pads, seed=97, step=1, sigma=1e-3, device=DEV)[0]
    ghat = synth.rank_grads(1, P, pads, seed=98, step=1, sigma=1e-3, device=DEV)[0][0]
    even = list(range(0, plan.n_buckets, 2))

    def make_state():
        return {"master": m0.clone(), "m": torch.zeros_like(m0), "v": torch.zeros_like(m0),
                "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0], "par": torch.zeros(P, dtype=BF16, device=DEV)}

    def body(st):
        for t in (1, 2):
            zs.zs_fused_step_buckets(plan, even, grads, st["master"], st["m"], st["v"], st["reps"], HP, t)
        zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, st["master"], st["m"], st["v"], [st["par"]],
                               zs.ZS_SHARDED, HP, 3)

    _run_both(make_state, body)


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_reduce_scatter_into_one_array(n_d):
    """The staged reduce-scatter-mean (every rank's tile staged, the mean streamed to one array)."""
    plan = zs.Plan([((1 << 25) + 7,)], n_d, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    grads = synth.rank_grads(n_d, P, pads, seed=99, step=1, sigma=1e-3, device=DEV)[0]

    def make_state():
        return {"out": torch.zeros(P, dtype=BF16, device=DEV)}

    def body(st):
        zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, [st["out"]], zs.ZS_SHARDED)

    _run_both(make_state, body)


@pytest.mark.parametrize("n_d", [2, 8, 16, 64])
def test_bulk_store_gather_copies_every_element(n_d):
    """The bulk-store gather (one source, N_d destinations): every destination equals the source on
    every element (the gather has no streaming twin behind the variant switch: it is a copy)."""
    plan = zs.Plan([((1 << 25) + 9,)], n_d, stage=2)
    P = plan.padded
    src = torch.empty(P, dtype=BF16, device=DEV).normal_(0, 1e-2)
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    torch.cuda.synchronize()
    zs.zs_all_gather(plan, [src], zs.ZS_SHARDED, reps)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for q in range(n_d):
        assert torch.equal(reps[q], src), "replica %d differs from the source" % q


def test_bucket_walk_large_scattered_buckets():
    """Every other 64 MiB bucket of a 2^27+7-element buffer: the two large bodies take one
    single-range launch each, the short last bucket the list kernel; against the streaming kernel."""
    n_d = 8
    plan = zs.Plan([((1 << 27) + 7,)], n_d, stage=2, bucket_bytes=64 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    assert plan.n_buckets == 5
    m0 = synth.master_init(P, pads, seed=100, device=DEV)
    grads = synth.rank_grads(n_d, P, pads, seed=101, step=1, sigma=1e-3, device=DEV)[0]

    def make_state():
        return {"master": m0.clone(), "m": torch.zeros_like(m0), "v": torch.zeros_like(m0),
                "reps": synth.rank_buffers(n_d, P, BF16, DEV)[0]}

    def body(st):
        for t in (1, 2):
            zs.zs_fused_step_buckets(plan, [4, 2, 0], grads, st["master"], st["m"], st["v"], st["reps"], HP, t)

    _run_both(make_state, body)
