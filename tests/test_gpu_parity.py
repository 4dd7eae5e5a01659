"""GPU parity: every device entry point of the C ABI against the CPU oracle.

Small cases run the oracle on the whole buffer; the full-size model shapes
(in the launch configuration the benchmark times) compare sampled chunks of
the flat space, which is exact because every step is element-wise.
"""

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth
from oracle import layout, numerics, steps

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


def _plans(shapes, n_d, units=None, bucket_bytes=0, stage=1):
    plan = zs.Plan(shapes, n_d, stage=stage, bucket_bytes=bucket_bytes, unit_of_param=units)
    ref = layout.make_plan(shapes, n_d, unit_of_param=units, bucket_bytes=bucket_bytes if bucket_bytes > 0 else None)
    return plan, ref


class State:
    """fp32 master/m/v (ZS_SHARDED) on the device."""

    def __init__(self, master):
        self.master = master.clone()
        self.m = torch.zeros_like(master)
        self.v = torch.zeros_like(master)

    def args(self):
        return self.master, self.m, self.v


def _oracle_state(ref, master_np):
    n_d = ref.n_d
    return (H.reshard(ref, master_np), [np.zeros(ref.shard_total, np.float32) for _ in range(n_d)],
            [np.zeros(ref.shard_total, np.float32) for _ in range(n_d)])


def _check_state(ref, st, om, omm, ov, what):
    H.check_f32(H.to_np_f32(st.master), H.unshard(ref, om), what + " master")
    H.check_f32(H.to_np_f32(st.m), H.unshard(ref, omm), what + " m")
    H.check_f32(H.to_np_f32(st.v), H.unshard(ref, ov), what + " v")


# ---------------------------------------------------------------- the tiny MLP, every path, 10 steps

@pytest.mark.parametrize("bucket_bytes", [0, 4096, 1000])
def test_mlp_tiny_zero1_zero2_fused_ten_steps(bucket_bytes):
    """W1 256x512, b1, W2 512x256, b2 on N_d = 4 ranks, 10 steps: the fused step,
    ZeRO-1 (in-place reduce-scatter, AdamW, in-place all-gather) and ZeRO-2
    (bucket-wise reduce-scatter from per-bucket staging into a sharded reduced
    gradient, AdamW, all-gather) each against the oracle's ZeRO step."""
    shapes, _ = synth.workload_params("mlp-tiny")
    n_d = 4
    plan, ref = _plans(shapes, n_d, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=0, device=DEV)
    sts = {k: State(master0) for k in ("fused", "zero1", "zero2")}
    reps = {k: synth.rank_buffers(n_d, P, BF16, DEV)[0] for k in sts}
    om, omm, ov = _oracle_state(ref, H.to_np_f32(master0))
    for t in range(1, 11):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=0, step=t, sigma=1e-3, device=DEV)
        g_np = [H.to_np_bf16(g) for g in grads]
        ref_reps, om, omm, ov = steps.zero_step(ref, g_np, om, omm, ov, HP, t)
        reduced_ref = steps.reduce_scatter_mean(ref, g_np)

        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *sts["fused"].args(), reps["fused"], HP, t)

        g1 = [g.clone() for g in grads]
        zs.zs_reduce_scatter_mean(plan, -1, g1, zs.ZS_RANK_FULL, g1, zs.ZS_RANK_FULL)
        zs.zs_adamw_shard_step(plan, -1, g1, zs.ZS_RANK_FULL, *sts["zero1"].args(), reps["zero1"],
                               zs.ZS_RANK_FULL, HP, t)
        zs.zs_all_gather(plan, reps["zero1"], zs.ZS_RANK_FULL, reps["zero1"])

        ghat = torch.zeros(P, dtype=BF16, device=DEV)
        for b in reversed(range(plan.n_buckets)):          # backward makes buckets ready last-to-first
            _, lo, hi = plan.bucket(b)
            staging = [g[lo:hi].clone() for g in grads]
            zs.zs_reduce_scatter_mean(plan, b, staging, zs.ZS_RANK_BUCKET, [ghat], zs.ZS_SHARDED)
            del staging                                     # the bucket's non-owned gradients are freed
        shards = torch.zeros(P, dtype=BF16, device=DEV)
        zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, *sts["zero2"].args(), [shards],
                               zs.ZS_SHARDED, HP, t)
        zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, reps["zero2"])
        torch.cuda.synchronize()

        for k in sts:
            _check_state(ref, sts[k], om, omm, ov, "%s t=%d" % (k, t))
            for q in range(n_d):
                H.check_bf16(H.to_np_bf16(reps[k][q]), ref_reps[q], "%s replica %d t=%d" % (k, q, t))
        # ZeRO-1 keeps the full gradient buffer: owned slice reduced, the rest untouched local gradients
        for r in range(n_d):
            lo, hi = layout.shard_range(ref, 0, r)
            g1r = H.to_np_bf16(g1[r])
            H.check_bf16(g1r[lo:hi], reduced_ref[r], "zero1 reduced slice r=%d" % r)
            assert np.array_equal(g1r[:lo], g_np[r][:lo]) and np.array_equal(g1r[hi:], g_np[r][hi:])
        H.check_bf16(H.to_np_bf16(ghat), H.unshard(ref, reduced_ref), "zero2 reduced gradient t=%d" % t)


# ---------------------------------------------------------------- gradient accumulation

@pytest.mark.parametrize("n_d", [1, 3, 8])
def test_accumulation_four_microbatches(n_d):
    shapes = [(1000, 3), (77,), (5, 5, 5)]
    plan, ref = _plans(shapes, n_d)
    P, pads = plan.padded, plan.pad_ranges()
    acc, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    ref_acc = [None] * n_d
    for j in range(4):
        micro, _ = synth.rank_grads(n_d, P, pads, seed=11, step=j, sigma=1e-3, device=DEV)
        zs.zs_accumulate_grad(plan, acc, micro, 0.25, first=(j == 0))
        for q in range(n_d):
            ref_acc[q] = steps.accumulate(ref_acc[q], H.to_np_bf16(micro[q]), 0.25, first=(j == 0))
    torch.cuda.synchronize()
    for q in range(n_d):
        H.check_bf16(H.to_np_bf16(acc[q]), ref_acc[q], "acc rank %d" % q)


def test_accumulation_in_place_and_equal_microbatches():
    """acc may be the micro buffer itself; four equal micro-batches give back the gradient."""
    plan, _ = _plans([(4099,)], 2)
    P, pads = plan.padded, plan.pad_ranges()
    g, _ = synth.rank_grads(2, P, pads, seed=5, step=0, sigma=1e-3, device=DEV)
    acc, _ = synth.rank_buffers(2, P, BF16, DEV)
    for j in range(4):
        zs.zs_accumulate_grad(plan, acc, g, 0.25, first=(j == 0))
    same = [x.clone() for x in g]
    zs.zs_accumulate_grad(plan, same, same, 1.0, first=True)
    torch.cuda.synchronize()
    for q in range(2):
        assert torch.equal(acc[q], g[q])
        assert torch.equal(same[q], g[q])


@pytest.mark.parametrize("n_d,numel", [(2, 3 * (1 << 22) + 13), (8, (1 << 22) + (1 << 20) + 3), (3, (1 << 20) + 8)])
@pytest.mark.parametrize("mode", ["auto", "ldg"])
def test_accumulation_large_buffers_match_oracle(n_d, numel, mode):
    """Accumulation over buffers of a million elements and more (3 x 2^22 + 13 elements, padded to
    3 x 2^22 + 14: a ragged end of 6 elements past the 16-byte vectors), four micro-batches at scale
    1/4 with outliers, then in place (the micro-batch buffer as its own accumulator): equal to the
    oracle bit for bit, with the default and the forced register-streaming (ldg) fused variant."""
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG if mode == "ldg" else zs.ZS_FUSED_AUTO)
    try:
        plan, _ = _plans([(numel,)], n_d)
        P, pads = plan.padded, plan.pad_ranges()
        acc, _ = synth.rank_buffers(n_d, P, BF16, DEV)
        ref_acc = [None] * n_d
        last = None
        for j in range(4):
            micro, _ = synth.rank_grads(n_d, P, pads, seed=17, step=j, sigma=1e-3, outlier_p=0.001, device=DEV)
            zs.zs_accumulate_grad(plan, acc, micro, 0.25, first=(j == 0))
            for q in range(n_d):
                ref_acc[q] = steps.accumulate(ref_acc[q], H.to_np_bf16(micro[q]), 0.25, first=(j == 0))
            last = micro
        # in place: the micro-batch buffer is its own accumulator
        last_np = [H.to_np_bf16(x) for x in last]
        zs.zs_accumulate_grad(plan, last, last, 0.5, first=False)
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        for q in range(n_d):
            H.check_bf16(H.to_np_bf16(acc[q]), ref_acc[q], "acc rank %d (%s)" % (q, mode))
            m = last_np[q]
            H.check_bf16(H.to_np_bf16(last[q]), steps.accumulate(m, m, 0.5, first=False), "in place rank %d" % q)
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


# ---------------------------------------------------------------- ZeRO-3 per unit

def _tiny_llama(n_layers=3, d=64, ffn=176, vocab=100):
    shapes, units = [(vocab, d)], [n_layers]
    for layer in range(n_layers):
        ls = [(d,), (d, d), (d, d), (d, d), (d, d), (d,), (ffn, d), (ffn, d), (d, ffn)]
        shapes += ls
        units += [layer] * len(ls)
    shapes += [(d,), (vocab, d)]
    units += [n_layers, n_layers]
    return shapes, units


@pytest.mark.parametrize("n_d", [16, 5, 2])
def test_zero3_units_two_steps(n_d):
    """Per unit: gather for forward, gather again for backward (both equal the
    shards before the update), reduce-scatter + AdamW on the shard; no gather after."""
    shapes, units = _tiny_llama()
    plan, ref = _plans(shapes, n_d, units=units, stage=3)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=3, device=DEV)
    st = State(master0)
    shards = torch.empty(P, dtype=BF16, device=DEV)
    shards.copy_(master0.to(BF16))       # the initial bf16 shards: the cast of the fp32 masters
    om, omm, ov = _oracle_state(ref, H.to_np_f32(master0))
    osh = H.reshard(ref, H.to_np_bf16(shards))
    for t in (1, 2):
        for u in range(plan.n_units):                                   # forward: layer order
            ud = plan.unit(u)
            full, _ = synth.rank_buffers(n_d, ud["padded"], BF16, DEV)
            zs.zs_zero3_gather_unit(plan, u, shards, full)
            want = steps.all_gather_unit(ref, u, osh)
            torch.cuda.synchronize()
            for q in range(n_d):
                H.check_bf16(H.to_np_bf16(full[q]), want[q], "fwd gather u=%d q=%d" % (u, q))
        for u in reversed(range(plan.n_units)):                         # backward: reverse order
            ud = plan.unit(u)
            full, _ = synth.rank_buffers(n_d, ud["padded"], BF16, DEV)
            zs.zs_zero3_gather_unit(plan, u, shards, full)
            upads = [(ud["numel"], ud["padded"])] if ud["padded"] > ud["numel"] else []
            grads, _ = synth.rank_grads(n_d, ud["padded"], upads, seed=30 + u, step=t, sigma=5e-4, device=DEV)
            zs.zs_zero3_rs_step_unit(plan, u, grads, *st.args(), shards, HP, t)
            fwd, bwd, osh, om, omm, ov = steps.zero3_unit_step(ref, u, osh, [H.to_np_bf16(g) for g in grads],
                                                               om, omm, ov, HP, t)
            torch.cuda.synchronize()
            for q in range(n_d):
                H.check_bf16(H.to_np_bf16(full[q]), bwd[q], "bwd gather u=%d q=%d" % (u, q))
        _check_state(ref, st, om, omm, ov, "zero3 t=%d" % t)
        H.check_bf16(H.to_np_bf16(shards), H.unshard(ref, osh), "zero3 shards t=%d" % t)


# ---------------------------------------------------------------- edge cases

EDGE = [
    # (shapes, n_d, bucket_bytes)
    ([(1,)], 1, 0),                         # one element, one rank
    ([(7,)], 3, 0),                         # padding to 9, non-power-of-two ranks
    ([(3,), (4,)], 8, 2),                   # more ranks than elements, one-element buckets
    ([(65_541,)], 8, 1000),                 # ragged tail, buckets off the 8-element grid
    ([(3 * 65_536 + 13,)], 5, 0),           # odd shard size (owner boundaries off the grid)
    ([(100_003,), (17, 3)], 16, 4096),
    ([(40_000,)], 32, 0),
    ([(9_999,)], 64, 0),                    # the largest rank count
    ([(123_457,)], 6, 2048),
]


@pytest.mark.parametrize("shapes,n_d,bucket_bytes", EDGE)
def test_edge_cases_all_paths(shapes, n_d, bucket_bytes):
    plan, ref = _plans(shapes, n_d, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=7, device=DEV)
    om, omm, ov = _oracle_state(ref, H.to_np_f32(master0))
    st_f, st_u, st_b = State(master0), State(master0), State(master0)
    reps_f = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    reps_u = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    reps_b = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    for t in (1, 2, 3):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=7, step=t, sigma=1e-3, outlier_p=0.01, device=DEV)
        g_np = [H.to_np_bf16(g) for g in grads]
        ref_reps, om, omm, ov = steps.zero_step(ref, g_np, om, omm, ov, HP, t)
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *st_f.args(), reps_f, HP, t)
        # fused, bucket by bucket from staging buffers (ZeRO-2 with the update as each bucket completes)
        for b in reversed(range(plan.n_buckets)):
            _, lo, hi = plan.bucket(b)
            staging = [g[lo:hi].clone() for g in grads]
            zs.zs_fused_step(plan, b, staging, zs.ZS_RANK_BUCKET, *st_b.args(), reps_b, HP, t)
        # unfused ZeRO-1, one rank at a time for the update
        g1 = [g.clone() for g in grads]
        zs.zs_reduce_scatter_mean(plan, -1, g1, zs.ZS_RANK_FULL, g1, zs.ZS_RANK_FULL)
        for r in range(n_d):
            zs.zs_adamw_shard_step(plan, r, g1, zs.ZS_RANK_FULL, *st_u.args(), reps_u, zs.ZS_RANK_FULL, HP, t)
        zs.zs_all_gather(plan, reps_u, zs.ZS_RANK_FULL, reps_u)
        torch.cuda.synchronize()
        for name, st, reps in (("fused", st_f, reps_f), ("bucketed", st_b, reps_b), ("unfused", st_u, reps_u)):
            _check_state(ref, st, om, omm, ov, "%s t=%d" % (name, t))
            for q in range(n_d):
                H.check_bf16(H.to_np_bf16(reps[q]), ref_reps[q], "%s replica %d t=%d" % (name, q, t))
        for lo, hi in pads:                                  # padding stays exactly zero
            assert not st_f.master[lo:hi].any() and not reps_f[0][lo:hi].float().any()


# ---------------------------------------------------------------- guard zones and rejected calls

def _guarded(n_elems, dtype, guard=2048, fill=0x5A):
    raw = torch.full(((n_elems + 2 * guard) * torch.tensor([], dtype=dtype).element_size(),), fill,
                     dtype=torch.uint8, device=DEV)
    t = raw.view(dtype)
    return t[guard:guard + n_elems], raw, guard * t.element_size()


def test_guard_zones_untouched():
    """Sentinel bytes before and after every buffer must survive every call (no
    out-of-bounds writes; compute-sanitizer is not available on this machine)."""
    shapes, n_d, bb = [(5_003,), (11,)], 3, 998
    plan, _ = _plans(shapes, n_d, bucket_bytes=bb)
    P = plan.padded
    bufs = []

    def mk(dtype):
        t, raw, g = _guarded(P, dtype)
        t.zero_()
        bufs.append((raw, g))
        return t

    grads = [mk(BF16) for _ in range(n_d)]
    for g in grads:
        g.normal_(0, 1e-3)
    reps = [mk(BF16) for _ in range(n_d)]
    master, m, v = mk(torch.float32), mk(torch.float32), mk(torch.float32)
    ghat, shards = mk(BF16), mk(BF16)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
    zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, master, m, v, [shards], zs.ZS_SHARDED, HP, 2)
    zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, reps)
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, grads, zs.ZS_RANK_FULL)
    zs.zs_adamw_shard_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, zs.ZS_RANK_FULL, HP, 3)
    zs.zs_all_gather(plan, reps, zs.ZS_RANK_FULL, reps)
    zs.zs_accumulate_grad(plan, grads, reps, 0.5, first=False)
    for b in range(plan.n_buckets):
        zs.zs_fused_step(plan, b, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 4)
    torch.cuda.synchronize()
    for raw, g in bufs:
        assert bool((raw[:g] == 0x5A).all()) and bool((raw[-g:] == 0x5A).all())


def test_rejected_calls_write_nothing():
    plan, _ = _plans([(4096,)], 4)
    P = plan.padded
    grads, _ = synth.rank_grads(4, P, [], seed=1, step=1, sigma=1e-3, device=DEV)
    reps, _ = synth.rank_buffers(4, P, BF16, DEV)
    master = synth.master_init(P, [], 1, device=DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    before = master.clone()
    misaligned = torch.zeros(P + 8, dtype=BF16, device=DEV)[1:P + 1]
    with pytest.raises(zs.ZsError) as e:
        zs.zs_fused_step(plan, -1, grads[:3] + [misaligned], zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    assert e.value.status == zs.ZS_ERR_INVALID and "aligned" in str(e.value)
    with pytest.raises(zs.ZsError):
        zs.zs_fused_step(plan, -1, grads[:3] + [0], zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)
    with pytest.raises(zs.ZsError):
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 0)
    with pytest.raises(zs.ZsError):
        zs.zs_adamw_shard_step(plan, 4, grads, zs.ZS_RANK_FULL, master, m, v, reps, zs.ZS_RANK_FULL, HP, 1)
    with pytest.raises(zs.ZsError):
        zs.zs_all_gather(plan, grads, zs.ZS_RANK_FULL, reps)          # in place needs src == replicas
    with pytest.raises(ValueError):
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master[:100], m, v, reps, HP, 1)  # too small
    torch.cuda.synchronize()
    assert torch.equal(master, before) and not m.any() and not any(r.float().any() for r in reps)


# ---------------------------------------------------------------- staged (bulk-copy) kernel

@pytest.fixture
def variant():
    yield zs.zs_set_fused_variant
    zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


@pytest.mark.parametrize("n_d,numel,bucket_bytes", [
    (2, 3 * 2048 * 8 + 5, 0), (4, 1_000_003, 0), (8, 262_912, 0), (8, 2_000_001, 1 << 20),
    (16, 700_001, 0), (32, 300_007, 0), (3, 50_001, 0)])
def test_staged_and_streaming_fused_kernels_agree_with_oracle(variant, n_d, numel, bucket_bytes):
    """The bulk-copy staged kernel and the register-streaming kernel give the oracle's
    results bit for bit, for whole-space and per-bucket launches with ragged tails."""
    plan, ref = _plans([(numel,)], n_d, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=8, device=DEV)
    om, omm, ov = _oracle_state(ref, H.to_np_f32(master0))
    states = {v: State(master0) for v in (zs.ZS_FUSED_LDG, zs.ZS_FUSED_TMA)}
    reps = {v: synth.rank_buffers(n_d, P, BF16, DEV)[0] for v in states}
    for t in (1, 2):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=8, step=t, sigma=1e-3, outlier_p=0.001, device=DEV)
        ref_reps, om, omm, ov = steps.zero_step(ref, [H.to_np_bf16(g) for g in grads], om, omm, ov, HP, t)
        for v in states:
            variant(v)
            if bucket_bytes:
                for b in reversed(range(plan.n_buckets)):
                    zs.zs_fused_step(plan, b, grads, zs.ZS_RANK_FULL, *states[v].args(), reps[v], HP, t)
            else:
                zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *states[v].args(), reps[v], HP, t)
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        for v in states:
            _check_state(ref, states[v], om, omm, ov, "variant %d t=%d" % (v, t))
            for q in range(n_d):
                H.check_bf16(H.to_np_bf16(reps[v][q]), ref_reps[q], "variant %d replica %d" % (v, q))


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_staged_reduce_scatter_matches_oracle(variant, n_d):
    """The staged reduce-scatter-mean (forced, every rank count with a shape) into one array, over the
    whole space and bucket by bucket from per-bucket staging buffers (offset views, bucket edges off
    the 8-element grid, so the fringes take the streaming kernel): the oracle's mean, bit for bit;
    the in-place ZeRO-1 form (streaming kernel) agrees on the owned slices."""
    numel = 1_100_003
    plan, ref = _plans([(numel,)], n_d, bucket_bytes=2 * 300_001, stage=2)
    P, pads = plan.padded, plan.pad_ranges()
    grads, _ = synth.rank_grads(n_d, P, pads, seed=65, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)
    want = steps.reduce_mean([H.to_np_bf16(g) for g in grads])
    variant(zs.ZS_FUSED_TMA)
    ghat = torch.full((P,), 7.0, dtype=BF16, device=DEV)
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    H.check_bf16(H.to_np_bf16(ghat), want, "whole space n_d=%d" % n_d)
    ghat2 = torch.full((P,), 7.0, dtype=BF16, device=DEV)
    for b in reversed(range(plan.n_buckets)):
        _, lo, hi = plan.bucket(b)
        staging = [g[lo:hi].clone() for g in grads]
        zs.zs_reduce_scatter_mean(plan, b, staging, zs.ZS_RANK_BUCKET, [ghat2], zs.ZS_SHARDED)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    assert torch.equal(ghat2, ghat)
    inplace = [g.clone() for g in grads]
    zs.zs_reduce_scatter_mean(plan, -1, inplace, zs.ZS_RANK_FULL, inplace, zs.ZS_RANK_FULL)
    torch.cuda.synchronize()
    S = plan.shard_per_rank
    for q in (0, n_d - 1):
        assert torch.equal(inplace[q][q * S:(q + 1) * S], ghat[q * S:(q + 1) * S])


@pytest.mark.parametrize("n_d", [2, 4, 8, 16, 32])
def test_staged_zero3_rs_step_matches_streaming(variant, n_d):
    """The single-output staged kernel (every rank count's own shape) equals the streaming kernel."""
    shapes, units = _tiny_llama(n_layers=2, d=256, ffn=704, vocab=1000)
    plan, _ = _plans(shapes, n_d, units=units, stage=3)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=9, device=DEV)
    out = {}
    for v in (zs.ZS_FUSED_LDG, zs.ZS_FUSED_TMA):
        variant(v)
        st = State(master0)
        shards = master0.to(BF16)
        for u in reversed(range(plan.n_units)):
            ud = plan.unit(u)
            grads, _ = synth.rank_grads(n_d, ud["padded"], [], seed=90 + u, step=1, sigma=5e-4, device=DEV)
            zs.zs_zero3_rs_step_unit(plan, u, grads, *st.args(), shards, HP, 1)
        torch.cuda.synchronize()
        out[v] = (st, shards)
    a, b = out[zs.ZS_FUSED_LDG], out[zs.ZS_FUSED_TMA]
    for x, y in zip(a[0].args(), b[0].args()):
        assert torch.equal(x, y)
    assert torch.equal(a[1], b[1])


def test_bounded_wait_times_out_and_reports():
    """A wait nothing completes gives up after its budget, records the status, and the
    context stays usable."""
    zs.zs_device_status(clear=True)
    zs.zs_selftest_wait_timeout(200_000)
    torch.cuda.synchronize()
    assert zs.zs_device_status(clear=True) == zs.ZS_DEVERR_SELFTEST
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    x = torch.ones(1024, device=DEV)
    assert float(x.sum()) == 1024.0
    with pytest.raises(zs.ZsError):
        zs.zs_selftest_wait_timeout(0)
    with pytest.raises(zs.ZsError):
        zs.zs_set_fused_variant(7)


# ---------------------------------------------------------------- ZeRO-3 step on two streams

@pytest.mark.parametrize("n_d,reshard,size", [(16, True, "tiny"), (5, True, "tiny"), (4, False, "tiny"), (2, True, "tiny"),
                                               (8, True, "walked"), (5, True, "walked"), (16, False, "walked")])
def test_zero3_step_two_streams_matches_oracle(n_d, reshard, size):
    """The whole ZeRO-3 step (forward gathers, backward gathers, reduce-scatter + update per
    unit) with communication on a side stream equals the oracle, and equals the same step
    with everything serialised on one stream, bit for bit.  "walked": layer units of 3.2 M
    elements and a root unit of 32.8 M (unit bases off the 8-element grid for N_d = 5), so
    the root unit's gathers and update are each walked in four overlapping launches."""
    if size == "tiny":
        shapes, units = _tiny_llama(n_layers=3, d=96, ffn=256, vocab=300)
    else:
        shapes, units = _tiny_llama(n_layers=2, d=512, ffn=1408, vocab=32000)
    plan, ref = _plans(shapes, n_d, units=units, stage=3)
    P, pads = plan.padded, plan.pad_ranges()
    U = plan.n_units
    biggest = max(plan.unit(u)["padded"] for u in range(U))
    master0 = synth.master_init(P, pads, seed=12, device=DEV)
    om, omm, ov = _oracle_state(ref, H.to_np_f32(master0))
    osh = H.reshard(ref, H.to_np_bf16(master0.to(BF16)))
    runs = {}
    for mode in ("overlap", "serial"):
        st = State(master0)
        shards = master0.to(BF16)
        n_slots = 2 if reshard else U
        pool = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(n_slots)]
        main = torch.cuda.current_stream()
        side = torch.cuda.Stream() if mode == "overlap" else main
        for t in (1, 2):
            ugrads = []
            for u in range(U):
                ud = plan.unit(u)
                upads = [(ud["numel"], ud["padded"])] if ud["padded"] > ud["numel"] else []
                ugrads.append(synth.rank_grads(n_d, ud["padded"], upads, seed=40 + u, step=t, sigma=5e-4,
                                               device=DEV)[0])
            zs.zs_zero3_step(plan, shards, *st.args(), ugrads, pool, reshard, HP, t, main_stream=main,
                             side_stream=side)
            torch.cuda.synchronize()
            if mode == "overlap":
                pre = [s_.copy() for s_ in osh]
                for u in reversed(range(U)):
                    _, _, osh, om, omm, ov = steps.zero3_unit_step(ref, u, osh, [H.to_np_bf16(g) for g in ugrads[u]],
                                                                   om, omm, ov, HP, t)
                _check_state(ref, st, om, omm, ov, "zero3_step t=%d" % t)
                H.check_bf16(H.to_np_bf16(shards), H.unshard(ref, osh), "zero3_step shards t=%d" % t)
                # the slots hold the last units gathered into them, from before the update
                for u in ((0, 1) if reshard else range(U)):
                    slot = (u & 1) if reshard else u
                    want = steps.all_gather_unit(ref, u, pre)
                    n_u = plan.unit(u)["padded"]
                    for q in range(n_d):
                        H.check_bf16(H.to_np_bf16(pool[slot][q][:n_u]), want[q], "pool slot %d q=%d" % (slot, q))
        runs[mode] = (st, shards)
    a, b = runs["overlap"], runs["serial"]
    for x, y in zip(a[0].args(), b[0].args()):
        assert torch.equal(x, y)
    assert torch.equal(a[1], b[1])


def test_zero3_step_rejects_small_pool():
    shapes, units = _tiny_llama(n_layers=2)
    plan, _ = _plans(shapes, 4, units=units, stage=3)
    P = plan.padded
    master = torch.zeros(P, device=DEV)
    ug = [synth.rank_buffers(4, plan.unit(u)["padded"], BF16, DEV)[0] for u in range(plan.n_units)]
    pool = [synth.rank_buffers(4, max(plan.unit(u)["padded"] for u in range(plan.n_units)), BF16, DEV)[0]]
    with pytest.raises(zs.ZsError):
        zs.zs_zero3_step(plan, master.to(BF16), master, master.clone(), master.clone(), ug, pool, True, HP, 1)
    with pytest.raises(zs.ZsError):
        zs.zs_zero3_step(plan, master.to(BF16), master, master.clone(), master.clone(), ug, pool * 2, False, HP, 1)


# ---------------------------------------------------------------- host-fed steps

@pytest.mark.parametrize("n_d,numel,bucket_bytes", [(8, 1_000_003, 1 << 18), (4, 262_912, 0), (3, 77_777, 10_000)])
def test_host_fed_steps_match_device_fused_step(n_d, numel, bucket_bytes):
    """zs_zero2_step_host (bucket-wise copies through a two-slot staging ring on a copy
    stream, overlapped with the per-bucket update) and zs_fused_step_host equal
    zs_fused_step on device-resident gradients, bit for bit, including the host copy of
    rank 0's replica."""
    plan, _ = _plans([(numel,)], n_d, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=13, device=DEV)
    sts = [State(master0) for _ in range(3)]
    reps = [synth.rank_buffers(n_d, P, BF16, DEV)[0] for _ in range(3)]
    biggest = max(hi - lo for _, lo, hi in (plan.bucket(b) for b in range(plan.n_buckets)))
    staging = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(2)]
    dev_grads = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    copy_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    for t in (1, 2, 3):
        grads, _ = synth.rank_grads(n_d, P, pads, seed=13, step=t, sigma=1e-3, device=DEV)
        host = [g.cpu().pin_memory() for g in grads]
        out1 = torch.empty(P, dtype=BF16).pin_memory()
        out2 = torch.empty(P, dtype=BF16).pin_memory()
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *sts[0].args(), reps[0], HP, t)
        zs.zs_zero2_step_host(plan, host, staging, *sts[1].args(), reps[1], HP, t, host_replica0=out1,
                              copy_stream=copy_stream, d2h_stream=d2h_stream)
        zs.zs_fused_step_host(plan, host, dev_grads, *sts[2].args(), reps[2], HP, t, host_replica0=out2)
        torch.cuda.synchronize()
        for k in (1, 2):
            for x, y in zip(sts[0].args(), sts[k].args()):
                assert torch.equal(x, y)
            for q in range(n_d):
                assert torch.equal(reps[0][q], reps[k][q])
        assert torch.equal(out1, reps[0][0].cpu()) and torch.equal(out2, reps[0][0].cpu())


@pytest.mark.parametrize("variant", [zs.ZS_FUSED_AUTO, zs.ZS_FUSED_TMA])
def test_fused_step_reads_and_writes_pinned_host_memory(variant):
    """Gradients in pinned host memory and rank 0's replica in pinned host memory: the kernel
    reads and writes them over the host link; results equal the all-device step bit for bit
    (the staged kernel is never used for such calls, whatever variant is selected)."""
    zs.zs_set_fused_variant(variant)
    try:
        plan, _ = _plans([(2_000_003,)], 8)
        P, pads = plan.padded, plan.pad_ranges()
        master0 = synth.master_init(P, pads, seed=14, device=DEV)
        a, b = State(master0), State(master0)
        reps_a = synth.rank_buffers(8, P, BF16, DEV)[0]
        reps_b = synth.rank_buffers(8, P, BF16, DEV)[0]
        host_rep0 = torch.empty(P, dtype=BF16).pin_memory()
        for t in (1, 2):
            grads, _ = synth.rank_grads(8, P, pads, seed=14, step=t, sigma=1e-3, device=DEV)
            host = [g.cpu().pin_memory() for g in grads]
            zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *a.args(), reps_a, HP, t)
            zs.zs_fused_step(plan, -1, host, zs.ZS_RANK_FULL, *b.args(), [host_rep0] + reps_b[1:], HP, t)
            torch.cuda.synchronize()
            for x, y in zip(a.args(), b.args()):
                assert torch.equal(x, y)
            assert torch.equal(host_rep0, reps_a[0].cpu())
            for q in range(1, 8):
                assert torch.equal(reps_a[q], reps_b[q])
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


@pytest.mark.parametrize("variant", [zs.ZS_FUSED_AUTO, zs.ZS_FUSED_TMA])
def test_bucket_walk_with_pinned_host_gradients(variant):
    """A bucket walk (every other bucket, then the rest) whose gradients are pinned host memory runs
    on the streaming kernel, range by range, and equals the all-device whole-range step."""
    zs.zs_set_fused_variant(variant)
    try:
        plan, _ = _plans([(2_000_003,)], 4, bucket_bytes=1 << 20)
        P, pads = plan.padded, plan.pad_ranges()
        master0 = synth.master_init(P, pads, seed=15, device=DEV)
        a, b = State(master0), State(master0)
        reps_a = synth.rank_buffers(4, P, BF16, DEV)[0]
        reps_b = synth.rank_buffers(4, P, BF16, DEV)[0]
        grads, _ = synth.rank_grads(4, P, pads, seed=15, step=1, sigma=1e-3, device=DEV)
        host = [g.cpu().pin_memory() for g in grads]
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *a.args(), reps_a, HP, 1)
        order = list(reversed(range(plan.n_buckets)))
        for part in (order[0::2], order[1::2]):
            zs.zs_fused_step_buckets(plan, part, host, *b.args(), reps_b, HP, 1)
        torch.cuda.synchronize()
        for x, y in zip(a.args(), b.args()):
            assert torch.equal(x, y)
        assert all(torch.equal(x, y) for x, y in zip(reps_a, reps_b))
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)


# ---------------------------------------------------------------- bulk-store gather

@pytest.mark.parametrize("n_d,numel", [(2, 3_000_001), (3, 1_500_007), (8, 4_194_305), (16, 2_100_003), (64, 1_048_583)])
def test_bulk_store_gathers_match_oracle(n_d, numel):
    """Gathers large enough for the bulk-store kernel (one source, N_d destinations): the
    all-gather from shards into full replicas, and the ZeRO-3 unit gather at a unit base that is
    not zero; ragged ends go through the element-wise fringe."""
    shapes = [(numel,), (1_048_576 + 24,)]
    plan, ref = _plans(shapes, n_d, units=[0, 1], stage=3)
    P, pads = plan.padded, plan.pad_ranges()
    shards = synth.master_init(P, pads, seed=60, device=DEV).to(BF16)
    osh = H.reshard(ref, H.to_np_bf16(shards))
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, reps)
    full_units = []
    for u in range(plan.n_units):
        full, _ = synth.rank_buffers(n_d, plan.unit(u)["padded"], BF16, DEV)
        zs.zs_zero3_gather_unit(plan, u, shards, full)
        full_units.append(full)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    want = steps.all_gather(ref, osh)
    for q in range(n_d):
        assert np.array_equal(H.to_np_bf16(reps[q]), want[q])
    for u in range(plan.n_units):
        want_u = steps.all_gather_unit(ref, u, osh)
        for q in (0, n_d // 2, n_d - 1):
            assert np.array_equal(H.to_np_bf16(full_units[u][q]), want_u[q])


@pytest.mark.parametrize("n_d,numel", [(8, 3_000_005), (3, 2_500_001), (8, 3 * (1 << 22) + 5), (2, (1 << 24) + 13)])
def test_staged_adamw_on_sharded_buffers(variant, n_d, numel):
    """zs_adamw_shard_step with the reduced gradient and the parameters in ZS_SHARDED arrays runs
    through the staged kernel with one rank, walked in overlapping launches (3 x 2^22 + 5 elements:
    three launches, the later two streaming while their predecessor drains), or from 2^24 elements on
    in one dynamic-order launch (the whole-buffer call at 2^24 + 13; its per-rank calls are walked);
    whole-unit and per-rank calls (ragged shard bounds) equal the oracle and the streaming kernel bit
    for bit."""
    plan, ref = _plans([(numel,)], n_d)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=61, device=DEV)
    ghat_np = numerics.bf16_rne((np.random.default_rng(61).standard_normal(P) * 1e-3).astype(np.float32))
    for lo, hi in pads:
        ghat_np[lo:hi] = 0
    ghat = H.from_np_bf16(ghat_np)
    z = np.zeros(P, np.float32)
    want_p, want_m, want_v, want_bits = steps.adamw(H.to_np_f32(master0), z, z, ghat_np, HP, 3)
    results = {}
    for v_, per_rank in ((zs.ZS_FUSED_AUTO, False), (zs.ZS_FUSED_AUTO, True), (zs.ZS_FUSED_LDG, False)):
        variant(v_)
        st = State(master0)
        params = torch.zeros(P, dtype=BF16, device=DEV)
        if per_rank:
            for r in range(n_d):
                zs.zs_adamw_shard_step(plan, r, [ghat], zs.ZS_SHARDED, *st.args(), [params], zs.ZS_SHARDED, HP, 3)
        else:
            zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, *st.args(), [params], zs.ZS_SHARDED, HP, 3)
        torch.cuda.synchronize()
        H.check_f32(H.to_np_f32(st.master), want_p, "master %d %s" % (v_, per_rank))
        H.check_f32(H.to_np_f32(st.m), want_m, "m %d %s" % (v_, per_rank))
        H.check_f32(H.to_np_f32(st.v), want_v, "v %d %s" % (v_, per_rank))
        H.check_bf16(H.to_np_bf16(params), want_bits, "params %d %s" % (v_, per_rank))
        results[(v_, per_rank)] = st
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE


def test_guard_zones_untouched_large_kernels():
    """Sentinels around every buffer of the large-range kernels (accumulation, staged fused step over
    one range and over a scattered bucket list, staged AdamW, bulk-store gathers, staged naive-DP step
    and the in-place all-reduce, FSDP2 copies): nothing is written outside the buffers."""
    n_d, numel = 8, 2_097_165
    plan, _ = _plans([(numel,)], n_d, stage=3)
    P = plan.padded
    bufs = []

    def mk(n, dtype):
        t, raw, g = _guarded(n, dtype)
        t.zero_()
        bufs.append((raw, g))
        return t

    grads = [mk(P, BF16) for _ in range(n_d)]
    for g in grads:
        g.normal_(0, 1e-3)
    reps = [mk(P, BF16) for _ in range(n_d)]
    full = [mk(P, BF16) for _ in range(n_d)]
    master, m, v = mk(P, torch.float32), mk(P, torch.float32), mk(P, torch.float32)
    ghat, shards = mk(P, BF16), mk(P, BF16)
    zs.zs_accumulate_grad(plan, reps, grads, 0.25, first=True)                           # accumulation
    zs.zs_accumulate_grad(plan, reps, grads, 0.25, first=False)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, 1)        # staged, broadcast
    zs.zs_zero3_rs_step_unit(plan, 0, grads, master, m, v, shards, HP, 2)               # staged, single output
    zs.zs_reduce_scatter_mean(plan, -1, grads, zs.ZS_RANK_FULL, [ghat], zs.ZS_SHARDED)
    zs.zs_adamw_shard_step(plan, -1, [ghat], zs.ZS_SHARDED, master, m, v, [shards], zs.ZS_SHARDED, HP, 3)
    zs.zs_all_gather(plan, [shards], zs.ZS_SHARDED, reps)                               # bulk gather
    zs.zs_zero3_gather_unit(plan, 0, shards, full)                                      # bulk gather
    bp = zs.Plan([(numel,)], n_d, stage=2, bucket_bytes=1 << 20)
    assert bp.n_buckets >= 4
    zs.zs_fused_step_buckets(bp, list(range(0, bp.n_buckets, 2)), grads, master, m, v, reps, HP, 4)  # list kernel
    dp = zs.Plan([(numel,)], n_d, stage=0)
    assert dp.padded == P
    dm, dmm, dv = ([mk(P, torch.float32) for _ in range(n_d)] for _ in range(3))
    zs.zs_dp_step(dp, grads, dm, dmm, dv, full, HP, 1)                                  # staged naive DP
    zs.zs_all_reduce_mean(dp, -1, grads)                                                # in place
    p2 = zs.Plan([(1023, 2048), (5,)], n_d, layout=zs.ZS_LAYOUT_FSDP2)
    params = [mk(1023 * 2048, BF16), mk(5, BF16)]
    params[0].normal_()
    flat = mk(p2.unit(0)["padded"], BF16)
    zs.zs_fsdp2_chunk_cat(p2, 0, params, flat)
    zs.zs_fsdp2_copy_out(p2, 0, flat, params)
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for raw, g in bufs:
        assert bool((raw[:g] == 0x5A).all()) and bool((raw[-g:] == 0x5A).all())


@pytest.mark.parametrize("bucket_bytes", [1 << 20, 4 << 20, 1000, 2 * 65544])
@pytest.mark.parametrize("mode", ["walk", "per_bucket", "per_bucket_two_streams"])
def test_fused_step_buckets_equals_whole_range(bucket_bytes, mode):
    """zs_fused_step_buckets over all buckets, descending, equals the whole-range step: walked as two
    lists of disjoint buckets, one launch per bucket, and one launch per bucket with the odd
    positions on a side stream.  Work enqueued on the caller's stream just before the call is
    seen, and work enqueued right after it sees the whole step (one launch per bucket lets a
    bucket's launch start before the previous bucket's ends; only the first launch on each stream
    waits for what came before the call); a repeated bucket is refused before anything runs.
    65,544-element buckets make the walk start with a short last bucket on the streaming kernel and
    go on with staged launches."""
    plan, _ = _plans([(3_000_011,)], 8, bucket_bytes=bucket_bytes)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=62, device=DEV)
    a, b = State(master0), State(master0)
    ra = synth.rank_buffers(8, P, BF16, DEV)[0]
    rb = synth.rank_buffers(8, P, BF16, DEV)[0]
    src, _ = synth.rank_grads(8, P, pads, seed=62, step=1, sigma=1e-3, device=DEV)
    grads = synth.rank_buffers(8, P, BF16, DEV)[0]
    side = torch.cuda.Stream() if mode == "per_bucket_two_streams" else None
    lm = zs.ZS_BUCKETS_ONE_WALK if mode == "walk" else zs.ZS_BUCKETS_PER_BUCKET
    zs.zs_fused_step(plan, -1, src, zs.ZS_RANK_FULL, *a.args(), ra, HP, 1)
    torch.cuda.synchronize()
    for q in range(8):
        grads[q].copy_(src[q])                      # on the caller's stream, still in flight at the call
    order = list(reversed(range(plan.n_buckets)))
    if mode == "walk":
        # every other bucket, then the rest: each call is a list of disjoint runs (the list kernel;
        # 1000-byte buckets give 3,000 runs per call, several list launches and a streaming fringe
        # at every run edge off the 8-element grid); all buckets at once would merge into one range
        for part in (order[0::2], order[1::2]):
            zs.zs_fused_step_buckets(plan, part, grads, *b.args(), rb, HP, 1, launch_mode=lm)
    else:
        zs.zs_fused_step_buckets(plan, order, grads, *b.args(), rb, HP, 1, launch_mode=lm, side_stream=side)
    after = [r.clone() for r in rb] + [x.clone() for x in b.args()]   # caller's stream, right after
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for x, y in zip(a.args(), b.args()):
        assert torch.equal(x, y)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))
    assert all(torch.equal(x, y) for x, y in zip(ra + list(a.args()), after))
    before = b.master.clone()
    with pytest.raises(zs.ZsError):
        zs.zs_fused_step_buckets(plan, [0, 1, 0], grads, *b.args(), rb, HP, 2, launch_mode=lm, side_stream=side)
    with pytest.raises(zs.ZsError):
        zs.zs_fused_step_buckets(plan, [0, 1], grads, *b.args(), rb, HP, 2, launch_mode=7)
    torch.cuda.synchronize()
    assert torch.equal(b.master, before)


def test_fused_step_buckets_all_at_once_merge_into_one_range():
    """All buckets of a plan in one walk (descending) touch each other, so they are stepped as one
    range: the same values as the whole-range step."""
    plan, _ = _plans([(2_500_003,)], 8, bucket_bytes=1 << 20)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=64, device=DEV)
    a, b = State(master0), State(master0)
    ra = synth.rank_buffers(8, P, BF16, DEV)[0]
    rb = synth.rank_buffers(8, P, BF16, DEV)[0]
    grads, _ = synth.rank_grads(8, P, pads, seed=64, step=1, sigma=1e-3, device=DEV)
    zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *a.args(), ra, HP, 1)
    zs.zs_fused_step_buckets(plan, list(reversed(range(plan.n_buckets))), grads, *b.args(), rb, HP, 1)
    torch.cuda.synchronize()
    for x, y in zip(a.args(), b.args()):
        assert torch.equal(x, y)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))


@pytest.mark.parametrize("n_d", [2, 4, 16, 32])
def test_fused_step_bucket_walk_every_rank_count(variant, n_d):
    """The list walk of the staged kernel (forced, so even a small list takes it) for every rank count
    with a staged shape, buckets in a shuffled order and a subset stepped first: equals stepping the
    same buckets one by one with the streaming kernel."""
    plan, _ = _plans([(700_001,)], n_d, bucket_bytes=2 * 40_000)
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=63, device=DEV)
    grads, _ = synth.rank_grads(n_d, P, pads, seed=63, step=1, sigma=1e-3, device=DEV)
    order = list(np.random.default_rng(n_d).permutation(plan.n_buckets))
    out = {}
    for v, lm in ((zs.ZS_FUSED_TMA, zs.ZS_BUCKETS_ONE_WALK), (zs.ZS_FUSED_LDG, zs.ZS_BUCKETS_PER_BUCKET)):
        variant(v)
        st = State(master0)
        reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
        zs.zs_fused_step_buckets(plan, order[:3], grads, *st.args(), reps, HP, 1, launch_mode=lm)
        zs.zs_fused_step_buckets(plan, order[3:], grads, *st.args(), reps, HP, 1, launch_mode=lm)
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        out[v] = (st, reps)
    (sa, ra), (sb, rb) = out[zs.ZS_FUSED_TMA], out[zs.ZS_FUSED_LDG]
    for x, y in zip(sa.args(), sb.args()):
        assert torch.equal(x, y)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))


@pytest.mark.parametrize("mode", ["walk", "per_bucket", "per_bucket_two_streams", "single_bucket_calls"])
def test_walk_of_unaligned_long_buckets(mode):
    """Buckets of 4,194,307 elements (longer than a walk piece, odd, so every bucket edge is off the
    8-element grid): each bucket is walked as staged pieces plus streaming fringes, the later staged
    launches not waiting before they start.  Equals the whole-range step bit for bit, with the
    gradients' copy enqueued just before the call and the results read just after it."""
    n = 3 * 4_194_307 + 5
    plan, _ = _plans([(n,)], 8, bucket_bytes=2 * 4_194_307)
    assert plan.n_buckets == 4
    P, pads = plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=65, device=DEV)
    a, b = State(master0), State(master0)
    ra = synth.rank_buffers(8, P, BF16, DEV)[0]
    rb = synth.rank_buffers(8, P, BF16, DEV)[0]
    src, _ = synth.rank_grads(8, P, pads, seed=65, step=1, sigma=1e-3, device=DEV)
    grads = synth.rank_buffers(8, P, BF16, DEV)[0]
    zs.zs_fused_step(plan, -1, src, zs.ZS_RANK_FULL, *a.args(), ra, HP, 1)
    torch.cuda.synchronize()
    for q in range(8):
        grads[q].copy_(src[q])
    order = list(reversed(range(plan.n_buckets)))
    if mode == "single_bucket_calls":
        for bk in order:
            zs.zs_fused_step(plan, bk, grads, zs.ZS_RANK_FULL, *b.args(), rb, HP, 1)
    elif mode == "walk":
        for part in (order[0::2], order[1::2]):
            zs.zs_fused_step_buckets(plan, part, grads, *b.args(), rb, HP, 1, launch_mode=zs.ZS_BUCKETS_ONE_WALK)
    else:
        side = torch.cuda.Stream() if mode == "per_bucket_two_streams" else None
        zs.zs_fused_step_buckets(plan, order, grads, *b.args(), rb, HP, 1, launch_mode=zs.ZS_BUCKETS_PER_BUCKET,
                                 side_stream=side)
    after = [r.clone() for r in rb] + [x.clone() for x in b.args()]
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for x, y in zip(a.args(), b.args()):
        assert torch.equal(x, y)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))
    assert all(torch.equal(x, y) for x, y in zip(ra + list(a.args()), after))
