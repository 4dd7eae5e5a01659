"""Full-size parity for the widening rows, in the launch configurations the benchmark's
widening leg times, sampled.

* the bucket-list step on the 2^28+7 buffer (1 MiB and 4 MiB buckets), walked by one launch and
  launched bucket by bucket on two streams;
* naive DP (all-reduce-mean + replicated AdamW) on GPT-2-small at N_d = 8;
* ZeRO-3 without resharding after forward on Llama-1.3B (24 layer units + root), N_d = 8;
* the FSDP2 Shard(0) layout on the same grouping: gradients converted per rank, the fused step
  on the group buffers, the gathered parameters converted back.

Each is checked against the oracle on chunks (element-wise steps make a chunk's result depend
on that chunk's inputs only) and against the sharded FSDP1 step it must equal bit for bit.
"""

import gc

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth

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


def _chunks(P, boundaries, seed, n_random=6, width=W):
    rng = np.random.default_rng(seed)
    out = [(0, min(P, width)), (max(0, P - width), P)]
    for b in boundaries:
        out.append((max(0, b - width // 2), min(P, b + width // 2)))
    for _ in range(n_random):
        s = int(rng.integers(0, max(1, P - width)))
        out.append((s, min(P, s + width)))
    return sorted(set(out))


def _np(t):
    t = t.detach().cpu().clone()
    return H.to_np_bf16(t) if t.dtype == BF16 else H.to_np_f32(t)


def _check_chunks(chunks, before, master, m, v, reps, t, what):
    for (lo, hi), (gc_, p0, m0, v0) in zip(chunks, before):
        _, p, m1, v1, bits = H.chunk_oracle(gc_, p0, m0, v0, HP, t)
        w = "%s [%d,%d)" % (what, lo, hi)
        H.check_f32(_np(master[lo:hi]), p, "master " + w)
        H.check_f32(_np(m[lo:hi]), m1, "m " + w)
        H.check_f32(_np(v[lo:hi]), v1, "v " + w)
        for q, r in enumerate(reps):
            H.check_bf16(_np(r[lo:hi]), bits, "replica %d %s" % (q, w))


@pytest.mark.parametrize("mib,mode", [(1, "walk"), (4, "walk"), (1, "two_streams"), (4, "two_streams")])
def test_bucket_list_full_size(mib, mode):
    """2^28+7 elements, N_d = 8: every bucket in descending order, walked by one launch or launched
    one by one with the odd positions on a side stream, equals the whole-range step bit for bit,
    and the oracle on chunks around bucket edges."""
    n_d = 8
    shapes = [(2 ** 28 + 7,)]
    whole = zs.Plan(shapes, n_d, stage=2)
    plan = zs.Plan(shapes, n_d, stage=2, bucket_bytes=mib << 20)
    P, pads = plan.padded, plan.pad_ranges()
    bounds = [plan.bucket(b)[1] for b in range(1, plan.n_buckets)]
    chunks = _chunks(P, bounds[:3] + bounds[-3:], seed=mib)
    master = synth.master_init(P, pads, 4, device=DEV)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, 4, 1, 1e-3)
    a = [master.clone(), torch.zeros_like(master), torch.zeros_like(master)]
    b = [master.clone(), torch.zeros_like(master), torch.zeros_like(master)]
    del master
    ra, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    rb, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    before = [([_np(g[lo:hi]) for g in grads], _np(b[0][lo:hi]), _np(b[1][lo:hi]), _np(b[2][lo:hi]))
              for lo, hi in chunks]
    zs.zs_fused_step(whole, -1, grads, zs.ZS_RANK_FULL, *a, ra, HP, 1)
    order = list(reversed(range(plan.n_buckets)))
    if mode == "walk":
        # two lists of disjoint buckets (all at once would merge into one range)
        for part in (order[0::2], order[1::2]):
            zs.zs_fused_step_buckets(plan, part, grads, *b, rb, HP, 1, launch_mode=zs.ZS_BUCKETS_ONE_WALK)
    else:
        zs.zs_fused_step_buckets(plan, order, grads, *b, rb, HP, 1, launch_mode=zs.ZS_BUCKETS_PER_BUCKET,
                                 side_stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    assert all(torch.equal(x, y) for x, y in zip(ra, rb))
    _check_chunks(chunks, before, *b, [rb[0], rb[-1]], 1, "buckets %d MiB %s" % (mib, mode))


def test_naive_dp_gpt2_full_size():
    """GPT-2-small, N_d = 8: every rank's replicated state and parameters after two naive-DP steps
    equal the sharded ZeRO step's, bit for bit; the oracle on chunks."""
    n_d = 8
    shapes, _ = synth.workload_params("gpt2-small")
    plan = zs.Plan(shapes, n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    chunks = _chunks(P, [plan.shard_per_rank * r for r in range(1, n_d)][:4], seed=11)
    master0 = synth.master_init(P, pads, 1, device=DEV)
    dp_master = [master0.clone() for _ in range(n_d)]
    dp_m = [torch.zeros_like(master0) for _ in range(n_d)]
    dp_v = [torch.zeros_like(master0) for _ in range(n_d)]
    dp_reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    z = [master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)]
    z_reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    for t in (1, 2):
        synth.fill_grads(grads, pads, 1, t, 1e-3)
        before = [([_np(g[lo:hi]) for g in grads], _np(dp_master[3][lo:hi]), _np(dp_m[3][lo:hi]),
                   _np(dp_v[3][lo:hi])) for lo, hi in chunks]
        zs.zs_dp_step(plan, grads, dp_master, dp_m, dp_v, dp_reps, HP, t)
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *z, z_reps, HP, t)
        torch.cuda.synchronize()
        _check_chunks(chunks, before, dp_master[3], dp_m[3], dp_v[3], [dp_reps[0], dp_reps[7]], t, "dp t=%d" % t)
        for q in range(n_d):
            assert torch.equal(dp_master[q], z[0]) and torch.equal(dp_m[q], z[1]) and torch.equal(dp_v[q], z[2])
            assert torch.equal(dp_reps[q], z_reps[q])


def test_zero3_no_reshard_llama13b_full_size():
    """Llama-1.3B in 25 units, N_d = 8: the ZeRO-3 step without resharding after forward (one
    gather per unit, every unit held in its own slot) equals the step with resharding bit for bit;
    each slot then holds its unit's parameters from before the update; the oracle on chunks."""
    n_d = 8
    shapes, units = synth.workload_params("llama-1.3b-units")
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, U = plan.padded, plan.n_units
    assert plan.numel == 1_345_423_360 and U == 25
    pads = plan.pad_ranges()
    biggest = max(plan.unit(u)["padded"] for u in range(U))
    master0 = synth.master_init(P, pads, 2, device=DEV)
    shards0 = master0.to(BF16)
    ugrads, _ = synth.rank_buffers(n_d, biggest, BF16, DEV)
    synth.fill_grads(ugrads, [], 2, 1, 5e-4)
    # every unit reads the first padded_u elements of the same per-rank buffers
    res = {}
    for reshard in (True, False):
        st = [master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)]
        shards = shards0.clone()
        slots = U if not reshard else 2
        pool = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(slots)]
        side = torch.cuda.Stream()
        zs.zs_zero3_step(plan, shards, *st, [ugrads] * U, pool, reshard, HP, 1, side_stream=side)
        torch.cuda.synchronize()
        res[reshard] = (st, shards, None if reshard else pool)
        del pool
    (sa, sha, _), (sb, shb, pool) = res[True], res[False]
    for x, y in zip(sa, sb):
        assert torch.equal(x, y)
    assert torch.equal(sha, shb)
    for u in (0, 12, U - 1):
        ud = plan.unit(u)
        for q in (0, n_d - 1):
            assert torch.equal(pool[u][q][:ud["padded"]], shards0[ud["base"]:ud["base"] + ud["padded"]])
    del res, pool
    # the oracle on chunks of three units (the unit's gradients are the first padded_u elements)
    g_np = [_np(g) for g in ugrads]
    for u in (0, 12, U - 1):
        ud = plan.unit(u)
        base, up = ud["base"], ud["padded"]
        for lo, hi in _chunks(up, [ud["shard"] * r for r in range(1, n_d)][:3], seed=u, n_random=2):
            _, p, m1, v1, bits = H.chunk_oracle([g[lo:hi] for g in g_np], _np(master0[base + lo:base + hi]),
                                                np.zeros(hi - lo, np.float32), np.zeros(hi - lo, np.float32), HP, 1)
            w = "u=%d [%d,%d)" % (u, lo, hi)
            H.check_f32(_np(sb[0][base + lo:base + hi]), p, "master " + w)
            H.check_f32(_np(sb[2][base + lo:base + hi]), v1, "v " + w)
            H.check_bf16(_np(shb[base + lo:base + hi]), bits, "shards " + w)


def test_fsdp2_layout_step_llama13b_full_size():
    """Llama-1.3B in 25 groups, N_d = 4, FSDP2 Shard(0) layout: each rank's per-parameter gradients
    converted into the group buffers, the fused step there, the gathered buffers converted back,
    give every parameter exactly the values of the FSDP1 step on the same gradients."""
    n_d = 4
    shapes, units = synth.workload_params("llama-1.3b-units")
    p1 = zs.Plan(shapes, n_d, stage=2, unit_of_param=units)
    p2 = zs.Plan(shapes, n_d, stage=2, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    P1, P2, U = p1.padded, p2.padded, p1.n_units
    members = [p1.unit_members(u) for u in range(U)]

    def views(flat, plan, k):
        # parameter k's values inside an FSDP1 flat buffer (its natural layout)
        _, off, n = plan.param(k)
        return flat[off:off + n].view(shapes[k])

    # FSDP1: gradients and bf16-valued master (so both layouts start from the same values)
    g1, _ = synth.rank_buffers(n_d, P1, BF16, DEV)
    synth.fill_grads(g1, p1.pad_ranges(), 2, 1, 5e-4)
    m_bf = synth.master_init(P1, p1.pad_ranges(), 2, device=DEV).to(BF16)
    s1 = [m_bf.float(), torch.zeros(P1, device=DEV), torch.zeros(P1, device=DEV)]
    r1, _ = synth.rank_buffers(n_d, P1, BF16, DEV)
    zs.zs_fused_step(p1, -1, g1, zs.ZS_RANK_FULL, *s1, r1, HP, 1)
    del s1
    # FSDP2: the same per-parameter values converted into the group buffers
    g2, _ = synth.rank_buffers(n_d, P2, BF16, DEV)
    m2_bf = torch.zeros(P2, dtype=BF16, device=DEV)
    for u in range(U):
        ud = p2.unit(u)
        sl = slice(ud["base"], ud["base"] + ud["padded"])
        zs.zs_fsdp2_chunk_cat(p2, u, [views(m_bf, p1, k) for k in members[u]], m2_bf[sl])
        for q in range(n_d):
            zs.zs_fsdp2_chunk_cat(p2, u, [views(g1[q], p1, k) for k in members[u]], g2[q][sl])
    del g1
    s2 = [m2_bf.float(), torch.zeros(P2, device=DEV), torch.zeros(P2, device=DEV)]
    del m2_bf
    r2, _ = synth.rank_buffers(n_d, P2, BF16, DEV)
    chunks = _chunks(P2, [p2.unit(u)["base"] for u in (1, 12, 24)], seed=5, n_random=4)
    before = [([_np(g[lo:hi]) for g in g2], _np(s2[0][lo:hi]), _np(s2[1][lo:hi]), _np(s2[2][lo:hi]))
              for lo, hi in chunks]
    zs.zs_fused_step(p2, -1, g2, zs.ZS_RANK_FULL, *s2, r2, HP, 1)
    torch.cuda.synchronize()
    _check_chunks(chunks, before, *s2, [r2[0], r2[-1]], 1, "fsdp2")
    del g2, s2
    # convert rank 0's and the last rank's gathered group buffers back and compare per parameter
    for q in (0, n_d - 1):
        back = [torch.empty(s, dtype=BF16, device=DEV) for s in shapes]
        for u in range(U):
            ud = p2.unit(u)
            zs.zs_fsdp2_copy_out(p2, u, r2[q][ud["base"]:ud["base"] + ud["padded"]], [back[k] for k in members[u]])
        torch.cuda.synchronize()
        for k in range(len(shapes)):
            assert torch.equal(back[k], views(r1[q], p1, k)), "parameter %d rank %d" % (k, q)
