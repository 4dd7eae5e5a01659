"""FSDP2 Shard(0) layout on the GPU: the layout conversions and a whole step.

The conversions are pure data movement and must equal the oracle's exactly; a
step on the FSDP2 layout (each rank's per-parameter gradients converted into
its group buffers, the fused reduce-scatter + AdamW + all-gather, the gathered
buffers converted back into parameters) must give every rank the parameters of
naive DP computed in the parameters' own layout, bit for bit.
"""

import random

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth
from oracle import fsdp2, numerics, steps

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


def _bf16_param(rng, shape, scale):
    n = int(np.prod(shape)) if shape else 1
    return numerics.bf16_rne((rng.standard_normal(n) * scale).astype(np.float32))


@pytest.mark.parametrize("n_d", [2, 8])
def test_chunk_cat_and_copy_out_aligned_groups(n_d):
    """Every piece of the first group 16-byte aligned in both layouts (the vector path throughout):
    pieces of several 16K-element tasks, a last rank with fewer rows (zero padding rows), a
    parameter with fewer rows than ranks; the second group has 5-element rows (element path)."""
    shapes = [(4096, 64), (1003, 128), (4, 64), (64, 8), (40, 5)]
    units = [0, 0, 0, 0, 1]
    plan = zs.Plan(shapes, n_d, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    ref = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
    nrng = np.random.default_rng(70 + n_d)
    vals = [_bf16_param(nrng, s_, 1.0) for s_ in shapes]
    for u in range(plan.n_units):
        members = [k for k in range(len(shapes)) if units[k] == u]
        dev_params = [H.from_np_bf16(vals[k]).reshape(shapes[k]) for k in members]
        flat = torch.full((plan.unit(u)["padded"],), -3.0, dtype=BF16, device=DEV)
        zs.zs_fsdp2_chunk_cat(plan, u, dev_params, flat)
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        want = fsdp2.chunk_cat(ref, u, vals)
        assert np.array_equal(H.to_np_bf16(flat), want)
        outs = [torch.full_like(x, 5.0) for x in dev_params]
        zs.zs_fsdp2_copy_out(plan, u, flat, outs)
        torch.cuda.synchronize()
        back = fsdp2.copy_out(ref, u, want)
        for x, k in zip(outs, members):
            assert np.array_equal(H.to_np_bf16(x.reshape(-1)), back[k])


@pytest.mark.parametrize("n_d", [3, 8])
def test_chunk_cat_and_copy_out_large_pieces_and_many_params(n_d):
    """Pieces spanning many 16K-element copy tasks, padding rows inside a task, rows of odd length
    (element-wise path) and a group of more parameters than one launch takes (70 > 64)."""
    big = [(1000, 33), (517, 64), (7,), (70000, 1), (4096, 8), ()]
    small = [(rng_d0, 3) for rng_d0 in range(1, 65)]
    shapes = big + small
    units = [0] * len(big) + [1] * len(small)
    plan = zs.Plan(shapes, n_d, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    ref = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
    nrng = np.random.default_rng(n_d)
    vals = [_bf16_param(nrng, s, 1.0) for s in shapes]
    for u in range(plan.n_units):
        members = [k for k in range(len(shapes)) if units[k] == u]
        dev_params = [H.from_np_bf16(vals[k]).reshape(shapes[k]) for k in members]
        flat = torch.full((plan.unit(u)["padded"],), -2.0, dtype=BF16, device=DEV)
        zs.zs_fsdp2_chunk_cat(plan, u, dev_params, flat)
        torch.cuda.synchronize()
        want = fsdp2.chunk_cat(ref, u, vals)
        assert np.array_equal(H.to_np_bf16(flat), want)
        outs = [torch.full_like(x, 3.0) for x in dev_params]
        zs.zs_fsdp2_copy_out(plan, u, flat, outs)
        torch.cuda.synchronize()
        back = fsdp2.copy_out(ref, u, want)
        for x, k in zip(outs, members):
            assert np.array_equal(H.to_np_bf16(x.reshape(-1)), back[k])


@pytest.mark.parametrize("seed", range(6))
def test_chunk_cat_and_copy_out_match_oracle(seed):
    rng = random.Random(seed)
    n = rng.randint(1, 7)
    shapes = [tuple(rng.randint(1, 300) if i == 0 else rng.randint(1, 40) for i in range(rng.randint(0, 3)))
              for _ in range(n)]
    units = sorted(rng.randint(0, 2) for _ in range(n))
    remap = {u: i for i, u in enumerate(sorted(set(units)))}
    units = [remap[u] for u in units]
    n_d = rng.choice([1, 2, 3, 4, 8, 16])
    plan = zs.Plan(shapes, n_d, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    ref = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
    nrng = np.random.default_rng(seed)
    vals = [_bf16_param(nrng, s, 1.0) for s in shapes]
    for u in range(plan.n_units):
        members = [k for k in range(n) if units[k] == u]
        dev_params = [H.from_np_bf16(vals[k]) for k in members]
        flat = torch.full((plan.unit(u)["padded"],), 1.5, dtype=BF16, device=DEV)   # not zero: padding must be written
        zs.zs_fsdp2_chunk_cat(plan, u, dev_params, flat)
        torch.cuda.synchronize()
        want = fsdp2.chunk_cat(ref, u, vals)
        assert np.array_equal(H.to_np_bf16(flat), want)
        outs = [torch.zeros_like(x) for x in dev_params]
        zs.zs_fsdp2_copy_out(plan, u, flat, outs)
        torch.cuda.synchronize()
        back = fsdp2.copy_out(ref, u, want)
        for x, k in zip(outs, members):
            assert np.array_equal(H.to_np_bf16(x), back[k])


@pytest.mark.parametrize("n_d", [2, 4, 5])
def test_fsdp2_step_equals_naive_dp_in_parameter_layout(n_d):
    shapes = [(300, 64), (64,), (3, 64, 7), (257, 64), (1,), ()]
    units = [0, 0, 1, 1, 2, 2]
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    ref = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
    P = plan.padded
    nrng = np.random.default_rng(n_d)
    master_nat = [(nrng.standard_normal(int(np.prod(s)) if s else 1) * 0.02).astype(np.float32) for s in shapes]
    # the state in the FSDP2 layout, assembled on the host by the oracle's layout function
    master_flat = np.concatenate([fsdp2.chunk_cat(ref, u, master_nat) for u in range(plan.n_units)])
    master = torch.from_numpy(master_flat).to(DEV)
    m, v = torch.zeros_like(master), torch.zeros_like(master)
    reps = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    grads = synth.rank_buffers(n_d, P, BF16, DEV)[0]
    om = [x.copy() for x in master_nat]
    omm = [np.zeros_like(x) for x in master_nat]
    ov = [np.zeros_like(x) for x in master_nat]
    for t in (1, 2):
        g_nat = [[_bf16_param(nrng, s, 1e-3) for s in shapes] for _ in range(n_d)]
        for q in range(n_d):
            for u in range(plan.n_units):
                base = plan.unit(u)["base"]
                members = [k for k in range(len(shapes)) if units[k] == u]
                zs.zs_fsdp2_chunk_cat(plan, u, [H.from_np_bf16(g_nat[q][k]) for k in members],
                                      grads[q][base:base + plan.unit(u)["padded"]])
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, master, m, v, reps, HP, t)
        torch.cuda.synchronize()
        # oracle: naive DP per parameter, in the parameter's own layout
        want_bits = []
        for k in range(len(shapes)):
            _, om[k], omm[k], ov[k] = steps.dp_step([g_nat[q][k] for q in range(n_d)], om[k], omm[k], ov[k], HP, t)
            want_bits.append(numerics.bf16_rne(om[k]))
        for q in range(n_d):
            for u in range(plan.n_units):
                base = plan.unit(u)["base"]
                members = [k for k in range(len(shapes)) if units[k] == u]
                outs = [torch.empty(int(np.prod(shapes[k])) if shapes[k] else 1, dtype=BF16, device=DEV) for k in members]
                zs.zs_fsdp2_copy_out(plan, u, reps[q][base:base + plan.unit(u)["padded"]], outs)
                torch.cuda.synchronize()
                for x, k in zip(outs, members):
                    H.check_bf16(H.to_np_bf16(x), want_bits[k], "rank %d param %d t=%d" % (q, k, t))
        want_flat = np.concatenate([fsdp2.chunk_cat(ref, u, om) for u in range(plan.n_units)])
        H.check_f32(H.to_np_f32(master), want_flat, "master t=%d" % t)
        for b, e in plan.pad_ranges():
            assert not master[b:e].any() and not reps[0][b:e].float().any()
