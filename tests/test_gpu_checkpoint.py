"""Sharded checkpoint on the GPU: save with one rank count, load with another, keep training.

Compared against the oracle's checkpoint (save = each rank's shards, load = the
unit's real elements re-padded and re-cut) and, after loading, against the
oracle's ZeRO step on the loaded state.
"""

import os

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth
from oracle import checkpoint, layout, numerics, steps

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


def _model():
    shapes, units = [(300, 96)], [3]
    for layer in range(3):
        ls = [(96,), (96, 96), (96, 96), (96, 96), (96, 96), (96,), (257, 96), (257, 96), (96, 257)]
        shapes += ls
        units += [layer] * len(ls)
    shapes += [(96,), (300, 96)]
    units += [3, 3]
    return shapes, units


def _state(plan, seed):
    P, pads = plan.padded, plan.pad_ranges()
    master = synth.master_init(P, pads, seed, device=DEV)
    m = synth.master_init(P, pads, seed + 1, device=DEV, sigma=1e-4)
    v = synth.master_init(P, pads, seed + 2, device=DEV, sigma=1e-6).abs()
    return master.to(BF16), master, m, v


@pytest.mark.parametrize("units_on", [True, False])
@pytest.mark.parametrize("n_src,n_dst", [(8, 3), (8, 16), (4, 4), (5, 2)])
def test_save_load_other_rank_count_then_step(tmp_path, units_on, n_src, n_dst):
    shapes, units = _model()
    units = units if units_on else None
    src = zs.Plan(shapes, n_src, stage=3 if units_on else 1, unit_of_param=units)
    ref_src = layout.make_plan(shapes, n_src, unit_of_param=units)
    arrays = _state(src, 21)
    names = ["params", "master", "m", "v"]
    zs.zs_checkpoint_save(src, str(tmp_path), *arrays, step=7)
    assert os.path.exists(tmp_path / "meta.txt")
    assert len([f for f in os.listdir(tmp_path) if f.startswith("rank-")]) == n_src

    # the oracle's save of the same input arrays (rank-local shards)
    host = [H.to_np_bf16(arrays[0])] + [H.to_np_f32(a) for a in arrays[1:]]
    saved = checkpoint.save(ref_src, [{n: steps.shard_of(ref_src, r, h) for n, h in zip(names, host)}
                                      for r in range(n_src)])

    dst = zs.Plan(shapes, n_dst, stage=3 if units_on else 1, unit_of_param=units)
    ref_dst = layout.make_plan(shapes, n_dst, unit_of_param=units)
    P = dst.padded
    out = [torch.full((P,), 7, dtype=BF16, device=DEV)] + [torch.full((P,), 7.0, device=DEV) for _ in range(3)]
    assert zs.zs_checkpoint_load(dst, str(tmp_path), *out) == 7
    want = {n: checkpoint.load(ref_dst, saved, n) for n in names}
    H.check_bf16(H.to_np_bf16(out[0]), H.unshard(ref_dst, want["params"]), "params")
    for i, n in enumerate(names[1:], 1):
        H.check_f32(H.to_np_f32(out[i]), H.unshard(ref_dst, want[n]), n)

    # one more training step on the loaded state, on both sides
    grads, _ = synth.rank_grads(n_dst, P, dst.pad_ranges(), seed=22, step=8, sigma=1e-3, device=DEV)
    reps = synth.rank_buffers(n_dst, P, BF16, DEV)[0]
    zs.zs_fused_step(dst, -1, grads, zs.ZS_RANK_FULL, out[1], out[2], out[3], reps, HP, 8)
    torch.cuda.synchronize()
    ref_reps, om, omm, ov = steps.zero_step(ref_dst, [H.to_np_bf16(g) for g in grads], want["master"], want["m"],
                                            want["v"], HP, 8)
    H.check_f32(H.to_np_f32(out[1]), H.unshard(ref_dst, om), "master after step")
    H.check_f32(H.to_np_f32(out[3]), H.unshard(ref_dst, ov), "v after step")
    H.check_bf16(H.to_np_bf16(reps[n_dst - 1]), ref_reps[n_dst - 1], "replica after step")


def test_load_refuses_other_model_and_broken_files(tmp_path):
    shapes, _ = _model()
    plan = zs.Plan(shapes, 4)
    arrays = _state(plan, 3)
    zs.zs_checkpoint_save(plan, str(tmp_path), *arrays, step=1)
    other = zs.Plan(shapes[:-1] + [(301, 96)], 4)
    P = other.padded
    bufs = [torch.zeros(P, dtype=BF16, device=DEV)] + [torch.zeros(P, device=DEV) for _ in range(3)]
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_load(other, str(tmp_path), *bufs)
    assert "another model" in str(e.value)
    assert not any(b.float().any() for b in bufs)                  # nothing written
    with open(tmp_path / "rank-00002.bin", "r+b") as f:             # truncate one rank file
        f.truncate(100)
    with pytest.raises(zs.ZsError) as e:
        zs.zs_checkpoint_load(plan, str(tmp_path), *[torch.zeros_like(a) for a in arrays])
    assert "wrong size" in str(e.value)
    with pytest.raises(zs.ZsError):
        zs.zs_checkpoint_load(plan, str(tmp_path / "missing"), *[torch.zeros_like(a) for a in arrays])


@pytest.mark.parametrize("src_layout,n_src,src_units,dst_layout,n_dst,dst_units", [
    ("fsdp1", 8, True, "fsdp2", 3, False),
    ("fsdp2", 4, True, "fsdp1", 5, True),
    ("fsdp2", 6, False, "fsdp2", 16, True),
    ("fsdp1", 2, False, "fsdp1", 7, True),
])
def test_load_into_another_layout_and_grouping(tmp_path, src_layout, n_src, src_units, dst_layout, n_dst, dst_units):
    """A save in one layout (FSDP1 FlatParameter or FSDP2 Shard(0)), rank count and unit grouping
    loads into another; every array equals the oracle's element-identity reload, bit for bit."""
    from oracle import fsdp2

    shapes, units = _model()
    lay = {"fsdp1": zs.ZS_LAYOUT_FSDP1, "fsdp2": zs.ZS_LAYOUT_FSDP2}

    def plans(kind, n_d, grouped):
        u = units if grouped else None
        ours = zs.Plan(shapes, n_d, stage=3 if grouped else 1, unit_of_param=u, layout=lay[kind])
        ref = layout.make_plan(shapes, n_d, unit_of_param=u) if kind == "fsdp1" else \
            fsdp2.make_plan(shapes, n_d, unit_of_param=u)
        return ours, ref

    src, ref_src = plans(src_layout, n_src, src_units)
    dst, ref_dst = plans(dst_layout, n_dst, dst_units)
    # inputs in the source layout, built on the host by the oracle from per-parameter values
    nrng = np.random.default_rng(n_src * 31 + n_dst)
    nat = {name: [(nrng.standard_normal(int(np.prod(s))) * sc).astype(np.float32) for s in shapes]
           for name, sc in (("master", 0.02), ("m", 1e-4), ("v", 1e-6))}
    nat["v"] = [np.abs(x) for x in nat["v"]]

    def lay_out(kind, ref, values):
        if kind == "fsdp2":
            return np.concatenate([fsdp2.chunk_cat(ref, u, values) for u in range(len(ref.units))])
        full = np.zeros(ref.padded, np.float32)
        for k, x in enumerate(values):
            full[ref.param_offset[k]:ref.param_offset[k] + x.size] = x
        return full

    host = {name: lay_out(src_layout, ref_src, nat[name]) for name in nat}
    params_bits = numerics.bf16_rne(host["master"])
    dev_arrays = [H.from_np_bf16(params_bits)] + [torch.from_numpy(host[n]).to(DEV) for n in ("master", "m", "v")]
    zs.zs_checkpoint_save(src, str(tmp_path), *dev_arrays, step=4)

    P = dst.padded
    out = [torch.full((P,), 3, dtype=BF16, device=DEV)] + [torch.full((P,), 3.0, device=DEV) for _ in range(3)]
    assert zs.zs_checkpoint_load(dst, str(tmp_path), *out) == 4
    saved = checkpoint.save_any(ref_src, src_layout, [
        {"params": _rank_slice(ref_src, src_layout, r, params_bits),
         **{n: _rank_slice(ref_src, src_layout, r, host[n]) for n in ("master", "m", "v")}}
        for r in range(n_src)])
    n_params = len(shapes)
    for i, name in enumerate(("params", "master", "m", "v")):
        want = checkpoint.load_any(saved, ref_dst, dst_layout, name, n_params)
        got = H.to_np_bf16(out[0]) if i == 0 else H.to_np_f32(out[i])
        full_want = np.concatenate([_unshard_any(ref_dst, dst_layout, want)])
        assert np.array_equal(got.view(np.uint16 if i == 0 else np.uint32),
                              full_want.view(np.uint16 if i == 0 else np.uint32)), name


def _rank_slice(ref, kind, r, full):
    """Rank r's shard (all units) of a flat array laid out by `ref`."""
    pieces = []
    for u in ref.units:
        shard = u.shard
        base = u.base
        pieces.append(full[base + r * shard:base + (r + 1) * shard])
    return np.concatenate(pieces)


def _unshard_any(ref, kind, rank_arrays):
    full = np.zeros(ref.padded, dtype=rank_arrays[0].dtype)
    offs, acc = [], 0
    for u in ref.units:
        offs.append(acc)
        acc += u.shard
    for ui, u in enumerate(ref.units):
        for r in range(ref.n_d):
            full[u.base + r * u.shard:u.base + (r + 1) * u.shard] = rank_arrays[r][offs[ui]:offs[ui] + u.shard]
    return full
