"""The C ABI without a GPU: the library loads, exports every declared symbol, its
planner and accounting equal the oracle's bit for bit, and bad arguments are
rejected before anything is enqueued."""

import ctypes
import os
import random
import re

import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import synth
from oracle import accounting, layout, steps

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "zs.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|const char\*)\s+(zs_\w+)\s*\(", text, re.M)))


def test_library_exports_every_declared_symbol():
    names = _declared_symbols()
    assert len(names) >= 18
    lib = ctypes.CDLL(zs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(zs.EXPORTED)


def _compare_plans(shapes, n_d, units=None, bucket_bytes=0, stage=1, sample_params=None):
    ours = zs.Plan(shapes, n_d, stage=stage, bucket_bytes=bucket_bytes, unit_of_param=units)
    ref = layout.make_plan(shapes, n_d, unit_of_param=units, bucket_bytes=bucket_bytes if bucket_bytes > 0 else None)
    assert ours.numel == ref.numel
    assert ours.padded == ref.padded
    assert ours.shard_per_rank == ref.shard_total
    assert ours.n_units == len(ref.units)
    for u, ru in enumerate(ref.units):
        d = ours.unit(u)
        assert (d["base"], d["numel"], d["padded"], d["shard"]) == (ru.base, ru.numel, ru.padded, ru.shard)
    assert ours.n_buckets == len(ref.buckets)
    for b, rb in enumerate(ref.buckets):
        assert ours.bucket(b) == rb
        for r in range(n_d):
            lo, hi = ours.bucket_rank_slice(b, r)
            rlo, rhi = layout.bucket_rank_slice(ref, b, r)
            assert (hi - lo) == max(0, rhi - rlo)
            if hi > lo:
                assert (lo, hi) == (rlo, rhi)
    ks = range(len(shapes)) if sample_params is None else sample_params
    for k in ks:
        assert ours.param(k) == (ref.param_unit[k], ref.param_offset[k], ref.param_numel[k])
        for r in range(n_d):
            assert ours.param_segment(k, r) == layout.param_segment(ref, k, r)
    for s in range(4):
        assert ours.memory_bytes(s) == accounting.memory_bytes(ref, s)
        assert ours.comm_bytes(s) == accounting.comm_bytes_sent(ref, s)
    assert ours.comm_bytes(3, reshard_after_forward=False) == accounting.comm_bytes_sent(ref, 3, reshard_after_forward=False)
    return ours, ref


def test_python_constants_match_the_header():
    """Every ZS_* integer constant of the binding has the value include/zs.h gives it."""
    text = open(os.path.join(ROOT, "include", "zs.h")).read()
    pairs = re.findall(r"#define\s+(ZS_[A-Z0-9_]+)\s+\(?(-?\d+)[uUlL]*\)?\s", text)
    pairs += re.findall(r"\b(ZS_[A-Z0-9_]+)\s*=\s*(-?\d+)", text)
    checked = 0
    for name, value in pairs:
        if hasattr(zs, name):
            assert getattr(zs, name) == int(value), name
            checked += 1
    assert checked >= 20
    names = {n for n, _ in pairs}
    for n in ("ZS_DEVERR_GATHER_WAIT", "ZS_BUCKETS_ONE_WALK", "ZS_BUCKETS_PER_BUCKET", "ZS_FUSED_TMA"):
        assert n in names and hasattr(zs, n), n


def test_plan_matches_oracle_on_tiny_plans():
    rng = random.Random(5)
    for _ in range(150):
        n = rng.randint(1, 5)
        shapes = [tuple(rng.randint(1, 6) for _ in range(rng.randint(0, 3))) for _ in range(n)]
        units = None
        if rng.random() < 0.5:
            units = sorted(rng.randint(0, 2) for _ in range(n))
            remap = {u: i for i, u in enumerate(sorted(set(units)))}
            units = [remap[u] for u in units]
        _compare_plans(shapes, rng.randint(1, 9), units=units, bucket_bytes=rng.choice([0, 2, 6, 16, 50]))


def test_plan_fsdp1_worked_example():
    p = zs.Plan([(4, 2)] * 3, 2)
    assert p.padded == 24 and p.shard_per_rank == 12
    assert p.param_segment(0, 0) == (0, 0, 8) and p.param_segment(0, 1)[2] == 0
    assert p.param_segment(1, 0) == (8, 8, 4) and p.param_segment(1, 1) == (12, 0, 4)
    assert p.param_segment(2, 0)[2] == 0 and p.param_segment(2, 1) == (16, 4, 8)


@pytest.mark.parametrize("name,cfg", [
    ("mlp-tiny", dict(n_d=4, bucket_bytes=0, stage=1)),
    ("gpt2-small", dict(n_d=8, bucket_bytes=25 << 20, stage=1)),
    ("llama-1.3b", dict(n_d=8, bucket_bytes=25 << 20, stage=2)),
    ("llama-7b", dict(n_d=16, bucket_bytes=0, stage=3)),
])
def test_plan_matches_oracle_on_workloads(name, cfg):
    shapes, units = synth.workload_params(name)
    sample = sorted(set([0, 1, 2, len(shapes) - 2, len(shapes) - 1] + list(range(3, len(shapes), 7))))
    ours, _ = _compare_plans(shapes, cfg["n_d"], units=units, bucket_bytes=cfg["bucket_bytes"],
                             stage=cfg["stage"], sample_params=sample)
    expected_numel = {"mlp-tiny": 262_912, "gpt2-small": 124_439_808, "llama-1.3b": 1_345_423_360,
                      "llama-7b": 6_738_415_616}[name]
    assert ours.numel == expected_numel


@pytest.mark.parametrize("n_d,pad", [(2, 1), (4, 1), (8, 1), (16, 9), (32, 25)])
def test_plan_sweep_padding(n_d, pad):
    for mib in (1, 64, 1024):
        ours, _ = _compare_plans([(2 ** 28 + 7,)], n_d, bucket_bytes=mib << 20)
        assert ours.padded - ours.numel == pad


def test_adamw_scalars_match_oracle():
    for t in (1, 2, 3, 10, 1000, 10 ** 6):
        for hp in (synth.HPARAMS, {"lr": 3e-4, "beta1": 0.8, "beta2": 0.999, "eps": 1e-6, "weight_decay": 0.0}):
            ours = zs.zs_adamw_scalars(hp, t)
            ref = steps.adamw_scalars(hp, t)
            keys = ["beta1", "beta2", "eps", "decay", "c1", "c2", "step_size", "sqrt_bc2"]
            assert [float(ref[k]) for k in keys] == ours


def test_plan_rejects_bad_arguments():
    with pytest.raises(zs.ZsError):
        zs.Plan([(4,)], 0)
    with pytest.raises(zs.ZsError):
        zs.Plan([(4,)], zs.ZS_MAX_RANKS + 1)
    with pytest.raises(zs.ZsError):
        zs.Plan([(4, 0)], 2)
    with pytest.raises(zs.ZsError):
        zs.Plan([(4,), (5,)], 2, unit_of_param=[0, 2])          # unit 1 unused
    with pytest.raises(zs.ZsError):
        zs.Plan([(4,)], 2, stage=7)
    with pytest.raises(zs.ZsError):
        zs.Plan([(4,)], 2, bucket_bytes=1)                      # less than one bf16 element
    p = zs.Plan([(4,)], 2)
    with pytest.raises(zs.ZsError):
        p.bucket(1)
    with pytest.raises(zs.ZsError):
        p.param_segment(0, 2)
    with pytest.raises(zs.ZsError):
        zs.zs_adamw_scalars(synth.HPARAMS, 0)
    assert "step" in zs.zs_last_error()


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes placeholder addresses; the GPU tests cover this with real buffers")
def test_device_calls_reject_bad_arguments_before_launch():
    """Every case must be refused by the argument checks (ZS_ERR_INVALID), so no
    launch is ever attempted with these placeholder addresses."""
    lib = ctypes.CDLL(zs.LIB_PATH)
    lib.zs_fused_step.restype = ctypes.c_int32
    p = zs.Plan([(64,)], 4)
    hp = zs.zs_adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1)
    good = [0x10000 * (q + 1) for q in range(4)]

    def arr(xs):
        return (ctypes.c_void_p * len(xs))(*xs)

    def fused(grads, replicas, master=0x90000, step=1, bucket=-1, kind=zs.ZS_RANK_FULL):
        return lib.zs_fused_step(p.handle, ctypes.c_int32(bucket), arr(grads), ctypes.c_int32(kind),
                                 ctypes.c_void_p(master), ctypes.c_void_p(0xA0000), ctypes.c_void_p(0xB0000),
                                 arr(replicas), ctypes.byref(hp), ctypes.c_int64(step), ctypes.c_void_p(0))

    reps = [0x100000 * (q + 1) for q in range(4)]
    assert fused([good[0], 0, good[2], good[3]], reps) == zs.ZS_ERR_INVALID        # missing rank
    assert "missing rank" in zs.zs_last_error()
    assert fused([good[0] + 2] + good[1:], reps) == zs.ZS_ERR_INVALID               # misaligned
    assert fused(good, reps, master=0x90004) == zs.ZS_ERR_INVALID                   # misaligned state
    assert fused(good, reps, step=0) == zs.ZS_ERR_INVALID                           # 0-based step
    assert fused(good, reps, bucket=1) == zs.ZS_ERR_INVALID                         # no such bucket
    assert fused(good, reps, kind=zs.ZS_RANK_BUCKET) == zs.ZS_ERR_INVALID           # bucket kind without bucket
    assert fused(good, good) == zs.ZS_ERR_INVALID                                   # replicas alias grads
    bad_hp = zs.zs_adamw_hparams(1e-3, 1.0, 0.95, 1e-8, 0.1)
    assert lib.zs_fused_step(p.handle, -1, arr(good), 0, ctypes.c_void_p(0x90000), ctypes.c_void_p(0xA0000),
                             ctypes.c_void_p(0xB0000), arr(reps), ctypes.byref(bad_hp), ctypes.c_int64(1),
                             ctypes.c_void_p(0)) == zs.ZS_ERR_INVALID
    assert lib.zs_fused_step(None, -1, arr(good), 0, None, None, None, arr(reps), ctypes.byref(hp),
                             ctypes.c_int64(1), None) == zs.ZS_ERR_INVALID

    # the accumulating step: the same checks plus its own operands
    lib.zs_fused_step_accumulate.restype = ctypes.c_int32
    micro = [0x200000 * (q + 1) for q in range(4)]

    def fused_acc(acc, mic, replicas, scale=0.25, kind=zs.ZS_RANK_FULL, bucket=-1, step=1):
        return lib.zs_fused_step_accumulate(p.handle, ctypes.c_int32(bucket), arr(acc), arr(mic), ctypes.c_int32(kind),
                                            ctypes.c_float(scale), ctypes.c_void_p(0x90000), ctypes.c_void_p(0xA0000),
                                            ctypes.c_void_p(0xB0000), arr(replicas), ctypes.byref(hp),
                                            ctypes.c_int64(step), ctypes.c_void_p(0))

    assert fused_acc(good, [micro[0], 0] + micro[2:], reps) == zs.ZS_ERR_INVALID    # missing micro rank
    assert "micro" in zs.zs_last_error()
    assert fused_acc(good, [micro[0] + 8] + micro[1:], reps) == zs.ZS_ERR_INVALID   # misaligned micro
    assert fused_acc(good, micro, reps, scale=float("nan")) == zs.ZS_ERR_INVALID    # scale not finite
    assert fused_acc(good, micro, micro) == zs.ZS_ERR_INVALID                       # replicas alias micro
    assert fused_acc(good, micro, good) == zs.ZS_ERR_INVALID                        # replicas alias acc
    assert fused_acc(good, micro, reps, kind=zs.ZS_RANK_BUCKET) == zs.ZS_ERR_INVALID
    assert fused_acc(good, micro, reps, step=0) == zs.ZS_ERR_INVALID
    assert fused_acc(good, micro, reps, bucket=3) == zs.ZS_ERR_INVALID              # no such bucket


def test_list_zero3_and_dp_calls_reject_bad_arguments_before_launch():
    """The bucket-list, ZeRO-3 and naive-DP entry points refuse bad arguments with ZS_ERR_INVALID before
    anything is enqueued (placeholder addresses: no case may reach a launch)."""
    lib = ctypes.CDLL(zs.LIB_PATH)
    for name in ("zs_fused_step_buckets", "zs_zero3_step", "zs_dp_step"):
        getattr(lib, name).restype = ctypes.c_int32
    p = zs.Plan([(64,)], 4, stage=2, bucket_bytes=32)          # 4 buckets of 16 elements
    hp = zs.zs_adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1)
    good = [0x10000 * (q + 1) for q in range(4)]
    reps = [0x100000 * (q + 1) for q in range(4)]
    S = ctypes.c_void_p

    def arr(xs):
        return (ctypes.c_void_p * len(xs))(*xs)

    def ids(xs):
        return (ctypes.c_int32 * max(len(xs), 1))(*xs)

    def walk(buckets, grads=good, mode=zs.ZS_BUCKETS_ONE_WALK, n=None):
        return lib.zs_fused_step_buckets(p.handle, ctypes.c_int32(len(buckets) if n is None else n), ids(buckets),
                                         arr(grads), S(0x90000), S(0xA0000), S(0xB0000), arr(reps),
                                         ctypes.byref(hp), ctypes.c_int64(1), ctypes.c_int32(mode), S(0), S(0))

    assert walk([0, 4]) == zs.ZS_ERR_INVALID                                   # no such bucket
    assert walk([1, 2, 1]) == zs.ZS_ERR_INVALID                                # repeated bucket
    assert "twice" in zs.zs_last_error()
    assert walk([0], mode=7) == zs.ZS_ERR_INVALID                              # unknown launch mode
    assert walk([0], n=-1) == zs.ZS_ERR_INVALID                                # negative count
    assert walk([0], grads=[good[0], 0, good[2], good[3]]) == zs.ZS_ERR_INVALID  # missing rank
    assert lib.zs_fused_step_buckets(p.handle, 2, None, arr(good), S(0x90000), S(0xA0000), S(0xB0000), arr(reps),
                                     ctypes.byref(hp), ctypes.c_int64(1), 0, S(0), S(0)) == zs.ZS_ERR_INVALID

    p3 = zs.Plan([(64,), (32,), (16,)], 4, stage=3, unit_of_param=[0, 1, 2])   # three units
    ug = arr(good * 3)
    pool1 = arr(reps)                                                          # one slot: too few
    assert lib.zs_zero3_step(p3.handle, S(0xC0000), S(0x90000), S(0xA0000), S(0xB0000), ug, pool1, 1, 1,
                             ctypes.byref(hp), ctypes.c_int64(1), S(0), S(0)) == zs.ZS_ERR_INVALID
    assert lib.zs_zero3_step(p3.handle, S(0xC0000), S(0x90000), S(0xA0000), S(0xB0000), ug, arr(reps + reps), 2, 0,
                             ctypes.byref(hp), ctypes.c_int64(1), S(0), S(0)) == zs.ZS_ERR_INVALID  # needs 3 slots
    assert lib.zs_zero3_step(p3.handle, S(0xC0000), S(0x90000), S(0xA0000), S(0xB0000), ug, arr(reps + reps), 2, 1,
                             ctypes.byref(hp), ctypes.c_int64(0), S(0), S(0)) == zs.ZS_ERR_INVALID  # 0-based step

    pd = zs.Plan([(64,)], 4, stage=0)
    st = arr([0x200000 * (q + 1) for q in range(4)])
    assert lib.zs_dp_step(pd.handle, arr(good), st, st, st, arr(reps), ctypes.byref(hp), ctypes.c_int64(0),
                          S(0)) == zs.ZS_ERR_INVALID                           # 0-based step
    assert lib.zs_dp_step(pd.handle, arr([good[0] + 4] + good[1:]), st, st, st, arr(reps), ctypes.byref(hp),
                          ctypes.c_int64(1), S(0)) == zs.ZS_ERR_INVALID          # misaligned gradient


def test_fused_variant_switch_validates():
    assert zs.zs_set_fused_variant(zs.ZS_FUSED_LDG) == zs.ZS_OK
    assert zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO) == zs.ZS_OK
    with pytest.raises(zs.ZsError):
        zs.zs_set_fused_variant(3)


def test_dependent_launch_switch():
    """The programmatic-dependent-launch switch is process-wide and never fails (no CUDA call)."""
    assert zs.zs_set_dependent_launch(False) == zs.ZS_OK
    assert zs.zs_set_dependent_launch(True) == zs.ZS_OK


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes placeholder addresses; the GPU tests cover this with real buffers")
def test_checkpoint_step_is_validated(tmp_path):
    """A save with a negative step count and a meta.txt whose step is negative or missing are refused
    before any device memory is touched (placeholder addresses: no case may reach a copy)."""
    lib = ctypes.CDLL(zs.LIB_PATH)
    lib.zs_checkpoint_save.restype = ctypes.c_int32
    lib.zs_checkpoint_load.restype = ctypes.c_int32
    p = zs.Plan([(64,)], 4, stage=1)
    a = [ctypes.c_void_p(0x10000 * (k + 1)) for k in range(4)]
    d = os.fsencode(str(tmp_path))
    assert lib.zs_checkpoint_save(p.handle, d, *a, ctypes.c_int64(-1), None) == zs.ZS_ERR_INVALID
    assert "step" in zs.zs_last_error()
    step = ctypes.c_int64(0)
    for bad in ("step -5\n", "step\n", "steps 3\n"):
        (tmp_path / "meta.txt").write_text("zs-checkpoint 2\nn_d 4\n" + bad + "layout 0\nparams 1\n")
        assert lib.zs_checkpoint_load(p.handle, d, *a, ctypes.byref(step), None) == zs.ZS_ERR_INVALID
        assert "bad step" in zs.zs_last_error(), bad


@pytest.mark.skipif(torch.cuda.is_available(), reason="passes placeholder addresses; the GPU tests cover this with real buffers")
def test_rank_shard_step_rejects_bad_arguments_before_launch():
    """zs_rank_shard_step (one rank's local update) refuses bad arguments with ZS_ERR_INVALID before it
    looks at any buffer (placeholder addresses: no case may reach a launch)."""
    lib = ctypes.CDLL(zs.LIB_PATH)
    lib.zs_rank_shard_step.restype = ctypes.c_int32
    p = zs.Plan([(64,)], 4, stage=2, bucket_bytes=32)
    hp = zs.zs_adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1)
    good = [0x10000 * (q + 1) for q in range(4)]

    def call(rank=0, bucket=0, slices=good, master=0x90000, step=1, hpp=hp):
        arr = (ctypes.c_void_p * len(slices))(*slices)
        return lib.zs_rank_shard_step(p.handle, ctypes.c_int32(rank), ctypes.c_int32(bucket), arr,
                                      ctypes.c_void_p(master), ctypes.c_void_p(0xA0000), ctypes.c_void_p(0xB0000),
                                      ctypes.c_void_p(0xC0000), ctypes.byref(hpp), ctypes.c_int64(step),
                                      ctypes.c_void_p(0))

    assert call(rank=4) == zs.ZS_ERR_INVALID and "rank" in zs.zs_last_error()
    assert call(rank=-1) == zs.ZS_ERR_INVALID
    assert call(bucket=p.n_buckets) == zs.ZS_ERR_INVALID and "bucket" in zs.zs_last_error()
    assert call(bucket=-2) == zs.ZS_ERR_INVALID
    assert call(slices=[good[0], 0, good[2], good[3]]) == zs.ZS_ERR_INVALID
    assert "missing rank" in zs.zs_last_error()
    assert call(slices=[good[0] + 2] + good[1:]) == zs.ZS_ERR_INVALID                # misaligned slice
    assert call(master=0x90004) == zs.ZS_ERR_INVALID                                 # misaligned state
    assert call(step=0) == zs.ZS_ERR_INVALID
    assert call(hpp=zs.zs_adamw_hparams(1e-3, 1.0, 0.95, 1e-8, 0.1)) == zs.ZS_ERR_INVALID
