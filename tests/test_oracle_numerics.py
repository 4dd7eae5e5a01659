"""Pins for the oracle's arithmetic (runs without a GPU).

bf16 rounding against torch's conversion; accumulation against the page's
4-micro-batch identity and a least-squares model; the rank mean against exact
rationals; AdamW against closed forms, float64 and torch.optim.AdamW; the
whole ZeRO step against naive DP and against the ZeRO-3 per-unit path.
Planted mistakes (in the oracle, on the CPU) must each trip at least one pin.
"""

import numpy as np
import pytest
import torch

import pins
from oracle import layout, numerics, steps


# ---------------------------------------------------------------- bf16

def _all_tie_and_edge_patterns():
    hi = np.arange(65536, dtype=np.uint32)
    lows = np.array([0x0000, 0x0001, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x4000, 0xC000], dtype=np.uint32)
    u = (hi[:, None] << 16) | lows[None, :]
    return u.reshape(-1)


def test_bf16_rne_matches_torch_on_every_exponent_and_tie():
    u = _all_tie_and_edge_patterns()
    rng = np.random.default_rng(0)
    u = np.concatenate([u, rng.integers(0, 2 ** 32, 1_000_000, dtype=np.uint64).astype(np.uint32)])
    x = u.view(np.float32)
    ours = numerics.bf16_rne(x)
    theirs = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], theirs[~nan])
    # NaN stays NaN
    back = numerics.f32_from_bf16(ours[nan])
    assert np.all(np.isnan(back))


def test_bf16_widening_is_exact_and_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = numerics.f32_from_bf16(bits)
    theirs = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == theirs.view(np.uint32)) | (np.isnan(ours) & np.isnan(theirs))
    assert same.all()
    finite = np.isfinite(ours)
    assert np.array_equal(numerics.bf16_rne(ours[finite]), bits[finite])


def test_bf16_ulp():
    one = numerics.bf16_rne(np.array([1.0, 1.5, 2.0, 3.0e-39], np.float32))
    ulp = numerics.bf16_ulp(one)
    assert ulp[0] == 2.0 ** -7 and ulp[1] == 2.0 ** -7 and ulp[2] == 2.0 ** -6
    assert ulp[3] == 2.0 ** -133


# ---------------------------------------------------------------- accumulation and mean

def test_accumulation_four_equal_microbatches():
    pins.pin_accumulation_four_equal_microbatches()


def test_accumulation_linear_model_full_batch():
    pins.pin_accumulation_linear_model()


def test_mean_against_exact_rationals():
    pins.pin_mean_against_exact_rationals()


def test_mean_of_equal_grads_is_exact():
    pins.pin_mean_of_equal_grads()


def test_mean_single_rank_is_identity():
    rng = np.random.default_rng(1)
    g = pins.rand_bf16(rng, 1000, 1.0)
    assert np.array_equal(steps.reduce_mean([g]), g)


# ---------------------------------------------------------------- AdamW

@pytest.mark.parametrize("pin", pins.ALL_ADAMW_PINS, ids=lambda f: f.__name__)
def test_adamw_pins(pin):
    pin()


def test_sharded_update_equals_unsharded():
    pins.pin_sharded_update_equals_unsharded()


def test_step_must_be_one_based():
    with pytest.raises(ValueError):
        steps.adamw_scalars(pins.HP, 0)


# ---------------------------------------------------------------- whole steps

def _random_state(rng, plan):
    n_d = plan.n_d
    pads = layout.pad_ranges(plan)
    full = (rng.standard_normal(plan.padded) * 0.02).astype(np.float32)
    for lo, hi in pads:
        full[lo:hi] = 0
    master = [steps.shard_of(plan, r, full) for r in range(n_d)]
    zeros = [np.zeros(plan.shard_total, np.float32) for _ in range(n_d)]
    return full, master, [z.copy() for z in zeros], [z.copy() for z in zeros]


def _random_grads(rng, plan):
    gs = []
    for _ in range(plan.n_d):
        g = pins.rand_bf16(rng, plan.padded, 1e-3)
        for lo, hi in layout.pad_ranges(plan):
            g[lo:hi] = 0
        gs.append(g)
    return gs


@pytest.mark.parametrize("n_d,bucket", [(1, 64), (2, 7), (3, 100), (4, 5), (8, 33)])
def test_zero_step_equals_naive_dp(n_d, bucket):
    """Sharded ZeRO-1/2 step (RS-mean, shard AdamW, AG) == naive DP (AR-mean, full AdamW on every replica)."""
    rng = np.random.default_rng(n_d)
    plan = layout.make_plan([(13, 7), (29,), (5, 5)], n_d, bucket_bytes=2 * bucket)
    full, master, m, v = _random_state(rng, plan)
    fm, fv = np.zeros(plan.padded, np.float32), np.zeros(plan.padded, np.float32)
    for t in range(1, 4):
        grads = _random_grads(rng, plan)
        replicas, master, m, v = steps.zero_step(plan, grads, master, m, v, pins.HP, t)
        dp_replicas, full, fm, fv = steps.dp_step(grads, full, fm, fv, pins.HP, t)
        for r in range(n_d):
            assert np.array_equal(replicas[r], dp_replicas[r])
            assert np.array_equal(master[r], steps.shard_of(plan, r, full))
            assert np.array_equal(m[r], steps.shard_of(plan, r, fm))
            assert np.array_equal(v[r], steps.shard_of(plan, r, fv))
        # every replica identical and equal to bf16(master); padding stays zero
        assert all(np.array_equal(replicas[0], rep) for rep in replicas)
        assert np.array_equal(replicas[0], numerics.bf16_rne(full))
        for lo, hi in layout.pad_ranges(plan):
            assert not replicas[0][lo:hi].any() and not full[lo:hi].any()


def test_bucket_order_does_not_change_the_result():
    rng = np.random.default_rng(3)
    plan = layout.make_plan([(100,), (37,)], 4, bucket_bytes=2 * 9)
    grads = _random_grads(rng, plan)
    a = steps.reduce_scatter_mean(plan, grads)
    b = steps.reduce_scatter_mean(plan, grads, bucket_order=list(range(len(plan.buckets))))
    for r in range(4):
        assert np.array_equal(a[r], b[r])


@pytest.mark.parametrize("n_d", [2, 4, 5])
def test_zero3_units_equal_flat_update(n_d):
    """ZeRO-3 per unit: gathering the updated shards gives the same parameters as a
    flat update with the same per-unit gradients (the units only change where
    the padding goes)."""
    rng = np.random.default_rng(20 + n_d)
    shapes = [(6, 5), (11,), (3, 3), (17,), (4, 4)]
    units = [0, 0, 1, 1, 2]
    plan = layout.make_plan(shapes, n_d, unit_of_param=units)
    full, master, m, v = _random_state(rng, plan)
    shards = [numerics.bf16_rne(master[r]) for r in range(n_d)]
    # flat reference over the same global padded space
    fm, fv = np.zeros(plan.padded, np.float32), np.zeros(plan.padded, np.float32)
    for t in (1, 2):
        unit_grads = []
        for ui, u in enumerate(plan.units):
            per_rank = []
            for _ in range(n_d):
                g = pins.rand_bf16(rng, u.padded, 1e-3)
                g[u.numel:] = 0
                per_rank.append(g)
            unit_grads.append(per_rank)
        gathered_before = [steps.all_gather_unit(plan, ui, shards) for ui in range(len(plan.units))]
        for ui in range(len(plan.units)):
            fwd, bwd, shards, master, m, v = steps.zero3_unit_step(plan, ui, shards, unit_grads[ui],
                                                                   master, m, v, pins.HP, t)
            # forward and backward gathers see the parameters from before the update
            for r in range(n_d):
                assert np.array_equal(fwd[r], gathered_before[ui][r])
                assert np.array_equal(bwd[r], gathered_before[ui][r])
        flat_grads = [np.concatenate([unit_grads[ui][q] for ui in range(len(plan.units))]) for q in range(n_d)]
        replicas, full, fm, fv = steps.dp_step(flat_grads, full, fm, fv, pins.HP, t)
        gathered = np.concatenate([steps.all_gather_unit(plan, ui, shards)[0] for ui in range(len(plan.units))])
        assert np.array_equal(gathered, replicas[0])
        for r in range(n_d):
            assert np.array_equal(master[r], steps.shard_of(plan, r, full))


# ---------------------------------------------------------------- planted mistakes

def _mutant_scalars(kind):
    real = steps.adamw_scalars

    def mutated(hp, t):
        s = dict(real(hp, t))
        if kind == "no_bias_correction":
            s["step_size"] = np.float32(hp["lr"])
            s["sqrt_bc2"] = np.float32(1.0)
        elif kind == "betas_swapped":
            s["beta1"], s["beta2"] = s["beta2"], s["beta1"]
            s["c1"], s["c2"] = s["c2"], s["c1"]
        elif kind == "decay_sign":
            s["decay"] = np.float32(1.0 + hp["lr"] * hp["weight_decay"])
        elif kind == "eps_dropped":
            s["eps"] = np.float32(0.0)
        elif kind == "t_off_by_one":
            return real(hp, t + 1)
        return s
    return mutated


@pytest.mark.parametrize("kind", ["no_bias_correction", "betas_swapped", "decay_sign", "eps_dropped",
                                  "t_off_by_one"])
@pytest.mark.filterwarnings("ignore:invalid value encountered in divide:RuntimeWarning")   # eps_dropped: 0 / 0
def test_planted_adamw_mistakes_are_caught(kind, monkeypatch):
    monkeypatch.setattr(steps, "adamw_scalars", _mutant_scalars(kind))
    failures = 0
    for pin in pins.ALL_ADAMW_PINS:
        try:
            pin()
        except (AssertionError, FloatingPointError):
            failures += 1
    assert failures >= 1, kind


def test_planted_mean_mistakes_are_caught(monkeypatch):
    real = steps.reduce_mean
    # dividing by N_d - 1 + 1 only for N_d=1 is right; drop the division altogether
    monkeypatch.setattr(steps, "reduce_mean",
                        lambda rs: numerics.bf16_rne(sum(numerics.f32_from_bf16(r) for r in rs)))
    with pytest.raises(AssertionError):
        pins.pin_mean_of_equal_grads()
    # fold that skips the last rank
    monkeypatch.setattr(steps, "reduce_mean", lambda rs: real(rs[:-1]) if len(rs) > 1 else real(rs))
    with pytest.raises(AssertionError):
        pins.pin_mean_against_exact_rationals()


def test_planted_accumulation_mistakes_are_caught(monkeypatch):
    real = steps.accumulate
    monkeypatch.setattr(steps, "accumulate", lambda a, g, s, first: real(a, g, 1.0, first))
    with pytest.raises(AssertionError):
        pins.pin_accumulation_linear_model()
    monkeypatch.setattr(steps, "accumulate", lambda a, g, s, first: real(a, g, s, True))
    with pytest.raises(AssertionError):
        pins.pin_accumulation_four_equal_microbatches()
