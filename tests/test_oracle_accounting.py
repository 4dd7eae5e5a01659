"""Pins for the oracle's memory and communication accounting (runs without a GPU).

The oracle counts buffers and transferred element ranges; these tests hold
the counts to the formulas printed in "Infra: Data Parallel", section
"Zero Redundancy Optimizer (ZeRO)" (memory figure; communication paragraphs
and flow-figure captions), read from the golden files.
"""

import os
import random
from fractions import Fraction

import pytest

from oracle import accounting, layout


def _read_formulas(golden_dir, name):
    consts, rows = {}, {}
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" not in line:
                key, val = line.split()
                consts[key] = int(val)
                continue
            head, expr = line.split(":", 1)
            stage = int(head.split()[0])
            rows[stage] = [e.strip() for e in expr.split(";")]
    return consts, rows


def _eval(expr, **names):
    env = {k: Fraction(v) for k, v in names.items()}
    return eval(expr, {"__builtins__": {}}, env)  # noqa: S307 - fixture expressions only


def _plans_divisible():
    rng = random.Random(1)
    out = []
    for _ in range(40):
        n_d = rng.choice([1, 2, 4, 8, 16])
        shapes = [(rng.randint(1, 40) * n_d,) for _ in range(rng.randint(1, 5))]
        out.append(layout.make_plan(shapes, n_d, bucket_bytes=2 * rng.randint(1, 100)))
    # the figure's own setting, N_d = 4, and the FSDP1 example
    out.append(layout.make_plan([(4, 2)] * 3, 4))
    return out


def test_memory_matches_figure_when_no_padding(golden_dir):
    consts, rows = _read_formulas(golden_dir, "zero_model_state_memory.txt")
    assert consts["k"] == 12 and consts["figure_n_d"] == 4
    for plan in _plans_divisible():
        assert plan.padded == plan.numel
        for stage, (expr,) in rows.items():
            want = _eval(expr, Psi=plan.numel, N_d=plan.n_d, k=consts["k"])
            for r in range(plan.n_d):
                assert accounting.memory_bytes(plan, stage, r) == want, (stage, plan.n_d)


def test_memory_with_padding_uses_padded_length(golden_dir):
    """With padding the sharded stages hold the padded FlatParameter (a reading:
    the figure leaves padding out); naive DP holds the unpadded model."""
    consts, rows = _read_formulas(golden_dir, "zero_model_state_memory.txt")
    plan = layout.make_plan([(2 ** 20 + 7,)], 8)
    assert plan.padded == 2 ** 20 + 8
    assert accounting.memory_bytes(plan, 0) == _eval(rows[0][0], Psi=plan.numel, N_d=8, k=12)
    for stage in (1, 2, 3):
        assert accounting.memory_bytes(plan, stage) == _eval(rows[stage][0], Psi=plan.padded, N_d=8, k=12)


def test_memory_ordering_and_zero3_scaling():
    plan = layout.make_plan([(4096,)] * 3, 8)
    b = [accounting.memory_bytes(plan, s) for s in range(4)]
    assert b[0] > b[1] > b[2] > b[3]
    assert b[3] * 8 == b[0]          # ZeRO-3 divides every model state by N_d


def test_comm_volume_matches_ring_model(golden_dir):
    _, rows = _read_formulas(golden_dir, "comm_volume_per_rank.txt")
    for plan in _plans_divisible():
        for stage, (expr, factor) in rows.items():
            want = _eval(expr, Psi=plan.numel) * _eval(factor, N_d=plan.n_d)
            for r in range(plan.n_d):
                assert accounting.comm_bytes_sent(plan, stage, r) == want, (stage, plan.n_d)


def test_comm_volume_summed_over_layers_and_buckets(golden_dir):
    """'One pass' sums every bucket or layer: splitting into buckets or units changes nothing."""
    _, rows = _read_formulas(golden_dir, "comm_volume_per_rank.txt")
    shapes = [(64,), (128,), (32,), (256,)]
    for bucket in (2, 30, 1000):
        for units in (None, [0, 1, 2, 3], [0, 0, 1, 1]):
            plan = layout.make_plan(shapes, 4, unit_of_param=units, bucket_bytes=bucket)
            for stage in (1, 2, 3):
                want = _eval(rows[stage][0], Psi=480) * Fraction(3, 4)
                assert accounting.comm_bytes_sent(plan, stage, 1) == want


def test_comm_reshard_after_forward_false_saves_one_gather():
    """reshard_after_forward=False keeps the gathered parameters into backward: one All-Gather fewer (4 Psi)."""
    plan = layout.make_plan([(1024,)], 8)
    assert accounting.comm_bytes_sent(plan, 3, 0, reshard_after_forward=False) == Fraction(4 * 1024 * 7, 8)


@pytest.mark.parametrize("n_d", [2, 3, 5, 8])
def test_comm_with_padding_uses_padded_length(n_d):
    plan = layout.make_plan([(1001,)], n_d)
    for stage, mult in ((0, 4), (1, 4), (2, 4), (3, 6)):
        assert accounting.comm_bytes_sent(plan, stage, 0) == mult * (plan.padded - plan.units[0].shard)
