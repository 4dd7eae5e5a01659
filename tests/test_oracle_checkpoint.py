"""Pins for the oracle's sharded checkpoint (runs without a GPU).

A checkpoint must preserve every parameter and optimizer value across save and
load with any rank count ("Infra: Data Parallel", subsection "Checkpoint"):
checked by building each parameter as its own array, sharding, saving, loading
with other rank counts, and reading each parameter back through its per-rank
views; plus the FSDP1 worked example of the layout figure with concrete values.
"""

import random

import numpy as np
import pytest

from oracle import checkpoint, layout


def _shard_params(plan, params):
    """Rank-local shards of per-parameter arrays, built element by element from the param views."""
    offs, acc = [], 0
    for u in plan.units:
        offs.append(acc)
        acc += u.shard
    out = [np.zeros(plan.shard_total, dtype=np.float32) for _ in range(plan.n_d)]
    for k, p in enumerate(params):
        ui = plan.param_unit[k]
        flat = p.reshape(-1)
        pos = 0
        for r in range(plan.n_d):
            begin, shard_off, length = layout.param_segment(plan, k, r)
            if length:
                assert begin - plan.param_offset[k] == pos
                out[r][offs[ui] + shard_off:offs[ui] + shard_off + length] = flat[pos:pos + length]
                pos += length
        assert pos == flat.size
    return out


def test_fsdp1_example_values_resharded():
    shapes = [(4, 2)] * 3
    params = [np.arange(8 * k, 8 * k + 8, dtype=np.float32).reshape(4, 2) for k in range(3)]
    p2 = layout.make_plan(shapes, 2)
    shards = _shard_params(p2, params)
    assert list(shards[0]) == list(range(12)) and list(shards[1]) == list(range(12, 24))
    saved = checkpoint.save(p2, [{"master": s} for s in shards])
    p4 = layout.make_plan(shapes, 4)
    got = checkpoint.load(p4, saved, "master")
    assert [list(g) for g in got] == [list(range(6 * r, 6 * r + 6)) for r in range(4)]
    p5 = layout.make_plan(shapes, 5)                          # 24 -> padded to 25
    got5 = checkpoint.load(p5, saved, "master")
    assert list(got5[4]) == [20, 21, 22, 23, 0]


def test_random_models_survive_any_chain_of_rank_counts():
    rng = random.Random(2)
    for _ in range(60):
        n = rng.randint(1, 6)
        shapes = [tuple(rng.randint(1, 5) for _ in range(rng.randint(1, 2))) for _ in range(n)]
        units = sorted(rng.randint(0, 2) for _ in range(n))
        remap = {u: i for i, u in enumerate(sorted(set(units)))}
        units = [remap[u] for u in units]
        params = [np.asarray(np.random.default_rng(rng.randint(0, 10 ** 6)).standard_normal(s), np.float32)
                  for s in shapes]
        chain = [rng.randint(1, 9) for _ in range(4)]
        plan = layout.make_plan(shapes, chain[0], unit_of_param=units)
        shards = _shard_params(plan, params)
        for n_d in chain[1:]:
            saved = checkpoint.save(plan, [{"master": s, "m": 2 * s} for s in shards])
            plan = layout.make_plan(shapes, n_d, unit_of_param=units)
            shards = checkpoint.load(plan, saved, "master")
            twice = checkpoint.load(plan, saved, "m")
            for r in range(n_d):
                assert np.array_equal(twice[r], 2 * shards[r])
            for k, p in enumerate(params):
                assert np.array_equal(checkpoint.param_values(plan, [{"x": s} for s in shards], k, "x"),
                                      p.reshape(-1))
            # padding is zero in the new layout
            offs = np.cumsum([0] + [u.shard for u in plan.units])
            for ui, u in enumerate(plan.units):
                full = np.concatenate([shards[r][offs[ui]:offs[ui] + u.shard] for r in range(n_d)])
                assert not full[u.numel:].any()


def test_load_rejects_another_model():
    p = layout.make_plan([(4,), (6,)], 2)
    saved = checkpoint.save(p, [{"master": np.zeros(p.shard_total, np.float32)} for _ in range(2)])
    with pytest.raises(ValueError):
        checkpoint.load(layout.make_plan([(4,), (7,)], 2), saved, "master")


def _fsdp2_shards(plan2, params):
    from oracle import fsdp2
    out = [[] for _ in range(plan2.n_d)]
    for ui, u in enumerate(plan2.units):
        flat = fsdp2.chunk_cat(plan2, ui, [p.reshape(-1) for p in params])
        for r in range(plan2.n_d):
            out[r].append(flat[r * u.shard:(r + 1) * u.shard])
    return [np.concatenate(x) for x in out]


def test_any_layout_to_any_layout():
    """Save in FSDP1 or FSDP2 with one rank count and unit grouping, load into the other layout with
    another rank count and grouping: every parameter reads back unchanged, padding is zero."""
    from oracle import fsdp2

    rng = random.Random(9)
    for _ in range(40):
        n = rng.randint(1, 6)
        shapes = [tuple(rng.randint(1, 6) for _ in range(rng.randint(1, 3))) for _ in range(n)]
        params = [np.random.default_rng(rng.randint(0, 10 ** 6)).standard_normal(s).astype(np.float32) + 3
                  for s in shapes]
        state = None
        for step in range(4):
            kind = rng.choice(["fsdp1", "fsdp2"])
            n_d = rng.randint(1, 7)
            units = sorted(rng.randint(0, 2) for _ in range(n))
            remap = {u: i for i, u in enumerate(sorted(set(units)))}
            units = [remap[u] for u in units]
            plan = layout.make_plan(shapes, n_d, unit_of_param=units) if kind == "fsdp1" else \
                fsdp2.make_plan(shapes, n_d, unit_of_param=units)
            if state is None:
                shards = _shard_params(plan, params) if kind == "fsdp1" else _fsdp2_shards(plan, params)
            else:
                shards = checkpoint.load_any(state, plan, kind, "x", n)
            for k, p in enumerate(params):
                saved_now = checkpoint.save_any(plan, kind, [{"x": s} for s in shards])
                assert np.array_equal(checkpoint.param_values_any(saved_now, k, "x"), p.reshape(-1))
            total = sum(s.size for s in shards)
            assert total == plan.padded
            assert np.count_nonzero(np.concatenate(shards)) == sum(p.size for p in params)   # padding is zero
            state = checkpoint.save_any(plan, kind, [{"x": s} for s in shards])
