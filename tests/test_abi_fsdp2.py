"""FSDP2 planner through the C ABI against the oracle (runs without a GPU)."""

import random

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
from oracle import fsdp2


def _check(shapes, n_d, units=None):
    ours = zs.Plan(shapes, n_d, unit_of_param=units, layout=zs.ZS_LAYOUT_FSDP2)
    ref = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
    assert ours.layout() == zs.ZS_LAYOUT_FSDP2
    assert ours.padded == ref.padded
    for u, ru in enumerate(ref.units):
        d = ours.unit(u)
        assert (d["base"], d["shard"], d["padded"], d["numel"]) == (ru.base, ru.shard, ru.padded(n_d), ru.numel)
    pads = []
    for k, p in enumerate(ref.params):
        for r in range(n_d):
            b, n = fsdp2.local_rows(ref, k, r)
            rows = ours.param_rows(k, r)
            assert (rows["row_begin"], rows["nrows"], rows["rows_per_rank"], rows["row_elems"]) == (b, n, p.chunk, p.row)
            seg = ours.param_segment(k, r)
            if n:
                assert seg == (fsdp2.flat_index(ref, k, b, 0), p.off, n * p.row)
            else:
                assert seg[2] == 0
    # padding: every flat index of the plan that no parameter element maps to
    real = {fsdp2.flat_index(ref, k, i, j) for k, p in enumerate(ref.params) for i in range(p.d0) for j in range(p.row)}
    want = [i for i in range(ref.padded) if i not in real]
    got = [i for b, e in ours.pad_ranges() for i in range(b, e)]
    assert got == want
    return ours


def test_pages_examples():
    p = _check([(8, 4)], 4)
    assert all(p.param_rows(0, r)["nrows"] == 2 for r in range(4)) and p.shard_per_rank == 8
    p = _check([(4, 2)] * 3, 2)
    assert p.shard_per_rank == 12


def test_random_models():
    rng = random.Random(8)
    for _ in range(120):
        n = rng.randint(1, 5)
        shapes = [tuple(rng.randint(1, 7) for _ in range(rng.randint(0, 3))) for _ in range(n)]
        units = None
        if rng.random() < 0.5:
            units = sorted(rng.randint(0, 2) for _ in range(n))
            remap = {u: i for i, u in enumerate(sorted(set(units)))}
            units = [remap[u] for u in units]
        _check(shapes, rng.randint(1, 9), units)


def test_memory_accounting_counts_the_padded_rows():
    p = zs.Plan([(10, 3), (7,)], 4, layout=zs.ZS_LAYOUT_FSDP2)
    # c = 3 rows of 3 and 2 rows of 1 per rank: S = 11 per rank
    assert p.shard_per_rank == 11
    assert p.memory_bytes(3) == 16 * 11
    assert p.comm_bytes(1) == 2 * 2 * 3 * 11
