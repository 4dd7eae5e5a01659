"""Pins for the oracle's FlatParameter layout (runs without a GPU).

* the FSDP1 worked example printed on "Infra: Data Parallel" (FSDP1 layout figure);
* brute force over every tiny plan against a set-based construction that
  deals elements out one by one (no offset arithmetic shared with the oracle);
* partition invariants of shards and buckets.
"""

import itertools
import os
import random

import pytest

from oracle import layout


def _read_fsdp1(golden_dir):
    spec = {"params": [], "segs": []}
    with open(os.path.join(golden_dir, "fsdp1_flatparameter_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            if tok[0] == "n_d":
                spec["n_d"] = int(tok[1])
            elif tok[0] == "param":
                spec["params"].append((tok[1], tuple(int(x) for x in tok[2:])))
            elif tok[0] == "total":
                spec["total"] = int(tok[1])
            elif tok[0] == "shard":
                spec["shard"] = int(tok[1])
            elif tok[0] == "seg":
                spec["segs"].append((tok[1], int(tok[2]), int(tok[3]), int(tok[4]), int(tok[5])))
    return spec


def test_fsdp1_worked_example(golden_dir):
    spec = _read_fsdp1(golden_dir)
    names = [n for n, _ in spec["params"]]
    plan = layout.make_plan([s for _, s in spec["params"]], spec["n_d"])
    assert plan.numel == spec["total"]
    assert plan.padded == spec["total"]            # 24 is already a multiple of 2
    assert plan.units[0].shard == spec["shard"]
    for name, rank, begin, off, length in spec["segs"]:
        got = layout.param_segment(plan, names.index(name), rank)
        if length == 0:
            assert got[2] == 0, (name, rank, got)
        else:
            assert got == (begin, off, length), (name, rank, got)
    # the cut runs through W2: both ranks hold a non-empty part of it
    w2 = names.index("W2")
    assert all(layout.param_segment(plan, w2, r)[2] > 0 for r in range(2))


# ---------------------------------------------------------------- brute force

def _dealt_layout(numels, n_d):
    """Independent construction: walk the elements one by one.

    Returns (padded, owner_of_flat_index list, param_of_flat_index list)
    where padding elements have param -1.
    """
    elems = []
    for k, n in enumerate(numels):
        for _ in range(n):
            elems.append(k)
    while len(elems) % n_d:                      # append padding until the ranks can share evenly
        elems.append(-1)
    per_rank = len(elems) // n_d
    owner = []
    rank, filled = 0, 0
    for _ in elems:                              # fill rank 0, then rank 1, ...
        if filled == per_rank:
            rank, filled = rank + 1, 0
        owner.append(rank)
        filled += 1
    return len(elems), owner, elems


def _check_plan_against_dealing(numels, n_d, bucket_elems):
    shapes = [(n,) for n in numels]
    plan = layout.make_plan(shapes, n_d, bucket_bytes=2 * bucket_elems)
    padded, owner, param_of = _dealt_layout(numels, n_d)
    assert plan.padded == padded
    assert plan.numel == sum(numels)
    assert layout.pad_ranges(plan) == ([(sum(numels), padded)] if padded > sum(numels) else [])
    for i in range(padded):
        assert layout.owner(plan, i) == (0, owner[i])
    # segments: the set of flat indices of param k held by rank r
    for k in range(len(numels)):
        for r in range(n_d):
            want = [i for i in range(padded) if param_of[i] == k and owner[i] == r]
            begin, off, length = layout.param_segment(plan, k, r)
            if not want:
                assert length == 0
                continue
            assert list(range(begin, begin + length)) == want
            first_of_rank = owner.index(r)
            assert off == begin - first_of_rank
    # buckets: contiguous, in order, cover [0, padded) exactly once, each at most bucket_elems long
    covered = []
    for (_, lo, hi) in plan.buckets:
        assert 0 < hi - lo <= bucket_elems
        covered.extend(range(lo, hi))
    assert covered == list(range(padded))
    assert all(hi - lo == bucket_elems for (_, lo, hi) in plan.buckets[:-1])
    # each bucket hands every rank exactly the bucket elements that rank owns
    for b, (_, lo, hi) in enumerate(plan.buckets):
        for r in range(n_d):
            s_lo, s_hi = layout.bucket_rank_slice(plan, b, r)
            want = [i for i in range(lo, hi) if owner[i] == r]
            assert list(range(s_lo, s_hi)) == want


def test_bruteforce_every_tiny_plan():
    """All splits of up to 3 params with sizes 1..5, every N_d 1..8, several bucket sizes."""
    count = 0
    for n_params in (1, 2, 3):
        for numels in itertools.product(range(1, 6), repeat=n_params):
            for n_d in range(1, 9):
                for bucket in (1, 3, 8, 64):
                    _check_plan_against_dealing(list(numels), n_d, bucket)
                    count += 1
    assert count > 1000


def test_bruteforce_random_plans_up_to_64():
    rng = random.Random(7)
    for _ in range(300):
        n_params = rng.randint(1, 4)
        numels = [rng.randint(1, 16) for _ in range(n_params)]
        n_d = rng.randint(1, 8)
        bucket = rng.randint(1, 70)
        _check_plan_against_dealing(numels, n_d, bucket)


def test_units_are_padded_and_sharded_separately():
    """Per-unit FlatParameters: each unit is its own padded buffer, laid out one after the other."""
    rng = random.Random(11)
    for _ in range(200):
        n_params = rng.randint(1, 6)
        numels = [rng.randint(1, 9) for _ in range(n_params)]
        units = sorted(rng.randint(0, 2) for _ in range(n_params))
        # unit ids must be 0..U-1 without gaps
        remap = {u: i for i, u in enumerate(sorted(set(units)))}
        units = [remap[u] for u in units]
        n_d = rng.randint(1, 5)
        plan = layout.make_plan([(n,) for n in numels], n_d, unit_of_param=units)
        base = 0
        for ui, u in enumerate(plan.units):
            members = [k for k in range(n_params) if units[k] == ui]
            sub = [numels[k] for k in members]
            padded, owner, _ = _dealt_layout(sub, n_d)
            assert u.base == base and u.padded == padded and u.numel == sum(sub)
            for j in range(padded):
                assert layout.owner(plan, base + j) == (ui, owner[j])
            # buckets never cross units
            for (bu, lo, hi) in plan.buckets:
                if bu == ui:
                    assert base <= lo < hi <= base + padded
            base += padded
        assert plan.padded == base


@pytest.mark.parametrize("n_d", [1, 2, 3, 4, 8])
def test_shards_partition_and_are_equal(n_d):
    plan = layout.make_plan([(5, 3), (7,), (2, 2, 2)], n_d)
    seen = []
    for r in range(n_d):
        lo, hi = layout.shard_range(plan, 0, r)
        assert hi - lo == plan.units[0].shard
        seen.extend(range(lo, hi))
    assert seen == list(range(plan.padded))
