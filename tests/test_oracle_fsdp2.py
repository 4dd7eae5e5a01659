"""Pins for the oracle's FSDP2 Shard(0) layout (runs without a GPU).

The two worked examples of the FSDP2 layout figure (golden file), brute force
over every element of random models against an independent row-dealing
construction, the round trip chunk_cat / copy_out, and the contrast with FSDP1
(FSDP1's cut runs through W2, FSDP2 keeps half of every weight on each rank).
"""

import os
import random

import numpy as np

from oracle import fsdp2, layout, numerics, steps


def _read_cases(golden_dir):
    cases, cur = [], None
    with open(os.path.join(golden_dir, "fsdp2_shard0_examples.txt")) as f:
        for line in f:
            tok = line.split()
            if not tok or tok[0].startswith("#"):
                continue
            if tok[0] == "case":
                cur = {"name": tok[1], "n_d": int(tok[3]), "params": [], "local": [], "rank_elems": []}
                cases.append(cur)
            elif tok[0] == "param":
                cur["params"].append((tok[1], tuple(int(x) for x in tok[2:])))
            elif tok[0] == "local":
                cur["local"].append((tok[1], int(tok[2]), tuple(int(x) for x in tok[3:])))
            elif tok[0] == "rank_elems":
                cur["rank_elems"].append((int(tok[1]), int(tok[2])))
    return cases


def test_pages_examples(golden_dir):
    for case in _read_cases(golden_dir):
        names = [n for n, _ in case["params"]]
        plan = fsdp2.make_plan([s for _, s in case["params"]], case["n_d"])
        for name, rank, shape in case["local"]:
            assert fsdp2.local_shape(plan, names.index(name), rank) == shape, (case["name"], name, rank)
        for rank, n in case["rank_elems"]:
            assert plan.units[0].shard == n
        for k, (_, shape) in enumerate(case["params"]):
            assert plan.params[k].shape == shape              # the global shape is kept


def test_fsdp1_and_fsdp2_cut_differently():
    shapes = [(4, 2)] * 3
    p1 = layout.make_plan(shapes, 2)
    p2 = fsdp2.make_plan(shapes, 2)
    # FSDP1: W2 is split between the ranks, W1 and W3 are whole on one rank each
    assert layout.param_segment(p1, 0, 1)[2] == 0 and layout.param_segment(p1, 2, 0)[2] == 0
    # FSDP2: every rank has rows of every weight
    for k in range(3):
        for r in range(2):
            assert fsdp2.local_rows(p2, k, r) == (2 * r, 2)


def _dealt(shapes, n_d, units):
    """Independent construction: deal each parameter's rows out to the ranks one by one."""
    owner_rows = {}
    for k, shape in enumerate(shapes):
        d0 = shape[0] if shape else 1
        per = -(-d0 // n_d)
        for i in range(d0):
            owner_rows[(k, i)] = (i // per, i % per)
    return owner_rows


def test_bruteforce_every_element_has_one_home():
    rng = random.Random(4)
    for _ in range(120):
        n = rng.randint(1, 5)
        shapes = [tuple(rng.randint(1, 7) for _ in range(rng.randint(0, 3))) for _ in range(n)]
        units = sorted(rng.randint(0, 2) for _ in range(n))
        remap = {u: i for i, u in enumerate(sorted(set(units)))}
        units = [remap[u] for u in units]
        n_d = rng.randint(1, 6)
        plan = fsdp2.make_plan(shapes, n_d, unit_of_param=units)
        dealt = _dealt(shapes, n_d, units)
        seen = set()
        for k, shape in enumerate(shapes):
            p = plan.params[k]
            u = plan.units[p.unit]
            for i in range(p.d0):
                for j in range(p.row):
                    idx = fsdp2.flat_index(plan, k, i, j)
                    r, local_row = dealt[(k, i)]
                    assert u.base + r * u.shard <= idx < u.base + (r + 1) * u.shard   # inside rank r's shard
                    assert idx not in seen
                    seen.add(idx)
            # every rank's piece of the parameter has the same number of rows (padding included)
            assert sum(p.chunk * p.row for _ in range(n_d)) >= p.d0 * p.row
        assert len(seen) == sum(u.numel for u in plan.units)
        # round trip through the grouped flat buffer; padding is zero
        vals = [np.random.default_rng(k).standard_normal(int(np.prod(s)) if s else 1).astype(np.float32) + 10
                for k, s in enumerate(shapes)]
        for ui in range(len(plan.units)):
            flat = fsdp2.chunk_cat(plan, ui, vals)
            back = fsdp2.copy_out(plan, ui, flat)
            for k, v in back.items():
                assert np.array_equal(v, vals[k])
            pos = {fsdp2.flat_index(plan, k, i, j) - plan.units[ui].base
                   for k, p in enumerate(plan.params) if p.unit == ui for i in range(p.d0) for j in range(p.row)}
            pad = [x for x in range(len(flat)) if x not in pos]
            assert not flat[pad].any()


def test_update_commutes_with_the_layout():
    """AdamW is element-wise: updating the FSDP2 flat buffer and copying out equals updating each
    parameter in its own layout."""
    shapes = [(7, 3), (5,), (2, 2, 2)]
    plan = fsdp2.make_plan(shapes, 3)
    rng = np.random.default_rng(0)
    p0 = [(rng.standard_normal(int(np.prod(s))) * 0.02).astype(np.float32) for s in shapes]
    g = [steps.reduce_mean([numerics.bf16_rne((rng.standard_normal(int(np.prod(s))) * 1e-3).astype(np.float32))
                            for _ in range(3)]) for s in shapes]
    hp = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}
    flat_p = fsdp2.chunk_cat(plan, 0, p0)
    flat_g = fsdp2.chunk_cat(plan, 0, g)
    z = np.zeros_like(flat_p)
    new_flat, _, _, _ = steps.adamw(flat_p, z, z, flat_g, hp, 1)
    back = fsdp2.copy_out(plan, 0, new_flat)
    for k in range(3):
        zk = np.zeros_like(p0[k])
        want, _, _, _ = steps.adamw(p0[k], zk, zk, g[k], hp, 1)
        assert np.array_equal(back[k], want)
