"""Sharded checkpoint save and load with a different rank count (oracle; test infrastructure only).

"Infra: Data Parallel" (F. Pu), section "Fully Sharded Data Parallel (FSDP)",
subsection "Checkpoint": every rank writes the shards it owns together with
the metadata needed to restore them; loading reads according to the target
run's sharding layout, so the number of ranks may differ between save and
load; optimizer state is saved alongside the weights.  The subsection says
FSDP1's flat layout supports this too.

With FSDP1 shards are contiguous pieces of each unit's padded FlatParameter,
so what identifies an element across layouts is its position among the unit's
real elements.  Saving keeps each rank's pieces; loading concatenates the
saved pieces of a unit, drops the old padding, appends the new padding (zeros)
and cuts the result for the new ranks.
"""

import numpy as np

from . import layout


def save(plan, rank_shards):
    """rank_shards[r][name] is rank r's shard array (rank-local, all units concatenated).

    Returns the saved form: {"n_d", "units": [(numel, padded, shard)], "ranks": [{name: array}]}.
    """
    return {
        "n_d": plan.n_d,
        "units": [(u.numel, u.padded, u.shard) for u in plan.units],
        "ranks": [{k: np.array(v, copy=True) for k, v in rank_shards[r].items()} for r in range(plan.n_d)],
    }


def unit_real_elements(saved, unit, name):
    """The real (unpadded) elements of one unit of one saved array, in flat order."""
    offs, acc = [], 0
    for (_, _, shard) in saved["units"]:
        offs.append(acc)
        acc += shard
    numel, padded, shard = saved["units"][unit]
    pieces = [saved["ranks"][r][name][offs[unit]:offs[unit] + shard] for r in range(saved["n_d"])]
    return np.concatenate(pieces)[:numel]


def load(plan, saved, name):
    """Rank-local shard arrays of `name` for the ranks of `plan` (same model, any rank count)."""
    if [u.numel for u in plan.units] != [u[0] for u in saved["units"]]:
        raise ValueError("the checkpoint was saved for a different model")
    out = []
    for r in range(plan.n_d):
        pieces = []
        for ui, u in enumerate(plan.units):
            real = unit_real_elements(saved, ui, name)
            padded = np.zeros(u.padded, dtype=real.dtype)
            padded[:u.numel] = real
            pieces.append(padded[r * u.shard:(r + 1) * u.shard])
        out.append(np.concatenate(pieces))
    return out


def param_values(plan, rank_shards, k, name):
    """All elements of parameter k gathered from the ranks' views (use_orig_params style)."""
    vals = []
    offs = []
    acc = 0
    for u in plan.units:
        offs.append(acc)
        acc += u.shard
    for r in range(plan.n_d):
        begin, shard_off, length = layout.param_segment(plan, k, r)
        if length:
            ui = plan.param_unit[k]
            vals.append(rank_shards[r][name][offs[ui] + shard_off:offs[ui] + shard_off + length])
    return np.concatenate(vals) if vals else np.zeros(0)
