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


# ---------------------------------------------------------------- any layout to any layout
# An element is identified by (parameter, position in the parameter's own row-major order),
# which neither the rank count, the unit grouping nor the layout changes.  Saving keeps each
# rank's shard of its layout; loading reads every parameter back element by element and lays it
# out for the target plan.

def save_any(plan, kind, rank_shards):
    """kind: "fsdp1" (a layout.Plan) or "fsdp2" (an fsdp2.Plan2); rank_shards[r][name] rank-local."""
    return {"kind": kind, "plan": plan, "ranks": [{k: np.array(v, copy=True) for k, v in rank_shards[r].items()}
                                                  for r in range(plan.n_d)]}


def param_values_any(saved, k, name):
    """Parameter k's values (row-major) from a save of either layout."""
    from . import fsdp2

    plan, ranks = saved["plan"], saved["ranks"]
    if saved["kind"] == "fsdp1":
        return param_values(plan, ranks, k, name)
    p = plan.params[k]
    offs, acc = [], 0
    for u in plan.units:
        offs.append(acc)
        acc += u.shard
    rows = []
    for r in range(plan.n_d):
        begin, count = fsdp2.local_rows(plan, k, r)
        if count:
            start = offs[p.unit] + p.off
            rows.append(ranks[r][name][start:start + count * p.row])
    return np.concatenate(rows)


def load_any(saved, plan, kind, name, n_params):
    """Rank-local shards of `name` for `plan` (kind "fsdp1" or "fsdp2") from a save of either layout."""
    from . import fsdp2

    values = [param_values_any(saved, k, name) for k in range(n_params)]
    full = []
    for ui in range(len(plan.units)):
        if kind == "fsdp2":
            full.append(fsdp2.chunk_cat(plan, ui, values))
        else:
            u = plan.units[ui]
            flat = np.zeros(u.padded, dtype=values[0].dtype)
            for k in range(n_params):
                if plan.param_unit[k] == ui:
                    off = plan.param_offset[k] - u.base
                    flat[off:off + values[k].size] = values[k]
            full.append(flat)
    out = []
    for r in range(plan.n_d):
        pieces = []
        for ui, u in enumerate(plan.units):
            shard = u.shard
            pieces.append(full[ui][r * shard:(r + 1) * shard])
        out.append(np.concatenate(pieces))
    return out
