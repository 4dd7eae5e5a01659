"""FSDP2 per-parameter Shard(0) layout (oracle; test infrastructure only).

"Infra: Data Parallel" (F. Pu), section "Fully Sharded Data Parallel (FSDP)",
FSDP2 layout figure and subsection "FSDP2": every parameter keeps its own
global shape and is cut along dimension 0 (Shard(0)), rank r keeping its rows;
a (8, 4) weight on 4 ranks leaves a local (2, 4) piece on each rank; three
(4, 2) weights on 2 ranks leave 12 elements per rank, two rows of each weight.
Parameters of one `fully_shard` group are still all-gathered and
reduce-scattered together.

Readings for what the pages leave open:
* uneven dimension 0: every rank gets ceil(d0 / N_d) rows, the last ranks
  fewer or none; their missing rows are zero padding, so every rank's piece of
  a parameter has ceil(d0 / N_d) rows and all ranks' shards are equally long;
* a 0-dimensional parameter is treated as one row of one element;
* grouped communication buffer: rank r's shard is the concatenation, in
  parameter order, of its (padded) pieces; the group's flat buffer is the
  ranks' shards one after another (rank-major), so a gather of the group is
  the same contiguous all-gather as FSDP1, and turning the gathered buffer back
  into the parameters' own layout is a permutation (copy_out);
* groups (units) are laid out one after another, as for FSDP1.
"""

from dataclasses import dataclass, field


def _dims(shape):
    shape = tuple(int(d) for d in shape)
    if not shape:
        return 1, 1, ()
    d0 = shape[0]
    row = 1
    for d in shape[1:]:
        row *= d
    return d0, row, shape


@dataclass
class Param2:
    unit: int
    d0: int
    row: int           # elements per dim-0 row
    chunk: int         # rows per rank, ceil(d0 / n_d)
    off: int           # offset of this parameter's piece inside a rank's shard of its unit
    shape: tuple


@dataclass
class Unit2:
    base: int
    shard: int         # elements per rank (sum of chunk * row over the unit's parameters)
    numel: int         # real elements of the unit

    def padded(self, n_d):
        return n_d * self.shard


@dataclass
class Plan2:
    n_d: int
    params: list = field(default_factory=list)
    units: list = field(default_factory=list)

    @property
    def padded(self):
        return sum(u.padded(self.n_d) for u in self.units)


def make_plan(shapes, n_d, unit_of_param=None):
    n = len(shapes)
    unit_of_param = list(unit_of_param) if unit_of_param is not None else [0] * n
    n_units = max(unit_of_param) + 1 if n else 0
    plan = Plan2(n_d=n_d, params=[None] * n)
    base = 0
    for u in range(n_units):
        off = 0
        numel = 0
        for k in range(n):
            if unit_of_param[k] != u:
                continue
            d0, row, shape = _dims(shapes[k])
            chunk = -(-d0 // n_d)
            plan.params[k] = Param2(unit=u, d0=d0, row=row, chunk=chunk, off=off, shape=shape)
            off += chunk * row
            numel += d0 * row
        plan.units.append(Unit2(base=base, shard=off, numel=numel))
        base += n_d * off
    return plan


def local_rows(plan, k, rank):
    """Rows [begin, begin + count) of parameter k that `rank` holds (count may be 0)."""
    p = plan.params[k]
    begin = min(rank * p.chunk, p.d0)
    end = min((rank + 1) * p.chunk, p.d0)
    return begin, end - begin


def local_shape(plan, k, rank):
    p = plan.params[k]
    _, count = local_rows(plan, k, rank)
    return (count,) + tuple(p.shape[1:]) if p.shape else ((1,) if count else (0,))


def flat_index(plan, k, i, j):
    """Global flat index of element (row i, column j) of parameter k."""
    p = plan.params[k]
    u = plan.units[p.unit]
    r = i // p.chunk
    return u.base + r * u.shard + p.off + (i - r * p.chunk) * p.row + j


def chunk_cat(plan, unit, values):
    """One rank's values of a unit's parameters (each flattened, natural layout) -> the unit's
    flat buffer (rank-major, padding rows zero)."""
    import numpy as np

    u = plan.units[unit]
    members = [k for k, p in enumerate(plan.params) if p.unit == unit]
    out = np.zeros(plan.n_d * u.shard, dtype=np.asarray(values[members[0]]).dtype)
    for k in members:
        p = plan.params[k]
        flat = np.asarray(values[k]).reshape(-1)
        for i in range(p.d0):
            r = i // p.chunk
            dst = r * u.shard + p.off + (i - r * p.chunk) * p.row
            out[dst:dst + p.row] = flat[i * p.row:(i + 1) * p.row]
    return out


def copy_out(plan, unit, flat):
    """The unit's flat buffer (rank-major) -> each parameter's values in natural layout (flattened)."""
    import numpy as np

    u = plan.units[unit]
    out = {}
    for k, p in enumerate(plan.params):
        if p.unit != unit:
            continue
        vals = np.zeros(p.d0 * p.row, dtype=np.asarray(flat).dtype)
        for i in range(p.d0):
            r = i // p.chunk
            src = r * u.shard + p.off + (i - r * p.chunk) * p.row
            vals[i * p.row:(i + 1) * p.row] = flat[src:src + p.row]
        out[k] = vals
    return out
