"""FlatParameter layout: concatenate, pad, shard, bucket (oracle; test infrastructure only).

Follows "Infra: Data Parallel" (F. Pu):

* FSDP section, FSDP1 layout figure and "FSDP1: pack first, then shard": the
  parameters of one FSDP unit are flattened and concatenated in the given
  order into a one-dimensional FlatParameter, which is then cut into N_d
  equal contiguous pieces, one per rank.  A piece may cross parameter
  boundaries; a rank that got no element of a parameter sees an empty view.
* The figure leaves padding out; the plainest reading that makes the pieces
  equal is to append the fewest zero elements that make the length a
  multiple of N_d (padded length = ceil(numel / N_d) * N_d), per unit.
* Bucketing (section "Naive Data Parallelism"): gradients are communicated in
  buckets.  Here a bucket is a contiguous range of floor(bucket_bytes / 2)
  bf16 gradient elements of one unit's padded range, the last one shorter.
* Units (FSDP1 unit, e.g. one Transformer block): each unit is its own
  FlatParameter.  The global flat index space is the concatenation of the
  units' padded ranges in unit order, so unit u starts at ``unit_base[u]``.

Everything is computed with plain Python integers and explicit loops.
"""

from dataclasses import dataclass, field


def numel_of(shape):
    n = 1
    for d in shape:
        n *= int(d)
    return n


@dataclass
class Unit:
    params: list          # indices of the parameters in this unit, in flat order
    base: int             # global flat index of the unit's first element
    numel: int            # real elements
    padded: int           # padded elements (multiple of n_d)
    shard: int            # padded // n_d


@dataclass
class Plan:
    n_d: int
    shapes: list
    unit_of_param: list
    bucket_elems: int
    units: list = field(default_factory=list)
    param_unit: list = field(default_factory=list)
    param_offset: list = field(default_factory=list)   # global flat index of each param's first element
    param_numel: list = field(default_factory=list)
    buckets: list = field(default_factory=list)        # (unit, begin, end), global flat indices

    @property
    def numel(self):
        return sum(u.numel for u in self.units)

    @property
    def padded(self):
        return sum(u.padded for u in self.units)

    @property
    def shard_total(self):
        """Elements one rank owns, summed over units."""
        return sum(u.shard for u in self.units)


def make_plan(shapes, n_d, unit_of_param=None, bucket_bytes=None):
    """Build the FlatParameter plan.

    shapes        : list of parameter shapes, in module order.
    n_d           : number of data-parallel ranks (>= 1).
    unit_of_param : unit id of each parameter (ids 0..U-1, non-decreasing is
                    not required); None puts every parameter in unit 0.
    bucket_bytes  : gradient bucket size in bytes of bf16 gradients; None or
                    a size >= the unit gives one bucket per unit.
    """
    if n_d < 1:
        raise ValueError("n_d must be >= 1")
    n_params = len(shapes)
    if unit_of_param is None:
        unit_of_param = [0] * n_params
    n_units = (max(unit_of_param) + 1) if n_params else 0
    plan = Plan(n_d=n_d, shapes=[tuple(s) for s in shapes], unit_of_param=list(unit_of_param), bucket_elems=0)

    plan.param_unit = list(unit_of_param)
    plan.param_offset = [0] * n_params
    plan.param_numel = [numel_of(s) for s in shapes]

    base = 0
    for u in range(n_units):
        members = [k for k in range(n_params) if unit_of_param[k] == u]
        offset = base
        for k in members:
            plan.param_offset[k] = offset
            offset += plan.param_numel[k]
        real = offset - base
        # fewest zero elements that make the unit's length a multiple of n_d
        padded = real
        while padded % n_d != 0:
            padded += 1
        plan.units.append(Unit(params=members, base=base, numel=real, padded=padded, shard=padded // n_d))
        base += padded

    if bucket_bytes is None:
        bucket_elems = max([u.padded for u in plan.units] + [1])
    else:
        bucket_elems = bucket_bytes // 2
        if bucket_elems < 1:
            raise ValueError("bucket must hold at least one bf16 element")
    plan.bucket_elems = bucket_elems
    for ui, u in enumerate(plan.units):
        start = 0
        while start < u.padded:
            end = min(start + bucket_elems, u.padded)
            plan.buckets.append((ui, u.base + start, u.base + end))
            start = end
    return plan


def shard_range(plan, unit, rank):
    """Global flat range [begin, end) that ``rank`` owns in ``unit``."""
    u = plan.units[unit]
    return u.base + rank * u.shard, u.base + (rank + 1) * u.shard


def owner(plan, i):
    """(unit, rank) owning global flat index i."""
    for ui, u in enumerate(plan.units):
        if u.base <= i < u.base + u.padded:
            return ui, (i - u.base) // u.shard
    raise IndexError(i)


def pad_ranges(plan):
    """Global flat ranges [begin, end) that hold padding (zeros)."""
    out = []
    for u in plan.units:
        if u.padded > u.numel:
            out.append((u.base + u.numel, u.base + u.padded))
    return out


def param_segment(plan, k, rank):
    """The part of parameter k that ``rank`` holds, as (flat_begin, shard_offset, length).

    flat_begin is a global flat index, shard_offset the position inside the
    rank's shard of the parameter's unit.  A rank holding no element of the
    parameter gets length 0 (the empty view of "use_orig_params"), reported
    as (0, 0, 0).
    """
    u = plan.param_unit[k]
    lo = plan.param_offset[k]
    hi = lo + plan.param_numel[k]
    s_lo, s_hi = shard_range(plan, u, rank)
    a = max(lo, s_lo)
    b = min(hi, s_hi)
    if a >= b:
        return 0, 0, 0
    return a, a - s_lo, b - a


def bucket_rank_slice(plan, b, rank):
    """Global flat range [begin, end) of bucket b that rank receives in the reduce-scatter (may be empty)."""
    ui, lo, hi = plan.buckets[b]
    s_lo, s_hi = shard_range(plan, ui, rank)
    a = max(lo, s_lo)
    c = min(hi, s_hi)
    if a >= c:
        return a, a
    return a, c
