"""Model-state memory and communication volume per rank, by counting (oracle; test infrastructure only).

"Infra: Data Parallel" (F. Pu), section "Zero Redundancy Optimizer (ZeRO)":

* memory figure: per-GPU bytes of model states (parameters and gradients at
  2 bytes per element, optimizer state at k = 12 bytes per element; no
  activations, no temporary communication buffers).
* communication paragraphs: bytes each rank sends under the ring model,
  summed over every bucket or layer of one step.

The functions below do not evaluate those formulas.  They list the buffers a
rank holds under each stage and add up their sizes, and they walk the
simulated collectives element range by element range and count what leaves
each rank.  The tests compare the counts with the page's formulas.

Stages: 0 = naive DP (no sharding, no padding), 1 = ZeRO-1, 2 = ZeRO-2,
3 = ZeRO-3 / FSDP full shard.
"""

from . import layout

BF16 = 2
FP32 = 4
OPT_STATES = 3      # master, m, v


def held_buffers(plan, stage, rank):
    """(name, elements, bytes_per_element) of every model-state buffer ``rank`` holds."""
    shard = sum(u.shard for u in plan.units)       # the rank's piece of every unit
    if stage == 0:
        n = plan.numel
        return [("params", n, BF16), ("grads", n, BF16),
                ("master", n, FP32), ("m", n, FP32), ("v", n, FP32)]
    states = [("master", shard, FP32), ("m", shard, FP32), ("v", shard, FP32)]
    if stage == 1:
        return [("params", plan.padded, BF16), ("grads", plan.padded, BF16)] + states
    if stage == 2:
        return [("params", plan.padded, BF16), ("grad_shard", shard, BF16)] + states
    if stage == 3:
        return [("param_shard", shard, BF16), ("grad_shard", shard, BF16)] + states
    raise ValueError(stage)


def memory_bytes(plan, stage, rank=0):
    return sum(n * b for _, n, b in held_buffers(plan, stage, rank))


def _rs_sent(plan, rank):
    """Elements ``rank`` sends in one reduce-scatter over every bucket: the bucket elements it does not own."""
    sent = 0
    for b, (ui, lo, hi) in enumerate(plan.buckets):
        own_lo, own_hi = layout.bucket_rank_slice(plan, b, rank)
        sent += (hi - lo) - max(0, own_hi - own_lo)
    return sent


def _ag_sent(plan, rank):
    """Elements ``rank`` sends in one all-gather of every unit: its shard, once to every other rank."""
    sent = 0
    for ui in range(len(plan.units)):
        lo, hi = layout.shard_range(plan, ui, rank)
        for peer in range(plan.n_d):
            if peer != rank:
                sent += hi - lo
    return sent


def _ring_allreduce_sent(plan, rank):
    """Naive DP: a ring all-reduce per unit, simulated step by step.

    The unit's padded range is cut into N_d chunks; in each of the N_d - 1
    reduce-scatter steps and N_d - 1 all-gather steps every rank passes one
    chunk to its right neighbour.
    """
    n_d = plan.n_d
    sent = 0
    for u in plan.units:
        chunk = [u.shard] * n_d
        for step in range(n_d - 1):                 # reduce-scatter phase
            sent += chunk[(rank - step) % n_d]
        for step in range(n_d - 1):                 # all-gather phase
            sent += chunk[(rank + 1 - step) % n_d]
    return sent


def comm_bytes_sent(plan, stage, rank=0, reshard_after_forward=True):
    """Bytes ``rank`` sends during one step (16-bit elements)."""
    if stage == 0:
        return BF16 * _ring_allreduce_sent(plan, rank)
    if stage in (1, 2):
        return BF16 * (_rs_sent(plan, rank) + _ag_sent(plan, rank))
    if stage == 3:
        gathers = 2 if reshard_after_forward else 1
        return BF16 * (_rs_sent(plan, rank) + gathers * _ag_sent(plan, rank))
    raise ValueError(stage)
