"""The steps of the sharded optimizer step, written out plainly (oracle; test infrastructure only).

Source: "Infra: Data Parallel" (F. Pu).

* Gradient accumulation (section "Naive Data Parallelism", paragraph on
  gradient accumulation and no_sync): micro-batch gradients are summed
  locally and synchronised only after the last one; with 4 equal micro-batches
  each loss is divided by 4 before backward, which (backward being linear)
  is each micro-batch gradient scaled by 1/4.
* ZeRO-1 (section "Zero Redundancy Optimizer (ZeRO)" and the ZeRO-1 flow
  figure): gradients are reduce-scattered with averaging so each rank gets the
  mean gradient of the part it owns; each rank runs AdamW on its own shard
  only (AdamW is element-wise, so a shard needs nothing else); the updated
  parameters are all-gathered so every rank holds the full model again.
* ZeRO-2 (same section, ZeRO-2 flow figure): the reduce-scatter happens
  bucket by bucket during backward and each rank keeps only the reduced
  slice it owns.  Values are the same as ZeRO-1.
* ZeRO-3 (same section, ZeRO-3 flow figure): parameters are sharded too; per
  unit, the full parameters are all-gathered before forward, freed, gathered
  again for backward, the gradients are reduce-scattered with averaging, and
  AdamW updates the local shard; there is no gather after the update.
* Naive DP (section "Naive Data Parallelism"): every rank all-reduces the
  gradients to their mean and runs the same update on a full replica.

The AdamW equations are not written on the pages (only its name, that it is
element-wise, and that master weights and both moments are fp32).  The reading
taken is the decoupled-weight-decay Adam of Loshchilov & Hutter with bias
correction, in the usual single-tensor form:

    p <- p * (1 - lr*wd)
    m <- beta1*m + (1-beta1)*g
    v <- beta2*v + (1-beta2)*g*g
    p <- p - (lr / (1-beta1^t)) * m / (sqrt(v)/sqrt(1-beta2^t) + eps)

with t the 1-based step.  The five step-dependent scalars are computed in
float64 from the fp32 hyper-parameters and then rounded to fp32; every
per-element operation below is one fp32 operation, rounded to nearest even,
with no fused multiply-add.  The reduced gradient is stored as bf16 (gradients
are 16-bit on the pages) and widened before the update.

Mean over ranks: fp32 sum of the ranks' gradients in ascending rank order,
starting from +0, divided by N_d, rounded to bf16.
"""

import math

import numpy as np

from . import layout
from .numerics import bf16_rne, f32_from_bf16

F32 = np.float32


# ---------------------------------------------------------------- element-wise pieces

def accumulate(acc_bits, micro_bits, scale, first):
    """One micro-batch into the local bf16 gradient buffer: acc <- bf16(acc + g*scale).

    ``first`` starts from +0 (the buffer holds nothing yet).
    """
    micro = f32_from_bf16(micro_bits)
    prev = np.zeros(micro.shape, dtype=F32) if first else f32_from_bf16(acc_bits)
    prod = micro * F32(scale)
    total = prev + prod
    return bf16_rne(total)


def reduce_mean(rank_slices):
    """Mean over ranks of the same slice: bf16( (sum_q fp32 g_q) / N_d ), ascending q."""
    n_d = len(rank_slices)
    total = np.zeros(np.asarray(rank_slices[0]).shape, dtype=F32)
    for q in range(n_d):
        total = total + f32_from_bf16(rank_slices[q])
    mean = total / F32(n_d)
    return bf16_rne(mean)


def adamw_scalars(hp, t):
    """Step-dependent AdamW scalars: float64 from the fp32 hyper-parameters, then fp32."""
    if t < 1:
        raise ValueError("step t is 1-based")
    lr = float(F32(hp["lr"]))
    b1 = float(F32(hp["beta1"]))
    b2 = float(F32(hp["beta2"]))
    eps = float(F32(hp["eps"]))
    wd = float(F32(hp["weight_decay"]))
    return {
        "beta1": F32(b1),
        "beta2": F32(b2),
        "eps": F32(eps),
        "decay": F32(1.0 - lr * wd),
        "c1": F32(1.0 - b1),
        "c2": F32(1.0 - b2),
        "step_size": F32(lr / (1.0 - math.pow(b1, t))),
        "sqrt_bc2": F32(math.sqrt(1.0 - math.pow(b2, t))),
    }


def adamw(master, m, v, grad_bits, hp, t):
    """Element-wise AdamW on fp32 state from a bf16 gradient.

    Returns new (master, m, v) as fp32 arrays and the bf16 parameter bits.
    Inputs are not modified.
    """
    s = adamw_scalars(hp, t)
    g = f32_from_bf16(grad_bits)
    p = np.asarray(master, dtype=F32) * s["decay"]
    m_new = s["beta1"] * np.asarray(m, dtype=F32) + s["c1"] * g
    gg = g * g
    v_new = s["beta2"] * np.asarray(v, dtype=F32) + s["c2"] * gg
    root = np.sqrt(v_new)
    denom = root / s["sqrt_bc2"] + s["eps"]
    ratio = m_new / denom
    p = p - s["step_size"] * ratio
    return p, m_new, v_new, bf16_rne(p)


# ---------------------------------------------------------------- rank-local shard coordinates

def unit_local_offsets(plan):
    """Position of each unit's piece inside one rank's shard array (length plan.shard_total)."""
    out, acc = [], 0
    for u in plan.units:
        out.append(acc)
        acc += u.shard
    return out


def shard_of(plan, rank, full):
    """Rank ``rank``'s shard (rank-local array) taken out of a full flat array."""
    pieces = []
    for ui in range(len(plan.units)):
        lo, hi = layout.shard_range(plan, ui, rank)
        pieces.append(np.asarray(full)[lo:hi])
    return np.concatenate(pieces) if pieces else np.zeros(0, dtype=np.asarray(full).dtype)


# ---------------------------------------------------------------- collectives on simulated ranks

def reduce_scatter_mean(plan, rank_grads, bucket_order=None):
    """Reduce-Scatter with averaging, bucket by bucket.

    rank_grads : list of N_d full local gradient buffers (bf16 bits, padded length).
    Returns the N_d rank-local reduced shards (bf16 bits, length plan.shard_total).
    Buckets are visited in ``bucket_order`` (default: descending, the order
    in which backward makes them ready); each bucket hands rank r the part of
    the bucket that lies in r's shard.
    """
    n_d = plan.n_d
    offs = unit_local_offsets(plan)
    out = [np.zeros(plan.shard_total, dtype=np.uint16) for _ in range(n_d)]
    order = list(range(len(plan.buckets)))[::-1] if bucket_order is None else bucket_order
    for b in order:
        ui = plan.buckets[b][0]
        for r in range(n_d):
            lo, hi = layout.bucket_rank_slice(plan, b, r)
            if hi <= lo:
                continue
            reduced = reduce_mean([np.asarray(rank_grads[q])[lo:hi] for q in range(n_d)])
            s_lo, _ = layout.shard_range(plan, ui, r)
            dst = offs[ui] + (lo - s_lo)
            out[r][dst:dst + (hi - lo)] = reduced
    return out


def all_gather(plan, rank_param_shards):
    """All-Gather: every rank gets the concatenation of all ranks' bf16 shards, per unit."""
    n_d = plan.n_d
    offs = unit_local_offsets(plan)
    full = np.zeros(plan.padded, dtype=np.uint16)
    for ui, u in enumerate(plan.units):
        for r in range(n_d):
            lo, hi = layout.shard_range(plan, ui, r)
            full[lo:hi] = rank_param_shards[r][offs[ui]:offs[ui] + u.shard]
    return [full.copy() for _ in range(n_d)]


def all_gather_unit(plan, unit, rank_param_shards):
    """ZeRO-3: gather one unit's full bf16 parameters on every rank (unit-local indexing)."""
    offs = unit_local_offsets(plan)
    u = plan.units[unit]
    full = np.zeros(u.padded, dtype=np.uint16)
    for r in range(plan.n_d):
        full[r * u.shard:(r + 1) * u.shard] = rank_param_shards[r][offs[unit]:offs[unit] + u.shard]
    return [full.copy() for _ in range(plan.n_d)]


# ---------------------------------------------------------------- whole steps

def zero_step(plan, rank_grads, rank_master, rank_m, rank_v, hp, t):
    """One ZeRO-1/2 optimizer step on simulated ranks.

    rank_grads              : N_d full local bf16 gradient buffers (after accumulation).
    rank_master/m/v         : N_d rank-local fp32 shard arrays.
    Returns (replicas, master, m, v): N_d full bf16 parameter replicas and the
    updated rank-local states.
    """
    reduced = reduce_scatter_mean(plan, rank_grads)
    new_master, new_m, new_v, shards = [], [], [], []
    for r in range(plan.n_d):
        p, m, v, bits = adamw(rank_master[r], rank_m[r], rank_v[r], reduced[r], hp, t)
        new_master.append(p)
        new_m.append(m)
        new_v.append(v)
        shards.append(bits)
    replicas = all_gather(plan, shards)
    return replicas, new_master, new_m, new_v


def zero3_unit_step(plan, unit, rank_param_shards, rank_layer_grads, rank_master, rank_m, rank_v, hp, t):
    """ZeRO-3 for one unit: gather for forward, gather again for backward, reduce-scatter, update.

    rank_param_shards : N_d rank-local bf16 shard arrays (length plan.shard_total).
    rank_layer_grads  : N_d unit-local full gradient buffers (length = unit's padded size),
                        the gradients each rank's backward produced for this unit.
    Returns (forward_full, backward_full, shards, master, m, v); only the
    unit's piece of the rank-local arrays changes.
    """
    offs = unit_local_offsets(plan)
    u = plan.units[unit]
    forward_full = all_gather_unit(plan, unit, rank_param_shards)    # then freed after forward
    backward_full = all_gather_unit(plan, unit, rank_param_shards)   # gathered again for backward
    shards, masters, ms, vs = [], [], [], []
    for r in range(plan.n_d):
        lo, hi = r * u.shard, (r + 1) * u.shard
        reduced = reduce_mean([np.asarray(rank_layer_grads[q])[lo:hi] for q in range(plan.n_d)])
        a, b = offs[unit], offs[unit] + u.shard
        p, m, v, bits = adamw(rank_master[r][a:b], rank_m[r][a:b], rank_v[r][a:b], reduced, hp, t)
        sh = np.array(rank_param_shards[r], copy=True)
        sh[a:b] = bits
        mm = np.array(rank_master[r], copy=True)
        mm[a:b] = p
        m1 = np.array(rank_m[r], copy=True)
        m1[a:b] = m
        v1 = np.array(rank_v[r], copy=True)
        v1[a:b] = v
        shards.append(sh)
        masters.append(mm)
        ms.append(m1)
        vs.append(v1)
    return forward_full, backward_full, shards, masters, ms, vs


def dp_step(rank_grads, master, m, v, hp, t):
    """Naive DP: all-reduce the gradients to their mean, then every rank runs the same full update.

    master/m/v are the (replicated) full fp32 states.  Returns (replicas, master, m, v).
    """
    n_d = len(rank_grads)
    mean = reduce_mean(rank_grads)
    reduced = [mean.copy() for _ in range(n_d)]       # every rank receives the same mean
    outs = [adamw(master, m, v, reduced[r], hp, t) for r in range(n_d)]
    p, m1, v1, _ = outs[0]
    return [o[3] for o in outs], p, m1, v1
