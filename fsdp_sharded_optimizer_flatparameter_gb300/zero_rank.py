"""Data-parallel ranks as separate processes: the sharded step's exchanges over torch.distributed.

"Infra: Data Parallel", ZeRO section (communication paragraphs, ZeRO-1/2/3 flow figures): rank r
owns the contiguous shard [base_u + r*S_u, base_u + (r+1)*S_u) of every unit.  A bucket's
reduce-scatter hands the owner of each part every rank's gradients for it; the owner averages them
and updates its shard of the optimizer state; an all-gather then spreads the updated parameter
shards.  Under ZeRO-3 a unit's parameters are gathered before forward and again before backward,
and nothing is gathered after the update.

The reduction is not left to the collective.  A bucket is exchanged with an all-to-all (every rank
sends each owner that owner's part of its bucket; bytes only, no arithmetic), and the owner folds the
N_d received slices in ascending rank order in the library's kernel (zs_rank_shard_step).  The
result is therefore bit-identical to the one-GPU step on simulated ranks and to the oracle, for any
rank count and whatever order the collective uses inside.  Per step and rank the exchanges send
2 (Psi' - S) bytes and the all-gather 2 S (N_d - 1) bytes, which is zs_plan_comm_bytes' count for
ZeRO-1/2 (the class keeps a running total in ``bytes_sent``).

Device buffers of one rank (all on its own GPU):
  grads        its full bf16 gradient buffer (Psi' elements; ZeRO-3: one unit's buffer);
  master, m, v its fp32 shard state in its local layout (every unit's shard back to back);
  param_shard  its bf16 parameter shard, same layout;
  replica      its full bf16 parameters (ZeRO-1/2), refreshed by the all-gather.
The collectives run on the process group's backend (NCCL between GPUs); with the default local
update the step's arithmetic runs in the library's kernels on the current stream.  A step issues
every bucket's exchange before the first update, so the exchanges stream on the collective's side
while the updates follow bucket by bucket, each after its own exchange.
"""

import torch
import torch.distributed as dist

from . import zs_rank_shard_step


class ZeroRank:
    """One rank of N_d, each its own process: exchange, local update (the library's
    zs_rank_shard_step, in local_update), gather."""

    def __init__(self, plan, group=None):
        self.plan, self.group = plan, group
        self.rank = dist.get_rank(group)
        self.n_d = dist.get_world_size(group)
        if self.n_d != plan.n_d:
            raise ValueError("the process group has %d ranks, the plan N_d = %d" % (self.n_d, plan.n_d))
        self.bytes_sent = 0
        # every owner's part of every bucket: the all-to-all's split sizes
        self._lens = [[hi - lo for lo, hi in (plan.bucket_rank_slice(b, q) for q in range(self.n_d))]
                      for b in range(plan.n_buckets)]
        self._unit_buckets = [[] for _ in range(plan.n_units)]
        for b in range(plan.n_buckets):
            self._unit_buckets[plan.bucket(b)[0]].append(b)

    def local_update(self, bucket, slices, master, m, v, param_shard, hp, step):
        """This rank's part of `bucket`: fold the received slices, AdamW on its own shard state."""
        zs_rank_shard_step(self.plan, self.rank, bucket, slices, master, m, v, param_shard, hp, step)

    def _exchange_start(self, bucket, grads, grads_base, async_op):
        lens = self._lens[bucket]
        _, lo, hi = self.plan.bucket(bucket)
        send = grads[lo - grads_base:hi - grads_base]
        mine = lens[self.rank]
        recv = torch.empty(self.n_d * mine, dtype=grads.dtype, device=grads.device)
        work = dist.all_to_all_single(recv, send, [mine] * self.n_d, lens, group=self.group, async_op=async_op)
        self.bytes_sent += 2 * (sum(lens) - lens[self.rank])
        return work, recv, mine

    def _slices(self, recv, mine, grads):
        if mine % 8 == 0:
            return [recv[q * mine:(q + 1) * mine] for q in range(self.n_d)]
        # the library takes 16-byte-aligned slices: a part that is not a multiple of 8 elements is laid
        # out again in rows of a multiple of 8 (one copy of the part; plans whose bucket parts are
        # multiples of 8 elements never take this path)
        stride = (mine + 7) // 8 * 8
        rows = torch.empty((self.n_d, stride), dtype=grads.dtype, device=grads.device)
        rows[:, :mine].copy_(recv.view(self.n_d, mine))
        return [rows[q, :mine] for q in range(self.n_d)]

    def exchange(self, bucket, grads, grads_base=0):
        """The reduce-scatter's data movement for one bucket: an all-to-all in which every rank sends
        each owner its part of the bucket.  Returns N_d slices, slice q holding rank q's gradients for
        this rank's part.  grads: element i of this rank's gradients at grads[i - grads_base]."""
        _, recv, mine = self._exchange_start(bucket, grads, grads_base, False)
        return self._slices(recv, mine, grads)

    def reduce_scatter_update(self, bucket, grads, master, m, v, param_shard, hp, step, grads_base=0):
        """Exchange one bucket, then average and apply AdamW to this rank's part of it."""
        self._buckets_update([bucket], grads, master, m, v, param_shard, hp, step, grads_base)

    def _buckets_update(self, buckets, grads, master, m, v, param_shard, hp, step, grads_base=0):
        # Every listed bucket's exchange is issued before the first update: an exchange only reads the
        # gradients and writes its own receive buffer, so the exchanges run on the collective's stream
        # while the updates follow one by one on the current stream, each after its own exchange.
        # The receive buffers alive at once hold N_d times this rank's part of the listed buckets (at
        # most one gradient buffer's worth for a whole step).
        pending = [(b, self._exchange_start(b, grads, grads_base, True)) for b in buckets]
        for b, (work, recv, mine) in pending:
            work.wait()
            if mine > 0:
                self.local_update(b, self._slices(recv, mine, grads), master, m, v, param_shard, hp, step)

    def all_gather(self, param_shard, replica):
        """Every rank's updated shard of every unit into this rank's full bf16 replica."""
        for u in range(self.plan.n_units):
            ud, off = self.plan.unit(u), self.plan.unit_local_offset(u)
            dist.all_gather_into_tensor(replica[ud["base"]:ud["base"] + ud["padded"]],
                                        param_shard[off:off + ud["shard"]], group=self.group)
            self.bytes_sent += 2 * ud["shard"] * (self.n_d - 1)

    def step(self, grads, master, m, v, param_shard, replica, hp, step, buckets=None):
        """One ZeRO-1/2 step: each bucket (default: all, last first, as backward makes them ready)
        exchanged and applied, then the all-gather of the parameter shards."""
        order = list(buckets) if buckets is not None else list(reversed(range(self.plan.n_buckets)))
        self._buckets_update(order, grads, master, m, v, param_shard, hp, step)
        self.all_gather(param_shard, replica)

    def gather_unit(self, unit, param_shard, full):
        """ZeRO-3: unit `unit`'s full bf16 parameters (unit-local indexing) from every rank's shard."""
        ud, off = self.plan.unit(unit), self.plan.unit_local_offset(unit)
        dist.all_gather_into_tensor(full[:ud["padded"]], param_shard[off:off + ud["shard"]], group=self.group)
        self.bytes_sent += 2 * ud["shard"] * (self.n_d - 1)

    def unit_step(self, unit, unit_grads, master, m, v, param_shard, hp, step):
        """ZeRO-3: the unit's gradients (unit-local buffer) exchanged bucket by bucket and applied to
        this rank's shard of the unit; nothing is gathered afterwards."""
        base = self.plan.unit(unit)["base"]
        self._buckets_update(list(reversed(self._unit_buckets[unit])), unit_grads, master, m, v, param_shard, hp,
                             step, grads_base=base)
