"""Shared pieces of the GPU parity tests: buffer set-up, oracle runs, and the gates.

Gates (the stated tolerance of the method): fp32 master/m/v within
max |relative error| <= 1e-6 (exact equality where the oracle's value is 0),
bf16 parameters within 1 bf16 ulp.  The kernels follow the oracle's operation
order, so the tests also count how many values are not bit-identical, and
``exact=True`` requires that count to be zero.
"""

import numpy as np
import torch

from oracle import layout, numerics, steps

REL_TOL = 1e-6


def to_np_bf16(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()


def to_np_f32(t):
    return t.detach().cpu().contiguous().numpy().copy()


def from_np_bf16(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def check_f32(got, want, what, exact=True):
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, what
    zero = want == 0
    assert np.array_equal(got[zero], want[zero]), "%s: nonzero where the oracle has 0" % what
    nz = ~zero
    if nz.any():
        rel = np.abs(got[nz].astype(np.float64) - want[nz]) / np.abs(want[nz].astype(np.float64))
        assert rel.max() <= REL_TOL, "%s: max rel err %.3g" % (what, rel.max())
    if exact:
        diff = int(np.count_nonzero(got.view(np.uint32) != want.view(np.uint32)))
        assert diff == 0, "%s: %d of %d values not bit-identical" % (what, diff, got.size)


def check_bf16(got, want, what, exact=True):
    got = np.asarray(got, np.uint16)
    want = np.asarray(want, np.uint16)
    assert got.shape == want.shape, what
    g = numerics.f32_from_bf16(got).astype(np.float64)
    w = numerics.f32_from_bf16(want).astype(np.float64)
    ulp = numerics.bf16_ulp(want)
    assert np.all(np.abs(g - w) <= ulp), "%s: more than 1 bf16 ulp off" % what
    if exact:
        diff = int(np.count_nonzero(got != want))
        assert diff == 0, "%s: %d of %d values not bit-identical" % (what, diff, got.size)


def unshard(plan, rank_arrays):
    """Oracle rank-local shard arrays -> one global-flat-index array (the ZS_SHARDED layout)."""
    offs = steps.unit_local_offsets(plan)
    out = np.zeros(plan.padded, dtype=np.asarray(rank_arrays[0]).dtype)
    for ui, u in enumerate(plan.units):
        for r in range(plan.n_d):
            lo, hi = layout.shard_range(plan, ui, r)
            out[lo:hi] = rank_arrays[r][offs[ui]:offs[ui] + u.shard]
    return out


def reshard(plan, full):
    return [steps.shard_of(plan, r, full) for r in range(plan.n_d)]


def chunk_oracle(grads_chunks, master, m, v, hp, t):
    """The fused step on one chunk of the flat space: mean over ranks, then AdamW (element-wise)."""
    ghat = steps.reduce_mean(grads_chunks)
    p, m1, v1, bits = steps.adamw(master, m, v, ghat, hp, t)
    return ghat, p, m1, v1, bits
