"""zs_zero2_step_host_noalloc against the oracle and against zs_zero2_step_host (GPU).

The no-allocation entry point serves callers that cannot allocate device
memory when they step the optimizer; it stages gradients in a fixed array
inside the library instead of a caller-provided ring.  Its results must equal
the oracle's step (reduce-mean over ranks, then AdamW, on the whole flat
space) and the staged entry point's, bit for bit, on two calls in a row (the
second call reuses the array the first one left behind), with the device
status word clear after each pair.  This file is collected last so that a run
stopping at the first failure has already run every other test; it also
passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import gpu_helpers as H
import synth

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"


def _run_pair(plan, steps=(1, 2)):
    n_d, P, pads = plan.n_d, plan.padded, plan.pad_ranges()
    master0 = synth.master_init(P, pads, seed=31, device=DEV)
    a = [master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)]
    b = [master0.clone(), torch.zeros_like(master0), torch.zeros_like(master0)]
    reps_a = synth.rank_buffers(n_d, P, torch.bfloat16, DEV)[0]
    reps_b = synth.rank_buffers(n_d, P, torch.bfloat16, DEV)[0]
    biggest = max(hi - lo for _, lo, hi in (plan.bucket(k) for k in range(plan.n_buckets)))
    staging = [synth.rank_buffers(n_d, biggest, torch.bfloat16, DEV)[0] for _ in range(2)]
    # the oracle's state, stepped beside the device (every step is element-wise over the flat space)
    o_p, o_m, o_v = H.to_np_f32(master0), np.zeros(P, np.float32), np.zeros(P, np.float32)
    for t in steps:
        grads, _ = synth.rank_grads(n_d, P, pads, seed=32, step=t, sigma=1e-3, outlier_p=0.001, device=DEV)
        host = [g.cpu().pin_memory() for g in grads]
        out_a = torch.empty(P, dtype=torch.bfloat16).pin_memory()
        out_b = torch.empty(P, dtype=torch.bfloat16).pin_memory()
        zs.zs_device_status(clear=True)
        zs.zs_zero2_step_host(plan, host, staging, *a, reps_a, HP, t, host_replica0=out_a)
        # through the C ABI directly: plain pointers, nothing allocated by the call
        lib = ctypes.CDLL(zs.LIB_PATH)
        fn = lib.zs_zero2_step_host_noalloc
        fn.restype = ctypes.c_int32
        arr = lambda xs: (ctypes.c_void_p * len(xs))(*[x.data_ptr() for x in xs])  # noqa: E731
        hp = zs.zs_adamw_hparams(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"])
        rc = fn(plan.handle, arr(host), ctypes.c_void_p(b[0].data_ptr()), ctypes.c_void_p(b[1].data_ptr()),
                ctypes.c_void_p(b[2].data_ptr()), arr(reps_b), ctypes.byref(hp), ctypes.c_int64(t),
                ctypes.c_void_p(out_b.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == zs.ZS_OK, zs.zs_last_error()
        torch.cuda.synchronize()
        assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
        _, o_p, o_m, o_v, o_bits = H.chunk_oracle([H.to_np_bf16(g) for g in host], o_p, o_m, o_v, HP, t)
        for y, want, name in zip(b, (o_p, o_m, o_v), ("master", "m", "v")):
            H.check_f32(H.to_np_f32(y), want, "no-alloc %s vs oracle t=%d" % (name, t))
        for q in range(n_d):
            H.check_bf16(H.to_np_bf16(reps_b[q]), o_bits, "no-alloc replica %d vs oracle t=%d" % (q, t))
        H.check_bf16(H.to_np_bf16(out_b), o_bits, "no-alloc host replica vs oracle t=%d" % t)
        for x, y, name in zip(a, b, ("master", "m", "v")):
            H.check_f32(H.to_np_f32(y), H.to_np_f32(x), "%s t=%d" % (name, t))
        for q in range(n_d):
            H.check_bf16(H.to_np_bf16(reps_b[q]), H.to_np_bf16(reps_a[q]), "replica %d t=%d" % (q, t))
        H.check_bf16(H.to_np_bf16(out_b), H.to_np_bf16(out_a), "host replica t=%d" % t)


@pytest.mark.parametrize("shapes,n_d,bucket_bytes", [
    ([(1_000_003,)], 8, 1 << 18),          # ragged tail, 128 Ki-element buckets
    ([(300, 96), (96,), (257, 96)], 3, 10_000),
])
def test_noalloc_matches_staged_entry_point_two_calls(shapes, n_d, bucket_bytes):
    plan = zs.Plan(shapes, n_d, stage=2, bucket_bytes=bucket_bytes)
    _run_pair(plan)


def test_noalloc_rejects_buckets_beyond_the_builtin_array():
    plan = zs.Plan([(1 << 22,)], 8, stage=2, bucket_bytes=8 << 20)       # 2 x 8 x 4 Mi elements x 2 B = 128 MiB
    P = plan.padded
    host = [torch.zeros(P, dtype=torch.bfloat16) for _ in range(8)]
    st = [torch.zeros(P, device=DEV) for _ in range(3)]
    reps = synth.rank_buffers(8, P, torch.bfloat16, DEV)[0]
    with pytest.raises(zs.ZsError) as e:
        zs.zs_zero2_step_host_noalloc(plan, host, *st, reps, HP, 1)
    assert str(32 << 20) in str(e.value)
