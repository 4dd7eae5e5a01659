"""Race checks of the overlapping launches at the benchmarked sizes (GPU).

The benchmarked fused step is one launch whose CTAs take their tiles in dynamic order from a
counter, and the ZeRO-3 step runs its gathers and updates on two streams, each unit's phase one such
launch (units of 2^24 elements and more) or walked in overlapping launches.  A race there would show
as a run-to-run difference, so each step below runs repeatedly from the same state and must equal,
bit for bit, a reference run of the same step:

* the Llama-1.3B ZeRO-2 step at N_d = 8, the call the benchmark times (one dynamic-order launch),
  ten times (1.3e10 element-steps), against the register-streaming kernel;
* the ZeRO-3 step on the Llama-1.3B units at N_d = 8 (25 units of ~50 M elements, each unit's
  gathers and update one dynamic-order launch, two streams, the 2-slot pool), five times, against
  the same step with programmatic dependent launch off (every launch waiting for the previous one
  to complete) on one stream;
* the naive-DP step and the in-place all-reduce on the GPT-2-small buffers at N_d = 8 (one
  dynamic-order launch each), against the register-streaming kernels.

The oracle itself is not needed here: every-element oracle parity of the headline call is in
test_gpu_fullsize_every_element.py, and of the naive-DP forms in test_gpu_dyn_order.py.
"""

import gc

import pytest
import torch

import fsdp_sharded_optimizer_flatparameter_gb300 as zs
import synth

pytestmark = pytest.mark.gpu

HP = synth.HPARAMS
DEV = "cuda"
BF16 = torch.bfloat16


@pytest.fixture(autouse=True)
def _free_memory():
    yield
    zs.zs_set_dependent_launch(True)
    gc.collect()
    torch.cuda.empty_cache()


def _need(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.skip("needs %.0f GB of free device memory, %.0f GB free" % (nbytes / 1e9, free / 1e9))


def test_llama13b_zero2_step_repeats_the_streaming_result():
    wl = synth.WORKLOADS["llama-1.3b-zero2"]
    shapes, _ = synth.workload_params(wl["model"])
    n_d = wl["n_d"]
    plan = zs.Plan(shapes, n_d, stage=wl["stage"], bucket_bytes=wl["bucket_bytes"])
    P, pads = plan.padded, plan.pad_ranges()
    _need(P * (2 * n_d * 3 + 12 * 3) + (4 << 30))
    grads, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    synth.fill_grads(grads, pads, wl["seed"], 1, wl["sigma"], wl["outlier_p"])
    state0 = [synth.master_init(P, pads, wl["seed"], device=DEV)]
    state0 += [torch.rand_like(state0[0]) * 1e-3, torch.rand_like(state0[0]) * 1e-6]   # moments not zero
    ref_st = [x.clone() for x in state0]
    ref_reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *ref_st, ref_reps, HP, 2)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    st = [x.clone() for x in state0]
    reps, _ = synth.rank_buffers(n_d, P, BF16, DEV)
    zs.zs_device_status(clear=True)
    for k in range(10):
        for x, y in zip(st, state0):
            x.copy_(y)
        for r in reps:
            r.zero_()
        zs.zs_fused_step(plan, -1, grads, zs.ZS_RANK_FULL, *st, reps, HP, 2)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(st, ref_st)), "run %d: state differs" % k
        assert all(torch.equal(x, y) for x, y in zip(reps, ref_reps)), "run %d: replicas differ" % k
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE


def test_llama13b_units_zero3_walk_repeats_the_serialised_step():
    n_d = 8
    shapes, units = synth.workload_params("llama-1.3b-units")
    plan = zs.Plan(shapes, n_d, stage=3, unit_of_param=units)
    P, U = plan.padded, plan.n_units
    biggest = max(plan.unit(u)["padded"] for u in range(U))
    _need(P * (12 * 3 + 2 * 3) + 3 * n_d * biggest * 2 * 2 + (4 << 30))
    ugrads, _ = synth.rank_buffers(n_d, biggest, BF16, DEV)
    synth.fill_grads(ugrads, [], 3, 1, 5e-4, 0.001)
    master0 = synth.master_init(P, plan.pad_ranges(), 3, device=DEV)
    state0 = [master0, torch.rand_like(master0) * 1e-3, torch.rand_like(master0) * 1e-6]
    shards0 = master0.to(BF16)
    pool = [synth.rank_buffers(n_d, biggest, BF16, DEV)[0] for _ in range(2)]
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()

    ref_st, ref_sh = [x.clone() for x in state0], shards0.clone()
    zs.zs_set_dependent_launch(False)
    zs.zs_zero3_step(plan, ref_sh, *ref_st, [ugrads] * U, pool, True, HP, 2, main_stream=main, side_stream=main)
    torch.cuda.synchronize()
    zs.zs_set_dependent_launch(True)
    st, sh = [x.clone() for x in state0], shards0.clone()
    zs.zs_device_status(clear=True)
    for k in range(5):
        for x, y in zip(st, state0):
            x.copy_(y)
        sh.copy_(shards0)
        zs.zs_zero3_step(plan, sh, *st, [ugrads] * U, pool, True, HP, 2, main_stream=main, side_stream=side)
        torch.cuda.synchronize()
        assert all(torch.equal(x, y) for x, y in zip(st, ref_st)), "run %d: state differs" % k
        assert torch.equal(sh, ref_sh), "run %d: shards differ" % k
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE


def test_gpt2_naive_dp_step_repeats_the_streaming_result():
    """The naive-DP step on the GPT-2-small buffers at N_d = 8 (one dynamic-order launch over 124 M
    elements, every rank's full state), five times from the same state, and the in-place all-reduce
    on the same gradients: bit for bit the register-streaming kernels' results."""
    n_d = 8
    shapes, _ = synth.workload_params("gpt2-small")
    plan = zs.Plan(shapes, n_d, stage=0)
    P, pads = plan.padded, plan.pad_ranges()
    _need(P * (2 * n_d * 4 + 12 * n_d * 3 + 12) + (4 << 30))
    grads, _ = synth.rank_grads(n_d, P, pads, seed=11, step=1, sigma=1e-3, outlier_p=0.001, device=DEV)
    master0 = synth.master_init(P, pads, 12, device=DEV)
    m0, v0 = torch.rand_like(master0) * 1e-3, torch.rand_like(master0) * 1e-6

    def state():
        return ([master0.clone() for _ in range(n_d)], [m0.clone() for _ in range(n_d)],
                [v0.clone() for _ in range(n_d)], synth.rank_buffers(n_d, P, BF16, DEV)[0])

    ref = state()
    ref_ar = [g.clone() for g in grads]
    zs.zs_set_fused_variant(zs.ZS_FUSED_LDG)
    try:
        zs.zs_dp_step(plan, grads, *ref, HP, 2)
        zs.zs_all_reduce_mean(plan, -1, ref_ar)
        torch.cuda.synchronize()
    finally:
        zs.zs_set_fused_variant(zs.ZS_FUSED_AUTO)
    zs.zs_device_status(clear=True)
    for k in range(5):
        got = state()
        zs.zs_dp_step(plan, grads, *got, HP, 2)
        torch.cuda.synchronize()
        for a, b in zip(got, ref):
            assert all(torch.equal(x, y) for x, y in zip(a, b)), "run %d: the naive-DP step differs" % k
        del got
    ar = [g.clone() for g in grads]
    zs.zs_all_reduce_mean(plan, -1, ar)
    torch.cuda.synchronize()
    assert all(torch.equal(x, y) for x, y in zip(ar, ref_ar)), "the all-reduce differs"
    assert zs.zs_device_status() == zs.ZS_DEVERR_NONE
