// ZeRO-3 / FSDP full-shard step over every unit, scheduled on two streams.
//
// "Infra: Data Parallel" (F. Pu), section "Zero Redundancy Optimizer (ZeRO)",
// ZeRO-3 paragraph and flow figure: before a unit's forward its full
// parameters are gathered and freed after use; in backward (reverse unit
// order) they are gathered again, the unit's gradients are reduce-scattered
// with averaging and each rank updates its own shard; nothing is gathered
// after the update.  Subsection "FSDP2": with reshard_after_forward off the
// gathered parameters are kept from forward to backward (one gather fewer).
//
// Communication (gathers, reduce-scatter + update) goes on `side`, the
// compute stream `main` only records and waits on events (the place where a
// model's forward and backward kernels would run).  Gathers go into a pool of
// slots, each slot holding N_d unit-sized buffers; with two slots the gather
// of the next unit overlaps the use of the current one (prefetch depth 1) and
// a slot is reused only after `main` has released it.  The library creates
// CUDA events (no device memory) and destroys them before returning; event
// destruction is deferred by the runtime until the recorded work completes.
#include <string>
#include <vector>

#include "launch.h"
#include "plan.h"
#include "trace.h"
#include "walk.h"

namespace {

int fail(const char* fn, const std::string& what) {
    zs::set_error(std::string(fn) + ": " + what);
    return ZS_ERR_INVALID;
}

struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (auto e : ev) cudaEventDestroy(e);
    }
    cudaError_t make(size_t n) {
        ev.reserve(n);
        for (size_t i = 0; i < n; ++i) {
            cudaEvent_t e;
            cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
            if (r != cudaSuccess) return r;
            ev.push_back(e);
        }
        return cudaSuccess;
    }
};

}  // namespace

extern "C" int zs_zero3_step(zs_plan_t plan, void* shards, float* master, float* m, float* v,
                             const void* const* unit_grads, void* const* pool, int32_t pool_slots,
                             int32_t reshard_after_forward, const zs_adamw_hparams* hp, int64_t step,
                             void* main_stream, void* side_stream) {
    static const char* fn = "zs_zero3_step";
    zs::clear_error();
    if (!plan) return fail(fn, "plan is NULL");
    const int nd = plan->n_d;
    const int U = (int)plan->units.size();
    if (!unit_grads || !pool) return fail(fn, "unit_grads / pool is NULL");
    const int need_slots = reshard_after_forward ? (U < 2 ? U : 2) : U;
    if (pool_slots < need_slots)
        return fail(fn, reshard_after_forward ? "pool needs 2 slots (1 for a single unit)"
                                              : "pool needs one slot per unit when reshard_after_forward is off");
    // argument checks of every launch first, so a bad pointer enqueues nothing
    for (int u = 0; u < U; ++u) {
        for (int q = 0; q < nd; ++q)
            if (!unit_grads[(size_t)u * nd + q] || ((uintptr_t)unit_grads[(size_t)u * nd + q] & 15))
                return fail(fn, "unit_grads entry NULL or not 16-byte aligned");
    }
    for (int s = 0; s < pool_slots * nd; ++s)
        if (!pool[s] || ((uintptr_t)pool[s] & 15)) return fail(fn, "pool entry NULL or not 16-byte aligned");
    if (!shards || ((uintptr_t)shards & 15) || !master || !m || !v || ((uintptr_t)master & 15) ||
        ((uintptr_t)m & 15) || ((uintptr_t)v & 15))
        return fail(fn, "state or shard pointer NULL or not 16-byte aligned");
    if (!hp || step < 1) return fail(fn, "hparams NULL or step < 1");
    float sc[8];
    if (zs_adamw_scalars(hp, step, sc) != ZS_OK) return ZS_ERR_INVALID;
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return fail(fn, "betas must lie in [0, 1)");
    const zs::AdamScalars s{sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};

    cudaStream_t mainS = (cudaStream_t)main_stream, sideS = (cudaStream_t)side_stream;
    // On one stream (main_stream == side_stream) stream order already gives every dependency below, so
    // no event is created, recorded or waited on, and each launch follows the previous one directly.
    const bool one = mainS == sideS;
    Events E;
    // per unit: gathered (fwd), released (fwd), gathered (bwd), backward done, released (bwd)
    cudaError_t err = one ? cudaSuccess : E.make((size_t)U * 5 + 2);
    if (err != cudaSuccess) {
        zs::set_error(std::string(fn) + ": " + cudaGetErrorString(err));
        return ZS_ERR_CUDA;
    }
    auto ev = [&](int u, int k) { return one ? nullptr : E.ev[(size_t)u * 5 + k]; };
    cudaEvent_t start = one ? nullptr : E.ev[(size_t)U * 5];
    cudaEvent_t done = one ? nullptr : E.ev[(size_t)U * 5 + 1];

    zs::BView shard_view;
    for (int q = 0; q < ZS_MAX_RANKS; ++q) shard_view.ptr.p[q] = (uint16_t*)shards;
    shard_view.off = 0;
    auto slot_view = [&](int slot, const zs::Unit& un) {
        zs::BView b{};
        for (int q = 0; q < nd; ++q) b.ptr.p[q] = (uint16_t*)pool[(size_t)slot * nd + q];
        b.off = un.base;
        return b;
    };
    auto grad_view = [&](int u) {
        zs::BView b{};
        for (int q = 0; q < nd; ++q) b.ptr.p[q] = (uint16_t*)unit_grads[(size_t)u * nd + q];
        b.off = plan->units[u].base;
        return b;
    };
    auto check = [&](cudaError_t e) {
        if (e != cudaSuccess && err == cudaSuccess) err = e;
    };
    auto record = [&](cudaEvent_t e, cudaStream_t on) {
        if (!one) check(cudaEventRecord(e, on));
    };
    auto wait = [&](cudaStream_t on, cudaEvent_t e) {
        if (!one && e) check(cudaStreamWaitEvent(on, e, 0));
    };
    // A unit's gather and its reduce-scatter + update are each a walk over the unit's range: pieces cut
    // at multiples of kWalkChunk (none shorter than a quarter of it), one launch each, the first
    // waiting for everything before it on the stream, the others streaming their pieces while the
    // previous one drains (the launch-order modes of launch.h; the pieces are disjoint and the staged
    // kernels read global memory through bulk copies only).
    // A unit of at least kDynMinElems elements at N_d <= 16 goes in one launch per phase whose CTAs take
    // the unit's tiles in dynamic order instead.  Measured on GB300 against the walk (of the measured
    // copy rate): Llama-1.3B units 96.0 -> 98.4 % (reshard_after_forward off: 97.2 -> 100.4 %), Llama-7B
    // 102.9 % either way, the 2^28+7 buffer's one-unit step 101.7 / 100.9 / 101.2 / 102.0 -> 102.6 /
    // 102.1 / 102.1 / 102.6 % for N_d = 2 / 4 / 8 / 16, but 101.8 -> 100.5 % at N_d = 32, which keeps
    // the walk.
    constexpr int64_t kWalkChunk = int64_t(1) << 23;
    auto walk = [&](const zs::Unit& un, auto&& launch) {
        if (err != cudaSuccess) return;
        if (un.padded >= zs::kDynMinElems && nd <= 16) {
            check(launch(zs::Range{un.base, un.base + un.padded, un.base, un.shard}, zs::kSyncDynamic));
            return;
        }
        check(zs::walk_range(un.base, un.base + un.padded, kWalkChunk, [&](int64_t a, int64_t b, int sync) {
            return launch(zs::Range{a, b, un.base, un.shard}, sync);
        }));
    };
    auto gather = [&](int slot, const zs::Unit& un) {
        walk(un, [&](const zs::Range& r, int sync) {
            return zs::launch_gather(shard_view, false, slot_view(slot, un), false, r, nd, sideS, sync);
        });
    };

    // the side stream starts after everything already enqueued on main
    record(start, mainS);
    wait(sideS, start);

    zs::TraceRange step_range("zs_zero3_step");
    // forward, unit order
    cudaEvent_t slot_free[2] = {nullptr, nullptr};   // main's release of each slot's last user (reshard on)
    for (int u = 0; u < U && err == cudaSuccess; ++u) {
        zs::TraceRange r_("zero3 forward gather unit %lld", (long long)u);
        const zs::Unit& un = plan->units[u];
        const int slot = reshard_after_forward ? (u & 1) : u;
        if (reshard_after_forward) wait(sideS, slot_free[slot]);
        gather(slot, un);
        record(ev(u, 0), sideS);
        wait(mainS, ev(u, 0));
        // forward(u) runs here on main; afterwards the gathered parameters are released
        record(ev(u, 1), mainS);
        if (reshard_after_forward) slot_free[slot] = ev(u, 1);
    }

    // backward, reverse unit order.  With resharding, each unit's gather goes into its slot once main
    // has released the slot's previous user, and the gather of the next unit (u - 1) is issued before
    // the reduce-scatter/update of unit u (backward prefetch): the side stream streams that gather
    // while main runs backward(u), instead of idling until backward(u) is done.
    auto backward_gather = [&](int u) {
        zs::TraceRange r_("zero3 backward gather unit %lld", (long long)u);
        const zs::Unit& un = plan->units[u];
        const int slot = u & 1;
        wait(sideS, slot_free[slot]);
        gather(slot, un);
        record(ev(u, 2), sideS);
    };
    if (reshard_after_forward && U > 0 && err == cudaSuccess) backward_gather(U - 1);
    for (int u = U - 1; u >= 0 && err == cudaSuccess; --u) {
        zs::TraceRange r_("zero3 backward reduce-scatter/update unit %lld", (long long)u);
        const zs::Unit& un = plan->units[u];
        if (reshard_after_forward) {
            wait(mainS, ev(u, 2));
            // backward(u) runs here on main and produces unit_grads[u]; then the slot is released
            record(ev(u, 4), mainS);
            slot_free[u & 1] = ev(u, 4);
            if (u > 0) backward_gather(u - 1);
        } else {
            wait(mainS, ev(u, 0));                           // still gathered from forward
        }
        record(ev(u, 3), mainS);                             // backward(u) done: its gradients exist
        wait(sideS, ev(u, 3));
        walk(un, [&](const zs::Range& r, int sync) {
            return zs::launch_fused(grad_view(u), master, m, v, shard_view, false, r, s, nd, sideS,
                                    zs::kStagedIfDevice, sync);
        });
    }
    // main continues (the next step's forward) only after the last update
    record(done, sideS);
    wait(mainS, done);
    if (err != cudaSuccess) {
        zs::set_error(std::string(fn) + ": " + cudaGetErrorString(err));
        return ZS_ERR_CUDA;
    }
    return ZS_OK;
}
