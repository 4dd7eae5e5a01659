// C ABI of the device operations: argument checks, buffer-kind resolution and
// launches.  Every check runs before anything is enqueued, so a rejected call
// writes nothing.  The library never allocates device memory and never
// synchronises; all work goes on the caller's stream.
#include <cmath>
#include <cstdio>
#include <string>
#include <vector>

#include "launch.h"
#include "plan.h"
#include "trace.h"

using zs::BView;
using zs::Ptrs;
using zs::Range;
using zs::set_error;

namespace {

constexpr uintptr_t kAlign = 16;

bool misaligned(const void* p) { return ((uintptr_t)p & (kAlign - 1)) != 0; }

int fail(const char* fn, const std::string& what) {
    set_error(std::string(fn) + ": " + what);
    return ZS_ERR_INVALID;
}

int cuda_status(const char* fn, cudaError_t e) {
    if (e == cudaSuccess) return ZS_OK;
    set_error(std::string(fn) + ": " + cudaGetErrorString(e));
    return ZS_ERR_CUDA;
}

// Checks a pointer array of `count` entries: present, non-NULL, 16-byte aligned.
int check_ptrs(const char* fn, const char* name, const void* const* ptrs, int count) {
    if (!ptrs) return fail(fn, std::string(name) + " is NULL");
    for (int q = 0; q < count; ++q) {
        if (!ptrs[q]) return fail(fn, std::string(name) + "[" + std::to_string(q) + "] is NULL (missing rank)");
        if (misaligned(ptrs[q])) return fail(fn, std::string(name) + "[" + std::to_string(q) + "] is not 16-byte aligned");
    }
    return ZS_OK;
}

int check_one(const char* fn, const char* name, const void* p) {
    if (!p) return fail(fn, std::string(name) + " is NULL");
    if (misaligned(p)) return fail(fn, std::string(name) + " is not 16-byte aligned");
    return ZS_OK;
}

// Resolves a bf16 buffer of the given kind into a view; `bucket_begin` and
// `unit_base` give the origin of ZS_RANK_BUCKET and ZS_RANK_UNIT buffers.
int make_view(const char* fn, const char* name, const void* const* ptrs, int32_t kind, int nd,
              int64_t bucket_begin, int64_t unit_base, BView* out) {
    int rc;
    switch (kind) {
        case ZS_SHARDED:
            if ((rc = check_ptrs(fn, name, ptrs, 1)) != ZS_OK) return rc;
            for (int q = 0; q < ZS_MAX_RANKS; ++q) out->ptr.p[q] = (uint16_t*)ptrs[0];
            out->off = 0;
            return ZS_OK;
        case ZS_RANK_FULL:
        case ZS_RANK_BUCKET:
        case ZS_RANK_UNIT:
            if ((rc = check_ptrs(fn, name, ptrs, nd)) != ZS_OK) return rc;
            for (int q = 0; q < ZS_MAX_RANKS; ++q) out->ptr.p[q] = q < nd ? (uint16_t*)ptrs[q] : nullptr;
            out->off = kind == ZS_RANK_FULL ? 0 : (kind == ZS_RANK_BUCKET ? bucket_begin : unit_base);
            return ZS_OK;
        default:
            return fail(fn, std::string(name) + ": unknown buffer kind");
    }
}

int check_hp(const char* fn, const zs_adamw_hparams* hp, int64_t step, zs::AdamScalars* s) {
    if (!hp) return fail(fn, "hparams is NULL");
    if (step < 1) return fail(fn, "step must be >= 1 (1-based)");
    const float vals[5] = {hp->lr, hp->beta1, hp->beta2, hp->eps, hp->weight_decay};
    for (float x : vals)
        if (!std::isfinite(x)) return fail(fn, "hyper-parameters must be finite");
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return fail(fn, "betas must lie in [0, 1)");
    float sc[8];
    zs_adamw_scalars(hp, step, sc);
    *s = {sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};
    return ZS_OK;
}

int check_plan(const char* fn, zs_plan_t plan) {
    if (!plan) return fail(fn, "plan is NULL");
    return ZS_OK;
}

int check_bucket(const char* fn, zs_plan_t plan, int32_t bucket, bool allow_all) {
    if (bucket == -1 && allow_all) return ZS_OK;
    if (bucket < 0 || bucket >= (int32_t)plan->buckets.size()) return fail(fn, "bucket out of range");
    return ZS_OK;
}

Range unit_range(const zs::Unit& u) { return {u.base, u.base + u.padded, u.base, u.shard}; }

// A gather from one array (the all-gather, the per-unit ZeRO-3 gather): a unit of kDynMinElems or more
// in one dynamic-order launch at N_d <= 8.  Measured on GB300 against the statically ordered launch
// (of the measured copy rate): 100.3-100.5 -> 102.0 % on the Llama-1.3B buffer at N_d = 8, 101.3 ->
// 101.6-101.8 / 100.2 -> 100.7-100.8 % on the 2^28+7 buffer at N_d = 2 / 4; at N_d = 16 / 32 the
// static shape (a 4-stage ring, 16 CTAs per SM) is ahead: 102.8-103.0 / 104.6 % against 101.1 /
// 103.5 %.
int gather_sync(int nd) { return nd <= 8 ? zs::kSyncDynamic : zs::kSyncStream; }


cudaStream_t as_stream(void* s) { return (cudaStream_t)s; }

#define ZS_TRY(expr)                 \
    do {                             \
        int _rc = (expr);            \
        if (_rc != ZS_OK) return _rc; \
    } while (0)

}  // namespace

extern "C" int zs_accumulate_grad(zs_plan_t plan, void* const* acc, const void* const* micro, float scale,
                                  int32_t first, void* stream) {
    static const char* fn = "zs_accumulate_grad";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    ZS_TRY(check_ptrs(fn, "acc", (const void* const*)acc, plan->n_d));
    ZS_TRY(check_ptrs(fn, "micro", micro, plan->n_d));
    if (!std::isfinite(scale)) return fail(fn, "scale must be finite");
    Ptrs a{}, mi{};
    for (int q = 0; q < plan->n_d; ++q) {
        a.p[q] = (uint16_t*)acc[q];
        mi.p[q] = (uint16_t*)micro[q];
    }
    if (plan->padded == 0) return ZS_OK;
    return cuda_status(fn, zs::launch_accumulate(a, mi, plan->n_d, plan->padded, scale, first ? 1 : 0,
                                                 as_stream(stream)));
}

extern "C" int zs_reduce_scatter_mean(zs_plan_t plan, int32_t bucket, const void* const* grads, int32_t grads_kind,
                                      void* const* out, int32_t out_kind, void* stream) {
    static const char* fn = "zs_reduce_scatter_mean";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    ZS_TRY(check_bucket(fn, plan, bucket, true));
    if (grads_kind != ZS_RANK_FULL && grads_kind != ZS_RANK_BUCKET) return fail(fn, "grads_kind must be RANK_FULL or RANK_BUCKET");
    if (grads_kind == ZS_RANK_BUCKET && bucket < 0) return fail(fn, "RANK_BUCKET gradients need a bucket index");
    if (out_kind != ZS_RANK_FULL && out_kind != ZS_SHARDED) return fail(fn, "out_kind must be RANK_FULL or SHARDED");
    const int nd = plan->n_d;
    const int64_t bbeg = bucket >= 0 ? plan->buckets[bucket].begin : 0;
    BView g, o;
    ZS_TRY(make_view(fn, "grads", grads, grads_kind, nd, bbeg, 0, &g));
    ZS_TRY(make_view(fn, "out", (const void* const*)out, out_kind, nd, 0, 0, &o));
    const bool by_owner = out_kind == ZS_RANK_FULL;
    if (bucket >= 0) {
        const auto& bk = plan->buckets[bucket];
        const auto& u = plan->units[bk.unit];
        return cuda_status(fn, zs::launch_rs_mean(g, o, by_owner, {bk.begin, bk.end, u.base, u.shard}, nd,
                                                  as_stream(stream)));
    }
    for (const auto& u : plan->units) {
        if (u.padded == 0) continue;
        ZS_TRY(cuda_status(fn, zs::launch_rs_mean(g, o, by_owner, unit_range(u), nd, as_stream(stream))));
    }
    return ZS_OK;
}

extern "C" int zs_adamw_shard_step(zs_plan_t plan, int32_t rank, const void* const* grad, int32_t grad_kind,
                                   float* master, float* m, float* v, void* const* params, int32_t params_kind,
                                   const zs_adamw_hparams* hp, int64_t step, void* stream) {
    static const char* fn = "zs_adamw_shard_step";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    const int nd = plan->n_d;
    if (rank < -1 || rank >= nd) return fail(fn, "rank out of range");
    if (grad_kind != ZS_RANK_FULL && grad_kind != ZS_SHARDED) return fail(fn, "grad_kind must be RANK_FULL or SHARDED");
    if (params_kind != ZS_RANK_FULL && params_kind != ZS_SHARDED) return fail(fn, "params_kind must be RANK_FULL or SHARDED");
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    BView g, pv;
    ZS_TRY(make_view(fn, "grad", grad, grad_kind, nd, 0, 0, &g));
    ZS_TRY(make_view(fn, "params", (const void* const*)params, params_kind, nd, 0, 0, &pv));
    for (const auto& u : plan->units) {
        Range r = unit_range(u);
        if (rank >= 0) {
            r.lo = u.base + (int64_t)rank * u.shard;
            r.hi = r.lo + u.shard;
        }
        if (r.hi <= r.lo) continue;
        ZS_TRY(cuda_status(fn, zs::launch_adamw(g, grad_kind == ZS_RANK_FULL, master, m, v, pv,
                                                params_kind == ZS_RANK_FULL, r, s, as_stream(stream))));
    }
    return ZS_OK;
}

extern "C" int zs_all_gather(zs_plan_t plan, const void* const* src, int32_t src_kind, void* const* replicas,
                             void* stream) {
    static const char* fn = "zs_all_gather";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    const int nd = plan->n_d;
    if (src_kind != ZS_RANK_FULL && src_kind != ZS_SHARDED) return fail(fn, "src_kind must be RANK_FULL or SHARDED");
    BView sv, dv;
    ZS_TRY(make_view(fn, "src", src, src_kind, nd, 0, 0, &sv));
    ZS_TRY(make_view(fn, "replicas", (const void* const*)replicas, ZS_RANK_FULL, nd, 0, 0, &dv));
    const bool in_place = src_kind == ZS_RANK_FULL;
    if (in_place) {
        for (int q = 0; q < nd; ++q)
            if (src[q] != replicas[q]) return fail(fn, "RANK_FULL source must be the replicas themselves (in place)");
    }
    for (const auto& u : plan->units) {
        if (u.padded == 0) continue;
        ZS_TRY(cuda_status(fn, zs::launch_gather(sv, in_place, dv, in_place, unit_range(u), nd, as_stream(stream),
                                                 gather_sync(nd))));
    }
    return ZS_OK;
}

static int fused_common(const char* fn, zs_plan_t plan, int32_t bucket, const void* const* grads, int32_t grads_kind,
                        float* master, float* m, float* v, void* const* replicas, const zs_adamw_hparams* hp,
                        int64_t step, cudaStream_t st) {
    ZS_TRY(check_plan(fn, plan));
    ZS_TRY(check_bucket(fn, plan, bucket, true));
    if (grads_kind != ZS_RANK_FULL && grads_kind != ZS_RANK_BUCKET) return fail(fn, "grads_kind must be RANK_FULL or RANK_BUCKET");
    if (grads_kind == ZS_RANK_BUCKET && bucket < 0) return fail(fn, "RANK_BUCKET gradients need a bucket index");
    const int nd = plan->n_d;
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    const int64_t bbeg = bucket >= 0 ? plan->buckets[bucket].begin : 0;
    BView g, o;
    ZS_TRY(make_view(fn, "grads", grads, grads_kind, nd, bbeg, 0, &g));
    ZS_TRY(make_view(fn, "replicas", (const void* const*)replicas, ZS_RANK_FULL, nd, 0, 0, &o));
    for (int q = 0; q < nd; ++q)
        for (int j = 0; j < nd; ++j)
            if (replicas[q] == grads[j]) return fail(fn, "replicas must not be the gradient buffers");
    Range r;
    if (bucket >= 0) {
        const auto& bk = plan->buckets[bucket];
        r = {bk.begin, bk.end, 0, 1};
    } else {
        r = {0, plan->padded, 0, 1};       // the fused step needs no owner: one pass over the flat space
    }
    if (r.hi <= r.lo) return ZS_OK;
    // gradients or replicas may be pinned host memory: launch_fused then keeps to the streaming kernel.
    // zs::launch_fused_walk runs a long range as one launch that takes its tiles in dynamic order and
    // walks a shorter one in chunks whose launches overlap.
    return cuda_status(fn, zs::launch_fused_walk(g, master, m, v, o, {r}, s, nd, st, zs::kStagedIfDevice));
}

extern "C" int zs_fused_step(zs_plan_t plan, int32_t bucket, const void* const* grads, int32_t grads_kind,
                             float* master, float* m, float* v, void* const* replicas, const zs_adamw_hparams* hp,
                             int64_t step, void* stream) {
    zs::TraceRange trace_("zs_fused_step");
    zs::clear_error();
    return fused_common("zs_fused_step", plan, bucket, grads, grads_kind, master, m, v, replicas, hp, step,
                        as_stream(stream));
}

extern "C" int zs_fused_step_accumulate(zs_plan_t plan, int32_t bucket, const void* const* acc,
                                        const void* const* micro, int32_t grads_kind, float scale, float* master,
                                        float* m, float* v, void* const* replicas, const zs_adamw_hparams* hp,
                                        int64_t step, void* stream) {
    static const char* fn = "zs_fused_step_accumulate";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    ZS_TRY(check_bucket(fn, plan, bucket, true));
    if (grads_kind != ZS_RANK_FULL && grads_kind != ZS_RANK_BUCKET) return fail(fn, "grads_kind must be RANK_FULL or RANK_BUCKET");
    if (grads_kind == ZS_RANK_BUCKET && bucket < 0) return fail(fn, "RANK_BUCKET gradients need a bucket index");
    if (!std::isfinite(scale)) return fail(fn, "scale must be finite");
    const int nd = plan->n_d;
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    const int64_t bbeg = bucket >= 0 ? plan->buckets[bucket].begin : 0;
    BView a, o;
    zs::AccumIn in;
    in.scale = scale;
    ZS_TRY(make_view(fn, "acc", acc, grads_kind, nd, bbeg, 0, &a));
    ZS_TRY(make_view(fn, "micro", micro, grads_kind, nd, bbeg, 0, &in.micro));
    ZS_TRY(make_view(fn, "replicas", (const void* const*)replicas, ZS_RANK_FULL, nd, 0, 0, &o));
    for (int q = 0; q < nd; ++q)
        for (int j = 0; j < nd; ++j)
            if (replicas[q] == acc[j] || replicas[q] == micro[j])
                return fail(fn, "replicas must not be the accumulator or micro-batch buffers");
    Range r = bucket >= 0 ? Range{plan->buckets[bucket].begin, plan->buckets[bucket].end, 0, 1}
                          : Range{0, plan->padded, 0, 1};
    if (r.hi <= r.lo) return ZS_OK;
    // walked like zs_fused_step; pinned host buffers keep to the streaming kernel
    return cuda_status(fn, zs::launch_fused_walk(a, master, m, v, o, {r}, s, nd, as_stream(stream),
                                                 zs::kStagedIfDevice, &in));
}

extern "C" int zs_fused_step_buckets(zs_plan_t plan, int32_t n_buckets, const int32_t* buckets,
                                     const void* const* grads, float* master, float* m, float* v,
                                     void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                                     int32_t launch_mode, void* stream, void* side_stream) {
    static const char* fn = "zs_fused_step_buckets";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    if (n_buckets < 0 || (n_buckets > 0 && !buckets)) return fail(fn, "bad bucket list");
    if (launch_mode != ZS_BUCKETS_ONE_WALK && launch_mode != ZS_BUCKETS_PER_BUCKET)
        return fail(fn, "launch_mode must be ZS_BUCKETS_ONE_WALK or ZS_BUCKETS_PER_BUCKET");
    std::vector<char> seen(plan->buckets.size(), 0);
    for (int32_t i = 0; i < n_buckets; ++i) {
        ZS_TRY(check_bucket(fn, plan, buckets[i], false));
        if (seen[buckets[i]]) return fail(fn, "a bucket appears twice (it would be updated twice)");
        seen[buckets[i]] = 1;
    }
    // validate everything once through the single-bucket path's checks, then launch bucket by bucket
    const int nd = plan->n_d;
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    BView g, o;
    ZS_TRY(make_view(fn, "grads", grads, ZS_RANK_FULL, nd, 0, 0, &g));
    ZS_TRY(make_view(fn, "replicas", (const void* const*)replicas, ZS_RANK_FULL, nd, 0, 0, &o));
    for (int q = 0; q < nd; ++q)
        for (int j = 0; j < nd; ++j)
            if (replicas[q] == grads[j]) return fail(fn, "replicas must not be the gradient buffers");
    std::vector<int32_t> todo;
    for (int32_t i = 0; i < n_buckets; ++i)
        if (plan->buckets[buckets[i]].end > plan->buckets[buckets[i]].begin) todo.push_back(buckets[i]);
    if (todo.empty()) return ZS_OK;
    // the same pointers serve every bucket: ask the runtime about them once
    const zs::StagedPolicy pol =
        zs::fused_ptrs_on_device(g, master, m, v, o, true, nd) ? zs::kStagedDeviceKnown : zs::kStagedNever;
    cudaStream_t a = as_stream(stream);
    if (launch_mode == ZS_BUCKETS_ONE_WALK) {
        std::vector<zs::Range> ranges;
        ranges.reserve(todo.size());
        for (int32_t b : todo) ranges.push_back({plan->buckets[b].begin, plan->buckets[b].end, 0, 1});
        return cuda_status(fn, zs::launch_fused_ranges(g, master, m, v, o, ranges, s, nd, a, pol));
    }
    cudaStream_t b = side_stream ? as_stream(side_stream) : a;
    const bool two = b != a && todo.size() > 1;
    cudaEvent_t fork = nullptr, join = nullptr;
    if (two) {
        // buckets are disjoint, so consecutive ones may overlap: odd positions run on the side stream,
        // which first waits for everything already enqueued on the caller's stream
        ZS_TRY(cuda_status(fn, cudaEventCreateWithFlags(&fork, cudaEventDisableTiming)));
        cudaError_t e = cudaEventCreateWithFlags(&join, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventRecord(fork, a);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(b, fork, 0);
        if (e != cudaSuccess) {
            cudaEventDestroy(fork);
            if (join) cudaEventDestroy(join);
            return cuda_status(fn, e);
        }
    }
    // The buckets of the list are distinct (checked above), hence disjoint, so on each stream they are
    // walked (zs::launch_fused_walk): the launches after the first need not wait for their predecessor
    // before they start; each streams its own bucket while the previous one drains, and completes
    // after it.  The first launch on each stream waits for everything enqueued before the call.
    std::vector<zs::Range> on_a, on_b;
    for (size_t i = 0; i < todo.size(); ++i) {
        const auto& bk = plan->buckets[todo[i]];
        ((two && (i & 1)) ? on_b : on_a).push_back({bk.begin, bk.end, 0, 1});
    }
    cudaError_t err = zs::launch_fused_walk(g, master, m, v, o, on_a, s, nd, a, pol);
    if (err == cudaSuccess && !on_b.empty()) err = zs::launch_fused_walk(g, master, m, v, o, on_b, s, nd, b, pol);
    if (two) {
        // join even after a failed launch, so later work on the caller's stream orders after the side stream
        cudaError_t e = cudaEventRecord(join, b);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(a, join, 0);
        if (err == cudaSuccess) err = e;
        cudaEventDestroy(fork);
        cudaEventDestroy(join);
    }
    return cuda_status(fn, err);
}

extern "C" int zs_rank_shard_step(zs_plan_t plan, int32_t rank, int32_t bucket, const void* const* slices,
                                  float* master, float* m, float* v, void* param_shard,
                                  const zs_adamw_hparams* hp, int64_t step, void* stream) {
    static const char* fn = "zs_rank_shard_step";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    const int nd = plan->n_d;
    if (rank < 0 || rank >= nd) return fail(fn, "rank out of range");
    ZS_TRY(check_bucket(fn, plan, bucket, true));
    ZS_TRY(check_ptrs(fn, "slices", slices, nd));
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    ZS_TRY(check_one(fn, "param_shard", param_shard));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    // the pieces of rank r's part: global [lo, hi), offset in the rank's local layout, offset in the slices
    struct Piece {
        int64_t lo, hi, local, in_slice;
    };
    std::vector<Piece> pieces;
    std::vector<int64_t> local_of_unit(plan->units.size());
    int64_t acc = 0;
    for (size_t u = 0; u < plan->units.size(); ++u) {
        local_of_unit[u] = acc;
        acc += plan->units[u].shard;
    }
    auto own = [&](size_t u, int64_t lo, int64_t hi, int64_t in_slice) {
        const auto& un = plan->units[u];
        const int64_t s_lo = un.base + (int64_t)rank * un.shard;
        const int64_t a = lo > s_lo ? lo : s_lo, b = hi < s_lo + un.shard ? hi : s_lo + un.shard;
        if (b > a) pieces.push_back({a, b, local_of_unit[u] + (a - s_lo), in_slice});
        return b > a ? b - a : 0;
    };
    if (bucket >= 0) {
        const auto& bk = plan->buckets[bucket];
        own(bk.unit, bk.begin, bk.end, 0);
    } else {
        int64_t off = 0;
        for (size_t u = 0; u < plan->units.size(); ++u) off += own(u, plan->units[u].base,
                                                                   plan->units[u].base + plan->units[u].padded, off);
    }
    if (pieces.empty()) return ZS_OK;
    cudaStream_t st = as_stream(stream);
    // the kernels address element i of the state as base + i: hand them bases shifted so that global
    // index lo lands on the piece's local offset (integer arithmetic; only in-range addresses are formed)
    auto shift = [](void* p, int64_t elems, size_t esize) {
        return (void*)((uintptr_t)p + (uintptr_t)(elems * (int64_t)esize));
    };
    BView g, o;
    {
        const void* sp[1] = {param_shard};
        ZS_TRY(make_view(fn, "param_shard", sp, ZS_SHARDED, nd, 0, 0, &o));
    }
    // ask the runtime once, about the real pointers, whether every buffer is device memory (the staged
    // kernel's bulk copies are pointed at device memory only)
    for (int q = 0; q < ZS_MAX_RANKS; ++q) g.ptr.p[q] = q < nd ? (uint16_t*)slices[q] : nullptr;
    const zs::StagedPolicy pol =
        zs::fused_ptrs_on_device(g, master, m, v, o, false, nd) ? zs::kStagedDeviceKnown : zs::kStagedNever;
    for (const Piece& pc : pieces) {
        for (int q = 0; q < ZS_MAX_RANKS; ++q)
            g.ptr.p[q] = q < nd ? (uint16_t*)slices[q] + pc.in_slice : nullptr;
        g.off = pc.lo;
        o.off = pc.lo - pc.local;
        const int64_t d = pc.local - pc.lo;
        ZS_TRY(cuda_status(fn, zs::launch_fused(g, (float*)shift(master, d, 4), (float*)shift(m, d, 4),
                                                (float*)shift(v, d, 4), o, false, {pc.lo, pc.hi, 0, 1}, s, nd, st,
                                                pol)));
    }
    return ZS_OK;
}

extern "C" int zs_fused_step_host(zs_plan_t plan, const void* const* host_grads, void* const* dev_grads,
                                  float* master, float* m, float* v, void* const* replicas,
                                  const zs_adamw_hparams* hp, int64_t step, void* host_replica0, void* stream) {
    static const char* fn = "zs_fused_step_host";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    const int nd = plan->n_d;
    if (!host_grads) return fail(fn, "host_grads is NULL");
    for (int q = 0; q < nd; ++q)
        if (!host_grads[q]) return fail(fn, "host_grads has a NULL entry (missing rank)");
    ZS_TRY(check_ptrs(fn, "dev_grads", (const void* const*)dev_grads, nd));
    ZS_TRY(check_ptrs(fn, "replicas", (const void* const*)replicas, nd));
    // validate everything the fused step checks before the first copy is enqueued
    {
        ZS_TRY(check_one(fn, "master", master));
        ZS_TRY(check_one(fn, "m", m));
        ZS_TRY(check_one(fn, "v", v));
        zs::AdamScalars s;
        ZS_TRY(check_hp(fn, hp, step, &s));
    }
    cudaStream_t st = as_stream(stream);
    const size_t bytes = (size_t)plan->padded * 2;
    for (int q = 0; q < nd && bytes; ++q)
        ZS_TRY(cuda_status(fn, cudaMemcpyAsync(dev_grads[q], host_grads[q], bytes, cudaMemcpyHostToDevice, st)));
    ZS_TRY(fused_common(fn, plan, -1, (const void* const*)dev_grads, ZS_RANK_FULL, master, m, v, replicas, hp, step, st));
    if (host_replica0 && bytes)
        ZS_TRY(cuda_status(fn, cudaMemcpyAsync(host_replica0, replicas[0], bytes, cudaMemcpyDeviceToHost, st)));
    return ZS_OK;
}

extern "C" int zs_zero3_gather_unit(zs_plan_t plan, int32_t unit, const void* shards, void* const* full,
                                    void* stream) {
    static const char* fn = "zs_zero3_gather_unit";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    if (unit < 0 || unit >= (int32_t)plan->units.size()) return fail(fn, "unit out of range");
    const auto& u = plan->units[unit];
    const void* sp[1] = {shards};
    BView sv, dv;
    ZS_TRY(make_view(fn, "shards", sp, ZS_SHARDED, plan->n_d, 0, 0, &sv));
    ZS_TRY(make_view(fn, "full", (const void* const*)full, ZS_RANK_UNIT, plan->n_d, 0, u.base, &dv));
    if (u.padded == 0) return ZS_OK;
    return cuda_status(fn, zs::launch_gather(sv, false, dv, false, unit_range(u), plan->n_d, as_stream(stream),
                                             gather_sync(plan->n_d)));
}

extern "C" int zs_zero3_rs_step_unit(zs_plan_t plan, int32_t unit, const void* const* grads, float* master,
                                     float* m, float* v, void* shards, const zs_adamw_hparams* hp, int64_t step,
                                     void* stream) {
    static const char* fn = "zs_zero3_rs_step_unit";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    if (unit < 0 || unit >= (int32_t)plan->units.size()) return fail(fn, "unit out of range");
    const auto& u = plan->units[unit];
    ZS_TRY(check_one(fn, "master", master));
    ZS_TRY(check_one(fn, "m", m));
    ZS_TRY(check_one(fn, "v", v));
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    const void* sp[1] = {shards};
    BView g, o;
    ZS_TRY(make_view(fn, "grads", grads, ZS_RANK_UNIT, plan->n_d, 0, u.base, &g));
    ZS_TRY(make_view(fn, "shards", sp, ZS_SHARDED, plan->n_d, 0, 0, &o));
    if (u.padded == 0) return ZS_OK;
    // a unit of kDynMinElems or more at N_d <= 16 in one dynamic-order launch, as in zs_zero3_step:
    // measured on GB300 against one statically ordered launch per call (of the measured copy rate),
    // 101.3 -> 103.8-103.9 % over the Llama-1.3B units at N_d = 8, 100.9 -> 104.7-104.8 % / 97.9-98.0 ->
    // 103.8-103.9 % on the 2^28+7-element unit at N_d = 16 / 2
    return cuda_status(fn, zs::launch_fused(g, master, m, v, o, false, unit_range(u), s, plan->n_d,
                                            as_stream(stream), zs::kStagedIfDevice,
                                            plan->n_d <= 16 ? zs::kSyncDynamic : zs::kSyncStream));
}

extern "C" int zs_set_fused_variant(int32_t variant) {
    zs::clear_error();
    if (variant != ZS_FUSED_AUTO && variant != ZS_FUSED_LDG && variant != ZS_FUSED_TMA)
        return fail("zs_set_fused_variant", "unknown variant");
    zs::set_fused_variant(variant);
    return ZS_OK;
}

extern "C" int zs_set_dependent_launch(int32_t enable) {
    zs::clear_error();
    zs::set_dependent_launch(enable != 0);
    return ZS_OK;
}

extern "C" int zs_device_status(uint32_t* code, int32_t clear) {
    static const char* fn = "zs_device_status";
    zs::clear_error();
    if (!code) return fail(fn, "code is NULL");
    unsigned int v = 0;
    ZS_TRY(cuda_status(fn, zs::read_device_error(&v, clear != 0)));
    *code = v;
    return ZS_OK;
}

extern "C" int zs_selftest_wait_timeout(int64_t limit_cycles, void* stream) {
    static const char* fn = "zs_selftest_wait_timeout";
    zs::clear_error();
    if (limit_cycles < 1 || limit_cycles > (int64_t(1) << 32)) return fail(fn, "limit_cycles out of range");
    return cuda_status(fn, zs::launch_wait_selftest((long long)limit_cycles, as_stream(stream)));
}

extern "C" int zs_all_reduce_mean(zs_plan_t plan, int32_t bucket, void* const* grads, void* stream) {
    static const char* fn = "zs_all_reduce_mean";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    ZS_TRY(check_bucket(fn, plan, bucket, true));
    BView g;
    ZS_TRY(make_view(fn, "grads", (const void* const*)grads, ZS_RANK_FULL, plan->n_d, 0, 0, &g));
    Range r = bucket >= 0 ? Range{plan->buckets[bucket].begin, plan->buckets[bucket].end, 0, 1}
                          : Range{0, plan->padded, 0, 1};
    if (r.hi <= r.lo) return ZS_OK;
    return cuda_status(fn, zs::launch_all_reduce_mean(g, r, plan->n_d, as_stream(stream)));
}

extern "C" int zs_dp_step(zs_plan_t plan, const void* const* grads, float* const* master, float* const* m,
                          float* const* v, void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                          void* stream) {
    static const char* fn = "zs_dp_step";
    zs::TraceRange trace_(fn);
    zs::clear_error();
    ZS_TRY(check_plan(fn, plan));
    const int nd = plan->n_d;
    zs::AdamScalars s;
    ZS_TRY(check_hp(fn, hp, step, &s));
    ZS_TRY(check_ptrs(fn, "master", (const void* const*)master, nd));
    ZS_TRY(check_ptrs(fn, "m", (const void* const*)m, nd));
    ZS_TRY(check_ptrs(fn, "v", (const void* const*)v, nd));
    BView g, o;
    ZS_TRY(make_view(fn, "grads", grads, ZS_RANK_FULL, nd, 0, 0, &g));
    ZS_TRY(make_view(fn, "replicas", (const void* const*)replicas, ZS_RANK_FULL, nd, 0, 0, &o));
    for (int q = 0; q < nd; ++q)
        for (int j = 0; j < nd; ++j)
            if (replicas[q] == grads[j]) return fail(fn, "replicas must not be the gradient buffers");
    if (plan->padded == 0) return ZS_OK;
    return cuda_status(fn, zs::launch_dp_step(g, o, master, m, v, {0, plan->padded, 0, 1}, s, nd, as_stream(stream)));
}
