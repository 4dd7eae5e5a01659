// ZeRO-2 step fed from host memory, bucket by bucket, through a two-slot staging ring.
//
// "Infra: Data Parallel" (F. Pu), section "Zero Redundancy Optimizer (ZeRO)",
// ZeRO-2 paragraph and flow figure: gradients are reduced bucket by bucket as
// they become ready, each rank keeps only the reduced slice it owns and the
// rest is freed at once, so no rank holds a full gradient buffer.  Here each
// bucket's gradients arrive from (pinned) host memory into one slot of a
// ring of two bucket-sized staging slots on `copy_stream`; as soon as a slot
// is filled the fused step (reduce-mean, AdamW on the shard, scatter into every
// replica) runs on `stream` for that bucket, which frees the slot; the
// updated slice of rank 0's replica goes back to the host on `d2h_stream`.
// Buckets are visited in descending order (backward makes the last layer's
// gradients ready first).  Copies of bucket b+1 overlap the update of bucket b.
#include <string>

#include "launch.h"
#include "plan.h"
#include "trace.h"

namespace {

int fail(const char* fn, const std::string& what) {
    zs::set_error(std::string(fn) + ": " + what);
    return ZS_ERR_INVALID;
}

bool bad(const void* p) { return !p || ((uintptr_t)p & 15); }

}  // namespace

extern "C" int zs_zero2_step_host(zs_plan_t plan, const void* const* host_grads, void* const* staging,
                                  int64_t staging_elems, float* master, float* m, float* v,
                                  void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                                  void* host_replica0, void* stream, void* copy_stream, void* d2h_stream) {
    static const char* fn = "zs_zero2_step_host";
    zs::clear_error();
    if (!plan) return fail(fn, "plan is NULL");
    const int nd = plan->n_d;
    if (!host_grads || !staging || !replicas) return fail(fn, "host_grads / staging / replicas is NULL");
    for (int q = 0; q < nd; ++q) {
        if (!host_grads[q]) return fail(fn, "host_grads has a NULL entry (missing rank)");
        if (bad(replicas[q])) return fail(fn, "replicas entry NULL or not 16-byte aligned");
    }
    for (int k = 0; k < 2 * nd; ++k)
        if (bad(staging[k])) return fail(fn, "staging entry NULL or not 16-byte aligned");
    int64_t biggest = 0;
    for (const auto& b : plan->buckets) biggest = b.end - b.begin > biggest ? b.end - b.begin : biggest;
    if (staging_elems < biggest) return fail(fn, "staging slots are smaller than the largest bucket");
    if (bad(master) || bad(m) || bad(v)) return fail(fn, "state pointer NULL or not 16-byte aligned");
    if (!hp || step < 1) return fail(fn, "hparams NULL or step < 1");
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return fail(fn, "betas must lie in [0, 1)");
    float sc[8];
    if (zs_adamw_scalars(hp, step, sc) != ZS_OK) return ZS_ERR_INVALID;
    const zs::AdamScalars s{sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};

    cudaStream_t cs = (cudaStream_t)stream;
    cudaStream_t h2d = (cudaStream_t)copy_stream;
    cudaStream_t d2h = d2h_stream ? (cudaStream_t)d2h_stream : h2d;
    cudaEvent_t ev[6] = {};   // start, filled[2], freed[2], updated
    cudaError_t err = cudaSuccess;
    auto check = [&](cudaError_t e) {
        if (e != cudaSuccess && err == cudaSuccess) err = e;
    };
    for (auto& e : ev) check(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    cudaEvent_t start = ev[0], filled[2] = {ev[1], ev[2]}, freed[2] = {ev[3], ev[4]}, updated = ev[5];
    bool slot_used[2] = {false, false};

    zs::BView out{};
    for (int q = 0; q < nd; ++q) out.ptr.p[q] = (uint16_t*)replicas[q];
    out.off = 0;
    if (err == cudaSuccess) {
        check(cudaEventRecord(start, cs));             // copies may not overtake earlier work on `stream`
        check(cudaStreamWaitEvent(h2d, start, 0));
        if (d2h != h2d) check(cudaStreamWaitEvent(d2h, start, 0));
    }
    zs::TraceRange step_range("zs_zero2_step_host");
    int k = 0;
    for (int b = (int)plan->buckets.size() - 1; b >= 0 && err == cudaSuccess; --b, ++k) {
        zs::TraceRange r_("zero2 bucket %lld", (long long)b);
        const auto& bk = plan->buckets[b];
        const int slot = k & 1;
        const size_t bytes = (size_t)(bk.end - bk.begin) * 2;
        if (slot_used[slot]) check(cudaStreamWaitEvent(h2d, freed[slot], 0));
        for (int q = 0; q < nd; ++q)
            check(cudaMemcpyAsync(staging[(size_t)slot * nd + q], (const uint16_t*)host_grads[q] + bk.begin, bytes,
                                  cudaMemcpyHostToDevice, h2d));
        check(cudaEventRecord(filled[slot], h2d));
        check(cudaStreamWaitEvent(cs, filled[slot], 0));
        zs::BView g{};
        for (int q = 0; q < nd; ++q) g.ptr.p[q] = (uint16_t*)staging[(size_t)slot * nd + q];
        g.off = bk.begin;
        check(zs::launch_fused(g, master, m, v, out, true, {bk.begin, bk.end, 0, 1}, s, nd, cs));
        check(cudaEventRecord(freed[slot], cs));
        slot_used[slot] = true;
        if (host_replica0) {
            check(cudaStreamWaitEvent(d2h, freed[slot], 0));
            check(cudaMemcpyAsync((uint16_t*)host_replica0 + bk.begin, (const uint16_t*)replicas[0] + bk.begin, bytes,
                                  cudaMemcpyDeviceToHost, d2h));
        }
    }
    // `stream` ends the step only when every copy has landed
    if (err == cudaSuccess) {
        check(cudaEventRecord(updated, d2h));
        check(cudaStreamWaitEvent(cs, updated, 0));
        if (d2h != h2d) {
            check(cudaEventRecord(start, h2d));
            check(cudaStreamWaitEvent(cs, start, 0));
        }
    }
    for (auto e : ev)
        if (e) cudaEventDestroy(e);
    if (err != cudaSuccess) {
        zs::set_error(std::string(fn) + ": " + cudaGetErrorString(err));
        return ZS_ERR_CUDA;
    }
    return ZS_OK;
}
