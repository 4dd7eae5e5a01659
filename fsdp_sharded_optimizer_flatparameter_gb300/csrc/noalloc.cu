// zs_zero2_step_host_noalloc: the host-fed bucket-wise step without any
// caller-provided or library-allocated device staging.
//
// Some callers cannot allocate device memory when they run the optimizer
// step: a framework that has handed all device memory to its own pool and does
// not let plug-ins call cudaMalloc, a latency-critical thread that must not pay
// cudaMalloc's implicit device synchronisation, or an embedding runtime that
// passes only stream and buffer pointers.  For them this entry point stages
// each bucket's gradients in a fixed array that lives in the library image
// itself (a file-scope __device__ array, kZsNoallocStagingBytes bytes), so the
// call needs no allocation at all.  Every GPU that loads the library keeps
// that array until the process exits.
//
// Host code cannot use the array's name as a device address (it names a
// host-side stand-in).  The first call on each device therefore looks the
// address up with cudaGetSymbolAddress, with that device current, checks the
// result and caches it per device; later calls reuse it.
#include <mutex>
#include <string>

#include "launch.h"
#include "plan.h"

namespace {

constexpr int64_t kZsNoallocStagingBytes = ZS_NOALLOC_STAGING_BYTES;
constexpr int kMaxDevices = 64;

// The staging ring shared by every call on a device (two slots of N_d bucket buffers).
__device__ __align__(256) uint16_t zs_noalloc_staging[kZsNoallocStagingBytes / 2];

std::mutex g_setup_mu;
void* g_staging_ptr[kMaxDevices] = {};

int fail(const char* fn, const std::string& what, int code = ZS_ERR_INVALID) {
    zs::set_error(std::string(fn) + ": " + what);
    return code;
}

// Device address of the staging array for the current device (looked up once per device).
int staging_address(const char* fn, uint16_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    if (dev < 0 || dev >= kMaxDevices) return fail(fn, "device ordinal out of range");
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_staging_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, zs_noalloc_staging);
        if (e != cudaSuccess || !p) return fail(fn, std::string("cudaGetSymbolAddress: ") + cudaGetErrorString(e), ZS_ERR_CUDA);
        g_staging_ptr[dev] = p;
    }
    *out = (uint16_t*)g_staging_ptr[dev];
    return ZS_OK;
}

}  // namespace

extern "C" int zs_zero2_step_host_noalloc(zs_plan_t plan, const void* const* host_grads, float* master, float* m,
                                          float* v, void* const* replicas, const zs_adamw_hparams* hp, int64_t step,
                                          void* host_replica0, void* stream) {
    static const char* fn = "zs_zero2_step_host_noalloc";
    zs::clear_error();
    if (!plan) return fail(fn, "plan is NULL");
    const int nd = plan->n_d;
    if (!host_grads || !replicas) return fail(fn, "host_grads / replicas is NULL");
    for (int q = 0; q < nd; ++q) {
        if (!host_grads[q]) return fail(fn, "host_grads has a NULL entry (missing rank)");
        if (!replicas[q] || ((uintptr_t)replicas[q] & 15)) return fail(fn, "replicas entry NULL or not 16-byte aligned");
    }
    if (!master || !m || !v || ((uintptr_t)master & 15) || ((uintptr_t)m & 15) || ((uintptr_t)v & 15))
        return fail(fn, "state pointer NULL or not 16-byte aligned");
    if (!hp || step < 1) return fail(fn, "hparams NULL or step < 1");
    if (!(hp->beta1 >= 0.0f && hp->beta1 < 1.0f && hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return fail(fn, "betas must lie in [0, 1)");
    // the ring: two slots of N_d buffers, each a multiple of 8 elements so every buffer stays 16-byte aligned
    int64_t biggest = 0;
    for (const auto& b : plan->buckets) biggest = b.end - b.begin > biggest ? b.end - b.begin : biggest;
    const int64_t slot_elems = (biggest + 7) & ~int64_t(7);
    const int64_t need_bytes = 2 * (int64_t)nd * slot_elems * 2;
    if (need_bytes > kZsNoallocStagingBytes)
        return fail(fn, "2 slots x " + std::to_string(nd) + " ranks x the largest bucket (" + std::to_string(biggest) +
                            " elements) need " + std::to_string(need_bytes) + " bytes of staging; the built-in array holds " +
                            std::to_string(kZsNoallocStagingBytes) + " (use smaller buckets or zs_zero2_step_host)");
    float sc[8];
    if (zs_adamw_scalars(hp, step, sc) != ZS_OK) return ZS_ERR_INVALID;
    const zs::AdamScalars s{sc[0], sc[1], sc[2], sc[3], sc[4], sc[5], sc[6], sc[7]};
    uint16_t* staging = nullptr;
    int rc = staging_address(fn, &staging);
    if (rc != ZS_OK) return rc;

    // Everything runs in order on `stream`: copy a bucket in, update it, copy the replica slice out.
    cudaStream_t st = (cudaStream_t)stream;
    zs::BView out{};
    for (int q = 0; q < nd; ++q) out.ptr.p[q] = (uint16_t*)replicas[q];
    out.off = 0;
    int k = 0;
    for (int b = (int)plan->buckets.size() - 1; b >= 0; --b, ++k) {
        const auto& bk = plan->buckets[b];
        const size_t bytes = (size_t)(bk.end - bk.begin) * 2;
        uint16_t* slot = staging + (size_t)(k & 1) * nd * slot_elems;
        zs::BView g{};
        for (int q = 0; q < nd; ++q) {
            g.ptr.p[q] = slot + (size_t)q * slot_elems;
            cudaError_t e = cudaMemcpyAsync(g.ptr.p[q], (const uint16_t*)host_grads[q] + bk.begin, bytes,
                                            cudaMemcpyHostToDevice, st);
            if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
        }
        g.off = bk.begin;
        cudaError_t e = zs::launch_fused(g, master, m, v, out, true, {bk.begin, bk.end, 0, 1}, s, nd, st);
        if (e == cudaSuccess && host_replica0)
            e = cudaMemcpyAsync((uint16_t*)host_replica0 + bk.begin, (const uint16_t*)replicas[0] + bk.begin, bytes,
                                cudaMemcpyDeviceToHost, st);
        if (e != cudaSuccess) return fail(fn, cudaGetErrorString(e), ZS_ERR_CUDA);
    }
    return ZS_OK;
}
