// FSDP2 per-parameter Shard(0) layout: copies between the parameters' own
// layout and a group's rank-major flat buffer.
//
// "Infra: Data Parallel" (F. Pu), FSDP section, FSDP2 layout figure and
// subsection "FSDP2": each parameter keeps its global shape and is cut along
// dimension 0, rank r holding rows [r*c, (r+1)*c) with c = ceil(d0 / N_d); the
// parameters of one group are still gathered and reduce-scattered together.
// The group's flat buffer is the ranks' shards one after another; rank r's
// shard is its pieces of the group's parameters in order, each padded to c
// rows with zeros.  So parameter k's rank-r piece is one contiguous run in
// both layouts: (rows of rank r) * row elements from row r*c of the parameter
// to offset r*S + piece_off_k of the buffer, followed (in the buffer) by the
// zero rows that pad it to c rows.
//
// zs_fsdp2_chunk_cat builds the buffer from the parameters (the reduce-scatter
// input built from each rank's gradients); zs_fsdp2_copy_out writes the
// gathered buffer back into the parameters.  A launch covers up to kPerLaunch
// parameters.  Every (parameter, rank) piece is cut into tasks of kTask
// elements of the buffer side and each CTA takes one task, so the work is
// balanced whatever the mix of parameter sizes (a 2-element norm next to a
// 65M-element embedding); the CTA finds its piece by binary search over the
// launch's prefix of task counts.  256 threads copy a task: runs whose two
// ends share their 16-byte phase move 8 bf16 values per access, every thread
// issuing all of its loads before its stores; other runs go element by
// element.  (A bulk-copy version - one warp, a ring of 32 KB tiles, one bulk
// load and one bulk store per task - measured 87 % of the copy rate on the
// Llama-1.3B groups against this kernel's 90 %: a group's launch is ~35 us
// and the ring's fill and drain do not pay for themselves.)
#include <string>

#include "device.cuh"
#include "plan.h"

namespace zs {

namespace {

constexpr int kPerLaunch = kFsdp2PerLaunch;
constexpr int kCopyThreads = 256;
constexpr int kBatch = 8;                                   // 16-byte accesses in flight per thread
constexpr int64_t kTask = kFsdp2Task;                       // 16384 elements per CTA
static_assert(kTask == (int64_t)kCopyThreads * kBatch * 8, "a task is one batch of every thread");
using Piece = Fsdp2Piece;
using CopyArgs = Fsdp2CopyArgs;

__device__ __forceinline__ void copy_run(uint16_t* dst, const uint16_t* src, int64_t n, int t, int stride) {
    if ((((uintptr_t)dst ^ (uintptr_t)src) & 15) == 0) {
        const int64_t head = (int64_t)(((16 - ((uintptr_t)dst & 15)) & 15) >> 1);
        const int64_t h = head < n ? head : n;
        for (int64_t i = t; i < h; i += stride) dst[i] = src[i];
        const int64_t nv = (n - h) >> 3;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + h);
        uint4* d4 = reinterpret_cast<uint4*>(dst + h);
        for (int64_t b = t; b < nv; b += (int64_t)kBatch * stride) {
            uint4 r[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int64_t i = b + (int64_t)k * stride;
                if (i < nv) r[k] = __ldcs(s4 + i);
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int64_t i = b + (int64_t)k * stride;
                if (i < nv) __stcs(d4 + i, r[k]);
            }
        }
        for (int64_t i = h + (nv << 3) + t; i < n; i += stride) dst[i] = src[i];
    } else {
        for (int64_t i = t; i < n; i += stride) dst[i] = src[i];
    }
}

__device__ __forceinline__ void zero_run(uint16_t* dst, int64_t n, int t, int stride) {
    for (int64_t i = t; i < n; i += stride) dst[i] = 0;
}

__global__ void __launch_bounds__(kCopyThreads) k_fsdp2_copy(const __grid_constant__ CopyArgs a) {
    dependent_launch_prologue();
    const int64_t task = blockIdx.x;
    int lo = 0, hi = a.n - 1;                                 // last j with first[j] <= task
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.first[mid] <= task) lo = mid; else hi = mid - 1;
    }
    const Piece& pc = a.p[lo];
    const int64_t k = task - a.first[lo];
    const int64_t r = k / pc.tasks;                           // rank
    const int64_t tk = k - r * pc.tasks;                      // task within the piece
    const int64_t begin = r * pc.chunk < pc.d0 ? r * pc.chunk : pc.d0;
    const int64_t end = (r + 1) * pc.chunk < pc.d0 ? (r + 1) * pc.chunk : pc.d0;
    const int64_t n = (end - begin) * pc.row;                 // real elements of this piece
    const int64_t len = pc.chunk * pc.row;                    // buffer elements of this piece
    const int64_t x0 = tk * kTask;
    const int64_t x1 = x0 + kTask < len ? x0 + kTask : len;
    uint16_t* buf = a.flat + r * a.shard + pc.off;
    uint16_t* par = pc.param + begin * pc.row;
    const int64_t c1 = x1 < n ? x1 : n;                       // [x0, c1) real, [max(x0, n), x1) padding
    const int t = threadIdx.x, stride = blockDim.x;
    if (a.to_flat) {
        if (c1 > x0) copy_run(buf + x0, par + x0, c1 - x0, t, stride);
        const int64_t z0 = x0 > n ? x0 : n;
        if (x1 > z0) zero_run(buf + z0, x1 - z0, t, stride);
    } else if (c1 > x0) {
        copy_run(par + x0, buf + x0, c1 - x0, t, stride);
    }
}

int fail(const char* fn, const std::string& what) {
    set_error(std::string(fn) + ": " + what);
    return ZS_ERR_INVALID;
}

int fsdp2_copy(const char* fn, zs_plan_t plan, int32_t unit, void* const* params, void* flat, int to_flat,
               cudaStream_t st) {
    clear_error();
    if (!plan) return fail(fn, "plan is NULL");
    if (plan->layout != ZS_LAYOUT_FSDP2) return fail(fn, "the plan does not use the FSDP2 layout");
    if (unit < 0 || unit >= (int32_t)plan->units.size()) return fail(fn, "unit out of range");
    if (!params || !flat) return fail(fn, "params / flat is NULL");
    std::vector<int32_t> members;
    for (int32_t k = 0; k < (int32_t)plan->param_numel.size(); ++k)
        if (plan->param_unit[k] == unit) members.push_back(k);
    for (size_t j = 0; j < members.size(); ++j)
        if (!params[j] || ((uintptr_t)params[j] & 1)) return fail(fn, "a parameter pointer is NULL or not 2-byte aligned");
    if ((uintptr_t)flat & 1) return fail(fn, "flat is not 2-byte aligned");
    const zs::Unit& un = plan->units[unit];
    for (size_t first = 0; first < members.size(); first += kPerLaunch) {
        const size_t cnt = members.size() - first < (size_t)kPerLaunch ? members.size() - first : (size_t)kPerLaunch;
        CopyArgs a{};
        a.first[0] = 0;
        for (size_t j = 0; j < cnt; ++j) {
            const int32_t k = members[first + j];
            const int64_t len = plan->param_chunk[k] * plan->param_row[k];
            const int64_t tasks = std::max<int64_t>(1, (len + kTask - 1) / kTask);
            a.p[j] = {(uint16_t*)params[first + j], plan->param_d0[k], plan->param_row[k], plan->param_chunk[k],
                      plan->param_piece_off[k], tasks};
            a.first[j + 1] = a.first[j] + tasks * plan->n_d;
        }
        a.n = (int)cnt;
        a.flat = (uint16_t*)flat;
        a.shard = un.shard;
        a.to_flat = to_flat;
        const int64_t total = a.first[cnt];
        if (total > 0x7fffffffLL) return fail(fn, "unit too large for one launch");
        cudaError_t e = launch_kernel(k_fsdp2_copy, dim3((unsigned)total), dim3(kCopyThreads), 0, st, a);
        if (e != cudaSuccess) {
            set_error(std::string(fn) + ": " + cudaGetErrorString(e));
            return ZS_ERR_CUDA;
        }
    }
    return ZS_OK;
}

}  // namespace

}  // namespace zs

extern "C" int zs_fsdp2_chunk_cat(zs_plan_t plan, int32_t unit, const void* const* params, void* flat, void* stream) {
    return zs::fsdp2_copy("zs_fsdp2_chunk_cat", plan, unit, (void* const*)params, flat, 1, (cudaStream_t)stream);
}

extern "C" int zs_fsdp2_copy_out(zs_plan_t plan, int32_t unit, const void* flat, void* const* params, void* stream) {
    return zs::fsdp2_copy("zs_fsdp2_copy_out", plan, unit, params, (void*)flat, 0, (cudaStream_t)stream);
}
