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
// parameters; blockIdx.y picks the parameter, blockIdx.z the rank and
// blockIdx.x / threadIdx.x stride over the run.  Runs whose two ends share
// their 16-byte phase move 8 bf16 values per access after a short scalar head.
#include <string>

#include "launch.h"
#include "plan.h"

namespace zs {

namespace {

constexpr int kPerLaunch = 64;
constexpr int kCopyThreads = 256;

struct Piece {
    uint16_t* param;        // the parameter's own layout (d0 x row elements)
    int64_t d0, row, chunk, off;
};

struct CopyArgs {
    Piece p[kPerLaunch];
    uint16_t* flat;         // the group's buffer (N_d * shard elements)
    int64_t shard;
    int to_flat;            // 1: parameters -> buffer (zero padding rows), 0: buffer -> parameters
};

__device__ __forceinline__ void copy_run(uint16_t* dst, const uint16_t* src, int64_t n, int64_t t, int64_t stride) {
    if ((((uintptr_t)dst ^ (uintptr_t)src) & 15) == 0) {
        const int64_t head = (int64_t)(((16 - ((uintptr_t)dst & 15)) & 15) >> 1);
        const int64_t h = head < n ? head : n;
        for (int64_t i = t; i < h; i += stride) dst[i] = src[i];
        const int64_t nv = (n - h) >> 3;
        const uint4* s4 = reinterpret_cast<const uint4*>(src + h);
        uint4* d4 = reinterpret_cast<uint4*>(dst + h);
        for (int64_t i = t; i < nv; i += stride) __stcs(d4 + i, __ldcs(s4 + i));
        for (int64_t i = h + (nv << 3) + t; i < n; i += stride) dst[i] = src[i];
    } else {
        for (int64_t i = t; i < n; i += stride) dst[i] = src[i];
    }
}

__device__ __forceinline__ void zero_run(uint16_t* dst, int64_t n, int64_t t, int64_t stride) {
    for (int64_t i = t; i < n; i += stride) dst[i] = 0;
}

__global__ void __launch_bounds__(kCopyThreads) k_fsdp2_copy(const __grid_constant__ CopyArgs a) {
    const Piece& pc = a.p[blockIdx.y];
    const int64_t r = blockIdx.z;
    const int64_t begin = r * pc.chunk < pc.d0 ? r * pc.chunk : pc.d0;
    const int64_t end = (r + 1) * pc.chunk < pc.d0 ? (r + 1) * pc.chunk : pc.d0;
    const int64_t n = (end - begin) * pc.row;                 // real elements of this piece
    uint16_t* buf = a.flat + r * a.shard + pc.off;
    uint16_t* par = pc.param + begin * pc.row;
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if (a.to_flat) {
        copy_run(buf, par, n, t, stride);
        zero_run(buf + n, pc.chunk * pc.row - n, t, stride);  // padding rows
    } else {
        copy_run(par, buf, n, t, stride);
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
    int sms = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    for (size_t first = 0; first < members.size(); first += kPerLaunch) {
        const size_t cnt = members.size() - first < (size_t)kPerLaunch ? members.size() - first : (size_t)kPerLaunch;
        CopyArgs a{};
        int64_t longest = 1;
        for (size_t j = 0; j < cnt; ++j) {
            const int32_t k = members[first + j];
            a.p[j] = {(uint16_t*)params[first + j], plan->param_d0[k], plan->param_row[k], plan->param_chunk[k],
                      plan->param_piece_off[k]};
            longest = std::max<int64_t>(longest, plan->param_chunk[k] * plan->param_row[k]);
        }
        a.flat = (uint16_t*)flat;
        a.shard = un.shard;
        a.to_flat = to_flat;
        // enough blocks along x for the longest run, about two waves over the whole grid
        int64_t bx = (longest / 8 + kCopyThreads - 1) / kCopyThreads;
        const int64_t cap = std::max<int64_t>(1, (int64_t)sms * 16 / (int64_t)(cnt * plan->n_d));
        bx = std::max<int64_t>(1, std::min(bx, cap));
        dim3 grid((unsigned)bx, (unsigned)cnt, (unsigned)plan->n_d);
        k_fsdp2_copy<<<grid, kCopyThreads, 0, st>>>(a);
        cudaError_t e = cudaGetLastError();
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
