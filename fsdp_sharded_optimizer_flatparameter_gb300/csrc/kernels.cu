// Streaming kernels of the sharded optimizer step (sm_103a).
//
// Every step of the method is element-wise over the global flat index
// ("Infra: Data Parallel", ZeRO section: AdamW is element-wise, so a rank can
// update any part of the parameters from that part's mean gradient and
// moments), so each kernel is a grid-stride loop over the index range of a
// bucket or unit.  The body works on vectors of 8 elements (one 16-byte
// access per bf16 rank slice, two per fp32 state array); a range whose ends
// are not multiples of 8 has its at most 14 fringe elements done one by one
// by block 0, and a range whose buffers cannot all be accessed in 16-byte
// units (a bucket or unit base, or an owner boundary, off the 8-element grid)
// runs element by element throughout.  The rank count N_d is a template
// parameter for the common powers of two so the rank loops unroll; other
// counts use the runtime value.  Nothing here waits on anything but the preceding
// kernel on the stream (the dependent-launch wait, no longer than stream order), so
// no kernel can hang.  The launchers below also choose, per call, the bulk-copy staged
// kernels (kernels_tma.cu) for large bodies whose buffers are all device memory.
#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>
#include <vector>

#include "device.cuh"
#include "walk.h"

namespace zs {

constexpr int kThreads = 256;

// ------------------------------------------------------------------ launch geometry

// Blocks for a grid-stride kernel: enough to cover the work, at most one full wave of resident
// blocks on the current device.  The wave is cached per (device, kernel) once the queries succeed; a
// failed query is returned to the caller and not cached.
static cudaError_t grid_for(const void* kernel, int64_t items, int* grid) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, int> cap_cache;     // (device, kernel) -> resident blocks
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = ((uint64_t)(uintptr_t)kernel) ^ ((uint64_t)(uint32_t)dev << 56);
    int cap;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cap_cache.find(key);
        if (it == cap_cache.end()) {
            int sms = 0, occ = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0);
            if (e != cudaSuccess) return e;
            if (sms < 1 || occ < 1) return cudaErrorInvalidConfiguration;
            cap = sms * occ;
            cap_cache.emplace(key, cap);
        } else {
            cap = it->second;
        }
    }
    int64_t want = (items + kThreads - 1) / kThreads;
    if (want < 1) want = 1;
    *grid = (int)(want < cap ? want : cap);
    return cudaSuccess;
}

// Split [lo, hi) into an 8-aligned vector body and a scalar fringe.
struct Split {
    int64_t lo, hi;      // whole range
    int64_t vlo;         // first element of the vector body
    int64_t nvec;        // vectors of 8 in the body (0: run everything one by one)
    int sync;            // LaunchSync (kSyncStream or kSyncWalkFirst: these kernels read through L1)
};

static Split split_range(int64_t lo, int64_t hi, bool vec_ok) {
    Split s{lo, hi, lo, 0, kSyncStream};
    if (!vec_ok) return s;
    const int64_t vlo = (lo + 7) & ~int64_t(7);
    const int64_t vhi = hi & ~int64_t(7);
    if (vhi > vlo) {
        s.vlo = vlo;
        s.nvec = (vhi - vlo) >> 3;
    }
    return s;
}

// Runs op.template run<8>(i) over the body and op.template run<1>(i) over the fringe.
template <class Op>
__device__ __forceinline__ void for_range(const Split& sp, const Op& op) {
    dependent_launch_prologue(sp.sync);
    if (sp.nvec > 0) {
        for (int64_t t = gtid(); t < sp.nvec; t += gstride()) op.template run<8>(sp.vlo + (t << 3));
        const int64_t nhead = sp.vlo - sp.lo;
        const int64_t tail0 = sp.vlo + (sp.nvec << 3);
        const int64_t nfringe = nhead + (sp.hi - tail0);
        if (blockIdx.x == 0 && (int64_t)threadIdx.x < nfringe) {
            const int64_t j = threadIdx.x;
            op.template run<1>(j < nhead ? sp.lo + j : tail0 + (j - nhead));
        }
    } else {
        for (int64_t i = sp.lo + gtid(); i < sp.hi; i += gstride()) op.template run<1>(i);
    }
    dependent_launch_epilogue(sp.sync);
}

__device__ __forceinline__ int owner_of(int64_t i, int64_t base, int64_t shard) { return (int)((i - base) / shard); }

// ------------------------------------------------------------------ gradient accumulation

struct AccumArgs {
    Ptrs acc, micro;
    float scale;
    int first;
};

// One rank's buffers (blockIdx.y selects the rank).
struct AccumOp {
    uint16_t* acc;
    const uint16_t* micro;
    float scale;
    int first;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        float g[VEC], prev[VEC];
        unpack(ld_bf<VEC>(micro + i), g);
        if (first) {
#pragma unroll
            for (int k = 0; k < VEC; ++k) prev[k] = 0.0f;
        } else {
            unpack(ld_bf<VEC>(acc + i), prev);
        }
#pragma unroll
        for (int k = 0; k < VEC; ++k) prev[k] = accumulate_elem(prev[k], g[k], scale);
        st_bf<VEC>(acc + i, pack(prev));
    }
};

__global__ void __launch_bounds__(kThreads) k_accumulate(AccumArgs a, Split sp) {
    const AccumOp op{a.acc.p[blockIdx.y], a.micro.p[blockIdx.y], a.scale, a.first};
    for_range(sp, op);
}

cudaError_t launch_accumulate(const Ptrs& acc, const Ptrs& micro, int nd, int64_t n, float scale, int first,
                              cudaStream_t st) {
    AccumArgs a{acc, micro, scale, first};
    Split sp = split_range(0, n, true);
    int gx = 0;
    cudaError_t e = grid_for((const void*)k_accumulate, sp.nvec > 0 ? sp.nvec : n, &gx);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_accumulate, dim3(gx, nd), dim3(kThreads), 0, st, a, sp);
}

// ------------------------------------------------------------------ reduce-scatter with averaging

template <int ND>
struct RsOp {
    BView g, out;
    int out_by_owner;
    int nd;
    float inv_nd;
    int64_t base, shard;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int n = ND > 0 ? ND : nd;
        float acc[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            float f[VEC];
            unpack(ld_bf<VEC>(g.ptr.p[q] + (i - g.off)), f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = mean_of_sum<ND>(acc[k], n, inv_nd);
        const int qo = out_by_owner ? owner_of(i, base, shard) : 0;
        st_bf<VEC>(out.ptr.p[qo] + (i - out.off), pack(acc));
    }
};

template <int ND>
__global__ void __launch_bounds__(kThreads) k_rs_mean(RsOp<ND> op, Split sp) { for_range(sp, op); }

template <int ND>
static cudaError_t rs_impl(const BView& g, const BView& out, bool by_owner, const Range& r, int nd, Split sp,
                           cudaStream_t st) {
    RsOp<ND> op{g, out, by_owner ? 1 : 0, nd, 1.0f / (float)nd, r.base, r.shard};
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_rs_mean<ND>, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_rs_mean<ND>, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

// ------------------------------------------------------------------ AdamW on a shard

struct AdamOp {
    BView grad, par;
    int grad_by_owner, par_by_owner;
    float *master, *m, *v;
    AdamScalars s;
    int64_t base, shard;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int q = (grad_by_owner | par_by_owner) ? owner_of(i, base, shard) : 0;
        float g[VEC], p[VEC], mm[VEC], vv[VEC];
        unpack(ld_bf<VEC>(grad.ptr.p[grad_by_owner ? q : 0] + (i - grad.off)), g);
        ld_f32<VEC>(master + i, p);
        ld_f32<VEC>(m + i, mm);
        ld_f32<VEC>(v + i, vv);
#pragma unroll
        for (int k = 0; k < VEC; ++k) adamw_elem(g[k], p[k], mm[k], vv[k], s);
        st_f32<VEC>(master + i, p);
        st_f32<VEC>(m + i, mm);
        st_f32<VEC>(v + i, vv);
        st_bf<VEC>(par.ptr.p[par_by_owner ? q : 0] + (i - par.off), pack(p));
    }
};

__global__ void __launch_bounds__(kThreads) k_adamw(AdamOp op, Split sp) { for_range(sp, op); }

// ------------------------------------------------------------------ all-gather (copy to every rank)

template <int ND>
struct GatherOp {
    BView src, dst;
    int src_by_owner, skip_owner;
    int nd;
    int64_t base, shard;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int n = ND > 0 ? ND : nd;
        const int o = (src_by_owner | skip_owner) ? owner_of(i, base, shard) : -1;
        const BfVec<VEC> w = ld_bf<VEC>(src.ptr.p[src_by_owner ? o : 0] + (i - src.off));
#pragma unroll
        for (int q = 0; q < n; ++q) {
            if (skip_owner && q == o) continue;
            st_bf<VEC>(dst.ptr.p[q] + (i - dst.off), w);
        }
    }
};

template <int ND>
__global__ void __launch_bounds__(kThreads) k_gather(GatherOp<ND> op, Split sp) { for_range(sp, op); }

template <int ND>
static cudaError_t gather_impl(const BView& src, bool src_by_owner, const BView& dst, bool skip_owner,
                               const Range& r, int nd, Split sp, cudaStream_t st) {
    GatherOp<ND> op{src, dst, src_by_owner ? 1 : 0, skip_owner ? 1 : 0, nd, r.base, r.shard};
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_gather<ND>, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_gather<ND>, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

// ------------------------------------------------------------------ fused: reduce-mean + AdamW + scatter

// The micro-batch operand of the accumulating form (ACC): present only there, so the plain form's
// kernel parameter stays as small as before.
template <bool ACC>
struct FusedMicro {};
template <>
struct FusedMicro<true> {
    BView micro;
    float scale;
};

template <int ND, bool BROADCAST, bool ACC = false>
struct FusedOp : FusedMicro<ACC> {
    BView g, out;
    float *master, *m, *v;
    AdamScalars s;
    int nd;
    float inv_nd;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int n = ND > 0 ? ND : nd;
        float acc[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            float f[VEC];
            unpack(ld_bf<VEC>(g.ptr.p[q] + (i - g.off)), f);
            if constexpr (ACC) {
                // rank q's gradient: its accumulator plus the last micro-batch, rounded to bf16 as the
                // accumulation stores it
                float b[VEC];
                unpack(ld_bf<VEC>(this->micro.ptr.p[q] + (i - this->micro.off)), b);
#pragma unroll
                for (int k = 0; k < VEC; ++k) f[k] = accumulate_elem(f[k], b[k], this->scale);
                unpack(pack(f), f);
            }
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
        float p[VEC], mm[VEC], vv[VEC], gr[VEC];
        ld_f32<VEC>(master + i, p);
        ld_f32<VEC>(m + i, mm);
        ld_f32<VEC>(v + i, vv);
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = mean_of_sum<ND>(acc[k], n, inv_nd);
        unpack(pack(acc), gr);                  // the reduced gradient is a bf16 value
#pragma unroll
        for (int k = 0; k < VEC; ++k) adamw_elem(gr[k], p[k], mm[k], vv[k], s);
        st_f32<VEC>(master + i, p);
        st_f32<VEC>(m + i, mm);
        st_f32<VEC>(v + i, vv);
        const BfVec<VEC> w = pack(p);
        if constexpr (BROADCAST) {
#pragma unroll
            for (int q = 0; q < n; ++q) {
                st_bf<VEC>(out.ptr.p[q] + (i - out.off), w);
            }
        } else {
            st_bf<VEC>(out.ptr.p[0] + (i - out.off), w);
        }
    }
};

template <int ND, bool BROADCAST, bool ACC>
__global__ void __launch_bounds__(kThreads) k_fused(FusedOp<ND, BROADCAST, ACC> op, Split sp) { for_range(sp, op); }

template <int ND, bool BROADCAST, bool ACC = false>
static cudaError_t fused_impl(const BView& g, float* master, float* m, float* v, const BView& out,
                              const AdamScalars& s, int nd, Split sp, cudaStream_t st, const AccumIn* acc = nullptr) {
    FusedOp<ND, BROADCAST, ACC> op;
    op.g = g;
    op.out = out;
    op.master = master;
    op.m = m;
    op.v = v;
    op.s = s;
    op.nd = nd;
    op.inv_nd = 1.0f / (float)nd;
    if constexpr (ACC) {
        op.micro = acc->micro;
        op.scale = acc->scale;
    }
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_fused<ND, BROADCAST, ACC>, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_fused<ND, BROADCAST, ACC>, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

// ------------------------------------------------------------------ dispatch

static bool aligned8(int64_t x) { return (x & 7) == 0; }
static bool all_device(const void* const* ps, int n);
static std::atomic<int> g_fused_variant{ZS_FUSED_AUTO};   // read by launches on any thread
// Smallest body worth a persistent staged launch (below it the register-streaming kernel is as fast).
constexpr int64_t kTmaMinElems = int64_t(1) << 20;
// Within a walk over disjoint buckets a staged launch overlaps its predecessor (kSyncWalkNext), so
// the staged kernel pays off for smaller bodies there.
constexpr int64_t kTmaWalkMinElems = int64_t(1) << 16;

#define ZS_DISPATCH_ND(nd, CALL)            \
    switch (nd) {                           \
        case 1: return CALL(1);             \
        case 2: return CALL(2);             \
        case 4: return CALL(4);             \
        case 8: return CALL(8);             \
        case 16: return CALL(16);           \
        case 32: return CALL(32);           \
        default: return CALL(0);            \
    }

static cudaError_t rs_ldg(const BView& g, const BView& out, bool out_by_owner, const Range& r, int nd,
                          const Split& sp, cudaStream_t st) {
#define ZS_RS(N) rs_impl<N>(g, out, out_by_owner, r, nd, sp, st)
    ZS_DISPATCH_ND(nd, ZS_RS)
#undef ZS_RS
}

cudaError_t launch_rs_mean(const BView& g, const BView& out, bool out_by_owner, const Range& r, int nd,
                           cudaStream_t st) {
    const bool vec = aligned8(g.off) && aligned8(out.off) &&
                     (!out_by_owner || (aligned8(r.base) && aligned8(r.shard)));
    const Split sp = split_range(r.lo, r.hi, vec);
    // one output array (ZeRO-2/3 shard, a bucket's staging): the staged kernel for the 8-aligned
    // body, all on device memory; the in-place ZeRO-1 form (each element to its owner's buffer) and
    // host buffers keep the streaming kernel
    if (!out_by_owner && (sp.nvec << 3) >= kTmaMinElems && g_fused_variant.load() != ZS_FUSED_LDG &&
        (nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32)) {
        const void* ps[ZS_MAX_RANKS + 1];
        for (int q = 0; q < nd; ++q) ps[q] = g.ptr.p[q];
        ps[nd] = out.ptr.p[0];
        if (all_device(ps, nd + 1)) {
            const int64_t body_hi = sp.vlo + (sp.nvec << 3);
            cudaError_t e = launch_rs_tma(g, out.ptr.p[0], out.off, sp.vlo, sp.nvec << 3, nd, st);
            if (e != cudaErrorNotSupported) {
                if (e != cudaSuccess) return e;
                if (sp.vlo > sp.lo) {
                    e = rs_ldg(g, out, false, r, nd, split_range(sp.lo, sp.vlo, false), st);
                    if (e != cudaSuccess) return e;
                }
                if (sp.hi > body_hi) e = rs_ldg(g, out, false, r, nd, split_range(body_hi, sp.hi, false), st);
                return e;
            }
        }
    }
    return rs_ldg(g, out, out_by_owner, r, nd, sp, st);
}

// The staged AdamW over the 8-aligned body [lo, hi) of one-array buffers as a walk: pieces cut as in
// launch_fused_walk (multiples of kFusedWalkChunk, none shorter than a quarter of it), one launch each,
// the first waiting for the stream's predecessor and the others streaming their pieces while the
// previous one drains (the launch-order modes of launch.h: the pieces are disjoint and the kernel
// reads global memory through bulk copies only).
static cudaError_t adamw_tma_walk(const BView& grad, float* master, float* m, float* v, const BView& par, int64_t lo,
                                  int64_t hi, const AdamScalars& s, cudaStream_t st) {
    if (hi - lo >= kDynMinElems)      // one launch, tiles in dynamic order
        return launch_fused_single_dyn(grad, master, m, v, par, lo, hi - lo, s, 1, st);
    return walk_range(lo, hi, kFusedWalkChunk, [&](int64_t a, int64_t b, int sync) {
        return launch_fused_tma(grad, master, m, v, par, false, a, b - a, s, 1, st, sync);
    });
}

cudaError_t launch_adamw(const BView& grad, bool grad_by_owner, float* master, float* m, float* v,
                         const BView& par, bool par_by_owner, const Range& r, const AdamScalars& s,
                         cudaStream_t st) {
    const bool by_owner = grad_by_owner || par_by_owner;
    const bool vec = aligned8(grad.off) && aligned8(par.off) &&
                     (!by_owner || (aligned8(r.base) && aligned8(r.shard)));
    const Split sp = split_range(r.lo, r.hi, vec);
    // reduced gradient and parameters both one array (ZeRO-2): the staged kernel with one rank is
    // exactly this update (the mean of one bf16 value is that value; a -0 gradient reads as +0,
    // which changes neither moment nor parameter)
    if (!by_owner && (sp.nvec << 3) >= kTmaMinElems && g_fused_variant.load() != ZS_FUSED_LDG) {
        const void* ps[5] = {grad.ptr.p[0], par.ptr.p[0], master, m, v};
        if (all_device(ps, 5)) {
            const int64_t body_hi = sp.vlo + (sp.nvec << 3);
            cudaError_t e = adamw_tma_walk(grad, master, m, v, par, sp.vlo, body_hi, s, st);
            if (e != cudaErrorNotSupported) {
                if (e != cudaSuccess) return e;
                AdamOp op{grad, par, 0, 0, master, m, v, s, r.base, r.shard};
                Split rest[2] = {split_range(sp.lo, sp.vlo, false), split_range(body_hi, sp.hi, false)};
                for (const Split& f : rest) {
                    if (f.hi <= f.lo) continue;
                    int grid = 0;
                    e = grid_for((const void*)k_adamw, f.hi - f.lo, &grid);
                    if (e != cudaSuccess) return e;
                    e = launch_kernel(k_adamw, dim3(grid), dim3(kThreads), 0, st, op, f);
                    if (e != cudaSuccess) return e;
                }
                return cudaSuccess;
            }
        }
    }
    AdamOp op{grad, par, grad_by_owner ? 1 : 0, par_by_owner ? 1 : 0, master, m, v, s, r.base, r.shard};
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_adamw, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_adamw, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

constexpr int64_t kBulkGatherMinElems = int64_t(1) << 20;

cudaError_t launch_gather(const BView& src, bool src_by_owner, const BView& dst, bool skip_owner,
                          const Range& r, int nd, cudaStream_t st, int sync) {
    const bool by_owner = src_by_owner || skip_owner;
    const bool vec = aligned8(src.off) && aligned8(dst.off) &&
                     (!by_owner || (aligned8(r.base) && aligned8(r.shard)));
    const Split sp = split_range(r.lo, r.hi, vec);
    // one source for every destination: the bulk-store kernel moves the 8-aligned body
    if (!by_owner && (sp.nvec << 3) >= kBulkGatherMinElems) {
        const void* ps[ZS_MAX_RANKS + 1];
        ps[0] = src.ptr.p[0];
        for (int q = 0; q < nd; ++q) ps[q + 1] = dst.ptr.p[q];
        if (all_device(ps, nd + 1)) {
            const int64_t body_hi = sp.vlo + (sp.nvec << 3);
            cudaError_t e = sync == kSyncDynamic && (sp.nvec << 3) >= kDynMinElems
                                ? launch_gather_bulk_dyn(src.ptr.p[0], src.off, dst.ptr, dst.off, sp.vlo, sp.nvec << 3, nd, st)
                                : launch_gather_bulk(src.ptr.p[0], src.off, dst.ptr, dst.off, sp.vlo, sp.nvec << 3, nd, st,
                                                     sync == kSyncDynamic ? (int)kSyncStream : sync);
            if (e != cudaSuccess) return e;
            Split rest[2] = {split_range(sp.lo, sp.vlo, false), split_range(body_hi, sp.hi, false)};
            for (const Split& f : rest) {
                if (f.hi <= f.lo) continue;
#define ZS_GF(N) gather_impl<N>(src, false, dst, false, r, nd, f, st)
                e = [&]() -> cudaError_t { ZS_DISPATCH_ND(nd, ZS_GF) }();
#undef ZS_GF
                if (e != cudaSuccess) return e;
            }
            return cudaSuccess;
        }
    }
    // the streaming kernel reads through L1, so it never starts before its predecessor completes; as
    // the first launch of a walk it also waits before letting its successor launch
    Split ss = sp;
    ss.sync = sync == kSyncWalkFirst ? kSyncWalkFirst : kSyncStream;
#define ZS_GA(N) gather_impl<N>(src, src_by_owner, dst, skip_owner, r, nd, ss, st)
    ZS_DISPATCH_ND(nd, ZS_GA)
#undef ZS_GA
}

void set_fused_variant(int v) { g_fused_variant.store(v); }
int fused_variant() { return g_fused_variant.load(); }

static std::atomic<int> g_dependent_launch{1};
void set_dependent_launch(int on) { g_dependent_launch.store(on ? 1 : 0); }
int dependent_launch() { return g_dependent_launch.load(); }

static cudaError_t launch_fused_ldg(const BView& g, float* master, float* m, float* v, const BView& out,
                                    bool broadcast, const Split& sp, const AdamScalars& s, int nd, cudaStream_t st,
                                    const AccumIn* acc = nullptr) {
    if (acc) {
        if (!broadcast) return cudaErrorNotSupported;
#define ZS_FA(N) fused_impl<N, true, true>(g, master, m, v, out, s, nd, sp, st, acc)
        ZS_DISPATCH_ND(nd, ZS_FA)
#undef ZS_FA
    }
    if (broadcast) {
#define ZS_FB(N) fused_impl<N, true>(g, master, m, v, out, s, nd, sp, st)
        ZS_DISPATCH_ND(nd, ZS_FB)
#undef ZS_FB
    } else {
#define ZS_FS(N) fused_impl<N, false>(g, master, m, v, out, s, nd, sp, st)
        ZS_DISPATCH_ND(nd, ZS_FS)
#undef ZS_FS
    }
}

// True when every pointer is device memory of this context.  The staged kernel's bulk copies are
// only ever pointed at device memory; host (pinned, mapped) or unknown pointers take the streaming
// kernel, whose plain loads and stores reach pinned host memory under unified addressing.
static bool all_device(const void* const* ps, int n) {
    for (int i = 0; i < n; ++i) {
        cudaPointerAttributes at;
        if (cudaPointerGetAttributes(&at, ps[i]) != cudaSuccess) {
            cudaGetLastError();                   // unregistered pointer: clear the error, refuse staging
            return false;
        }
        if (at.type != cudaMemoryTypeDevice) return false;
    }
    return true;
}

bool fused_ptrs_on_device(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast,
                          int nd, const AccumIn* acc) {
    const void* ps[3 * ZS_MAX_RANKS + 3];
    int n = 0;
    for (int q = 0; q < nd; ++q) ps[n++] = g.ptr.p[q];
    if (acc)
        for (int q = 0; q < nd; ++q) ps[n++] = acc->micro.ptr.p[q];
    for (int q = 0; q < (broadcast ? nd : 1); ++q) ps[n++] = out.ptr.p[q];
    ps[n++] = master;
    ps[n++] = m;
    ps[n++] = v;
    return all_device(ps, n);
}

cudaError_t launch_fused(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast,
                         const Range& r, const AdamScalars& s, int nd, cudaStream_t st, StagedPolicy staged_policy,
                         int sync, const AccumIn* acc) {
    if (acc && !broadcast) return cudaErrorNotSupported;
    const bool vec = aligned8(g.off) && aligned8(out.off) && (!acc || aligned8(acc->micro.off));
    Split sp = split_range(r.lo, r.hi, vec);
    if (sync == kSyncDynamic) {
        // one output (the ZeRO-3 update): a long body in one dynamic-order launch, then the fringes;
        // anything else in plain stream order
        sync = kSyncStream;
        const int64_t body_hi = sp.vlo + (sp.nvec << 3);
        if (!broadcast && !acc && (sp.nvec << 3) >= kDynMinElems && fused_dyn_shape(nd) &&
            g_fused_variant.load() != ZS_FUSED_LDG && staged_policy != kStagedNever &&
            (staged_policy == kStagedDeviceKnown || fused_ptrs_on_device(g, master, m, v, out, false, nd))) {
            cudaError_t e = launch_fused_single_dyn(g, master, m, v, out, sp.vlo, sp.nvec << 3, s, nd, st);
            if (e == cudaSuccess && sp.vlo > sp.lo)
                e = launch_fused_ldg(g, master, m, v, out, false, split_range(sp.lo, sp.vlo, false), s, nd, st);
            if (e == cudaSuccess && sp.hi > body_hi)
                e = launch_fused_ldg(g, master, m, v, out, false, split_range(body_hi, sp.hi, false), s, nd, st);
            return e;
        }
    }
    const int variant = g_fused_variant.load();
    const int64_t min_staged = sync == kSyncStream ? kTmaMinElems : kTmaWalkMinElems;
    const bool want_tma = variant == ZS_FUSED_TMA || (variant == ZS_FUSED_AUTO && (sp.nvec << 3) >= min_staged);
    bool staged = want_tma && sp.nvec > 0 && staged_policy != kStagedNever &&
                  (acc ? fused_walk_shape(nd, true) : (nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32));
    // only a staged candidate pays for the pointer queries, and only when the caller has not
    if (staged && staged_policy == kStagedIfDevice)
        staged = fused_ptrs_on_device(g, master, m, v, out, broadcast, nd, acc);
    if (!staged) {
        // the streaming kernel reads through L1, so it never starts before its predecessor completes
        sp.sync = sync == kSyncWalkFirst ? kSyncWalkFirst : kSyncStream;
        return launch_fused_ldg(g, master, m, v, out, broadcast, sp, s, nd, st, acc);
    }
    // staged body, then the at most 14 fringe elements one by one
    const int64_t body_hi = sp.vlo + (sp.nvec << 3);
    cudaError_t e = launch_fused_tma(g, master, m, v, out, broadcast, sp.vlo, sp.nvec << 3, s, nd, st, sync, acc);
    if (e != cudaSuccess) return e;
    if (sp.vlo > sp.lo) {
        e = launch_fused_ldg(g, master, m, v, out, broadcast, split_range(sp.lo, sp.vlo, false), s, nd, st, acc);
        if (e != cudaSuccess) return e;
    }
    if (sp.hi > body_hi)
        e = launch_fused_ldg(g, master, m, v, out, broadcast, split_range(body_hi, sp.hi, false), s, nd, st, acc);
    return e;
}

cudaError_t launch_fused_walk(const BView& g, float* master, float* m, float* v, const BView& out,
                              const std::vector<Range>& ranges, const AdamScalars& s, int nd, cudaStream_t st,
                              StagedPolicy staged_policy, const AccumIn* acc) {
    // Cut points are multiples of the chunk (8-aligned, so a range's pieces keep its own fringes
    // only), none closer than a quarter chunk to a range end, so no piece is a sliver.  Only staged
    // launches overlap: buffers the staged kernel may not touch (pinned host memory) or the streaming
    // variant leave every range whole.
    if (staged_policy == kStagedIfDevice)
        staged_policy = fused_ptrs_on_device(g, master, m, v, out, true, nd, acc) ? kStagedDeviceKnown : kStagedNever;
    const bool chunked = fused_walk_shape(nd, acc != nullptr) && staged_policy != kStagedNever &&
                         g_fused_variant.load() != ZS_FUSED_LDG;
    // One long range (the whole flat space, or touching buckets merged): one launch that takes its tiles
    // in dynamic order, then the fringes off the 8-element grid.
    if (chunked && ranges.size() == 1 && fused_dyn_shape(nd)) {
        const Range& r = ranges[0];
        const Split sp = split_range(r.lo, r.hi, aligned8(g.off) && aligned8(out.off) && (!acc || aligned8(acc->micro.off)));
        if ((sp.nvec << 3) >= kDynMinElems) {
            const int64_t body_hi = sp.vlo + (sp.nvec << 3);
            cudaError_t e = launch_fused_tma_dyn(g, master, m, v, out, sp.vlo, sp.nvec << 3, s, nd, st, acc);
            if (e == cudaSuccess && sp.vlo > sp.lo)
                e = launch_fused_ldg(g, master, m, v, out, true, split_range(sp.lo, sp.vlo, false), s, nd, st, acc);
            if (e == cudaSuccess && sp.hi > body_hi)
                e = launch_fused_ldg(g, master, m, v, out, true, split_range(body_hi, sp.hi, false), s, nd, st, acc);
            return e;
        }
    }
    bool first = true;
    for (const Range& r : ranges) {
        if (r.hi <= r.lo) continue;
        const cudaError_t e = walk_range(r.lo, r.hi, chunked ? kFusedWalkChunk : 0, [&](int64_t a, int64_t b, int sync) {
            return launch_fused(g, master, m, v, out, true, {a, b, r.base, r.shard}, s, nd, st, staged_policy, sync, acc);
        }, first ? (int)kSyncWalkFirst : (int)kSyncWalkNext);
        if (e != cudaSuccess) return e;
        first = false;
    }
    return cudaSuccess;
}

cudaError_t launch_fused_ranges(const BView& g, float* master, float* m, float* v, const BView& out,
                                const std::vector<Range>& ranges, const AdamScalars& s, int nd, cudaStream_t st,
                                StagedPolicy staged_policy) {
    // The order of disjoint ranges is not observable, so ranges that touch are merged (a run of
    // neighbouring buckets, in either order, becomes one range, walked); what stays disjoint is walked
    // range by range, except short runs, which share list launches.
    std::vector<Range> merged;
    for (const Range& r : ranges)
        if (r.hi > r.lo) merged.push_back(r);
    std::sort(merged.begin(), merged.end(), [](const Range& x, const Range& y) { return x.lo < y.lo; });
    size_t w = 0;
    for (size_t i = 0; i < merged.size(); ++i) {
        if (w > 0 && merged[w - 1].hi == merged[i].lo) merged[w - 1].hi = merged[i].hi;
        else merged[w++] = merged[i];
    }
    merged.resize(w);
    if (merged.empty()) return cudaSuccess;
    if (merged.size() == 1) return launch_fused_walk(g, master, m, v, out, merged, s, nd, st, staged_policy);
    const bool vec = aligned8(g.off) && aligned8(out.off);
    std::vector<Split> splits;
    splits.reserve(merged.size());
    int64_t body_total = 0;
    for (const Range& r : merged) {
        splits.push_back(split_range(r.lo, r.hi, vec));
        body_total += splits.back().nvec << 3;
    }
    const int variant = g_fused_variant.load();
    // the list is one launch, so the staged kernel's ramp is paid once for all of it
    bool staged = body_total > 0 && staged_policy != kStagedNever &&
                  (variant == ZS_FUSED_TMA || (variant == ZS_FUSED_AUTO && body_total >= kTmaMinElems)) &&
                  (nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32);
    if (staged && staged_policy == kStagedIfDevice) staged = fused_ptrs_on_device(g, master, m, v, out, true, nd);
    if (!staged) {
        for (const Split& sp : splits) {
            cudaError_t e = launch_fused_ldg(g, master, m, v, out, true, sp, s, nd, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    // Ranges with a body of at least kTmaWalkMinElems are walked (one or more launches each, which
    // overlap: the walk shape streams them at the copy rate, 1 MiB buckets included); the short runs
    // left go through one list launch per kTmaListMax bodies, which pays one ramp for all of them
    // instead of one launch each.
    std::vector<Range> walked;
    std::vector<std::pair<int64_t, int64_t>> bodies;
    bodies.reserve(splits.size());
    cudaError_t e = cudaSuccess;
    for (size_t k = 0; k < splits.size(); ++k) {
        const Split& sp = splits[k];
        if ((sp.nvec << 3) >= kTmaWalkMinElems && fused_walk_shape(nd)) walked.push_back(merged[k]);
        else if (sp.nvec > 0) bodies.emplace_back(sp.vlo, sp.nvec << 3);
    }
    if (!walked.empty()) {
        e = launch_fused_walk(g, master, m, v, out, walked, s, nd, st, kStagedDeviceKnown);
        if (e != cudaSuccess) return e;
    }
    if (!bodies.empty()) {
        e = launch_fused_tma_list(g, master, m, v, out, bodies, s, nd, st);
        if (e != cudaSuccess) return e;
    }
    // fringes of the listed runs (ends off the 8-element grid): at most 14 elements per range; the
    // walked ranges' fringes were launched by the walk
    for (size_t k = 0; k < splits.size(); ++k) {
        const Split& sp = splits[k];
        if ((sp.nvec << 3) >= kTmaWalkMinElems && fused_walk_shape(nd)) continue;
        const int64_t body_hi = sp.nvec > 0 ? sp.vlo + (sp.nvec << 3) : sp.lo;
        const int64_t head_hi = sp.nvec > 0 ? sp.vlo : sp.hi;
        if (head_hi > sp.lo) {
            e = launch_fused_ldg(g, master, m, v, out, true, split_range(sp.lo, head_hi, false), s, nd, st);
            if (e != cudaSuccess) return e;
        }
        if (sp.nvec > 0 && sp.hi > body_hi) {
            e = launch_fused_ldg(g, master, m, v, out, true, split_range(body_hi, sp.hi, false), s, nd, st);
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace zs

namespace zs {

// ------------------------------------------------------------------ naive data parallelism
// "Infra: Data Parallel", section "Naive Data Parallelism": every rank keeps a full replica of
// parameters, gradients and optimizer state; the gradients are all-reduced to their mean and every
// rank applies the same update to its own copy.

template <int ND>
struct AllReduceOp {
    BView g;
    int nd;
    float inv_nd;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int n = ND > 0 ? ND : nd;
        float acc[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            float f[VEC];
            unpack(ld_bf<VEC>(g.ptr.p[q] + (i - g.off)), f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = mean_of_sum<ND>(acc[k], n, inv_nd);
        const BfVec<VEC> w = pack(acc);
#pragma unroll
        for (int q = 0; q < n; ++q) st_bf<VEC>(g.ptr.p[q] + (i - g.off), w);
    }
};

template <int ND>
__global__ void __launch_bounds__(kThreads) k_all_reduce_mean(AllReduceOp<ND> op, Split sp) { for_range(sp, op); }

struct FPtrs {
    float* p[ZS_MAX_RANKS];
};

template <int ND>
struct DpStepOp {
    BView g, out;
    FPtrs master, m, v;
    AdamScalars s;
    int nd;
    float inv_nd;
    template <int VEC>
    __device__ __forceinline__ void run(int64_t i) const {
        const int n = ND > 0 ? ND : nd;
        float acc[VEC], gr[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            float f[VEC];
            unpack(ld_bf<VEC>(g.ptr.p[q] + (i - g.off)), f);
#pragma unroll
            for (int k = 0; k < VEC; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
#pragma unroll
        for (int k = 0; k < VEC; ++k) acc[k] = mean_of_sum<ND>(acc[k], n, inv_nd);
        unpack(pack(acc), gr);                  // every rank receives the same bf16 mean
        // and runs the same update on its own full state; two ranks per pass, both ranks' loads
        // issued before either's stores (the stores may alias nothing the loads read, but the
        // compiler cannot know that, so the order is written out)
#pragma unroll 1
        for (int q = 0; q < n; q += 2) {
            const bool two = q + 1 < n;
            float p[2][VEC], mm[2][VEC], vv[2][VEC];
            ld_f32<VEC>(master.p[q] + i, p[0]);
            ld_f32<VEC>(m.p[q] + i, mm[0]);
            ld_f32<VEC>(v.p[q] + i, vv[0]);
            if (two) {
                ld_f32<VEC>(master.p[q + 1] + i, p[1]);
                ld_f32<VEC>(m.p[q + 1] + i, mm[1]);
                ld_f32<VEC>(v.p[q + 1] + i, vv[1]);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (h == 1 && !two) break;
#pragma unroll
                for (int k = 0; k < VEC; ++k) adamw_elem(gr[k], p[h][k], mm[h][k], vv[h][k], s);
                st_f32<VEC>(master.p[q + h] + i, p[h]);
                st_f32<VEC>(m.p[q + h] + i, mm[h]);
                st_f32<VEC>(v.p[q + h] + i, vv[h]);
                st_bf<VEC>(out.ptr.p[q + h] + (i - out.off), pack(p[h]));
            }
        }
    }
};

template <int ND>
__global__ void __launch_bounds__(kThreads) k_dp_step(DpStepOp<ND> op, Split sp) { for_range(sp, op); }

template <int ND>
static cudaError_t all_reduce_impl(const BView& g, int nd, Split sp, cudaStream_t st) {
    AllReduceOp<ND> op{g, nd, 1.0f / (float)nd};
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_all_reduce_mean<ND>, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_all_reduce_mean<ND>, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

template <int ND>
static cudaError_t dp_step_impl(const BView& g, const BView& out, float* const* master, float* const* m,
                                float* const* v, const AdamScalars& s, int nd, Split sp, cudaStream_t st) {
    DpStepOp<ND> op{};
    op.g = g;
    op.out = out;
    for (int q = 0; q < nd; ++q) {
        op.master.p[q] = master[q];
        op.m.p[q] = m[q];
        op.v.p[q] = v[q];
    }
    op.s = s;
    op.nd = nd;
    op.inv_nd = 1.0f / (float)nd;
    int grid = 0;
    cudaError_t ge = grid_for((const void*)k_dp_step<ND>, sp.nvec > 0 ? sp.nvec : sp.hi - sp.lo, &grid);
    if (ge != cudaSuccess) return ge;
    return launch_kernel(k_dp_step<ND>, dim3(grid), dim3(kThreads), 0, st, op, sp);
}

cudaError_t launch_all_reduce_mean(const BView& g, const Range& r, int nd, cudaStream_t st) {
    const Split sp = split_range(r.lo, r.hi, aligned8(g.off));
    // a body of at least kTmaMinElems in device memory: the staged kernel, in one dynamic-order launch
    // from kDynMinElems on where the rank count has a dynamic-order shape, else walked (pieces cut as in launch_fused_walk, the first waiting for the
    // stream's predecessor, the others streaming while the previous one drains); fringes, short
    // ranges, host memory and other rank counts stream
    const int64_t body = sp.nvec << 3;
    if (body >= kTmaMinElems && g_fused_variant.load() != ZS_FUSED_LDG &&
        (nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32)) {
        const void* ps[ZS_MAX_RANKS];
        for (int q = 0; q < nd; ++q) ps[q] = g.ptr.p[q];
        if (all_device(ps, nd)) {
            const int64_t body_hi = sp.vlo + body;
            cudaError_t e = body >= kDynMinElems && ar_dyn_shape(nd)
                                ? launch_all_reduce_tma(g, sp.vlo, body, nd, st, kSyncDynamic)
                                : walk_range(sp.vlo, body_hi, kFusedWalkChunk, [&](int64_t a, int64_t b, int sync) {
                                      return launch_all_reduce_tma(g, a, b - a, nd, st, sync);
                                  });
            Split rest[2] = {split_range(sp.lo, sp.vlo, false), split_range(body_hi, sp.hi, false)};
            for (const Split& f : rest) {
                if (e != cudaSuccess || f.hi <= f.lo) continue;
#define ZS_ARF(N) all_reduce_impl<N>(g, nd, f, st)
                e = [&]() -> cudaError_t { ZS_DISPATCH_ND(nd, ZS_ARF) }();
#undef ZS_ARF
            }
            return e;
        }
    }
#define ZS_AR(N) all_reduce_impl<N>(g, nd, sp, st)
    ZS_DISPATCH_ND(nd, ZS_AR)
#undef ZS_AR
}

static cudaError_t dp_step_ldg(const BView& g, const BView& out, float* const* master, float* const* m,
                               float* const* v, const Split& sp, const AdamScalars& s, int nd, cudaStream_t st) {
#define ZS_DP(N) dp_step_impl<N>(g, out, master, m, v, s, nd, sp, st)
    ZS_DISPATCH_ND(nd, ZS_DP)
#undef ZS_DP
}

cudaError_t launch_dp_step(const BView& g, const BView& out, float* const* master, float* const* m, float* const* v,
                           const Range& r, const AdamScalars& s, int nd, cudaStream_t st) {
    // The staged kernel streams one rank's state at a time through its ring (an earlier staged
    // variant that held every rank's state of a tile at once measured 88 % of the copy rate at
    // N_d = 8, the register-streaming kernel 92-93 %).  The fused-variant switch selects here too.
    const Split sp = split_range(r.lo, r.hi, aligned8(g.off) && aligned8(out.off));
    const int variant = g_fused_variant.load();
    bool staged = sp.nvec > 0 && (variant == ZS_FUSED_TMA || (variant == ZS_FUSED_AUTO && (sp.nvec << 3) >= kTmaMinElems)) &&
                  (nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32);
    if (staged) {
        const void* ps[5 * ZS_MAX_RANKS];
        int n = 0;
        for (int q = 0; q < nd; ++q) {
            ps[n++] = g.ptr.p[q];
            ps[n++] = out.ptr.p[q];
            ps[n++] = master[q];
            ps[n++] = m[q];
            ps[n++] = v[q];
        }
        staged = all_device(ps, n);
    }
    if (!staged) return dp_step_ldg(g, out, master, m, v, sp, s, nd, st);
    // where the rank count has a walk shape, a body of kDynMinElems or more in one dynamic-order launch
    // (the walk's shapes), a shorter one walked (pieces cut as in launch_fused_walk, the first waiting for the stream's
    // predecessor, the others streaming while the previous one drains), else one launch; then the fringes
    const int64_t body_hi = sp.vlo + (sp.nvec << 3);
    cudaError_t e = cudaSuccess;
    if ((sp.nvec << 3) >= kDynMinElems && dp_walk_shape(nd)) {
        e = launch_dp_tma(g, out, master, m, v, sp.vlo, sp.nvec << 3, s, nd, st, kSyncDynamic);
    } else if (dp_walk_shape(nd)) {
        e = walk_range(sp.vlo, body_hi, kFusedWalkChunk, [&](int64_t a, int64_t b, int sync) {
            return launch_dp_tma(g, out, master, m, v, a, b - a, s, nd, st, sync);
        });
    } else {
        e = launch_dp_tma(g, out, master, m, v, sp.vlo, sp.nvec << 3, s, nd, st);
    }
    if (e != cudaSuccess) return e;
    if (sp.vlo > sp.lo) {
        e = dp_step_ldg(g, out, master, m, v, split_range(sp.lo, sp.vlo, false), s, nd, st);
        if (e != cudaSuccess) return e;
    }
    if (sp.hi > body_hi) e = dp_step_ldg(g, out, master, m, v, split_range(body_hi, sp.hi, false), s, nd, st);
    return e;
}

}  // namespace zs
