// Kernels with bulk-copy (TMA engine) staging, sm_103a: the fused step over one range
// (k_fused_tma) and over a list of ranges (k_fused_tma_list), the reduce-scatter-mean alone
// (k_rs_tma), the gather from one source into N_d destinations with bulk stores
// (k_gather_bulk), and the naive-DP step over N_d full replicated states (k_dp_tma).
//
// The fused step: same arithmetic as the register-streaming fused kernel (reduce-mean over
// ranks, AdamW, bf16 cast, store into every replica: "Infra: Data Parallel",
// ZeRO section), different data movement.  The flat range is cut into tiles
// of T elements.  Each CTA is persistent (one wave of resident CTAs) and owns a ring of
// STAGES shared-memory stages; a stage holds one tile of every rank's bf16
// gradients and of the fp32 master, m and v.  One producer thread issues the
// N_d + 3 one-dimensional bulk copies of a tile (cp.async.bulk, completion
// counted in bytes on the stage's "full" mbarrier, L2 evict-first); NCW
// consumer warps wait for the stage, each thread computes VPT consecutive
// elements from shared memory, streams its results straight to global memory
// and releases the stage on its "empty" mbarrier.  With up to STAGES-1 tiles
// in flight per CTA the loads keep up to ~200 KB of reads outstanding per SM
// independent of register pressure.  The tile shape per rank count and output form (warps,
// elements per thread, ring depth, CTAs per SM) was picked by measurement; ring depth is not
// monotone in benefit on GB300 (for N_d = 8 broadcast, 8 stages of 1024 elements beat both 6-7
// and 16 stages).
//
// Every wait is bounded (clock64 budget).  A wait that runs out sets
// g_zs_device_error, the CTA stops taking tiles, the producer waits (again
// bounded) for the copies it still has in flight, and the kernel returns.
//
// Stage reuse (every staged kernel here).  A consumer thread reads a stage with ordinary
// shared-memory loads (the generic proxy), then arrives on the stage's "empty" barrier
// (mbarrier.arrive.release.cta).  The producer's acquire wait on that barrier sees the phase
// complete once every consumer has arrived, and only then refills the stage with bulk copies,
// which write through the async proxy.  Two rules of the PTX memory model bear on whether a refill
// can land under a consumer's loads:
//   (1) the arrive's release orders the thread's earlier memory accesses before the arrive, for a
//       thread that acquires the barrier's phase, within the generic proxy;
//   (2) accesses to one location through different proxies are ordered only across a proxy fence
//       (fence.proxy.async); a bulk copy's own completion carries one, but nothing orders a
//       generic-proxy read before a later async-proxy write to the same shared memory.
// So release/acquire alone does not promise that a consumer's loads have returned before the
// refill writes the stage, and on GB300 they did not always: a staged all-reduce whose consumers
// arrived right after their loads read, for a few elements in 10^5, the data of the tile S
// positions later in the same stage.  The protocol these kernels rely on is therefore a data
// dependency, not the memory model: a consumer arrives on an empty barrier only after
// instructions that consume every value it loaded from that stage (the global stores of its
// results; a thread that loaded nothing, past the end of a tile, arrives at once, and a thread
// of the list kernel past the end of a tile discards what it loaded).  The arrive cannot issue
// before the loads it depends on have delivered their data, whatever the proxies.  A change that
// moves an arrive above the consuming stores (releasing after the state stores only, say) must
// keep that dependency; tests/test_stage_release.py checks the source for it.
#include <atomic>
#include <memory>
#include <mutex>
#include <type_traits>
#include <unordered_map>
#include <utility>
#include <vector>

#include "device.cuh"

namespace zs {

__device__ unsigned int g_zs_device_error;   // 0 = fine; otherwise a ZS_DEVERR_* code

namespace {

// Launch geometry of a staged kernel on the current device: the SM count and how many CTAs of
// `threads` threads and `smem` bytes of dynamic shared memory fit on one SM.  The first launch of a
// kernel on a device raises its dynamic shared-memory limit (an attribute held per device) and asks
// the runtime; the answer is cached per (device, kernel), so later launches make none of these
// calls (the bucket-by-bucket and per-group paths launch many short kernels back to back).  Every
// runtime error is returned.
cudaError_t staged_geometry(const void* kern, int threads, int smem, int* sms, int* per_sm) {
    static std::mutex mu;
    static std::unordered_map<uint64_t, std::pair<int, int>> cache;   // (device, kernel) -> (sms, per_sm)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t key = ((uint64_t)(uintptr_t)kern) ^ ((uint64_t)(uint32_t)dev << 56);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) {
        *sms = it->second.first;
        *per_sm = it->second.second;
        return cudaSuccess;
    }
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int n_sm = 0, occ = 0;
    e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, smem);
    if (e != cudaSuccess) return e;
    if (n_sm < 1 || occ < 1) return cudaErrorInvalidConfiguration;     // the kernel does not fit on an SM
    cache.emplace(key, std::make_pair(n_sm, occ));
    *sms = n_sm;
    *per_sm = occ;
    return cudaSuccess;
}

// Host-side guard of the bulk-copy rules before a staged launch: a one-dimensional bulk copy must
// start at a 16-byte-aligned address and move a multiple of 16 bytes.  The staged kernels copy tiles
// of whole 8-element groups starting at body start + k * T (T a multiple of 8), so it suffices that
// the body [lo, lo + n) has lo and n multiples of 8 and that element lo of every array the kernel
// touches is 16-byte aligned.  The callers guarantee this; a launch that would break it is refused
// (cudaErrorMisalignedAddress) instead of faulting the GPU.
bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }
bool body_ok(int64_t lo, int64_t n) { return (lo & 7) == 0 && (n & 7) == 0 && n > 0; }
template <class T>
bool at_ok(const T* base, int64_t elems) {
    return aligned16((const void*)((uintptr_t)base + (uintptr_t)(elems * (int64_t)sizeof(T))));
}

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}

// The arrive and the wait spell out the semantics PTX gives them by default (release and acquire
// at CTA scope), so what the stage protocol below rests on is visible at the call.
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(su32(b)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete; false once `limit` cycles have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, long long limit) {
    if (mbar_try_wait(b, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(b, parity)) {
        if (clock64() - t0 > limit) return false;
    }
    return true;
}

__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// One-dimensional bulk copy global -> shared; bytes and both addresses multiples of 16.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            su32(dst)),
        "l"(src), "r"(bytes), "r"(su32(bar)), "l"(pol)
        : "memory");
}

__device__ __forceinline__ void flag_error(unsigned int code) { atomicCAS(&g_zs_device_error, 0u, code); }

// One-dimensional bulk copy shared -> global, tracked in this thread's bulk async-group.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(su32(src)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until this thread's committed bulk stores have finished reading shared memory / have completed.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// VPT consecutive bf16 values from shared memory as fp32.
template <int VPT>
__device__ __forceinline__ void lds_bf(const uint16_t* p, float (&f)[VPT]) {
    if constexpr (VPT == 8) {
        const uint4 w = *reinterpret_cast<const uint4*>(p);
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
        f[4] = bf16_lo(w.z); f[5] = bf16_hi(w.z); f[6] = bf16_lo(w.w); f[7] = bf16_hi(w.w);
    } else {
        const uint2 w = *reinterpret_cast<const uint2*>(p);
        f[0] = bf16_lo(w.x); f[1] = bf16_hi(w.x); f[2] = bf16_lo(w.y); f[3] = bf16_hi(w.y);
    }
}

template <int VPT>
__device__ __forceinline__ void lds_f32(const float* p, float (&f)[VPT]) {
#pragma unroll
    for (int k = 0; k < VPT; k += 4) {
        const float4 a = *reinterpret_cast<const float4*>(p + k);
        f[k] = a.x; f[k + 1] = a.y; f[k + 2] = a.z; f[k + 3] = a.w;
    }
}

template <int VPT>
__device__ __forceinline__ void stg_f32(float* p, const float (&f)[VPT]) {
#pragma unroll
    for (int k = 0; k < VPT; k += 4) __stcs(reinterpret_cast<float4*>(p + k), make_float4(f[k], f[k + 1], f[k + 2], f[k + 3]));
}

}  // namespace

struct TmaArgs {
    Ptrs g;               // rank gradients; element i of rank q at g.p[q] + (i - g_off)
    int64_t g_off;
    Ptrs out;             // outputs; BROADCAST: every rank's replica, else out.p[0] only
    int64_t out_off;
    float *master, *m, *v;
    AdamScalars s;
    int64_t lo, n;        // body [lo, lo + n): lo, n and lo - g_off, lo - out_off multiples of 8
    int nd;
    float inv_nd;
    long long wait_limit; // cycles a wait may take before the kernel gives up
    long long drain_limit;// cycles to wait for copies still in flight after giving up
    int sync;             // LaunchSync: order against the previous kernel on the stream
    unsigned int* order;  // dynamic tile order (k_fused_tma_dyn): the launch's tile counter and finish
                          // counter, order[0] and order[1]; null for the static order
};

// The fused step with the last micro-batch's accumulation folded in (AccumIn): `a.g` holds the
// accumulators, `micro` the micro-batch gradients; rank q's gradient is bf16(acc_q + micro_q * scale).
struct TmaAccArgs {
    TmaArgs a;
    Ptrs micro;           // element i of rank q at micro.p[q] + (i - micro_off); lo - micro_off a multiple of 8
    int64_t micro_off;
    float scale;
};

// A list of bodies stepped by one launch (the buckets of one call, in the caller's order): body r
// is [lo[r], lo[r] + n[r]) with the same alignment rules as TmaArgs' body, and first[r] is the
// number of tiles of the bodies before it (first[nr] = all tiles).  The kernel walks the
// concatenation of the bodies' tiles, so a CTA's tiles follow the list order.
constexpr int kTmaListMax = 128;   // bodies per launch (the table is staged in shared memory)
struct TmaListArgs {
    TmaArgs a;            // everything but lo and n
    int nr;
    int64_t total_tiles;  // first[nr]
    int64_t lo[kTmaListMax];
    int64_t n[kTmaListMax];
    int32_t first[kTmaListMax + 1];
};

namespace {

// A list launch copies the body table from the kernel parameter into shared memory once per CTA,
// reading the parameter with compile-time indices only: indexing a __grid_constant__ parameter with
// a run-time index turns every parameter access of the kernel into a generic load, which measured
// ~4 % slower on GB300.  Each thread then walks its CTA's tiles in increasing order, keeping the
// current body in registers and reading the shared table only when a tile lies past it.
struct ListTable {
    int64_t lo[kTmaListMax];
    int64_t n[kTmaListMax];
    int32_t first[kTmaListMax + 1];
};
constexpr int kListTableBytes = (int)((sizeof(ListTable) + 127) / 128 * 128);

__device__ __forceinline__ void list_table_fill(const TmaListArgs& l, ListTable* t, int lane) {
#pragma unroll
    for (int q = 0; q < kTmaListMax; ++q) {
        if ((q & 31) == lane) {
            t->lo[q] = l.lo[q];
            t->n[q] = l.n[q];
            t->first[q] = l.first[q];
        }
    }
    if (lane == 0) t->first[kTmaListMax] = l.first[kTmaListMax];
}

}  // namespace

// Tile and ring geometry: T elements per tile, as many stages as fit in
// BUDGET bytes of shared memory (at most MAXST), 256 bytes of barriers first.
template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
struct TmaShape {
    static constexpr int kT = NCW * 32 * VPT;                           // elements per tile
    static constexpr int kStageBytes = kT * (2 * ND + 12);
    static constexpr int kFit = (BUDGET - 256) / kStageBytes;
    static constexpr int kStages = kFit > MAXST ? MAXST : kFit;
    static constexpr int kSmem = 256 + kStages * kStageBytes;
    static_assert(kStages >= 2, "tile too large for a 2-stage ring");
    static_assert(2 * kStages * 8 <= 256, "barriers must fit in the first 256 bytes");
};

// ACC: every rank's gradient tile is formed from two staged tiles, its accumulator (a.g) and the
// last micro-batch (micro), so a stage holds 2 N_d bf16 tiles ahead of the fp32 state.
//
// DYN: the tiles are taken in dynamic order.  The producer takes its next tile from the launch's tile
// counter (a.order[0], an atomic add, so the whole grid works through the range front to back and
// its accesses stay close together) and publishes the tile index in the stage's record before the
// stage's copies; a record past the last tile tells the consumers that the CTA is done.
template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST, int BUDGET, bool ACC = false, bool DYN = false>
__device__ __forceinline__ void fused_tma_body(const TmaArgs& a, const Ptrs& micro, int64_t micro_off, float scale) {
    constexpr int NG = ACC ? 2 * ND : ND;                 // bf16 tiles per stage
    using Sh = TmaShape<NG, NCW, VPT, MAXST, BUDGET>;
    constexpr int T = Sh::kT;
    constexpr int S = Sh::kStages;
    static_assert(!DYN || S <= 8, "the dynamic order's stage records sit behind the barriers");
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    int64_t* rec = reinterpret_cast<int64_t*>(smem + 128);   // DYN: the tile of each stage
    uint8_t* stages = smem + 256;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int64_t ntiles = (a.n + T - 1) / T;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = evict_first_policy();
            int64_t j = 0;
            bool ok = true;
            for (int64_t tile = DYN ? 0 : blockIdx.x; DYN || tile < ntiles; tile += gridDim.x, ++j) {
                const int s = (int)(j % S);
                if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), a.wait_limit)) {
                    flag_error(ZS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                if constexpr (DYN) {
                    tile = (int64_t)atomicAdd(a.order, 1u);
                    rec[s] = tile;                        // published by the arrive below (release)
                    if (tile >= ntiles) {
                        mbar_arrive(&full[s]);            // no copies: the consumers read the end mark
                        break;
                    }
                }
                const int64_t i0 = a.lo + tile * T;
                const int64_t rem = a.n - tile * T;
                const uint32_t len = (uint32_t)(rem < T ? rem : T);
                uint8_t* st = stages + (size_t)s * Sh::kStageBytes;
                mbar_expect_tx(&full[s], len * (2u * NG + 12u));
#pragma unroll
                for (int q = 0; q < ND; ++q)
                    bulk_load(st + (size_t)q * T * 2, a.g.p[q] + (i0 - a.g_off), len * 2u, &full[s], pol);
                if constexpr (ACC) {
#pragma unroll
                    for (int q = 0; q < ND; ++q)
                        bulk_load(st + (size_t)(ND + q) * T * 2, micro.p[q] + (i0 - micro_off), len * 2u, &full[s], pol);
                }
                float* sf = reinterpret_cast<float*>(st + (size_t)NG * T * 2);
                bulk_load(sf, a.master + i0, len * 4u, &full[s], pol);
                bulk_load(sf + T, a.m + i0, len * 4u, &full[s], pol);
                bulk_load(sf + 2 * T, a.v + i0, len * 4u, &full[s], pol);
            }
            if (!ok) {
                // drain: wait (bounded) for the copies issued into stages not yet consumed
                const int64_t issued = j;
                for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k)
                    mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
            }
        }
        return;
    }

    // ---------------- consumers
    const int ct = threadIdx.x - 32;                  // 0 .. NCW*32-1
    const int e = ct * VPT;                           // this thread's first element in a tile
    const int n = ND;
    int64_t j = 0;
    for (int64_t tile = DYN ? 0 : blockIdx.x; DYN || tile < ntiles; tile += gridDim.x, ++j) {
        const int s = (int)(j % S);
        if (!mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_CONSUMER_WAIT);
            return;
        }
        if constexpr (DYN) {
            tile = rec[s];
            if (tile >= ntiles) return;                   // the producer's end mark
        }
        const int64_t i0 = a.lo + tile * T;
        const int64_t rem = a.n - tile * T;
        const int len = (int)(rem < T ? rem : T);
        if (e < len) {
            const uint8_t* st = stages + (size_t)s * Sh::kStageBytes;
            const uint16_t* sg = reinterpret_cast<const uint16_t*>(st);
            const float* sf = reinterpret_cast<const float*>(st + (size_t)NG * T * 2);
            float acc[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) acc[k] = 0.0f;
#pragma unroll
            for (int q = 0; q < n; ++q) {
                float f[VPT];
                lds_bf<VPT>(sg + (size_t)q * T + e, f);
                if constexpr (ACC) {
                    // rank q's gradient: accumulator plus micro-batch, rounded to bf16 as stored
                    float b[VPT];
                    lds_bf<VPT>(sg + (size_t)(ND + q) * T + e, b);
#pragma unroll
                    for (int k = 0; k < VPT; ++k) f[k] = bf16_to_f32(f32_to_bf16(accumulate_elem(f[k], b[k], scale)));
                }
#pragma unroll
                for (int k = 0; k < VPT; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
            }
            float p[VPT], mm[VPT], vv[VPT];
            lds_f32<VPT>(sf + e, p);
            lds_f32<VPT>(sf + T + e, mm);
            lds_f32<VPT>(sf + 2 * T + e, vv);
            uint32_t gw[VPT / 2];
#pragma unroll
            for (int k = 0; k < VPT; k += 2)
                gw[k / 2] = pack_bf16x2(mean_of_sum<ND>(acc[k], n, a.inv_nd), mean_of_sum<ND>(acc[k + 1], n, a.inv_nd));
#pragma unroll
            for (int k = 0; k < VPT; k += 2) {
                adamw_elem(bf16_lo(gw[k / 2]), p[k], mm[k], vv[k], a.s);
                adamw_elem(bf16_hi(gw[k / 2]), p[k + 1], mm[k + 1], vv[k + 1], a.s);
            }
            const int64_t i = i0 + e;
            stg_f32<VPT>(a.master + i, p);
            stg_f32<VPT>(a.m + i, mm);
            stg_f32<VPT>(a.v + i, vv);
            uint32_t pw[VPT / 2];
#pragma unroll
            for (int k = 0; k < VPT; k += 2) pw[k / 2] = pack_bf16x2(p[k], p[k + 1]);
            if constexpr (VPT == 8) {
                const uint4 w = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                if constexpr (BROADCAST) {
#pragma unroll
                    for (int q = 0; q < n; ++q) __stcs(reinterpret_cast<uint4*>(a.out.p[q] + (i - a.out_off)), w);
                } else {
                    __stcs(reinterpret_cast<uint4*>(a.out.p[0] + (i - a.out_off)), w);
                }
            } else {
                const uint2 w = make_uint2(pw[0], pw[1]);
                if constexpr (BROADCAST) {
#pragma unroll
                    for (int q = 0; q < n; ++q) __stcs(reinterpret_cast<uint2*>(a.out.p[q] + (i - a.out_off)), w);
                } else {
                    __stcs(reinterpret_cast<uint2*>(a.out.p[0] + (i - a.out_off)), w);
                }
            }
            // The stage is released after the stores, which consume everything read from it (the
            // stage reuse protocol at the top of this file); measured cost: none (11.27 against
            // 11.30 ms per step).
            mbar_arrive(&empty[s]);
        } else {
            mbar_arrive(&empty[s]);
        }
    }
}

// The step over one range; the body returns early (producer lanes, a wait that ran out) into the
// launch-order epilogue, which a kSyncWalkNext launch needs on every exit path.
template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST = 16, int BUDGET = 227 * 1024>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma(const __grid_constant__ TmaArgs a) {
    dependent_launch_prologue(a.sync);
    fused_tma_body<ND, NCW, VPT, BROADCAST, MAXST, BUDGET>(a, a.g, 0, 0.0f);
    dependent_launch_epilogue(a.sync);
}

// The broadcast step with the last micro-batch's accumulation folded in (TmaAccArgs).
// The broadcast step over one range in one persistent launch that takes its tiles in dynamic order
// (DYN in the body).  The launch's counters, order[0] (tiles handed out) and order[1] (CTAs
// finished), start at zero; the last CTA to finish sets both back to zero for the next launch that
// draws the same pair.
__device__ __forceinline__ void dyn_order_finish(unsigned int* order) {
    __syncthreads();                                      // every thread of the CTA is past the body
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(order + 1, 1u) == gridDim.x - 1) {  // the last CTA: no producer draws any more
            atomicExch(order, 0u);
            atomicExch(order + 1, 0u);
        }
    }
}

template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma_dyn(const __grid_constant__ TmaArgs a) {
    dependent_launch_prologue(kSyncStream);
    fused_tma_body<ND, NCW, VPT, true, MAXST, BUDGET, false, true>(a, a.g, 0, 0.0f);
    dyn_order_finish(a.order);
}

// The same with the last micro-batch's accumulation folded in (as k_fused_tma_acc).
template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma_acc_dyn(const __grid_constant__ TmaAccArgs x) {
    dependent_launch_prologue(kSyncStream);
    fused_tma_body<ND, NCW, VPT, true, MAXST, BUDGET, true, true>(x.a, x.micro, x.micro_off, x.scale);
    dyn_order_finish(x.a.order);
}

// The single-output step (the ZeRO-3 reduce-scatter + update of one unit) in one dynamic-order launch.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma_single_dyn(const __grid_constant__ TmaArgs a) {
    dependent_launch_prologue(kSyncStream);
    fused_tma_body<ND, NCW, VPT, false, MAXST, BUDGET, false, true>(a, a.g, 0, 0.0f);
    dyn_order_finish(a.order);
}

template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma_acc(const __grid_constant__ TmaAccArgs x) {
    dependent_launch_prologue(x.a.sync);
    fused_tma_body<ND, NCW, VPT, true, MAXST, BUDGET, true>(x.a, x.micro, x.micro_off, x.scale);
    dependent_launch_epilogue(x.a.sync);
}

// The broadcast step over a list of disjoint bodies in one launch (bodies that touch are merged
// on the host, so this serves scattered subsets of buckets).  The producer walks the bodies in
// table order, taking the tiles t of their concatenation with t = blockIdx.x mod gridDim.x, and
// publishes each stage's tile (first element, length) in shared memory before arriving on the
// stage's full barrier; after its last tile it publishes length 0 and arrives without data, which
// ends the consumers' loop.  The consumers' per-tile work is that of k_fused_tma; they read the
// tile from shared memory instead of computing it (the kernel stays a separate loop from
// k_fused_tma's: folding both into one generic loop cost the single-range kernel ~3 % on GB300).
template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_fused_tma_list(const __grid_constant__ TmaListArgs l) {
    dependent_launch_prologue();
    const TmaArgs& a = l.a;
    using Sh = TmaShape<ND, NCW, VPT, MAXST, BUDGET>;
    constexpr int T = Sh::kT;
    constexpr int S = Sh::kStages;
    static_assert(2 * S * 8 + 12 * S <= 256, "barriers and the tile table share the first 256 bytes");
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    int64_t* meta_i0 = reinterpret_cast<int64_t*>(smem + 2 * S * 8);
    uint32_t* meta_len = reinterpret_cast<uint32_t*>(smem + 2 * S * 8 + 8 * S);
    ListTable* table = reinterpret_cast<ListTable*>(smem + 256);
    uint8_t* stages = smem + 256 + kListTableBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) list_table_fill(l, table, lane);
    __syncthreads();

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = evict_first_policy();
            const int64_t G = gridDim.x;
            int64_t j = 0;
            bool ok = true;
            for (int r = 0; r < l.nr && ok; ++r) {
                const int64_t f0 = table->first[r], f1 = table->first[r + 1];
                const int64_t blo = table->lo[r], bn = table->n[r];
                for (int64_t k = ((int64_t)blockIdx.x - f0 % G + G) % G; f0 + k < f1; k += G, ++j) {
                    const int s = (int)(j % S);
                    if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), a.wait_limit)) {
                        flag_error(ZS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    const int64_t i0 = blo + k * T;
                    const int64_t rem = bn - k * T;
                    const uint32_t len = (uint32_t)(rem < T ? rem : T);
                    meta_i0[s] = i0;                     // ordered before the arrive below (release)
                    meta_len[s] = len;
                    uint8_t* st = stages + (size_t)s * Sh::kStageBytes;
                    mbar_expect_tx(&full[s], len * (2u * ND + 12u));
#pragma unroll
                    for (int q = 0; q < ND; ++q)
                        bulk_load(st + (size_t)q * T * 2, a.g.p[q] + (i0 - a.g_off), len * 2u, &full[s], pol);
                    float* sf = reinterpret_cast<float*>(st + (size_t)ND * T * 2);
                    bulk_load(sf, a.master + i0, len * 4u, &full[s], pol);
                    bulk_load(sf + T, a.m + i0, len * 4u, &full[s], pol);
                    bulk_load(sf + 2 * T, a.v + i0, len * 4u, &full[s], pol);
                }
            }
            if (ok) {
                // the end: a stage with length 0 and no data
                const int s = (int)(j % S);
                if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), a.wait_limit)) {
                    flag_error(ZS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                } else {
                    meta_len[s] = 0;
                    mbar_arrive(&full[s]);
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies issued into stages not yet consumed
                const int64_t issued = j;
                for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k)
                    mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
            }
        }
        return;
    }

    // ---------------- consumers
    const int ct = threadIdx.x - 32;                  // 0 .. NCW*32-1
    const int e = ct * VPT;                           // this thread's first element in a tile
    const int n = ND;
    for (int64_t j = 0;; ++j) {
        const int s = (int)(j % S);
        if (!mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_CONSUMER_WAIT);
            return;
        }
        // the stage's data is read and computed on before its tile record is needed (a thread past the
        // tile's end works on stale values of the stage and stores nothing), so the shared-memory
        // reads of the record and of the data are issued together
        const int64_t i0 = meta_i0[s];
        const int len = (int)meta_len[s];
        const uint8_t* st = stages + (size_t)s * Sh::kStageBytes;
        const uint16_t* sg = reinterpret_cast<const uint16_t*>(st);
        const float* sf = reinterpret_cast<const float*>(st + (size_t)ND * T * 2);
        float acc[VPT];
#pragma unroll
        for (int k = 0; k < VPT; ++k) acc[k] = 0.0f;
#pragma unroll
        for (int q = 0; q < n; ++q) {
            float f[VPT];
            lds_bf<VPT>(sg + (size_t)q * T + e, f);
#pragma unroll
            for (int k = 0; k < VPT; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
        float p[VPT], mm[VPT], vv[VPT];
        lds_f32<VPT>(sf + e, p);
        lds_f32<VPT>(sf + T + e, mm);
        lds_f32<VPT>(sf + 2 * T + e, vv);
        if (len == 0) return;                            // the closing stage
        uint32_t gw[VPT / 2];
#pragma unroll
        for (int k = 0; k < VPT; k += 2)
            gw[k / 2] = pack_bf16x2(mean_of_sum<ND>(acc[k], n, a.inv_nd), mean_of_sum<ND>(acc[k + 1], n, a.inv_nd));
#pragma unroll
        for (int k = 0; k < VPT; k += 2) {
            adamw_elem(bf16_lo(gw[k / 2]), p[k], mm[k], vv[k], a.s);
            adamw_elem(bf16_hi(gw[k / 2]), p[k + 1], mm[k + 1], vv[k + 1], a.s);
        }
        if (e < len) {
            const int64_t i = i0 + e;
            stg_f32<VPT>(a.master + i, p);
            stg_f32<VPT>(a.m + i, mm);
            stg_f32<VPT>(a.v + i, vv);
            uint32_t pw[VPT / 2];
#pragma unroll
            for (int k = 0; k < VPT; k += 2) pw[k / 2] = pack_bf16x2(p[k], p[k + 1]);
            if constexpr (VPT == 8) {
                const uint4 w = make_uint4(pw[0], pw[1], pw[2], pw[3]);
#pragma unroll
                for (int q = 0; q < n; ++q) __stcs(reinterpret_cast<uint4*>(a.out.p[q] + (i - a.out_off)), w);
            } else {
                const uint2 w = make_uint2(pw[0], pw[1]);
#pragma unroll
                for (int q = 0; q < n; ++q) __stcs(reinterpret_cast<uint2*>(a.out.p[q] + (i - a.out_off)), w);
            }
        }
        mbar_arrive(&empty[s]);                          // after the stores: see k_fused_tma
    }
}

// ------------------------------------------------------------------ gather with bulk stores
// One source, N_d destinations (the all-gather from shards and the ZeRO-3 unit gather:
// "Infra: Data Parallel", ZeRO section).  Each CTA is one warp with a ring of S shared-memory
// stages of T bf16 elements: lane 0 loads a tile with one bulk copy, then lanes 0..31 issue the
// N_d bulk stores of that tile (shared -> each destination) in parallel; a stage is refilled once
// every lane's stores have read it.  The tile shape was measured on GB300 (tiles of 4K-32K
// elements, 2-6 stages, 1-16 CTAs per SM in the grid, every N_d): 16K-element tiles in a 4-stage
// ring (128 KB, so one CTA resident per SM, up to 4 x 32 KB x N_d bytes of stores in flight) with a
// grid of 16 CTAs per SM streamed at 99.6-107 % of the measured copy rate for N_d = 2..32, against
// 94.5-100.7 % for 8K-element tiles in 2 stages; a read-light stream (1 read : N_d writes) can pass
// a 1:1 copy's rate.

struct GatherBulkArgs {
    const uint16_t* src;
    int64_t src_off;      // element i of the source at src + (i - src_off)
    Ptrs dst;
    int64_t dst_off;      // element i of destination q at dst.p[q] + (i - dst_off)
    int64_t lo, n;        // body [lo, lo + n): multiples of 8, and lo - src_off, lo - dst_off too
    int nd;
    int T;                // elements per tile (multiple of 8)
    long long wait_limit, drain_limit;
    int sync;             // LaunchSync: the loads are bulk copies, so a later launch of a walk may stream at once
    unsigned int* order;  // k_gather_bulk_dyn: the launch's tile and finish counters
};

template <int S>
__global__ void __launch_bounds__(32) k_gather_bulk(const __grid_constant__ GatherBulkArgs a) {
    dependent_launch_prologue(a.sync);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    uint16_t* buf = reinterpret_cast<uint16_t*>(smem + 128);
    const int lane = threadIdx.x;
    const int T = a.T;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const int64_t ntiles = (a.n + T - 1) / T;
    auto tile_len = [&](int64_t tl) -> uint32_t {
        const int64_t rem = a.n - tl * T;
        return (uint32_t)(rem < T ? rem : T);
    };
    auto load = [&](int64_t tl, int64_t j) {             // lane 0 only
        const int s = (int)(j % S);
        const uint32_t len = tile_len(tl);
        mbar_expect_tx(&bar[s], len * 2u);
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         su32(buf + (size_t)s * T)),
                     "l"(a.src + (a.lo + tl * T - a.src_off)), "r"(len * 2u), "r"(su32(&bar[s]))
                     : "memory");
    };
    int64_t issued = 0, next = blockIdx.x;
    for (; issued < S && next < ntiles; ++issued, next += gridDim.x)
        if (lane == 0) load(next, issued);
    int64_t j = 0;
    bool ok = true;
    for (int64_t tl = blockIdx.x; tl < ntiles; tl += gridDim.x, ++j) {
        const int s = (int)(j % S);
        if (!mbar_wait(&bar[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_GATHER_WAIT);
            ok = false;
            break;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int64_t i = a.lo + tl * T;
        const uint32_t bytes = tile_len(tl) * 2u;
        for (int q = lane; q < a.nd; q += 32) bulk_store(a.dst.p[q] + (i - a.dst_off), buf + (size_t)s * T, bytes);
        bulk_commit();
        if (next < ntiles) {
            bulk_wait_read_all();                        // every lane's stores have read the stage
            __syncwarp();
            if (lane == 0) load(next, issued);
            ++issued;
            next += gridDim.x;
        }
    }
    if (!ok && lane == 0)                                // loads still in flight into the ring
        for (int64_t k = j; k < issued; ++k) mbar_wait(&bar[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
    bulk_wait_all();
    dependent_launch_epilogue(a.sync);
}

// The gather in one dynamic-order launch: lane 0 takes each next tile from the launch's tile counter
// (a.order[0]) and records it in the stage (rec[s]) before the stage's bulk load; the warp reads the
// record after a __syncwarp.  A record past the last tile ends the CTA; the last CTA to finish sets
// the counters back to zero (dyn_order_finish).
template <int S>
__global__ void __launch_bounds__(32) k_gather_bulk_dyn(const __grid_constant__ GatherBulkArgs a) {
    static_assert(S <= 8, "barriers and records share the first 128 bytes");
    dependent_launch_prologue(kSyncStream);
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int64_t* rec = reinterpret_cast<int64_t*>(smem + 64);
    uint16_t* buf = reinterpret_cast<uint16_t*>(smem + 128);
    const int lane = threadIdx.x;
    const int T = a.T;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&bar[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    const int64_t ntiles = (a.n + T - 1) / T;
    auto take = [&](int s) {                             // lane 0: the next tile into stage s
        const int64_t tl = (int64_t)atomicAdd(a.order, 1u);
        rec[s] = tl;
        if (tl < ntiles) {
            const int64_t rem = a.n - tl * T;
            const uint32_t len = (uint32_t)(rem < T ? rem : T);
            mbar_expect_tx(&bar[s], len * 2u);
            asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                             su32(buf + (size_t)s * T)),
                         "l"(a.src + (a.lo + tl * T - a.src_off)), "r"(len * 2u), "r"(su32(&bar[s]))
                         : "memory");
        }
    };
    if (lane == 0)
        for (int s = 0; s < S; ++s) take(s);
    __syncwarp();
    int64_t j = 0;
    bool ok = true;
    for (;; ++j) {
        const int s = (int)(j % S);
        const int64_t tl = rec[s];
        if (tl >= ntiles) break;
        if (!mbar_wait(&bar[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_GATHER_WAIT);
            ok = false;
            break;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        const int64_t i = a.lo + tl * T;
        const int64_t rem = a.n - tl * T;
        const uint32_t bytes = (uint32_t)(rem < T ? rem : T) * 2u;
        for (int q = lane; q < a.nd; q += 32) bulk_store(a.dst.p[q] + (i - a.dst_off), buf + (size_t)s * T, bytes);
        bulk_commit();
        bulk_wait_read_all();                            // every lane's stores have read the stage
        __syncwarp();
        if (lane == 0) take(s);
        __syncwarp();
    }
    if (!ok && lane == 0)                                // loads still in flight into the ring
        for (int64_t k = j; k < j + S; ++k)
            if (rec[k % S] < ntiles) mbar_wait(&bar[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
    bulk_wait_all();
    dyn_order_finish(a.order);
}

namespace {

int64_t host_tiles(const TmaArgs& a, int T) { return (a.n + T - 1) / T; }

template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST, int BUDGET>
auto pick_kernel(const TmaArgs*) { return k_fused_tma<ND, NCW, VPT, BROADCAST, MAXST, BUDGET>; }
template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST, int BUDGET>
auto pick_kernel(const TmaListArgs*) {
    static_assert(BROADCAST, "lists are stepped by the broadcast form only");
    return k_fused_tma_list<ND, NCW, VPT, MAXST, BUDGET>;
}
int64_t host_tiles(const TmaListArgs& l, int) { return l.total_tiles; }
template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST, int BUDGET>
auto pick_kernel(const TmaAccArgs*) {
    static_assert(BROADCAST, "the accumulating step has the broadcast form only");
    return k_fused_tma_acc<ND, NCW, VPT, MAXST, BUDGET>;
}
int64_t host_tiles(const TmaAccArgs& x, int T) { return (x.a.n + T - 1) / T; }

// walk: a launch of a walk over disjoint ranges whose CTAs leave room for the next launch's.  A body
// of at most one tile per resident CTA then takes one CTA per SM, so the next launch of the walk
// finds a free slot on every SM while this one runs (measured on GB300 with the walk shape, 1 MiB
// buckets at N_d = 8: 98.5 % of the copy rate against 87.8 % with every slot filled); larger bodies
// fill every slot.
template <int ND, int NCW, int VPT, bool BROADCAST, int MAXST, int BUDGET, class Args>
cudaError_t tma_impl(const Args& a, cudaStream_t st, bool walk = false) {
    using Sh = TmaShape<std::is_same<Args, TmaAccArgs>::value ? 2 * ND : ND, NCW, VPT, MAXST, BUDGET>;
    constexpr int kSmem = Sh::kSmem + (std::is_same<Args, TmaListArgs>::value ? kListTableBytes : 0);
    static_assert(kSmem <= 232448, "shared memory above the per-CTA limit");
    auto kern = pick_kernel<ND, NCW, VPT, BROADCAST, MAXST, BUDGET>(static_cast<const Args*>(nullptr));
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)kern, 32 * (NCW + 1), kSmem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = host_tiles(a, Sh::kT);
    if (ntiles < 1) return cudaSuccess;
    if (walk && ntiles <= (int64_t)sms * per_sm) per_sm = 1;
    const int64_t cap = (int64_t)sms * per_sm;          // persistent: one wave of resident CTAs
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    return launch_kernel(kern, dim3(grid), dim3(32 * (NCW + 1)), kSmem, st, a);
}

template <int V>
using IC = std::integral_constant<int, V>;
template <bool V>
using BC = std::integral_constant<bool, V>;

// Calls f(ND, NCW, VPT, BROADCAST, MAXST, BUDGET) (as integral constants) with the measured shape for
// this rank count and output form; cudaErrorNotSupported when there is none.
// Shapes per rank count, chosen by measurement on GB300 (a grid of warps x elements per thread x
// ring depth per rank count and output form, on 2^28-element buffers, then the leaders re-timed
// three times interleaved): consumer warps, elements per thread, stage cap, shared-memory budget
// (the ring takes min(cap, what fits); 115712 bytes lets two CTAs share an SM).  The single-output
// form (ZeRO-3 update, standalone AdamW with N_d = 1) is read-heavy: at N_d = 8 the broadcast
// shape reaches only ~74 % there, while three small CTAs per SM (2 warps x 512, 4 stages) stream
// at the copy rate.  At N_d = 1 (one AdamW per 28 bytes moved) the consumers' arithmetic sets the
// pace: 8 consumer warps per SM (one CTA, 2048-element tiles, 8 stages) reached 98.8 % of the copy
// rate on the Llama-1.3B shard arrays against 96.8 % for two 4-warp CTAs and 53.5 % for one.
template <class F>
cudaError_t with_shape(bool broadcast, int nd, F&& f) {
#define ZS_TMA(ND_, NCW_, VPT_, MAXST_, BUDGET_, BROADCAST_) \
    return f(IC<ND_>{}, IC<NCW_>{}, IC<VPT_>{}, BC<BROADCAST_>{}, IC<MAXST_>{}, IC<BUDGET_>{})
    // The relative placement of the N_d rank buffers and the state arrays in memory moves the best
    // broadcast shape by a few per cent, so each shape below was confirmed on the benchmark's own
    // 2^28+7-element buffers (N_d = 4: 6 warps x 8, T = 1536, 4 stages, 99.9 % of the copy rate
    // against 93-95 % with 8 x 8, 3 stages; other candidates that led in stand-alone sweeps did not
    // hold up there for N_d = 2, 16 and 32).
    if (broadcast) {
        switch (nd) {
            case 2: ZS_TMA(2, 8, 8, 4, 232448, true);     // T 2048, 4 stages, 1 CTA/SM
            case 4: ZS_TMA(4, 6, 8, 4, 232448, true);     // T 1536, 4 stages, 1 CTA/SM
            case 8: ZS_TMA(8, 4, 8, 8, 232448, true);     // T 1024, 8 stages, 1 CTA/SM
            case 16: ZS_TMA(16, 8, 4, 3, 232448, true);   // T 1024, 3 stages, 1 CTA/SM
            case 32: ZS_TMA(32, 2, 8, 3, 232448, true);   // T 512, 3 stages, 1 CTA/SM
            default: return cudaErrorNotSupported;
        }
    }
    switch (nd) {
        case 1: ZS_TMA(1, 8, 8, 8, 232448, false);        // T 2048, 8 stages, 1 CTA/SM
        case 2: ZS_TMA(2, 8, 8, 4, 232448, false);        // T 2048, 4 stages, 1 CTA/SM
        case 4: ZS_TMA(4, 8, 8, 3, 232448, false);        // T 2048, 3 stages, 1 CTA/SM
        case 8: ZS_TMA(8, 2, 8, 4, 232448, false);        // T 512, 4 stages, 3 CTAs/SM
        case 16: ZS_TMA(16, 4, 8, 2, 115712, false);      // T 1024, 2 stages, 2 CTAs/SM
        case 32: ZS_TMA(32, 4, 4, 2, 115712, false);      // T 512, 2 stages, 2 CTAs/SM
        default: return cudaErrorNotSupported;
    }
#undef ZS_TMA
}

// The broadcast shape for the launches of a walk (kSyncWalkFirst / kSyncWalkNext), where consecutive
// launches overlap: a two-stage ring in under half an SM's shared memory, so a launch's CTAs share
// each SM with the next launch's.  N_d = 8: 8 consumer warps x 8 elements, T = 2048 (114,944 B).
// Measured on GB300 (Llama-1.3B buffer, N_d = 8, the step walked in 4 Mi-element launches): 103.5 %
// of the copy rate, against 98.5 % for one persistent launch of the whole-range shape over the same
// bytes and 95 % for this shape in one persistent launch; among walk shapes (T = 1024 with 3-4
// stages, T = 512 with 4-8 stages, 4 or 8 consumer warps) it led for every bucket size from 1 to
// 64 MiB.  The other rank counts, on the 2^28+7 buffer (whole step walked / one launch per 1, 4,
// 16 MiB bucket, of the copy rate; the whole-range shape's single launch in brackets):
//   N_d = 2:  8 warps x 8, T 2048, 2 stages: 102.9 / 97.5 / 99.4 / 102.6 %  (98.2 %)
//   N_d = 4:  8 warps x 8, T 2048, 2 stages: 102.4 / 87.8 / 97.8 / 102.3 %  (100.5 %)
//   N_d = 16: 8 warps x 4, T 1024, 2 stages: 101.1 / 97.6 / 101.6 / 101.2 % (94.4 %)
//   N_d = 32: 4 warps x 4, T 512, 2 stages:  99.7 / 99.4 / 99.2 / 99.8 %    (93.6 %)
// each the best of four candidates (2-4 stages, 2-8 consumer warps) at its rank count.
template <class F>
cudaError_t with_walk_shape(int nd, F&& f) {
    switch (nd) {
        case 2: return f(IC<2>{}, IC<8>{}, IC<8>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 4: return f(IC<4>{}, IC<8>{}, IC<8>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 8: return f(IC<8>{}, IC<8>{}, IC<8>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 16: return f(IC<16>{}, IC<8>{}, IC<4>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 32: return f(IC<32>{}, IC<4>{}, IC<4>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        default: return cudaErrorNotSupported;
    }
}

// The single-output walk shapes (the ZeRO-3 reduce-scatter + update of one unit, walked in launches of
// 8 Mi elements): two-stage rings in under half an SM's shared memory, the broadcast walk shapes'
// tiles (N_d = 2, 4, 8: 8 warps x 8, T 2048; 16: 8 x 4, T 1024; 32: 4 x 4, T 512).
template <class F>
cudaError_t with_single_walk_shape(int nd, F&& f) {
    switch (nd) {
        case 2: return f(IC<2>{}, IC<8>{}, IC<8>{}, BC<false>{}, IC<2>{}, IC<115712>{});
        case 4: return f(IC<4>{}, IC<8>{}, IC<8>{}, BC<false>{}, IC<2>{}, IC<115712>{});
        case 8: return f(IC<8>{}, IC<8>{}, IC<8>{}, BC<false>{}, IC<2>{}, IC<115712>{});
        case 16: return f(IC<16>{}, IC<8>{}, IC<4>{}, BC<false>{}, IC<2>{}, IC<115712>{});
        case 32: return f(IC<32>{}, IC<4>{}, IC<4>{}, BC<false>{}, IC<2>{}, IC<115712>{});
        default: return cudaErrorNotSupported;
    }
}

// The walk shapes of the accumulating step (k_fused_tma_acc): a stage holds 2 N_d bf16 tiles, so
// each rank count takes the tile of the plain walk shape with twice its rank count (two-stage ring
// under half an SM's shared memory): N_d = 2, 4: 8 warps x 8 (T 2048); 8: 8 x 4 (T 1024); 16: 4 x 4
// (T 512); 32: 2 x 4 (T 256).
template <class F>
cudaError_t with_acc_walk_shape(int nd, F&& f) {
    switch (nd) {
        case 2: return f(IC<2>{}, IC<8>{}, IC<8>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 4: return f(IC<4>{}, IC<8>{}, IC<8>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 8: return f(IC<8>{}, IC<8>{}, IC<4>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 16: return f(IC<16>{}, IC<4>{}, IC<4>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        case 32: return f(IC<32>{}, IC<2>{}, IC<4>{}, BC<true>{}, IC<2>{}, IC<115712>{});
        default: return cudaErrorNotSupported;
    }
}

TmaArgs make_args(const BView& g, float* master, float* m, float* v, const BView& out, const AdamScalars& s,
                  int nd) {
    TmaArgs a;
    a.g = g.ptr;
    a.g_off = g.off;
    a.out = out.ptr;
    a.out_off = out.off;
    a.master = master;
    a.m = m;
    a.v = v;
    a.s = s;
    a.lo = 0;
    a.n = 0;
    a.nd = nd;
    a.inv_nd = 1.0f / (float)nd;
    a.wait_limit = 4000000000LL;                     // ~2 s at the 2.07 GHz maximum SM clock
    a.drain_limit = 4000000000LL;
    a.sync = kSyncStream;
    a.order = nullptr;
    return a;
}

}  // namespace

// Returns cudaErrorNotSupported when no staged variant exists for this rank count.
cudaError_t launch_fused_tma(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast,
                             int64_t lo, int64_t n, const AdamScalars& s, int nd, cudaStream_t st, int sync,
                             const AccumIn* acc) {
    if (acc && !broadcast) return cudaErrorNotSupported;
    bool ok = body_ok(lo, n) && at_ok(master, lo) && at_ok(m, lo) && at_ok(v, lo);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(g.ptr.p[q], lo - g.off);
    for (int q = 0; q < (broadcast ? nd : 1) && ok; ++q) ok = at_ok(out.ptr.p[q], lo - out.off);
    for (int q = 0; acc && q < nd && ok; ++q) ok = at_ok(acc->micro.ptr.p[q], lo - acc->micro.off);
    if (!ok) return cudaErrorMisalignedAddress;
    TmaArgs a = make_args(g, master, m, v, out, s, nd);
    a.lo = lo;
    a.n = n;
    a.sync = sync;
    if (acc) {
        TmaAccArgs x;
        x.a = a;
        x.micro = acc->micro.ptr;
        x.micro_off = acc->micro.off;
        x.scale = acc->scale;
        // one shape per rank count, walked or not: a single launch of it over a whole range runs one
        // wave of resident CTAs
        return with_acc_walk_shape(nd, [&](auto ND, auto NCW, auto VPT, auto BR, auto MS, auto BU) {
            return tma_impl<decltype(ND)::value, decltype(NCW)::value, decltype(VPT)::value, decltype(BR)::value,
                            decltype(MS)::value, decltype(BU)::value>(x, st, sync != kSyncStream);
        });
    }
    // AdamW alone on sharded arrays (one rank, one output) in the launches of a walk: 8 consumer
    // warps x 8 elements (T 2048) and a 2-stage ring of 57,600 B, so up to three CTAs share an SM and a
    // launch's CTAs run beside the next launch's.  Measured on GB300 (the Llama-1.3B shard arrays,
    // 1,345,423,360 elements, pieces of 4 Mi elements): 102.5 % of the copy rate, against 96.4 % for
    // one persistent launch of the whole-range shape (8 stages, one CTA per SM) and 72.8 % for that
    // shape walked; T 2048 with 3 or 4 stages 102.4 / 101.9 %, three T 1024 shapes 101.5-101.6 %,
    // 16 warps x 8 with 2 stages 101.7 %; pieces of 2 Mi elements 89.8 %, of 8 Mi 101.9 %.
    if (!broadcast && nd == 1 && sync != kSyncStream) return tma_impl<1, 8, 8, false, 2, 115712>(a, st, true);
    if (!broadcast && sync != kSyncStream && fused_walk_shape(nd)) {
        return with_single_walk_shape(nd, [&](auto ND, auto NCW, auto VPT, auto BR, auto MS, auto BU) {
            return tma_impl<decltype(ND)::value, decltype(NCW)::value, decltype(VPT)::value, decltype(BR)::value,
                            decltype(MS)::value, decltype(BU)::value>(a, st, true);
        });
    }
    if (broadcast && sync != kSyncStream && fused_walk_shape(nd)) {
        return with_walk_shape(nd, [&](auto ND, auto NCW, auto VPT, auto BR, auto MS, auto BU) {
            return tma_impl<decltype(ND)::value, decltype(NCW)::value, decltype(VPT)::value, decltype(BR)::value,
                            decltype(MS)::value, decltype(BU)::value>(a, st, true);
        });
    }
    return with_shape(broadcast, nd, [&](auto ND, auto NCW, auto VPT, auto BR, auto MS, auto BU) {
        return tma_impl<decltype(ND)::value, decltype(NCW)::value, decltype(VPT)::value, decltype(BR)::value,
                        decltype(MS)::value, decltype(BU)::value>(a, st);
    });
}

bool fused_walk_shape(int nd, bool /*acc: the same rank counts*/) {
    return nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32;
}

// ------------------------------------------------------------------ dynamic tile order
// Counter pairs of the dynamic-order launches, one pair per launch in flight: launches draw pairs in
// turn, so up to kDynOrderSlots of them may run at once on a device, on any streams.  Module memory,
// zero at load (every device that loads the library holds its own array).
constexpr unsigned int kDynOrderSlots = 1024;
__device__ unsigned int g_zs_dyn_order[2 * kDynOrderSlots];

namespace {

// The next counter pair on the current device (its address looked up once per device).
cudaError_t dyn_order_pair(unsigned int** out) {
    static std::mutex mu;
    static std::unordered_map<int, unsigned int*> base;
    static std::atomic<unsigned int> next{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    unsigned int* b = nullptr;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = base.find(dev);
        if (it == base.end()) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_zs_dyn_order);
            if (e != cudaSuccess) return e;
            it = base.emplace(dev, static_cast<unsigned int*>(p)).first;
        }
        b = it->second;
    }
    *out = b + 2 * (next.fetch_add(1u) % kDynOrderSlots);
    return cudaSuccess;
}

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool BROADCAST>
auto dyn_kernel(const TmaArgs*) {
    if constexpr (BROADCAST)
        return k_fused_tma_dyn<ND, NCW, VPT, MAXST, BUDGET>;
    else
        return k_fused_tma_single_dyn<ND, NCW, VPT, MAXST, BUDGET>;
}
template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool BROADCAST>
auto dyn_kernel(const TmaAccArgs*) {
    static_assert(BROADCAST, "the accumulating step has the broadcast form only");
    return k_fused_tma_acc_dyn<ND, NCW, VPT, MAXST, BUDGET>;
}
TmaArgs& base_args(TmaArgs& a) { return a; }
TmaArgs& base_args(TmaAccArgs& x) { return x.a; }

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool BROADCAST = true, class Args>
cudaError_t dyn_impl(Args a, cudaStream_t st) {
    using Sh = TmaShape<std::is_same<Args, TmaAccArgs>::value ? 2 * ND : ND, NCW, VPT, MAXST, BUDGET>;
    auto kern = dyn_kernel<ND, NCW, VPT, MAXST, BUDGET, BROADCAST>(static_cast<const Args*>(nullptr));
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)kern, 32 * (NCW + 1), Sh::kSmem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    TmaArgs& b = base_args(a);
    const int64_t ntiles = (b.n + Sh::kT - 1) / Sh::kT;
    if (ntiles < 1) return cudaSuccess;
    const int64_t cap = (int64_t)sms * per_sm;          // persistent: one wave of resident CTAs
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    e = dyn_order_pair(&b.order);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, dim3(grid), dim3(32 * (NCW + 1)), Sh::kSmem, st, a);
}

}  // namespace

bool fused_dyn_shape(int nd) { return nd == 2 || nd == 4 || nd == 8 || nd == 16 || nd == 32; }

// The single-output step (ZeRO-3 reduce-scatter + update; out.p[0] the shard array; with one rank, the
// update alone on a reduced gradient) over the 8-aligned body [lo, lo + n) in one dynamic-order launch,
// with the single-output walk shapes' tiles and rings (two-stage rings under half an SM).
cudaError_t launch_fused_single_dyn(const BView& g, float* master, float* m, float* v, const BView& out, int64_t lo,
                                    int64_t n, const AdamScalars& s, int nd, cudaStream_t st) {
    bool ok = body_ok(lo, n) && at_ok(master, lo) && at_ok(m, lo) && at_ok(v, lo) && at_ok(out.ptr.p[0], lo - out.off);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(g.ptr.p[q], lo - g.off);
    if (!ok) return cudaErrorMisalignedAddress;
    TmaArgs a = make_args(g, master, m, v, out, s, nd);
    a.lo = lo;
    a.n = n;
    switch (nd) {
        // the update alone, in the walk's shape: 104.9 / 103.0 % of the measured copy rate on the
        // Llama-1.3B / GPT-2-small buffers against 102.9-103.0 / 101.0-101.1 % walked (GB300)
        case 1: return dyn_impl<1, 8, 8, 2, 115712, false>(a, st);
        case 2: return dyn_impl<2, 8, 8, 2, 115712, false>(a, st);
        case 4: return dyn_impl<4, 8, 8, 2, 115712, false>(a, st);
        case 8: return dyn_impl<8, 8, 8, 2, 115712, false>(a, st);
        case 16: return dyn_impl<16, 8, 4, 2, 115712, false>(a, st);
        case 32: return dyn_impl<32, 4, 4, 2, 115712, false>(a, st);
        default: return cudaErrorNotSupported;
    }
}

// The broadcast fused step over the 8-aligned body [lo, lo + n) in one dynamic-order launch.  Shapes from
// a measured comparison on GB300 (the 2^28+7-element buffer, against the walk of 4 Mi-element launches
// on the same box, of the measured copy rate): N_d = 2, 4: 4 consumer warps x 8 (T 1024), 4 stages:
// 103.3 / 103.0 % (walk 101.9 / 101.2 %); N_d = 8: 4 x 8, 4 stages: 102.0 % (100.5 %; on the
// Llama-1.3B buffer 103.4-103.8 % against 101.7-101.9 %); N_d = 16: 8 x 4 (T 1024), 2 stages: 102.0 %
// (99.4 %); N_d = 32: 4 x 4 (T 512), 2 stages: 102.0 % (97.5 %).  Rings of at most half an SM's shared
// memory, two CTAs per SM.
cudaError_t launch_fused_tma_dyn(const BView& g, float* master, float* m, float* v, const BView& out, int64_t lo,
                                 int64_t n, const AdamScalars& s, int nd, cudaStream_t st, const AccumIn* acc) {
    bool ok = body_ok(lo, n) && at_ok(master, lo) && at_ok(m, lo) && at_ok(v, lo);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(g.ptr.p[q], lo - g.off) && at_ok(out.ptr.p[q], lo - out.off);
    for (int q = 0; acc && q < nd && ok; ++q) ok = at_ok(acc->micro.ptr.p[q], lo - acc->micro.off);
    if (!ok) return cudaErrorMisalignedAddress;
    TmaArgs a = make_args(g, master, m, v, out, s, nd);
    a.lo = lo;
    a.n = n;
    if (acc) {
        TmaAccArgs x;
        x.a = a;
        x.micro = acc->micro.ptr;
        x.micro_off = acc->micro.off;
        x.scale = acc->scale;
        // A stage holds 2 N_d bf16 tiles: rings under half an SM.  N_d = 8 measured on GB300 (GPT-2-small,
        // the accumulating step alone, of the measured copy rate): 8 warps x 4 (T 1024), 2 stages 103.2 %,
        // 4 x 8 102.8 %, T 512 with 4 stages 101.5 %, T 2048 in a whole SM 101.3 %, against 101.0 % for
        // the walk on the same box; the other rank counts take tiles of the same bytes per stage.
        switch (nd) {
            case 2: return dyn_impl<2, 4, 8, 4, 115712>(x, st);
            case 4: return dyn_impl<4, 4, 8, 4, 115712>(x, st);
            case 8: return dyn_impl<8, 8, 4, 4, 115712>(x, st);
            case 16: return dyn_impl<16, 4, 4, 4, 115712>(x, st);
            case 32: return dyn_impl<32, 2, 4, 4, 115712>(x, st);
            default: return cudaErrorNotSupported;
        }
    }
    switch (nd) {
        case 2: return dyn_impl<2, 4, 8, 4, 115712>(a, st);
        case 4: return dyn_impl<4, 4, 8, 4, 115712>(a, st);
        case 8: return dyn_impl<8, 4, 8, 4, 115712>(a, st);
        case 16: return dyn_impl<16, 8, 4, 4, 115712>(a, st);
        case 32: return dyn_impl<32, 4, 4, 4, 115712>(a, st);
        default: return cudaErrorNotSupported;
    }
}

namespace {

// Launches the list kernel over `bodies`, kTmaListMax bodies (and at most 2^31 - 1 tiles) per launch.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
cudaError_t tma_list_impl(TmaListArgs& l, const std::vector<std::pair<int64_t, int64_t>>& bodies, cudaStream_t st) {
    using Sh = TmaShape<ND, NCW, VPT, MAXST, BUDGET>;
    size_t i = 0;
    while (i < bodies.size()) {
        int nr = 0;
        int64_t tiles = 0;
        l.first[0] = 0;
        for (; i < bodies.size() && nr < kTmaListMax; ++i) {
            const int64_t t = (bodies[i].second + Sh::kT - 1) / Sh::kT;
            if (t < 1) continue;
            if (tiles + t > 0x7fffffffLL) {                       // tile counts are 32-bit in the list
                if (nr == 0) return cudaErrorInvalidValue;
                break;
            }
            l.lo[nr] = bodies[i].first;
            l.n[nr] = bodies[i].second;
            tiles += t;
            l.first[++nr] = (int32_t)tiles;
        }
        l.nr = nr;
        l.total_tiles = tiles;
        if (nr == 0) continue;
        cudaError_t e = tma_impl<ND, NCW, VPT, true, MAXST, BUDGET>(l, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace

// Broadcast form over a list of bodies in one launch per kTmaListMax bodies.
cudaError_t launch_fused_tma_list(const BView& g, float* master, float* m, float* v, const BView& out,
                                  const std::vector<std::pair<int64_t, int64_t>>& bodies, const AdamScalars& s,
                                  int nd, cudaStream_t st) {
    if (bodies.empty()) return cudaSuccess;
    for (const auto& b : bodies) {
        bool ok = body_ok(b.first, b.second) && at_ok(master, b.first) && at_ok(m, b.first) && at_ok(v, b.first);
        for (int q = 0; q < nd && ok; ++q)
            ok = at_ok(g.ptr.p[q], b.first - g.off) && at_ok(out.ptr.p[q], b.first - out.off);
        if (!ok) return cudaErrorMisalignedAddress;
    }
    // the argument block is ~11 KB: built on the heap
    std::unique_ptr<TmaListArgs> l(new TmaListArgs());
    l->a = make_args(g, master, m, v, out, s, nd);
    return with_shape(true, nd, [&](auto ND, auto NCW, auto VPT, auto BR, auto MS, auto BU) -> cudaError_t {
        if constexpr (decltype(BR)::value)
            return tma_list_impl<decltype(ND)::value, decltype(NCW)::value, decltype(VPT)::value,
                                 decltype(MS)::value, decltype(BU)::value>(*l, bodies, st);
        else
            return cudaErrorNotSupported;                     // only the broadcast form walks lists
    });
}

// ------------------------------------------------------------------ staged reduce-scatter-mean
// The reduce-scatter with averaging alone, into one output array ("Infra: Data Parallel", ZeRO
// section): out[i] = bf16(fold over ranks of fp32 g_q[i], ascending from +0, times 1/N_d or divided
// by N_d), the same arithmetic as the fused kernel's first half.  The ring of k_fused_tma without the
// optimizer state: the producer stages every rank's bf16 tile with one bulk copy each, consumers fold
// from shared memory and stream the 16-bit results out.

struct RsTmaArgs {
    Ptrs g;               // rank gradients; element i of rank q at g.p[q] + (i - g_off)
    int64_t g_off;
    uint16_t* out;        // element i at out + (i - out_off)
    int64_t out_off;
    int64_t lo, n;        // body [lo, lo + n): lo, n, lo - g_off and lo - out_off multiples of 8
    int nd;
    float inv_nd;
    long long wait_limit, drain_limit;
    int sync;             // LaunchSync (the in-place all-reduce's walk; the reduce-scatter keeps stream order)
    unsigned int* order;  // the dynamic-order launch's counter pair (k_ar_tma_dyn), else unused
};

template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
struct RsShape {
    static constexpr int kT = NCW * 32 * VPT;
    static constexpr int kStageBytes = kT * 2 * ND;
    static constexpr int kFit = (BUDGET - 256) / kStageBytes;
    static constexpr int kStages = kFit > MAXST ? MAXST : kFit;
    static constexpr int kSmem = 256 + kStages * kStageBytes;
    static_assert(kStages >= 2, "tile too large for a 2-stage ring");
    static_assert(2 * kStages * 8 <= 256, "barriers must fit in the first 256 bytes");
};

// ALL: the in-place all-reduce with averaging of naive DP ("Infra: Data Parallel", Naive Data
// Parallelism): the mean goes back into every rank's own buffer (a.g) instead of one output array.  A
// tile's copies into shared memory complete before any consumer stores into it, and tiles are
// disjoint, so in place is safe.  DYN: tiles in dynamic order, as in fused_tma_body.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool ALL, bool DYN = false>
__device__ __forceinline__ void rs_tma_body(const RsTmaArgs& a) {
    using Sh = RsShape<ND, NCW, VPT, MAXST, BUDGET>;
    constexpr int T = Sh::kT;
    constexpr int S = Sh::kStages;
    static_assert(!DYN || S <= 8, "the dynamic order's stage records sit behind the barriers");
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + S;
    int64_t* rec = reinterpret_cast<int64_t*>(smem + 128);   // DYN: the tile of each stage
    uint8_t* stages = smem + 256;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    const int64_t ntiles = (a.n + T - 1) / T;

    if (warp == 0) {
        // ---------------- producer
        if (lane == 0) {
            const uint64_t pol = evict_first_policy();
            int64_t j = 0;
            bool ok = true;
            for (int64_t tile = DYN ? 0 : blockIdx.x; DYN || tile < ntiles; tile += gridDim.x, ++j) {
                const int s = (int)(j % S);
                if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), a.wait_limit)) {
                    flag_error(ZS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                if constexpr (DYN) {
                    tile = (int64_t)atomicAdd(a.order, 1u);
                    rec[s] = tile;                        // published by the arrive below (release)
                    if (tile >= ntiles) {
                        mbar_arrive(&full[s]);            // no copies: the consumers read the end mark
                        break;
                    }
                }
                const int64_t i0 = a.lo + tile * T;
                const int64_t rem = a.n - tile * T;
                const uint32_t len = (uint32_t)(rem < T ? rem : T);
                uint8_t* st = stages + (size_t)s * Sh::kStageBytes;
                mbar_expect_tx(&full[s], len * 2u * ND);
#pragma unroll
                for (int q = 0; q < ND; ++q)
                    bulk_load(st + (size_t)q * T * 2, a.g.p[q] + (i0 - a.g_off), len * 2u, &full[s], pol);
            }
            if (!ok) {
                const int64_t issued = j;
                for (int64_t k = issued > S ? issued - S : 0; k < issued; ++k)
                    mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
            }
        }
        return;
    }

    // ---------------- consumers
    const int ct = threadIdx.x - 32;
    const int e = ct * VPT;
    int64_t j = 0;
    for (int64_t tile = DYN ? 0 : blockIdx.x; DYN || tile < ntiles; tile += gridDim.x, ++j) {
        const int s = (int)(j % S);
        if (!mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_CONSUMER_WAIT);
            return;
        }
        if constexpr (DYN) {
            tile = rec[s];
            if (tile >= ntiles) return;                   // the producer's end mark
        }
        const int64_t i0 = a.lo + tile * T;
        const int64_t rem = a.n - tile * T;
        const int len = (int)(rem < T ? rem : T);
        if (e < len) {
            const uint16_t* sg = reinterpret_cast<const uint16_t*>(stages + (size_t)s * Sh::kStageBytes);
            float acc[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) acc[k] = 0.0f;
#pragma unroll
            for (int q = 0; q < ND; ++q) {
                float f[VPT];
                lds_bf<VPT>(sg + (size_t)q * T + e, f);
#pragma unroll
                for (int k = 0; k < VPT; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
            }
            uint32_t w[VPT / 2];
#pragma unroll
            for (int k = 0; k < VPT; k += 2)
                w[k / 2] = pack_bf16x2(mean_of_sum<ND>(acc[k], ND, a.inv_nd), mean_of_sum<ND>(acc[k + 1], ND, a.inv_nd));
            if constexpr (ALL) {
#pragma unroll
                for (int q = 0; q < ND; ++q) {
                    uint16_t* o = a.g.p[q] + (i0 + e - a.g_off);
                    if constexpr (VPT == 8)
                        __stcs(reinterpret_cast<uint4*>(o), make_uint4(w[0], w[1], w[2], w[3]));
                    else
                        __stcs(reinterpret_cast<uint2*>(o), make_uint2(w[0], w[1]));
                }
            } else {
                uint16_t* o = a.out + (i0 + e - a.out_off);
                if constexpr (VPT == 8)
                    __stcs(reinterpret_cast<uint4*>(o), make_uint4(w[0], w[1], w[2], w[3]));
                else
                    __stcs(reinterpret_cast<uint2*>(o), make_uint2(w[0], w[1]));
            }
            mbar_arrive(&empty[s]);                      // after the stores: see k_fused_tma
        } else {
            mbar_arrive(&empty[s]);
        }
    }
}

template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_rs_tma(const __grid_constant__ RsTmaArgs a) {
    dependent_launch_prologue();
    rs_tma_body<ND, NCW, VPT, MAXST, BUDGET, false>(a);
}

// The in-place all-reduce, launched as the pieces of a walk (a.sync); the body returns early
// (producer lanes, a wait that ran out) into the launch-order epilogue.
template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_ar_tma(const __grid_constant__ RsTmaArgs a) {
    dependent_launch_prologue(a.sync);
    rs_tma_body<ND, NCW, VPT, MAXST, BUDGET, true>(a);
    dependent_launch_epilogue(a.sync);
}

// The in-place all-reduce over one range in one persistent launch taking its tiles in dynamic order.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_ar_tma_dyn(const __grid_constant__ RsTmaArgs a) {
    dependent_launch_prologue(kSyncStream);
    rs_tma_body<ND, NCW, VPT, MAXST, BUDGET, true, true>(a);
    dyn_order_finish(a.order);
}

// The reduce-scatter into one array over one range in one persistent launch, dynamic tile order.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET>
__global__ void __launch_bounds__(32 * (NCW + 1)) k_rs_tma_dyn(const __grid_constant__ RsTmaArgs a) {
    dependent_launch_prologue(kSyncStream);
    rs_tma_body<ND, NCW, VPT, MAXST, BUDGET, false, true>(a);
    dyn_order_finish(a.order);
}

namespace {

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool ALL, bool DYN>
auto rs_kernel() {
    if constexpr (DYN && ALL) {
        return k_ar_tma_dyn<ND, NCW, VPT, MAXST, BUDGET>;
    } else if constexpr (DYN) {
        return k_rs_tma_dyn<ND, NCW, VPT, MAXST, BUDGET>;
    } else if constexpr (ALL) {
        return k_ar_tma<ND, NCW, VPT, MAXST, BUDGET>;
    } else {
        return k_rs_tma<ND, NCW, VPT, MAXST, BUDGET>;
    }
}

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool ALL = false, bool DYN = false>
cudaError_t rs_tma_impl(RsTmaArgs a, cudaStream_t st) {
    using Sh = RsShape<ND, NCW, VPT, MAXST, BUDGET>;
    auto kern = rs_kernel<ND, NCW, VPT, MAXST, BUDGET, ALL, DYN>();
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)kern, 32 * (NCW + 1), Sh::kSmem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.n + Sh::kT - 1) / Sh::kT;
    if (ntiles < 1) return cudaSuccess;
    const int64_t cap = (int64_t)sms * per_sm;
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    if constexpr (DYN) {
        e = dyn_order_pair(&a.order);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(kern, dim3(grid), dim3(32 * (NCW + 1)), Sh::kSmem, st, a);
}

}  // namespace

static RsTmaArgs rs_args(const BView& g, int64_t lo, int64_t n, int nd) {
    RsTmaArgs a;
    a.g = g.ptr;
    a.g_off = g.off;
    a.out = nullptr;
    a.out_off = 0;
    a.lo = lo;
    a.n = n;
    a.nd = nd;
    a.inv_nd = 1.0f / (float)nd;
    a.wait_limit = 4000000000LL;
    a.drain_limit = 4000000000LL;
    a.sync = kSyncStream;
    a.order = nullptr;
    return a;
}

// Returns cudaErrorNotSupported when no staged shape exists for this rank count.  At N_d = 8, 16 and
// 32 a body of kDynMinElems or more is one launch taking its tiles in dynamic order, in the same
// shapes: measured on GB300 (of the measured copy rate) 101.9 -> 106.5 % on the Llama-1.3B buffer at
// N_d = 8, 100.8 -> 102.1 / 93.7 -> 103.0 % on the 2^28+7 buffer at N_d = 16 / 32.  At N_d = 2 and 4
// the tiles carry 5-6 KB each, too little per draw from the one tile counter (38.5 / 34.7 % against
// 97.1-97.6 / 98.4-98.6 %), so those keep the static order.
cudaError_t launch_rs_tma(const BView& g, uint16_t* out, int64_t out_off, int64_t lo, int64_t n, int nd,
                          cudaStream_t st) {
    bool ok = body_ok(lo, n) && at_ok(out, lo - out_off);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(g.ptr.p[q], lo - g.off);
    if (!ok) return cudaErrorMisalignedAddress;
    RsTmaArgs a = rs_args(g, lo, n, nd);
    a.out = out;
    a.out_off = out_off;
    if (n >= kDynMinElems && nd >= 8) {
        switch (nd) {
            case 8: return rs_tma_impl<8, 8, 8, 2, 232448, false, true>(a, st);
            case 16: return rs_tma_impl<16, 8, 8, 2, 232448, false, true>(a, st);
            case 32: return rs_tma_impl<32, 2, 4, 2, 232448, false, true>(a, st);
            default: return cudaErrorNotSupported;
        }
    }
    // shapes per rank count from a measured sweep on GB300 (consumer warps x elements per thread x
    // ring depth, 2^27-element buffers): 96 / 99 / 100 / 102 / 102 % of the measured copy rate for
    // N_d = 2 / 4 / 8 / 16 / 32, against ~94 % for the register-streaming kernel
    switch (nd) {
        case 2: return rs_tma_impl<2, 4, 8, 2, 232448>(a, st);     // T 1024, 2 stages, 12 CTAs/SM
        case 4: return rs_tma_impl<4, 4, 4, 2, 232448>(a, st);     // T 512, 2 stages, 12 CTAs/SM
        case 8: return rs_tma_impl<8, 8, 8, 2, 232448>(a, st);     // T 2048, 2 stages, 3 CTAs/SM
        case 16: return rs_tma_impl<16, 8, 8, 2, 232448>(a, st);   // T 2048, 2 stages, 1 CTA/SM
        case 32: return rs_tma_impl<32, 2, 4, 2, 232448>(a, st);   // T 256, 2 stages, 6 CTAs/SM
        default: return cudaErrorNotSupported;
    }
}

// The in-place all-reduce with averaging over the 8-aligned body [lo, lo + n) of every rank's buffer, as
// one launch of a walk (`sync`); cudaErrorNotSupported when no staged shape exists for this rank
// count.  Two-stage rings with at least two CTAs per SM, so a launch's CTAs run beside the next
// launch's.  Measured on GB300 (GPT-2-small buffers, 124,439,808 elements per rank, walked in 4 Mi-element
// launches; of the measured copy rate, the register-streaming kernel in brackets): N_d = 2, 4 with 8
// warps x 8 (T 2048): 101.4 / 98.0 % (92.0 / 93.3 %; the reduce-scatter's smaller tiles 90.7 / 95.6 %,
// five other shapes 89.5-101.2 / 94.2-97.5 %); N_d = 8, 16, 32 with the reduce-scatter's tiles (T 2048,
// 8 x 4 at T 1024 for 16, T 256): 102.1 / 101.1 / 100.2 % (93.6 / 94.4 / 98.3 %).
cudaError_t launch_all_reduce_tma(const BView& g, int64_t lo, int64_t n, int nd, cudaStream_t st, int sync) {
    bool ok = body_ok(lo, n);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(g.ptr.p[q], lo - g.off);
    if (!ok) return cudaErrorMisalignedAddress;
    RsTmaArgs a = rs_args(g, lo, n, nd);
    if (sync == kSyncDynamic) {
        // One launch over the whole range, tiles in dynamic order, with the walk's tiles and rings.
        // Measured on GB300 against the walk (GPT-2-small buffers, of the measured copy rate): N_d = 4 /
        // 8 / 16 / 32: 102.3 / 103.2 / 103.1 / 102.5 % (walk 98.1-98.4 / 101.8-101.9 / 101.1-101.2 /
        // 100.2 %); N_d = 2: 100.8 % against 101.1-101.3 %, so that rank count keeps the walk.
        switch (nd) {
            case 4: return rs_tma_impl<4, 8, 8, 2, 232448, true, true>(a, st);
            case 8: return rs_tma_impl<8, 8, 8, 2, 232448, true, true>(a, st);
            case 16: return rs_tma_impl<16, 8, 4, 2, 232448, true, true>(a, st);
            case 32: return rs_tma_impl<32, 2, 4, 2, 232448, true, true>(a, st);
            default: return cudaErrorNotSupported;
        }
    }
    a.sync = sync;
    switch (nd) {
        case 2: return rs_tma_impl<2, 8, 8, 2, 232448, true>(a, st);
        case 4: return rs_tma_impl<4, 8, 8, 2, 232448, true>(a, st);
        case 8: return rs_tma_impl<8, 8, 8, 2, 232448, true>(a, st);
        case 16: return rs_tma_impl<16, 8, 4, 2, 232448, true>(a, st);
        case 32: return rs_tma_impl<32, 2, 4, 2, 232448, true>(a, st);
        default: return cudaErrorNotSupported;
    }
}

bool ar_dyn_shape(int nd) { return nd == 4 || nd == 8 || nd == 16 || nd == 32; }

// ------------------------------------------------------------------ naive-DP step, staged
// "Infra: Data Parallel", section "Naive Data Parallelism": every rank keeps the full fp32 state
// and applies the same AdamW update with the all-reduced bf16 mean.  Per tile of T elements the
// producer stages every rank's bf16 gradients (two grads buffers, so the next tile's arrive while
// this one's ranks are updated), then each rank's master, m and v in turn through a ring of S
// state stages.  Consumers fold the mean once per tile and keep it in registers as bf16, then
// update each rank's state as that rank's stage arrives and stream the results (state, replica)
// straight to global memory.  The arithmetic is the register-streaming naive-DP kernel's; the
// state of N_d ranks is 96 of the 112 bytes read per element at N_d = 8, so the ring stages one
// rank's state at a time instead of holding every rank's state of a tile at once.

struct DpTmaArgs {
    Ptrs g;               // rank gradients; element i of rank q at g.p[q] + (i - g_off)
    int64_t g_off;
    Ptrs out;             // rank replicas; element i of rank q at out.p[q] + (i - out_off)
    int64_t out_off;
    float* master[ZS_MAX_RANKS];     // rank q's full fp32 state, element i at master[q] + i
    float* m[ZS_MAX_RANKS];
    float* v[ZS_MAX_RANKS];
    AdamScalars s;
    int64_t lo, n;        // body [lo, lo + n): lo, n, lo - g_off and lo - out_off multiples of 8
    int nd;
    float inv_nd;
    long long wait_limit, drain_limit;
    int sync;             // LaunchSync: the loads are bulk copies, so a later launch of a walk may stream at once
    unsigned int* order;  // the dynamic-order launch's counter pair (k_dp_tma_dyn), else unused
};

// Consumers index the ranks at run time (one copy of the update code, not N_d): the rank pointers
// are copied from the kernel parameter into shared memory once per CTA, with compile-time indices.
template <int ND>
struct DpTable {
    uint16_t* out[ND];
    float* master[ND];
    float* m[ND];
    float* v[ND];
};

template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024>
struct DpShape {
    static constexpr int kT = NCW * 32 * VPT;                               // elements per tile
    static constexpr int kBarBytes = 512;
    static constexpr int kHead = kBarBytes + (int)((sizeof(DpTable<ND>) + 127) / 128 * 128);
    static constexpr int kGradBytes = kT * 2 * ND;                          // one grads buffer
    static constexpr int kStageBytes = kT * 12;                             // one rank's master, m, v
    static constexpr int kFit = (BUDGET - kHead - 2 * kGradBytes) / kStageBytes;
    static constexpr int kStages = kFit > MAXST ? MAXST : kFit;
    static constexpr int kSmem = kHead + 2 * kGradBytes + kStages * kStageBytes;
    static_assert(kStages >= 2, "tile too large for a 2-stage ring");
    static_assert((4 + 2 * kStages) * 8 + 16 <= kBarBytes, "barriers and tile records must fit in their block");
};

// DYN: tiles in dynamic order, as in fused_tma_body; the producer draws a tile per grads buffer and
// publishes it in the buffer's record, which the buffer's full barrier releases to the consumers.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET, bool DYN = false>
__device__ __forceinline__ void dp_tma_body(const DpTmaArgs& a) {
    using Sh = DpShape<ND, NCW, VPT, MAXST, BUDGET>;
    constexpr int T = Sh::kT;
    constexpr int S = Sh::kStages;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* gfull = reinterpret_cast<uint64_t*>(smem);     // [2] grads buffer b loaded
    uint64_t* gempty = gfull + 2;                            // [2] grads buffer b folded
    uint64_t* full = gfull + 4;                              // [S] state stage s loaded
    uint64_t* empty = full + S;                              // [S] state stage s consumed
    int64_t* rec = reinterpret_cast<int64_t*>(smem + Sh::kBarBytes - 16);   // [2] DYN: grads buffer b's tile
    DpTable<ND>* tab = reinterpret_cast<DpTable<ND>*>(smem + Sh::kBarBytes);
    uint16_t* gbuf = reinterpret_cast<uint16_t*>(smem + Sh::kHead);
    uint8_t* stages = smem + Sh::kHead + 2 * Sh::kGradBytes;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&gfull[b], 1);
            mbar_init(&gempty[b], NCW * 32);
        }
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW * 32);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
#pragma unroll
        for (int q = 0; q < ND; ++q) {
            if ((q & 31) == lane) {
                tab->out[q] = a.out.p[q];
                tab->master[q] = a.master[q];
                tab->m[q] = a.m[q];
                tab->v[q] = a.v[q];
            }
        }
    }
    __syncthreads();

    const int64_t ntiles = (a.n + T - 1) / T;

    if (warp == 0) {
        // ---------------- producer: grads of a tile, then each rank's state of the tile
        if (lane == 0) {
            const uint64_t pol = evict_first_policy();
            int64_t j = 0;        // state stages issued
            int64_t gi = 0;       // grads buffers issued (= tiles started)
            bool ok = true;
            for (int64_t tile = DYN ? 0 : blockIdx.x; (DYN || tile < ntiles) && ok; tile += gridDim.x) {
                const int b = (int)(gi & 1);
                if (gi >= 2 && !mbar_wait(&gempty[b], (uint32_t)(((gi >> 1) - 1) & 1), a.wait_limit)) {
                    flag_error(ZS_DEVERR_PRODUCER_WAIT);
                    ok = false;
                    break;
                }
                if constexpr (DYN) {
                    tile = (int64_t)atomicAdd(a.order, 1u);
                    rec[b] = tile;                        // published by the arrive below (release)
                    if (tile >= ntiles) {
                        mbar_arrive(&gfull[b]);           // no copies: the consumers read the end mark
                        break;
                    }
                }
                const int64_t i0 = a.lo + tile * T;
                const int64_t rem = a.n - tile * T;
                const uint32_t len = (uint32_t)(rem < T ? rem : T);
                uint16_t* gb = gbuf + (size_t)b * ND * T;
                mbar_expect_tx(&gfull[b], len * 2u * ND);
#pragma unroll
                for (int q = 0; q < ND; ++q)
                    bulk_load(gb + (size_t)q * T, a.g.p[q] + (i0 - a.g_off), len * 2u, &gfull[b], pol);
                ++gi;
#pragma unroll
                for (int q = 0; q < ND; ++q, ++j) {
                    const int s = (int)(j % S);
                    if (j >= S && !mbar_wait(&empty[s], (uint32_t)(((j / S) - 1) & 1), a.wait_limit)) {
                        flag_error(ZS_DEVERR_PRODUCER_WAIT);
                        ok = false;
                        break;
                    }
                    float* sf = reinterpret_cast<float*>(stages + (size_t)s * Sh::kStageBytes);
                    mbar_expect_tx(&full[s], len * 12u);
                    bulk_load(sf, a.master[q] + i0, len * 4u, &full[s], pol);
                    bulk_load(sf + T, a.m[q] + i0, len * 4u, &full[s], pol);
                    bulk_load(sf + 2 * T, a.v[q] + i0, len * 4u, &full[s], pol);
                }
            }
            if (!ok) {
                // drain: wait (bounded) for the copies issued into buffers not yet consumed
                for (int64_t k = gi > 2 ? gi - 2 : 0; k < gi; ++k)
                    mbar_wait(&gfull[k & 1], (uint32_t)((k >> 1) & 1), a.drain_limit);
                for (int64_t k = j > S ? j - S : 0; k < j; ++k)
                    mbar_wait(&full[k % S], (uint32_t)((k / S) & 1), a.drain_limit);
            }
        }
        return;
    }

    // ---------------- consumers
    const int ct = threadIdx.x - 32;                  // 0 .. NCW*32-1
    const int e = ct * VPT;                           // this thread's first element in a tile
    int64_t j = 0, t = 0;
    for (int64_t tile = DYN ? 0 : blockIdx.x; DYN || tile < ntiles; tile += gridDim.x, ++t) {
        const int b = (int)(t & 1);
        if (!mbar_wait(&gfull[b], (uint32_t)((t >> 1) & 1), a.wait_limit)) {
            flag_error(ZS_DEVERR_CONSUMER_WAIT);
            return;
        }
        if constexpr (DYN) {
            tile = rec[b];
            if (tile >= ntiles) return;                   // the producer's end mark
        }
        const int64_t i0 = a.lo + tile * T;
        const int64_t rem = a.n - tile * T;
        const int len = (int)(rem < T ? rem : T);
        uint32_t gw[VPT / 2] = {};                    // the tile's mean, bf16 pairs, kept for every rank
        if (e < len) {
            const uint16_t* gb = gbuf + (size_t)b * ND * T;
            float acc[VPT];
#pragma unroll
            for (int k = 0; k < VPT; ++k) acc[k] = 0.0f;
#pragma unroll
            for (int q = 0; q < ND; ++q) {
                float f[VPT];
                lds_bf<VPT>(gb + (size_t)q * T + e, f);
#pragma unroll
                for (int k = 0; k < VPT; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
            }
#pragma unroll
            for (int k = 0; k < VPT; k += 2)
                gw[k / 2] = pack_bf16x2(mean_of_sum<ND>(acc[k], ND, a.inv_nd), mean_of_sum<ND>(acc[k + 1], ND, a.inv_nd));
        }
#pragma unroll 1
        for (int q = 0; q < ND; ++q, ++j) {
            const int s = (int)(j % S);
            if (!mbar_wait(&full[s], (uint32_t)((j / S) & 1), a.wait_limit)) {
                flag_error(ZS_DEVERR_CONSUMER_WAIT);
                return;
            }
            if (e < len) {
                const float* sf = reinterpret_cast<const float*>(stages + (size_t)s * Sh::kStageBytes);
                float p[VPT], mm[VPT], vv[VPT];
                lds_f32<VPT>(sf + e, p);
                lds_f32<VPT>(sf + T + e, mm);
                lds_f32<VPT>(sf + 2 * T + e, vv);
#pragma unroll
                for (int k = 0; k < VPT; k += 2) {
                    adamw_elem(bf16_lo(gw[k / 2]), p[k], mm[k], vv[k], a.s);
                    adamw_elem(bf16_hi(gw[k / 2]), p[k + 1], mm[k + 1], vv[k + 1], a.s);
                }
                const int64_t i = i0 + e;
                stg_f32<VPT>(tab->master[q] + i, p);
                stg_f32<VPT>(tab->m[q] + i, mm);
                stg_f32<VPT>(tab->v[q] + i, vv);
                uint32_t pw[VPT / 2];
#pragma unroll
                for (int k = 0; k < VPT; k += 2) pw[k / 2] = pack_bf16x2(p[k], p[k + 1]);
                uint16_t* o = tab->out[q] + (i - a.out_off);
                if constexpr (VPT == 8)
                    __stcs(reinterpret_cast<uint4*>(o), make_uint4(pw[0], pw[1], pw[2], pw[3]));
                else
                    __stcs(reinterpret_cast<uint2*>(o), make_uint2(pw[0], pw[1]));
                mbar_arrive(&empty[s]);                  // after the stores: see k_fused_tma
            } else {
                mbar_arrive(&empty[s]);
            }
        }
        // the grads buffer too is released only after stores that used what was read from it
        mbar_arrive(&gempty[b]);
    }
}

// The naive-DP step over one range; MINB CTAs per SM at least (a walk shape runs two, so a launch's
// CTAs share each SM with the next launch's).  The body returns early (producer lanes, a wait that
// ran out) into the launch-order epilogue.
template <int ND, int NCW, int VPT, int MAXST = 16, int BUDGET = 227 * 1024, int MINB = 1>
__global__ void __launch_bounds__(32 * (NCW + 1), MINB) k_dp_tma(const __grid_constant__ DpTmaArgs a) {
    dependent_launch_prologue(a.sync);
    dp_tma_body<ND, NCW, VPT, MAXST, BUDGET>(a);
    dependent_launch_epilogue(a.sync);
}

// The naive-DP step over one range in one persistent launch taking its tiles in dynamic order.
template <int ND, int NCW, int VPT, int MAXST, int BUDGET, int MINB>
__global__ void __launch_bounds__(32 * (NCW + 1), MINB) k_dp_tma_dyn(const __grid_constant__ DpTmaArgs a) {
    dependent_launch_prologue(kSyncStream);
    dp_tma_body<ND, NCW, VPT, MAXST, BUDGET, true>(a);
    dyn_order_finish(a.order);
}

namespace {

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, int MINB, bool DYN>
auto dp_kernel() {
    if constexpr (DYN)
        return k_dp_tma_dyn<ND, NCW, VPT, MAXST, BUDGET, MINB>;
    else
        return k_dp_tma<ND, NCW, VPT, MAXST, BUDGET, MINB>;
}

template <int ND, int NCW, int VPT, int MAXST, int BUDGET, int MINB = 1, bool DYN = false>
cudaError_t dp_tma_impl(DpTmaArgs a, cudaStream_t st) {
    using Sh = DpShape<ND, NCW, VPT, MAXST, BUDGET>;
    static_assert(Sh::kSmem <= 232448, "shared memory above the per-CTA limit");
    auto kern = dp_kernel<ND, NCW, VPT, MAXST, BUDGET, MINB, DYN>();
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)kern, 32 * (NCW + 1), Sh::kSmem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (a.n + Sh::kT - 1) / Sh::kT;
    if (ntiles < 1) return cudaSuccess;
    const int64_t cap = (int64_t)sms * per_sm;          // persistent: one wave of resident CTAs
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    if constexpr (DYN) {
        e = dyn_order_pair(&a.order);
        if (e != cudaSuccess) return e;
    }
    return launch_kernel(kern, dim3(grid), dim3(32 * (NCW + 1)), Sh::kSmem, st, a);
}

}  // namespace

// Staged naive-DP step over the 8-aligned body [lo, lo + n); cudaErrorNotSupported for rank
// counts without a staged shape.
cudaError_t launch_dp_tma(const BView& g, const BView& out, float* const* master, float* const* m,
                          float* const* v, int64_t lo, int64_t n, const AdamScalars& s, int nd, cudaStream_t st,
                          int sync) {
    bool ok = body_ok(lo, n);
    for (int q = 0; q < nd && ok; ++q)
        ok = at_ok(g.ptr.p[q], lo - g.off) && at_ok(out.ptr.p[q], lo - out.off) && at_ok(master[q], lo) &&
             at_ok(m[q], lo) && at_ok(v[q], lo);
    if (!ok) return cudaErrorMisalignedAddress;
    DpTmaArgs a{};
    a.g = g.ptr;
    a.g_off = g.off;
    a.out = out.ptr;
    a.out_off = out.off;
    for (int q = 0; q < nd && q < ZS_MAX_RANKS; ++q) {
        a.master[q] = master[q];
        a.m[q] = m[q];
        a.v[q] = v[q];
    }
    a.s = s;
    a.lo = lo;
    a.n = n;
    a.nd = nd;
    a.inv_nd = 1.0f / (float)nd;
    a.wait_limit = 4000000000LL;                     // ~2 s at the 2.07 GHz maximum SM clock
    a.drain_limit = 4000000000LL;
    a.sync = sync;
    if (sync == kSyncDynamic) {
        // One launch over the whole range, tiles in dynamic order, in the walk's shapes (two CTAs per
        // SM).  Measured on GB300 against the walk (GPT-2-small buffers, of the measured copy rate):
        // N_d = 2 / 4 / 8 / 16: 103.8 / 103.6 / 103.7 / 103.1 % (walk 101.5-101.6 / 100.1-100.7 / 99.7 /
        // 99.4 %).  N_d = 32 in its whole-range shape: 90.3 % against 93.1 % for the statically ordered
        // launch, so that rank count keeps it (dp_walk_shape).
        switch (nd) {
            case 2: return dp_tma_impl<2, 8, 8, 16, 115712, 2, true>(a, st);
            case 4: return dp_tma_impl<4, 8, 8, 16, 115712, 2, true>(a, st);
            case 8: return dp_tma_impl<8, 8, 4, 16, 115712, 2, true>(a, st);
            case 16: return dp_tma_impl<16, 8, 4, 16, 115712, 2, true>(a, st);
            default: return cudaErrorNotSupported;
        }
    }
    if (sync != kSyncStream) {
        // The launches of a walk: two CTAs per SM, each with half an SM's shared memory, 8 consumer
        // warps each.  Measured on GB300 (GPT-2-small buffers walked in 4 Mi-element launches, of the
        // measured copy rate; the whole-range shapes' single launch in brackets): N_d = 2: 8 x 8, T 2048,
        // 4 stages: 101.5 % (90.5 %); 4: 8 x 8, 3 stages: 100.8 % (96.7 %); 8: 8 x 4, T 1024, 6 stages:
        // 99.9 % (98.2 %); 16: 8 x 4, 4 stages: 99.3 % (97.8 %).  N_d = 32 (4 x 4, T 512, 7 stages:
        // 90.2 % against 94.1 %) keeps its single launch (dp_walk_shape).
        switch (nd) {
            case 2: return dp_tma_impl<2, 8, 8, 16, 115712, 2>(a, st);
            case 4: return dp_tma_impl<4, 8, 8, 16, 115712, 2>(a, st);
            case 8: return dp_tma_impl<8, 8, 4, 16, 115712, 2>(a, st);
            case 16: return dp_tma_impl<16, 8, 4, 16, 115712, 2>(a, st);
            default: return cudaErrorNotSupported;
        }
    }
    // Shapes per rank count from a measured sweep on GB300 (GPT-2-small buffers, 124.4 M elements;
    // consumer warps x elements per thread x ring depth x CTAs per SM).  The update is ALU-heavy
    // here (one AdamW per 28 bytes moved, twice the fused step's density), so the consumers set the
    // pace: 4 consumer warps per SM reached only 53 % at N_d = 8, 8 warps 97 %.  Of the measured copy
    // rate, staged / streaming: N_d = 2: 90 / 89 %, 4: 97 / 95 %, 8: 97-98 / 92 %, 16: 95 / 91 %,
    // 32: 94 / 91 %.
    switch (nd) {
        case 2: return dp_tma_impl<2, 16, 8, 16, 232448>(a, st);   // T 4096, 4 stages, 1 CTA/SM
        case 4: return dp_tma_impl<4, 8, 8, 16, 232448>(a, st);    // T 2048, 8 stages, 1 CTA/SM
        case 8: return dp_tma_impl<8, 8, 8, 16, 232448>(a, st);    // T 2048, 6 stages, 1 CTA/SM
        case 16: return dp_tma_impl<16, 8, 8, 16, 232448>(a, st);  // T 2048, 4 stages, 1 CTA/SM
        case 32: return dp_tma_impl<32, 8, 4, 16, 232448>(a, st);  // T 1024, 8 stages, 1 CTA/SM
        default: return cudaErrorNotSupported;
    }
}

bool dp_walk_shape(int nd) { return nd == 2 || nd == 4 || nd == 8 || nd == 16; }

// Self-test of the bounded wait: waits on an mbarrier nothing arrives at, with
// a budget of `limit` cycles, then records ZS_DEVERR_SELFTEST and returns.
__global__ void k_wait_selftest(long long limit) {
    dependent_launch_prologue();
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit)) flag_error(ZS_DEVERR_SELFTEST);
}

cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st) {
    return launch_kernel(k_wait_selftest, dim3(1), dim3(32), 0, st, limit_cycles);
}

// Bulk-store gather over the 8-aligned body [lo, lo + n): tiles of 16384 elements in a 4-stage ring
// (131 KB, so one one-warp CTA resident per SM), a grid of 16 CTAs per SM (chosen by measurement on
// GB300).
cudaError_t launch_gather_bulk(const uint16_t* src, int64_t src_off, const Ptrs& dst, int64_t dst_off, int64_t lo,
                               int64_t n, int nd, cudaStream_t st, int sync) {
    bool ok = body_ok(lo, n) && at_ok(src, lo - src_off);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(dst.p[q], lo - dst_off);
    if (!ok) return cudaErrorMisalignedAddress;
    GatherBulkArgs a{};
    a.src = src;
    a.src_off = src_off;
    a.dst = dst;
    a.dst_off = dst_off;
    a.lo = lo;
    a.n = n;
    a.nd = nd;
    a.T = 16384;
    a.wait_limit = 4000000000LL;
    a.drain_limit = 4000000000LL;
    a.sync = sync;
    if (sync != kSyncStream) {
        // a launch of a walk: a 2-stage ring (65,664 B, three CTAs per SM) and one wave of resident
        // CTAs, so a launch's CTAs share each SM with the next launch's
        constexpr int S2 = 2;
        const int smem2 = 128 + S2 * a.T * 2;
        int sms = 0, per_sm = 0;
        cudaError_t e = staged_geometry((const void*)k_gather_bulk<S2>, 32, smem2, &sms, &per_sm);
        if (e != cudaSuccess) return e;
        const int64_t ntiles = (n + a.T - 1) / a.T;
        const int64_t cap = (int64_t)sms * per_sm;
        const int grid = (int)(ntiles < cap ? ntiles : cap);
        return launch_kernel(k_gather_bulk<S2>, dim3(grid), dim3(32), smem2, st, a);
    }
    constexpr int S = 4;
    const int smem = 128 + S * a.T * 2;
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)k_gather_bulk<S>, 32, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (n + a.T - 1) / a.T;
    const int64_t cap = (int64_t)sms * 16;
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    return launch_kernel(k_gather_bulk<S>, dim3(grid), dim3(32), smem, st, a);
}

// The single-source gather over the 8-aligned body [lo, lo + n) in one dynamic-order launch: 16,384-element
// tiles in a 2-stage ring (65,664 B, three CTAs per SM), one wave of resident CTAs.
cudaError_t launch_gather_bulk_dyn(const uint16_t* src, int64_t src_off, const Ptrs& dst, int64_t dst_off, int64_t lo,
                                   int64_t n, int nd, cudaStream_t st) {
    bool ok = body_ok(lo, n) && at_ok(src, lo - src_off);
    for (int q = 0; q < nd && ok; ++q) ok = at_ok(dst.p[q], lo - dst_off);
    if (!ok) return cudaErrorMisalignedAddress;
    GatherBulkArgs a{};
    a.src = src;
    a.src_off = src_off;
    a.dst = dst;
    a.dst_off = dst_off;
    a.lo = lo;
    a.n = n;
    a.nd = nd;
    a.T = 16384;
    a.wait_limit = 4000000000LL;
    a.drain_limit = 4000000000LL;
    a.sync = kSyncStream;
    constexpr int S = 2;
    const int smem = 128 + S * a.T * 2;
    int sms = 0, per_sm = 0;
    cudaError_t e = staged_geometry((const void*)k_gather_bulk_dyn<S>, 32, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t ntiles = (n + a.T - 1) / a.T;
    const int64_t cap = (int64_t)sms * per_sm;
    const int grid = (int)(ntiles < cap ? ntiles : cap);
    e = dyn_order_pair(&a.order);
    if (e != cudaSuccess) return e;
    return launch_kernel(k_gather_bulk_dyn<S>, dim3(grid), dim3(32), smem, st, a);
}

cudaError_t read_device_error(unsigned int* out, bool clear) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_zs_device_error, sizeof(unsigned int));
    if (e != cudaSuccess || !clear) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_zs_device_error, &zero, sizeof(unsigned int));
}

}  // namespace zs
