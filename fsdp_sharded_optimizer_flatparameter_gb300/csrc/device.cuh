// Device helpers shared by the kernels of the sharded optimizer step.
//
// Numerics follow the definition of the step in "Infra: Data Parallel"
// (F. Pu), section "Zero Redundancy Optimizer (ZeRO)": 16-bit (bf16)
// parameters and gradients, fp32 master weights and moments.  Every fp32
// operation is written with an explicitly rounded intrinsic (__fadd_rn,
// __fmul_rn, __fdiv_rn, __fsqrt_rn) so the compiler cannot contract a
// multiply and an add into an FMA: each operation is rounded once, to
// nearest even, in the order written.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace zs {

// ------------------------------------------------------------------ bf16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float((uint32_t)h << 16); }

// Two fp32 values -> two bf16 (round to nearest even) packed as lo | hi << 16.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

__device__ __forceinline__ uint16_t f32_to_bf16(float x) {
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(x));
    return h;
}

// ------------------------------------------------------------------ vectors of VEC elements
// VEC = 8: one 16-byte access per bf16 vector, two per fp32 vector (the
// caller guarantees 16-byte alignment).  VEC = 1: scalar accesses.
// Loads and stores use the streaming (evict-first) cache policy: every byte
// is touched once per step.

template <int VEC> struct BfVec;            // VEC bf16 values packed in 32-bit words
template <> struct BfVec<8> { uint4 w; };
template <> struct BfVec<1> { uint16_t h; };

template <int VEC>
__device__ __forceinline__ BfVec<VEC> ld_bf(const uint16_t* p);
template <>
__device__ __forceinline__ BfVec<8> ld_bf<8>(const uint16_t* p) { return {__ldcs(reinterpret_cast<const uint4*>(p))}; }
template <>
__device__ __forceinline__ BfVec<1> ld_bf<1>(const uint16_t* p) { return {__ldcs(reinterpret_cast<const unsigned short*>(p))}; }

template <int VEC>
__device__ __forceinline__ void st_bf(uint16_t* p, const BfVec<VEC>& v);
template <>
__device__ __forceinline__ void st_bf<8>(uint16_t* p, const BfVec<8>& v) { __stcs(reinterpret_cast<uint4*>(p), v.w); }
template <>
__device__ __forceinline__ void st_bf<1>(uint16_t* p, const BfVec<1>& v) { __stcs(reinterpret_cast<unsigned short*>(p), v.h); }

__device__ __forceinline__ void unpack(const BfVec<8>& v, float (&f)[8]) {
    f[0] = bf16_lo(v.w.x); f[1] = bf16_hi(v.w.x);
    f[2] = bf16_lo(v.w.y); f[3] = bf16_hi(v.w.y);
    f[4] = bf16_lo(v.w.z); f[5] = bf16_hi(v.w.z);
    f[6] = bf16_lo(v.w.w); f[7] = bf16_hi(v.w.w);
}
__device__ __forceinline__ void unpack(const BfVec<1>& v, float (&f)[1]) { f[0] = bf16_to_f32(v.h); }

__device__ __forceinline__ BfVec<8> pack(const float (&f)[8]) {
    BfVec<8> v;
    v.w.x = pack_bf16x2(f[0], f[1]);
    v.w.y = pack_bf16x2(f[2], f[3]);
    v.w.z = pack_bf16x2(f[4], f[5]);
    v.w.w = pack_bf16x2(f[6], f[7]);
    return v;
}
__device__ __forceinline__ BfVec<1> pack(const float (&f)[1]) { return {f32_to_bf16(f[0])}; }

template <int VEC>
__device__ __forceinline__ void ld_f32(const float* p, float (&f)[VEC]) {
    if constexpr (VEC == 8) {
        float4 a = __ldcs(reinterpret_cast<const float4*>(p));
        float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
        f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
        f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
    } else {
        f[0] = __ldcs(p);
    }
}

template <int VEC>
__device__ __forceinline__ void st_f32(float* p, const float (&f)[VEC]) {
    if constexpr (VEC == 8) {
        __stcs(reinterpret_cast<float4*>(p), make_float4(f[0], f[1], f[2], f[3]));
        __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(f[4], f[5], f[6], f[7]));
    } else {
        __stcs(p, f[0]);
    }
}

// ------------------------------------------------------------------ the method's arithmetic

// Mean over ranks of an fp32 sum: sum / N_d, correctly rounded.  For a power
// of two the quotient equals sum * (1/N_d) exactly (both are the correctly
// rounded value of the same real number), which avoids the division.
template <int ND>
__device__ __forceinline__ float mean_of_sum(float sum, int nd, float inv_nd) {
    if constexpr (ND > 0 && (ND & (ND - 1)) == 0) {
        return __fmul_rn(sum, inv_nd);
    } else {
        return __fdiv_rn(sum, (float)nd);
    }
}

// Gradient accumulation of one element: the running sum plus the micro-batch's gradient times the
// scale, each operation rounded in fp32 ("Infra: Data Parallel", gradient accumulation); the caller
// stores the result as bf16 (or, folded into a step, rounds it to bf16 before use).
__device__ __forceinline__ float accumulate_elem(float acc, float micro, float scale) {
    return __fadd_rn(acc, __fmul_rn(micro, scale));
}

// AdamW on one element (decoupled weight decay, bias corrections folded into
// step_size and sqrt_bc2); g is the fp32 value of the bf16 reduced gradient.
__device__ __forceinline__ void adamw_elem(float g, float& p, float& m, float& v, const AdamScalars& s) {
    const float pd = __fmul_rn(p, s.decay);
    m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.c1, g));
    v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.c2, __fmul_rn(g, g)));
    const float den = __fadd_rn(__fdiv_rn(__fsqrt_rn(v), s.sqrt_bc2), s.eps);
    p = __fsub_rn(pd, __fmul_rn(s.step_size, __fdiv_rn(m, den)));
}

// Programmatic dependent launch (sm_90 and later).  The library launches its kernels with
// programmatic stream serialization allowed: the next kernel on a stream may be scheduled once
// every CTA of the current one has started, so its CTAs are resident when the current one ends
// instead of being launched after it.  Each kernel therefore first lets its successor launch and
// then waits (griddepcontrol.wait: until every prerequisite grid has completed and its memory
// operations are visible) before it touches global memory, which keeps stream order for every
// byte; it waits no longer than plain stream order would.  Launched without the attribute, both
// instructions do nothing.
// A walk over disjoint ranges (the launches of one bucket-by-bucket call) relaxes this with the
// modes of LaunchSync: its first launch waits before it lets the next one launch, and its later
// staged launches start on their own ranges at once and wait only before their CTA 0 exits
// (dependent_launch_epilogue), so a launch's CTAs stream while its predecessor drains and the walk
// still completes in order.  The wait never deadlocks: a kernel is launched early only after every
// CTA of its predecessor has started, so the grid it waits for needs no further resources.
__device__ __forceinline__ void dependent_launch_prologue(int sync = kSyncStream) {
    if (sync == kSyncWalkFirst) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else if (sync == kSyncWalkNext) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

// A kSyncWalkNext launch completes only after its predecessor: CTA 0 waits for the predecessor
// before it exits, and a grid completes when its last CTA exits.  The other CTAs exit as soon as
// their work is done, so a CTA that drew fewer tiles frees its SM for the next launch at once.
__device__ __forceinline__ void dependent_launch_epilogue(int sync) {
    if (sync == kSyncWalkNext && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)
        asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Grid-stride loop helpers.
__device__ __forceinline__ int64_t gtid() { return (int64_t)blockIdx.x * blockDim.x + threadIdx.x; }
__device__ __forceinline__ int64_t gstride() { return (int64_t)gridDim.x * blockDim.x; }

}  // namespace zs
