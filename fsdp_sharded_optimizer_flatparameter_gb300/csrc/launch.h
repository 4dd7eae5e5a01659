// Host-side launchers of the step's kernels (internal; not part of the C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>
#include <vector>

#include "zs.h"

namespace zs {

// N_d rank pointers to bf16 words.
struct Ptrs {
    uint16_t* p[ZS_MAX_RANKS];
};

// A bf16 buffer kind resolved to addresses: rank q's element at global flat
// index i lives at ptr.p[q] + (i - off).  A ZS_SHARDED array repeats its one
// pointer in every slot with off = 0.
struct BView {
    Ptrs ptr;
    int64_t off;
};

// The step-dependent fp32 scalars of AdamW (see zs_adamw_scalars).
struct AdamScalars {
    float beta1, beta2, eps, decay, c1, c2, step_size, sqrt_bc2;
};

// How a kernel orders itself against the previous kernel on its stream under programmatic
// dependent launch (see dependent_launch_prologue in device.cuh).
//   kSyncStream    every launch by default: let the successor launch, then wait for the
//                  predecessor before touching global memory (plain stream order for every byte).
//   kSyncWalkFirst the first launch of a walk over disjoint ranges: wait for the predecessor,
//                  then let the successor launch, so no later launch of the walk starts before
//                  everything enqueued ahead of the walk has completed.
//   kSyncWalkNext  a later staged launch of such a walk: let the successor launch at once and read
//                  and write its own range without waiting; CTA 0 waits for the predecessor before
//                  exiting, so the launch completes after every launch before it.  Valid only when the
//                  kernel touches no byte that an earlier launch of the walk touches, and it reads
//                  global memory only through bulk copies (which read L2, never a stale L1 line).
//   kSyncDynamic   (launch_fused with one output, launch_gather) one launch over the whole range whose
//                  CTAs take their tiles in dynamic order from a counter pair (kDynMinElems and more
//                  elements on device buffers, else plain stream order); in stream order otherwise.
enum LaunchSync : int { kSyncStream = 0, kSyncWalkFirst = 1, kSyncWalkNext = 2, kSyncDynamic = 3 };

// A global range [lo, hi) inside one unit (base, shard); owner(i) = (i - base) / shard.
struct Range {
    int64_t lo, hi;
    int64_t base, shard;
};

cudaError_t launch_accumulate(const Ptrs& acc, const Ptrs& micro, int nd, int64_t n, float scale, int first,
                              cudaStream_t st);
cudaError_t launch_rs_mean(const BView& g, const BView& out, bool out_by_owner, const Range& r, int nd,
                           cudaStream_t st);
cudaError_t launch_adamw(const BView& grad, bool grad_by_owner, float* master, float* m, float* v,
                         const BView& par, bool par_by_owner, const Range& r, const AdamScalars& s,
                         cudaStream_t st);
// `sync`: a launch-order mode of a walk over disjoint ranges (kSyncWalkFirst / kSyncWalkNext) for the
// bulk-store kernel; the streaming kernel keeps stream order (a first launch of a walk still waits
// before it lets its successor launch).
cudaError_t launch_gather(const BView& src, bool src_by_owner, const BView& dst, bool skip_owner,
                          const Range& r, int nd, cudaStream_t st, int sync = kSyncStream);
// The last micro-batch's accumulation folded into the broadcast fused step: rank q's gradient is
// bf16(acc_q[i] + micro_q[i] * scale) (the accumulation rule, computed in the kernel and not stored),
// where the fused launch's gradient view holds the accumulators acc_q and `micro` the micro-batch.
struct AccumIn {
    BView micro;
    float scale;
};

// The fused step over r.  The staged kernel runs only for the 8-aligned body of a range of a
// supported rank count whose buffers are all device memory; elsewhere the register-streaming kernel.
// With `acc` (broadcast only) the gradients are formed from accumulators and a micro-batch.
// Which fused kernel a launch may use.  kStagedIfDevice asks the runtime about every pointer;
// kStagedDeviceKnown is for callers that already did (fused_ptrs_on_device) for the same pointers.
enum StagedPolicy { kStagedNever = 0, kStagedIfDevice = 1, kStagedDeviceKnown = 2 };
// `sync` (LaunchSync) orders the launch against its predecessor; a walk over disjoint buckets passes
// kSyncWalkFirst for its first launch on a stream and kSyncWalkNext for later ones, and then also
// takes the staged kernel for bodies down to kTmaWalkMinElems.
cudaError_t launch_fused(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast,
                         const Range& r, const AdamScalars& s, int nd, cudaStream_t st,
                         StagedPolicy staged_policy = kStagedIfDevice, int sync = kSyncStream,
                         const AccumIn* acc = nullptr);
// True when every pointer a fused launch over these views touches is device memory.
bool fused_ptrs_on_device(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast, int nd,
                          const AccumIn* acc = nullptr);

// Whether the broadcast staged kernel has a walk shape for this rank count: a shape whose launches
// share each SM with the next launch of a walk, for kSyncWalkFirst / kSyncWalkNext launches.
bool fused_walk_shape(int nd, bool acc = false);
// Whether the broadcast staged kernel has a dynamic-order shape for this rank count: one persistent
// launch whose CTAs take tiles from a counter, for one range of at least kDynMinElems elements.
bool fused_dyn_shape(int nd);
constexpr int64_t kDynMinElems = int64_t(1) << 24;
cudaError_t launch_fused_tma_dyn(const BView& g, float* master, float* m, float* v, const BView& out, int64_t lo,
                                 int64_t n, const AdamScalars& s, int nd, cudaStream_t st,
                                 const AccumIn* acc = nullptr);
// The single-output form (one output array; nd = 1: the update alone) in one dynamic-order launch.
cudaError_t launch_fused_single_dyn(const BView& g, float* master, float* m, float* v, const BView& out, int64_t lo,
                                    int64_t n, const AdamScalars& s, int nd, cudaStream_t st);
cudaError_t launch_gather_bulk_dyn(const uint16_t* src, int64_t src_off, const Ptrs& dst, int64_t dst_off, int64_t lo,
                                   int64_t n, int nd, cudaStream_t st);
// The broadcast fused step over disjoint ranges as a walk: ranges longer than kFusedWalkChunk are cut
// at multiples of it, each piece is one launch, the first on the stream kSyncWalkFirst and the others
// kSyncWalkNext, so every launch streams its piece while the previous one drains.  Without a walk
// shape for nd, one launch per range in stream order.
constexpr int64_t kFusedWalkChunk = int64_t(1) << 22;
cudaError_t launch_fused_walk(const BView& g, float* master, float* m, float* v, const BView& out,
                              const std::vector<Range>& ranges, const AdamScalars& s, int nd, cudaStream_t st,
                              StagedPolicy staged_policy, const AccumIn* acc = nullptr);
// Bulk-copy staged fused kernel over the 8-aligned body [lo, lo + n); returns
// cudaErrorNotSupported when no staged variant exists for this rank count.
cudaError_t launch_fused_tma(const BView& g, float* master, float* m, float* v, const BView& out, bool broadcast,
                             int64_t lo, int64_t n, const AdamScalars& s, int nd, cudaStream_t st,
                             int sync = kSyncStream, const AccumIn* acc = nullptr);
// The broadcast staged kernel over a list of bodies ([lo, lo + n): the TMA alignment rules of
// launch_fused_tma for each) in one launch per kTmaListMax (128) bodies, tiles walked in list order.
cudaError_t launch_fused_tma_list(const BView& g, float* master, float* m, float* v, const BView& out,
                                  const std::vector<std::pair<int64_t, int64_t>>& bodies, const AdamScalars& s,
                                  int nd, cudaStream_t st);
// The broadcast fused step over several ranges: touching ranges merge; with the staged kernel each
// range with a body of at least kTmaWalkMinElems is walked (launch_fused_walk) and the short runs
// share list launches (their fringe elements by the streaming kernel); else one streaming launch per
// range.
cudaError_t launch_fused_ranges(const BView& g, float* master, float* m, float* v, const BView& out,
                                const std::vector<Range>& ranges, const AdamScalars& s, int nd, cudaStream_t st,
                                StagedPolicy staged_policy = kStagedIfDevice);
cudaError_t launch_wait_selftest(long long limit_cycles, cudaStream_t st);
// Staged reduce-scatter-mean of the body [lo, lo + n) into one array (element i at out + (i -
// out_off)); the TMA alignment rules of launch_fused_tma.  cudaErrorNotSupported for rank counts
// without a staged shape.
cudaError_t launch_rs_tma(const BView& g, uint16_t* out, int64_t out_off, int64_t lo, int64_t n, int nd,
                          cudaStream_t st);
// FSDP2 layout copies (csrc/fsdp2.cu): one launch covers up to kFsdp2PerLaunch parameters of a
// group; every (parameter, rank) piece is cut into tasks of kFsdp2Task buffer elements, task t of
// the launch belonging to the last piece j with first[j] <= t (rank = (t - first[j]) / tasks).
constexpr int kFsdp2PerLaunch = 64;
constexpr int64_t kFsdp2Task = 16384;
struct Fsdp2Piece {
    uint16_t* param;        // the parameter's own layout (d0 x row elements)
    int64_t d0, row, chunk, off;
    int64_t tasks;          // tasks per rank: ceil(chunk * row / kFsdp2Task)
};
struct Fsdp2CopyArgs {
    Fsdp2Piece p[kFsdp2PerLaunch];
    int64_t first[kFsdp2PerLaunch + 1];
    int n;                  // pieces in this launch
    uint16_t* flat;         // the group's buffer (N_d * shard elements)
    int64_t shard;
    int to_flat;            // 1: parameters -> buffer (zero padding rows), 0: buffer -> parameters
};
// One source to N_d destinations with bulk stores, over the 8-aligned body [lo, lo + n); `sync` as for
// the fused kernel (the kernel reads through bulk copies only, so it may be a later launch of a walk).
cudaError_t launch_gather_bulk(const uint16_t* src, int64_t src_off, const Ptrs& dst, int64_t dst_off, int64_t lo,
                               int64_t n, int nd, cudaStream_t st, int sync = kSyncStream);
cudaError_t launch_all_reduce_mean(const BView& g, const Range& r, int nd, cudaStream_t st);
// Bulk-copy staged in-place all-reduce over the 8-aligned body [lo, lo + n) of every rank's buffer
// (device memory), one launch of a walk (`sync`), or with kSyncDynamic one launch over the whole body
// taking its tiles in dynamic order (rank counts with ar_dyn_shape); cudaErrorNotSupported without a
// staged shape.
bool ar_dyn_shape(int nd);
cudaError_t launch_all_reduce_tma(const BView& g, int64_t lo, int64_t n, int nd, cudaStream_t st, int sync);
// Staged naive-DP step over the 8-aligned body [lo, lo + n) (the TMA alignment rules of
// launch_fused_tma; every rank's master, m and v 16-byte aligned); cudaErrorNotSupported for rank
// counts without a staged shape.  `sync` as for the fused kernel (the kernel reads through bulk copies
// only, so it may be a later launch of a walk); walk launches need a walk shape (dp_walk_shape).  With
// kSyncDynamic, one launch over the whole body taking its tiles in dynamic order (rank counts with a walk
// shape).
bool dp_walk_shape(int nd);
cudaError_t launch_dp_tma(const BView& g, const BView& out, float* const* master, float* const* m,
                          float* const* v, int64_t lo, int64_t n, const AdamScalars& s, int nd, cudaStream_t st,
                          int sync = kSyncStream);
// The naive-DP step over r: the staged kernel for the 8-aligned body of a large range whose buffers
// are all device memory (the few fringe elements, and everything else, by the streaming kernel).
cudaError_t launch_dp_step(const BView& g, const BView& out, float* const* master, float* const* m, float* const* v,
                           const Range& r, const AdamScalars& s, int nd, cudaStream_t st);
cudaError_t read_device_error(unsigned int* out, bool clear);

// Which fused kernel zs_fused_step / zs_zero3_rs_step_unit use (ZS_FUSED_*).
void set_fused_variant(int v);
int fused_variant();

// Whether launches allow programmatic dependent launch (see dependent_launch_prologue).
void set_dependent_launch(int on);
int dependent_launch();

// Launches kern<<<grid, block, smem, st>>>(args...) with programmatic stream serialization allowed
// when dependent launch is on; a failed launch is returned and cleared from the runtime's last-error
// state, as cudaGetLastError after <<<>>> did.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = dependent_launch() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
    if (e != cudaSuccess) cudaGetLastError();
    return e;
}

}  // namespace zs
