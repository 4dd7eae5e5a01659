// The pieces of a walk: a range cut into launches that overlap one another (the launch-order modes
// kSyncWalkFirst / kSyncWalkNext of launch.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "launch.h"

namespace zs {

// Calls launch(lo, hi, sync) for each piece of [lo, hi): cuts at multiples of `chunk` (so cuts keep the
// 8-element grid when `chunk` is a multiple of 8), none closer than chunk / 4 to either end of the
// range, so no piece is a sliver; the first piece gets first_sync (kSyncWalkFirst for a walk on its
// own), the others kSyncWalkNext.  `chunk` <= 0 leaves the range whole.  Stops at the first error.
template <class F>
cudaError_t walk_range(int64_t lo, int64_t hi, int64_t chunk, F&& launch, int first_sync = kSyncWalkFirst) {
    bool first = true;
    while (lo < hi) {
        int64_t end = hi;
        if (chunk > 0) {
            const int64_t cut = (lo + chunk / 4 + chunk) / chunk * chunk;    // first multiple past lo + chunk/4
            if (cut < hi - chunk / 4) end = cut;
        }
        const cudaError_t e = launch(lo, end, first ? first_sync : (int)kSyncWalkNext);
        if (e != cudaSuccess) return e;
        first = false;
        lo = end;
    }
    return cudaSuccess;
}

}  // namespace zs
