// Named host ranges for profilers (NVTX, header-only).  A range marks the host-side enqueue of
// one phase (a unit's gather, a bucket's update); profilers line them up with the kernels they
// launched.  Without a profiler attached the calls return at once.
#pragma once

#include <cstdio>

#include <nvtx3/nvToolsExt.h>

namespace zs {

struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    TraceRange(const char* fmt, long long a) {
        char buf[96];
        std::snprintf(buf, sizeof(buf), fmt, a);
        nvtxRangePushA(buf);
    }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace zs
