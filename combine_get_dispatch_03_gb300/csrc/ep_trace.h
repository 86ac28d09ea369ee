// ep_trace.h -- NVTX ranges over the C ABI's entry points.
//
// Each entry point opens a range named after itself for as long as it runs, so that a profiler
// reading NVTX (Nsight Systems, or `ncu --nvtx --nvtx-include "ep_combine/"`) groups the kernels
// that one call enqueues.  NVTX is header-only; with no tool attached its calls return at once.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace ep {

class TraceRange {
public:
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace ep

#define EP_TRACE() ::ep::TraceRange ep_trace_range_(__func__)
