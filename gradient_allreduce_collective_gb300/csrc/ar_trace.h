// ar_trace.h — an NVTX range around each library call, so that nsys and ncu
// timelines show which call launched which kernels. NVTX v3 is header-only:
// with no tool attached a range costs a check of one function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace gar {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace gar

#define AR_TRACE(name) const gar::TraceRange ar_trace_range_(name)
