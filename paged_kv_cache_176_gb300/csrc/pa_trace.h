// pa_trace.h -- NVTX ranges around the library's entry points, so a timeline
// tool (ncu's range filters, a system profiler) can attribute device work to
// the call that enqueued it. nvtx3 is header-only: without a tool attached
// the calls do nothing.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace pa {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace pa
