// gdn_trace.h -- host-side tracing of the C-ABI calls.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace gdn {

// An NVTX range over the host side of one C-ABI call (a profiler attached to
// the process shows each call as a named range; without one, push and pop do
// nothing).
struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace gdn
