// One NVTX range per C-ABI call, named after the entry point, so that a timeline
// (Nsight Systems, or ncu --nvtx) shows which call enqueued which kernels.  NVTX v3 is
// header-only: without a tool attached the push / pop calls return at once.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace tp {

struct TraceRange {
  explicit TraceRange(const char* name) { nvtxRangePushA(name); }
  ~TraceRange() { nvtxRangePop(); }
  TraceRange(const TraceRange&) = delete;
  TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace tp

#define TP_TRACE() ::tp::TraceRange tp_trace_range_(__func__)
