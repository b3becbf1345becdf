// NVTX ranges over the library's host calls, so that a timeline profiler
// shows each call's launches under its name.  NVTX v3 is header-only; without
// a profiler attached a range costs a few nanoseconds.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace specv {

struct TraceRange {
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace specv
