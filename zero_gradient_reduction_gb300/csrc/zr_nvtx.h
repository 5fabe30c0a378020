// A named NVTX range over the span of a host call, so that Nsight tools show each
// step on the CPU timeline beside its kernels. NVTX is header-only: with no tool
// attached a range costs a few nanoseconds.
#pragma once
#include <nvtx3/nvToolsExt.h>

namespace zr {
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};
}  // namespace zr
