// NVTX ranges over the library's entry points: each call shows up as a named
// range on the host timeline of a profiler (Nsight Systems, Nsight Compute's
// range filters).  NVTX v3 is header-only; with no tool attached a range costs
// a check of a function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace tv {

struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace tv

// A range named after the enclosing entry point, closed when it returns.
#define TV_NVTX_RANGE(name) ::tv::NvtxRange tv_nvtx_range_(name)
