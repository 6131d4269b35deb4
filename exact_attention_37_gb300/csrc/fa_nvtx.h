// NVTX ranges around the C-ABI calls.  Builds with -DFA_NVTX mark every call with
// a range named after it (shown by profilers that read NVTX, nearly free when
// none is attached: the header-only NVTX library loads a tool only if one is
// registered); other builds compile the marker to nothing.
#pragma once

#ifdef FA_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace fa {

struct NvtxRange {
#ifdef FA_NVTX
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
#else
  explicit NvtxRange(const char*) {}
#endif
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace fa
