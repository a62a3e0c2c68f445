// trace.h -- NVTX ranges around the library's kernel launches, so that a
// profiler (nsys, or ncu --nvtx --nvtx-include) can attribute and filter them:
//   pkv::decode.schedule   the device plan's schedule kernel
//   pkv::decode.phase1     phase 1 (split attention)
//   pkv::decode.combine    phase 2 (cross-split combine)
//   pkv::mla.prefill       MLA staging kernel + tensor-core prefill kernel
// Header-only NVTX v3: with no tool attached a range costs a few branches.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pkv {

class TraceRange {
  public:
    explicit TraceRange(const char* name) { nvtxRangePushA(name); }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange&) = delete;
    TraceRange& operator=(const TraceRange&) = delete;
};

}  // namespace pkv
