// NVTX ranges around the host side of each entry point, so that a profiler's
// timeline shows planning, updates and launches by name. NVTX v3 is header-only:
// without a tool attached the calls return at once.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace pkv {

struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

}  // namespace pkv
