// nvtx.h — optional NVTX ranges around the C entry points, so that a profiler's timeline
// shows each call (its validation, planning and launch) by name.  Compiled in only when
// the library is built with PKV_NVTX defined; otherwise PKV_RANGE costs nothing.  (NVTX
// calls are themselves near free when no tool is attached.)
#pragma once

#ifdef PKV_NVTX
#include <nvtx3/nvToolsExt.h>

namespace pkv {
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace pkv
#define PKV_RANGE(name) const ::pkv::NvtxRange pkv_nvtx_range_(name)
#else
#define PKV_RANGE(name) ((void)0)
#endif
