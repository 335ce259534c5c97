// Sep-Attention backward (tcgen05).  Not built yet: every request reports
// "not supported".
#include "common.cuh"
#include "layout.h"

namespace sep {

size_t attn_bwd_tc_workspace(int, int, int, int, int) { return 256; }

int launch_attn_bwd_tc(IndexPtrs, const void*, const void*, const void*, const void*,
                       const float*, const void*, void*, void*, void*, int, int, int, int, int,
                       float, void*, int*, void*) {
  return static_cast<int>(cudaErrorNotSupported);
}

}  // namespace sep
