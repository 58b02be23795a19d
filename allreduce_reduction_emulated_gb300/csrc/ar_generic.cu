// ar_generic.cu -- the pipelined all-reduce / reduce-scatter for any rank
// count, 128-thread blocks; calls capped below the SM count go to the
// 768-thread width in ar_generic_wide.cu (a translation unit of its own, so
// the two widths compile in parallel).
#include "ar_generic.cuh"

namespace ar {

static bool capped(const Call& c) { return c.max_blocks > 0 && c.max_blocks < c.sms; }

cudaError_t launch_generic(const Call& c, LaunchInfo* info) {
  if (capped(c)) return launch_generic_wide(c, info);
  return generic_dispatch<kThreads>(c, info);
}

cudaError_t launch_reduce_scatter_vec(const Call& c, LaunchInfo* info) {
  if (capped(c)) return launch_reduce_scatter_vec_wide(c, info);
  return scatter_dispatch<kThreads>(c, info);
}

}  // namespace ar
