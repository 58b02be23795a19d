// ar_generic_wide.cu -- the pipelined all-reduce / reduce-scatter in 768-thread
// blocks, at most one per SM, for calls capped to a few SMs.
#include "ar_generic.cuh"

namespace ar {

cudaError_t launch_generic_wide(const Call& c, LaunchInfo* info) { return generic_dispatch<kWideThreads>(c, info); }

cudaError_t launch_reduce_scatter_vec_wide(const Call& c, LaunchInfo* info) {
  return scatter_dispatch<kWideThreads>(c, info);
}

}  // namespace ar
