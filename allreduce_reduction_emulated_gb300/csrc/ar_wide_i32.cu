// ar_wide_i32.cu -- the rank-specialised kernels in their wide shape (1024
// threads per block, one block per SM) for calls capped to a few SMs, for one
// data type (separate translation units so the data types compile in parallel).
#include "ar_static.cuh"

namespace ar {

cudaError_t launch_wide_i32(const Call& c, LaunchInfo* info) { return launch_static_dt<kI32, true>(c, info); }

}  // namespace ar
