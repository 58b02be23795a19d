// ar_static_i32.cu -- rank-specialised ring / tree kernels for one data type
// (separate translation units so the three data types compile in parallel).
#include "ar_static.cuh"

namespace ar {

cudaError_t launch_static_i32(const Call& c, LaunchInfo* info) { return launch_static_dt<kI32>(c, info); }

}  // namespace ar
