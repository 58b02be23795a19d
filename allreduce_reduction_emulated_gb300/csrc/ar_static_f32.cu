// ar_static_f32.cu -- rank-specialised ring / tree kernels for one data type
// (separate translation units so the three data types compile in parallel).
#include "ar_static.cuh"

namespace ar {

cudaError_t launch_static_f32(const Call& c, LaunchInfo* info) { return launch_static_dt<kF32>(c, info); }

}  // namespace ar
