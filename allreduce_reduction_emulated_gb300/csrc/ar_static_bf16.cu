// ar_static_bf16.cu -- rank-specialised ring / tree kernels for one data type
// (separate translation units so the three data types compile in parallel).
#include "ar_static.cuh"

namespace ar {

cudaError_t launch_static_bf16(const Call& c, LaunchInfo* info) { return launch_static_dt<kBF16>(c, info); }

}  // namespace ar
