// ar_wide_bf16.cu -- the rank-specialised kernels in their wide shape (1024
// threads per block, one block per SM) for calls capped to a few SMs, for one
// data type (separate translation units so the data types compile in parallel).
#include "ar_static.cuh"

namespace ar {

cudaError_t launch_wide_bf16(const Call& c, LaunchInfo* info) { return launch_static_dt<kBF16, true>(c, info); }

}  // namespace ar
