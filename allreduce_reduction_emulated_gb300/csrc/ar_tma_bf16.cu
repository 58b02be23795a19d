// ar_tma_bf16.cu -- the TMA-pipelined rank-specialised all-reduce for one data
// type (separate translation units so the three data types compile in parallel).
#include "ar_tma.cuh"

namespace ar {

cudaError_t launch_tma_bf16(const Call& c, LaunchInfo* info) { return tma::launch_dt<kBF16>(c, info); }

}  // namespace ar
