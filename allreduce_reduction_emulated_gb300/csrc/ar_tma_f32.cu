// ar_tma_f32.cu -- the TMA-pipelined rank-specialised all-reduce for one data
// type (separate translation units so the three data types compile in parallel).
#include "ar_tma.cuh"

namespace ar {

cudaError_t launch_tma_f32(const Call& c, LaunchInfo* info) { return tma::launch_dt<kF32>(c, info); }

}  // namespace ar
