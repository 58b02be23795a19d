// ar_launch.h -- internal interface between the C ABI (ar_api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace ar {

// Ranks up to this count run a kernel specialised on the exact rank count
// (all P input vectors held in registers); larger P runs the staged kernel.
constexpr int kMaxStaticRanks = 8;

// One all-reduce call as the kernels see it.
struct Call {
  int P;
  const void* const* send;  // host array of P device pointers
  void* const* recv;        // host array of P device pointers
  size_t count;             // elements per rank
  int dtype, op, algo;      // ar_dtype_t, ar_op_t, resolved ar_algo_t (never AUTO)
  float scale;
  cudaStream_t stream;
  int sms;                  // multiprocessors of the device
  // TREE for P > kMaxStaticRanks: tree 0's then tree 1's ranks in the order
  // their folds consume them (preorder; device memory, P entries each)
  const int16_t* tree_push;
  // LL protocol state
  unsigned long long* staging;  // P slots of stage_stride 8-byte words
  size_t stage_stride;
  int* status;                  // device status word (ar_status_t)
  // reduce-scatter / all-gather: elements per shard (recvcount / sendcount);
  // count is then the length of the larger buffers (P * shard)
  size_t shard;
  int group;                    // hierarchical order: ranks per group
  int max_blocks;               // > 0: at most this many CTAs (grid-stride loops)
  // LL / LL128 epoch state on the device ({last epoch, finished blocks}) and
  // the staging words it covers (cleared when the epoch wraps)
  unsigned int* epoch_state;
  size_t stage_words;
  uint32_t spin_limit;
  int skip_produce;
};

// What was launched, for AR_DEBUG logging.
struct LaunchInfo {
  const char* kernel = "";
  int grid = 0;
  int block = 0;
  size_t smem = 0;
};

// Programmatic dependent launch for a call that has the whole GPU: the kernel
// may be scheduled while the kernel before it on the stream drains, and waits
// on the device (pdl_enter) for that kernel's completion before it touches
// memory, so the stream's order is kept and only the launch gap is hidden
// (8 x 64 MiB fp32 ring: 157.7 -> 155.0 us per call back to back).  A call
// capped to a few SMs is launched plainly: its blocks would otherwise wait on
// SMs that other work is using (bucket all-reduces on 48 SMs beside gradient
// GEMMs: 27.05 ms per step launched this way, 25.01 ms plainly).
inline bool use_pdl(const Call& c) { return c.max_blocks <= 0 || c.max_blocks >= c.sms; }

template <class... K, class... A>
cudaError_t launch_kernel(void (*kernel)(K...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                          bool pdl, A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

// Elements per 16-byte vector.
inline int vec_elems(int dtype) { return dtype == 1 ? 8 : 4; }
inline size_t elem_bytes(int dtype) { return dtype == 1 ? 2 : 4; }

// rank-specialised kernels (P <= kMaxStaticRanks): all-reduce, or the ring
// reduce-scatter when c.shard != 0 (shards of whole 16-byte vectors)
cudaError_t launch_static_f32(const Call& c, LaunchInfo* info);
cudaError_t launch_static_bf16(const Call& c, LaunchInfo* info);
cudaError_t launch_static_i32(const Call& c, LaunchInfo* info);
// the same kernels in their wide shape (1024 threads per block, at most
// c.max_blocks blocks and one per SM, grid-stride): for calls that share the GPU
cudaError_t launch_wide_f32(const Call& c, LaunchInfo* info);
cudaError_t launch_wide_bf16(const Call& c, LaunchInfo* info);
cudaError_t launch_wide_i32(const Call& c, LaunchInfo* info);
// the same all-reduce (P <= kMaxStaticRanks, ring or tree; or the ring
// reduce-scatter when c.shard != 0) as a TMA bulk-copy pipeline, one block per
// SM on c.max_blocks SMs: for calls that share the GPU
cudaError_t launch_tma_f32(const Call& c, LaunchInfo* info);
cudaError_t launch_tma_bf16(const Call& c, LaunchInfo* info);
cudaError_t launch_tma_i32(const Call& c, LaunchInfo* info);
// the TMA kernel is chosen when every block gets at least this many bytes per
// rank (its tiles are 6 or 8 KiB; a block with fewer bytes has little to pipeline)
constexpr size_t kTmaTileBytes = 4096;
// the all-gather (any P) as a TMA pipeline on c.max_blocks SMs; its tile size
cudaError_t launch_all_gather_tma(const Call& c, LaunchInfo* info);
constexpr size_t kTmaGatherTileBytes = 32768;
cudaError_t launch_generic(const Call& c, LaunchInfo* info);
// the same pipelined kernels in 768-thread blocks, at most one per SM (calls
// capped below the SM count; launch_generic and launch_reduce_scatter_vec
// forward to them)
cudaError_t launch_generic_wide(const Call& c, LaunchInfo* info);
cudaError_t launch_reduce_scatter_vec_wide(const Call& c, LaunchInfo* info);
cudaError_t launch_ll(const Call& c, LaunchInfo* info);
// LL128: 128-byte lines of 120 payload bytes + a flag word (staging, stage_stride)
cudaError_t launch_ll128(const Call& c, LaunchInfo* info);
size_t ll128_stage_words(size_t bytes_per_rank);
// reduce-scatter with shards of whole 16-byte vectors, any P (pipelined ring kernel)
cudaError_t launch_reduce_scatter_vec(const Call& c, LaunchInfo* info);
// reduce-scatter of any shard length, element by element (same order)
cudaError_t launch_reduce_scatter_elem(const Call& c, LaunchInfo* info);
// all-gather: every rank's shard copied to all P receive buffers
cudaError_t launch_all_gather(const Call& c, LaunchInfo* info);

// Ring chunk length in vectors and first vector of tree 1, for `count`.
inline uint64_t ring_chunk_vectors(size_t count, int P, int dtype) {
  const uint64_t V = (uint64_t)vec_elems(dtype);
  const uint64_t per = (count + (uint64_t)P - 1) / (uint64_t)P;
  return (per + V - 1) / V;
}
inline uint64_t tree_split_vectors(size_t count, int dtype) {
  const uint64_t V = (uint64_t)vec_elems(dtype);
  uint64_t h = ((count + 1) / 2 + V - 1) / V * V;
  if (h > count) h = count;
  return (h + V - 1) / V;
}

}  // namespace ar
