// ar_collectives.cu -- the two halves of the ring all-reduce as standalone
// collectives ("NCCL, NIXL, and Distributed GPU Communication", sections
// "Reduce-scatter" and "All-gather"):
//   reduce-scatter -- element-wise kernel for shards that are not whole
//                     16-byte vectors (whole-vector shards run the ring
//                     kernels in scatter mode: ar_static.cuh for P <= 8,
//                     ar_tma.cuh when capped to a few SMs, ar_generic.cu
//                     above 8 ranks);
//   all-gather     -- rank s's sendcount elements copied to offset
//                     s * sendcount of every rank's receive buffer: one read
//                     and P writes per element, 16-byte vectors when every
//                     shard offset is 16-byte aligned, else element by element.
#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

constexpr int kThreads = 256;
// The vector all-gather: one load and P stores per thread, in 1024-thread
// blocks (8 x 8 MiB pieces back to back: 88.9 us per call against 89.6 in
// 256-thread blocks; two or four vectors per thread were slower).
constexpr int kAgThreads = 1024;

struct CollParams {
  const void* send[AR_MAX_RANKS];
  void* recv[AR_MAX_RANKS];
  int P;
  uint64_t shard;   // elements per shard
  uint64_t total;   // work items (elements or vectors) over all shards
  float scale;
  int do_scale;
};

template <int DT>
__device__ __forceinline__ typename Lanes<DT>::T load_elem(const void* base, uint64_t e) {
  if constexpr (DT == kF32) return static_cast<const float*>(base)[e];
  else if constexpr (DT == kI32) return static_cast<const int32_t*>(base)[e];
  else return bf16_lo((uint32_t) static_cast<const uint16_t*>(base)[e]);
}

template <int DT>
__device__ __forceinline__ void store_elem(void* base, uint64_t e, typename Lanes<DT>::T y, float scale,
                                           bool do_scale) {
  if constexpr (DT == kI32) {
    static_cast<int32_t*>(base)[e] = y;
  } else {
    if (do_scale) y = __fmul_rn(y, scale);
    if constexpr (DT == kF32) static_cast<float*>(base)[e] = y;
    else static_cast<uint16_t*>(base)[e] = (uint16_t)(pack_bf16x2(y, 0.0f) & 0xffffu);
  }
}

// Element e of the P * shard inputs: shard s = e / shard, folded in the ring
// order of chunk s (x_s, x_{s+1}, ...), result to rank s at e - s * shard.
template <int DT, int OP>
__global__ void __launch_bounds__(kThreads) reduce_scatter_elem_kernel(const __grid_constant__ CollParams p) {
  pdl_enter();
  __shared__ const void* s_send[AR_MAX_RANKS];
  for (int r = threadIdx.x; r < p.P; r += kThreads) s_send[r] = p.send[r];
  __syncthreads();
  const int P = p.P;
  for (uint64_t e = (uint64_t)blockIdx.x * kThreads + threadIdx.x; e < p.total;
       e += (uint64_t)gridDim.x * kThreads) {
    const int s = (int)(e / p.shard);
    typename Lanes<DT>::T acc = load_elem<DT>(s_send[s], e);
    int r = s;
    for (int k = 1; k < P; ++k) {
      r = r + 1 == P ? 0 : r + 1;
      acc = combine<DT, OP>(acc, load_elem<DT>(s_send[r], e));
    }
    store_elem<DT>(p.recv[s], e - (uint64_t)s * p.shard, acc, p.scale, p.do_scale != 0);
  }
}

// Vector v of the P * (shard / V) source vectors: rank s = v / (shard / V).
__global__ void __launch_bounds__(kAgThreads) all_gather_vec_kernel(const __grid_constant__ CollParams p) {
  pdl_enter();
  __shared__ uint4* s_recv[AR_MAX_RANKS];
  for (int r = threadIdx.x; r < p.P; r += kAgThreads) s_recv[r] = static_cast<uint4*>(p.recv[r]);
  __syncthreads();
  const int P = p.P;
  const uint64_t per = p.shard;  // vectors per shard here
  for (uint64_t v = (uint64_t)blockIdx.x * kAgThreads + threadIdx.x; v < p.total;
       v += (uint64_t)gridDim.x * kAgThreads) {
    const int s = (int)(v / per);
    const uint4 x = ld_stream(static_cast<const uint4*>(p.send[s]) + (v - (uint64_t)s * per));
    for (int r = 0; r < P; ++r) st_stream(s_recv[r] + v, x);
  }
}

template <typename W>
__global__ void __launch_bounds__(kThreads) all_gather_elem_kernel(const __grid_constant__ CollParams p) {
  pdl_enter();
  __shared__ W* s_recv[AR_MAX_RANKS];
  for (int r = threadIdx.x; r < p.P; r += kThreads) s_recv[r] = static_cast<W*>(p.recv[r]);
  __syncthreads();
  const int P = p.P;
  for (uint64_t e = (uint64_t)blockIdx.x * kThreads + threadIdx.x; e < p.total;
       e += (uint64_t)gridDim.x * kThreads) {
    const int s = (int)(e / p.shard);
    const W x = static_cast<const W*>(p.send[s])[e - (uint64_t)s * p.shard];
    for (int r = 0; r < P; ++r) s_recv[r][e] = x;
  }
}

unsigned grid_for(uint64_t items, int max_blocks, int threads = kThreads) {
  uint64_t g = (items + threads - 1) / threads;
  if (max_blocks > 0 && g > (uint64_t)max_blocks) g = (uint64_t)max_blocks;
  return (unsigned)(g < 1 ? 1 : (g > 0x7fffffffull ? 0x7fffffffull : g));
}

void fill(CollParams& p, const Call& c) {
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = c.send[r];
    p.recv[r] = c.recv[r];
  }
  p.P = c.P;
  p.shard = c.shard;
  p.scale = c.scale;
  p.do_scale = (c.dtype != kI32 && c.scale != 1.0f) ? 1 : 0;
}

template <int DT>
cudaError_t launch_rs_elem_dt(const Call& c, CollParams& p) {
  const unsigned g = grid_for(p.total, c.max_blocks);
  const bool pdl = use_pdl(c);
  switch (c.op) {
    case kSum: (void)launch_kernel(reduce_scatter_elem_kernel<DT, kSum>, dim3(g), dim3(kThreads), 0, c.stream, pdl, p); break;
    case kMin: (void)launch_kernel(reduce_scatter_elem_kernel<DT, kMin>, dim3(g), dim3(kThreads), 0, c.stream, pdl, p); break;
    case kMax: (void)launch_kernel(reduce_scatter_elem_kernel<DT, kMax>, dim3(g), dim3(kThreads), 0, c.stream, pdl, p); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_reduce_scatter_elem(const Call& c, LaunchInfo* info) {
  CollParams p;
  fill(p, c);
  p.total = (uint64_t)c.P * c.shard;
  info->kernel = "elementwise_reduce_scatter";
  info->grid = (int)grid_for(p.total, c.max_blocks);
  info->block = kThreads;
  switch (c.dtype) {
    case kF32: return launch_rs_elem_dt<kF32>(c, p);
    case kBF16: return launch_rs_elem_dt<kBF16>(c, p);
    case kI32: return launch_rs_elem_dt<kI32>(c, p);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_all_gather(const Call& c, LaunchInfo* info) {
  CollParams p;
  fill(p, c);
  const size_t es = elem_bytes(c.dtype);
  info->block = kThreads;
  if (c.algo == 1) {  // every pointer and the shard size are whole 16-byte units
    p.shard = c.shard * es / 16;  // vectors per shard
    p.total = (uint64_t)c.P * p.shard;
    const unsigned g = grid_for(p.total, c.max_blocks, kAgThreads);
    (void)launch_kernel(all_gather_vec_kernel, dim3(g), dim3(kAgThreads), 0, c.stream, use_pdl(c), p);
    info->kernel = "all_gather_vec";
    info->grid = (int)g;
    info->block = kAgThreads;
  } else {
    p.total = (uint64_t)c.P * c.shard;
    const unsigned g = grid_for(p.total, c.max_blocks);
    if (es == 2) (void)launch_kernel(all_gather_elem_kernel<uint16_t>, dim3(g), dim3(kThreads), 0, c.stream, use_pdl(c), p);
    else (void)launch_kernel(all_gather_elem_kernel<uint32_t>, dim3(g), dim3(kThreads), 0, c.stream, use_pdl(c), p);
    info->kernel = "all_gather_elem";
    info->grid = (int)g;
  }
  return cudaGetLastError();
}

}  // namespace ar
