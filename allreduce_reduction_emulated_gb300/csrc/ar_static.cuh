// ar_static.cuh -- ring-order and tree-order all-reduce kernels specialised
// on the exact rank count NP (1..8).
//
// One fused pass: each thread loads one 16-byte vector from each of the NP
// send buffers, folds the NP vectors in registers in the algorithm's order
// (the ring's rotation or the tree's nested expression, both resolved at
// compile time), applies the scale / narrowing epilogue once and stores the
// result vector to all NP receive buffers.  The ring and tree "steps" are a
// combination order here, not data movement: every input byte is read once
// and every output byte written once, the minimum 2 * NP * count * size
// bytes of HBM traffic.  The reduce-scatter variant (SCATTER) folds the same
// ring order (shard c = chunk c, from rank c) and stores each result vector
// only to its shard's owner: NP * count reads, count writes.
#pragma once

#include "ar_device.cuh"
#include "ar_launch.h"

namespace ar {

#ifndef AR_STATIC_THREADS
#define AR_STATIC_THREADS 256
#endif
#ifndef AR_STATIC_UNROLL
#define AR_STATIC_UNROLL 2
#endif
#ifndef AR_STATIC_PERSISTENT
#define AR_STATIC_PERSISTENT 0
#endif

constexpr int kStaticThreads = AR_STATIC_THREADS;
constexpr int kStaticUnroll = AR_STATIC_UNROLL;  // vectors per rank in flight per thread
// The all-reduce's shape: the same 512-vector tile per block, one vector per
// rank per thread in 512-thread blocks.  Back to back on 8 x 64 MiB fp32 it
// measured 154.5 us per call against 155.3 for 256 threads x 2 vectors; the
// reduce-scatter (8 loads per store) keeps 256 x 2, 0.3% faster there.
#ifndef AR_ALLREDUCE_THREADS
#define AR_ALLREDUCE_THREADS 512
#endif
#ifndef AR_ALLREDUCE_UNROLL
#define AR_ALLREDUCE_UNROLL 1
#endif
constexpr int kAllreduceThreads = AR_ALLREDUCE_THREADS;
constexpr int kAllreduceUnroll = AR_ALLREDUCE_UNROLL;
// 1: grid = resident blocks, grid-stride loop; 0: one tile of vectors per block
// (default: measured ~11% faster on 8 x 64 MiB, the persistent loop loses its
// last wave to imbalance)
constexpr bool kStaticPersistent = AR_STATIC_PERSISTENT != 0;

template <int NP>
struct StaticParams {
  const uint4* send[NP];
  uint4* recv[NP];
  uint64_t nfull;  // whole 16-byte vectors per rank
  uint64_t split;  // ring: vectors per chunk; tree: first vector folded along tree 1
  float scale;
  int do_scale;
  int tail;        // elements in the trailing partial vector (0 = none)
};

// Ring order for a vector of chunk C: x_C, then x_{C+1}, ..., x_{C+NP-1}.
template <int NP, int DT, int OP, int C>
__device__ __forceinline__ Acc<DT> ring_from(const uint4 (&r)[NP]) {
  Acc<DT> acc = widen<DT>(r[C]);
#pragma unroll
  for (int k = 1; k < NP; ++k) fold<DT, OP>(acc, widen<DT>(r[(C + k) % NP]));
  return acc;
}

// Selects the chunk's fold at run time; every branch has static register
// indices, so the rotation costs no dynamic indexing.
template <int NP, int DT, int OP, int C = 0>
__device__ __forceinline__ Acc<DT> ring_fold(const uint4 (&r)[NP], int c) {
  if constexpr (C == NP - 1) {
    return ring_from<NP, DT, OP, C>(r);
  } else {
    if (c == C) return ring_from<NP, DT, OP, C>(r);
    return ring_fold<NP, DT, OP, C + 1>(r, c);
  }
}

// Tree T's value at label V: ((own (+) left) (+) right).
template <int NP, int DT, int OP, int T, int V>
__device__ __forceinline__ Acc<DT> tree_node(const uint4 (&r)[NP]) {
  Acc<DT> acc = widen<DT>(r[tree_owner(V, NP, T)]);
  constexpr int kLeft = tree_left(V);
  constexpr int kRight = tree_right(V, NP);
  if constexpr (kLeft != 0) fold<DT, OP>(acc, tree_node<NP, DT, OP, T, kLeft>(r));
  if constexpr (kRight != 0) fold<DT, OP>(acc, tree_node<NP, DT, OP, T, kRight>(r));
  return acc;
}

// Ring chunk of vector v (chunks of split vectors), 32-bit division when it fits.
__device__ __forceinline__ int chunk_of(uint64_t v, uint64_t split) {
  return (v < 0xffffffffull && split < 0xffffffffull) ? (int)((uint32_t)v / (uint32_t)split)
                                                      : (int)(v / split);
}

template <int NP, int DT, int OP, int ALGO>
__device__ __forceinline__ Acc<DT> reduce_vec(const uint4 (&r)[NP], uint64_t v, uint64_t split) {
  if constexpr (ALGO == kRing) {
    return ring_fold<NP, DT, OP>(r, chunk_of(v, split));
  } else {
    if (v < split) return tree_node<NP, DT, OP, 0, tree_root(NP)>(r);
    return tree_node<NP, DT, OP, 1, tree_root(NP)>(r);
  }
}

// The wide shape for calls capped to a few SMs (AR_OPT_MAX_BLOCKS): blocks of
// 1024 threads, one vector per rank per thread in flight, one block per SM and
// a grid-stride loop.  A 256-thread block keeps 256 * 2 * NP vectors in
// flight and moves about 45 GB/s per SM; 1024 threads keep twice that and
// measured ~100 GB/s per SM for the 8-rank reduce-scatter on 64 SMs.
constexpr int kWideThreads = 1024;
constexpr int kWideUnroll = 1;

// SCATTER (ring only): recv[c] is shard c's owner buffer, written at the
// shard-relative position; there is no partial trailing vector.
template <int NP, int DT, int OP, int ALGO, bool SCATTER = false, int THREADS = kStaticThreads,
          int U = kStaticUnroll>
__global__ void __launch_bounds__(THREADS)
    static_allreduce_kernel(const __grid_constant__ StaticParams<NP> p) {
  pdl_enter();
  const uint64_t n = p.nfull;
  const uint64_t step = (uint64_t)gridDim.x * (THREADS * U);
  for (uint64_t base = (uint64_t)blockIdx.x * (THREADS * U) + threadIdx.x; base < n;
       base += step) {
    uint4 r[U][NP];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + (uint64_t)u * THREADS;
      if (v < n) {
#pragma unroll
        for (int k = 0; k < NP; ++k) r[u][k] = ld_stream(p.send[k] + v);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint64_t v = base + (uint64_t)u * THREADS;
      if (v < n) {
        if constexpr (SCATTER) {
          const int c = chunk_of(v, p.split);
          const uint4 o = narrow<DT>(ring_fold<NP, DT, OP>(r[u], c), p.scale, p.do_scale != 0);
          st_stream(p.recv[c] + (v - (uint64_t)c * p.split), o);
        } else {
          const uint4 o =
              narrow<DT>(reduce_vec<NP, DT, OP, ALGO>(r[u], v, p.split), p.scale, p.do_scale != 0);
#pragma unroll
          for (int k = 0; k < NP; ++k) st_stream(p.recv[k] + v, o);
        }
      }
    }
  }
  if (!SCATTER && p.tail != 0 && blockIdx.x == 0 && threadIdx.x == 0) {
    uint4 r[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) r[k] = load_partial<DT>(p.send[k] + n, p.tail);
    const uint4 o =
        narrow<DT>(reduce_vec<NP, DT, OP, ALGO>(r, n, p.split), p.scale, p.do_scale != 0);
#pragma unroll
    for (int k = 0; k < NP; ++k) store_partial<DT>(p.recv[k] + n, o, p.tail);
  }
}

// WIDE: the 1024-thread shape, grid capped at c.max_blocks and the SM count.
template <int DT, int NP, int OP, int ALGO, bool SCATTER = false, bool WIDE = false>
cudaError_t launch_static_one(const Call& c, LaunchInfo* info) {
  constexpr int U = WIDE ? kWideUnroll : SCATTER ? kStaticUnroll : kAllreduceUnroll;
  constexpr int kThreads = WIDE ? kWideThreads : SCATTER ? kStaticThreads : kAllreduceThreads;
  auto kernel = static_allreduce_kernel<NP, DT, OP, ALGO, SCATTER, kThreads, U>;
  StaticParams<NP> p;
  for (int k = 0; k < NP; ++k) {
    p.send[k] = static_cast<const uint4*>(c.send[k]);
    p.recv[k] = static_cast<uint4*>(c.recv[k]);
  }
  const uint64_t V = (uint64_t)vec_elems(DT);
  p.nfull = c.count / V;
  p.tail = (int)(c.count % V);
  p.split = ALGO == kRing ? ring_chunk_vectors(c.count, NP, DT) : tree_split_vectors(c.count, DT);
  if constexpr (SCATTER) {
    if (c.shard % V != 0 || c.count != (size_t)NP * c.shard) return cudaErrorInvalidValue;
    p.split = c.shard / V;  // whole vectors per shard
    p.tail = 0;
  }
  p.scale = c.scale;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  static const int blocks_per_sm = [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kThreads, 0) != cudaSuccess)
      b = 1;
    return b > 0 ? b : 1;
  }();
  const uint64_t need = (p.nfull + kThreads * U - 1) / (kThreads * U);
  uint64_t cap = kStaticPersistent || WIDE ? (uint64_t)c.sms * (uint64_t)blocks_per_sm : 0x7fffffffull;
  if (c.max_blocks > 0 && (uint64_t)c.max_blocks < cap) cap = (uint64_t)c.max_blocks;
  const int grid = (int)(need < 1 ? 1 : (need < cap ? need : cap));
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(kThreads), 0, c.stream, use_pdl(c), p);
  info->kernel = WIDE ? (SCATTER ? "wide_reduce_scatter" : ALGO == kRing ? "wide_ring" : "wide_tree")
                      : (SCATTER ? "static_reduce_scatter" : ALGO == kRing ? "static_ring" : "static_tree");
  info->grid = grid;
  info->block = kThreads;
  info->smem = 0;
  return cudaGetLastError();
}

template <int DT, int NP, bool WIDE>
cudaError_t launch_static_np(const Call& c, LaunchInfo* info) {
  if (c.shard != 0) {  // reduce-scatter
    switch (c.op) {
      case kSum: return launch_static_one<DT, NP, kSum, kRing, true, WIDE>(c, info);
      case kMin: return launch_static_one<DT, NP, kMin, kRing, true, WIDE>(c, info);
      case kMax: return launch_static_one<DT, NP, kMax, kRing, true, WIDE>(c, info);
      default: return cudaErrorInvalidValue;
    }
  }
  const int key = c.op * 4 + c.algo;
  switch (key) {
    case kSum * 4 + kRing: return launch_static_one<DT, NP, kSum, kRing, false, WIDE>(c, info);
    case kSum * 4 + kTree: return launch_static_one<DT, NP, kSum, kTree, false, WIDE>(c, info);
    case kMin * 4 + kRing: return launch_static_one<DT, NP, kMin, kRing, false, WIDE>(c, info);
    case kMin * 4 + kTree: return launch_static_one<DT, NP, kMin, kTree, false, WIDE>(c, info);
    case kMax * 4 + kRing: return launch_static_one<DT, NP, kMax, kRing, false, WIDE>(c, info);
    case kMax * 4 + kTree: return launch_static_one<DT, NP, kMax, kTree, false, WIDE>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT, bool WIDE = false>
cudaError_t launch_static_dt(const Call& c, LaunchInfo* info) {
  switch (c.P) {
    case 1: return launch_static_np<DT, 1, WIDE>(c, info);
    case 2: return launch_static_np<DT, 2, WIDE>(c, info);
    case 3: return launch_static_np<DT, 3, WIDE>(c, info);
    case 4: return launch_static_np<DT, 4, WIDE>(c, info);
    case 5: return launch_static_np<DT, 5, WIDE>(c, info);
    case 6: return launch_static_np<DT, 6, WIDE>(c, info);
    case 7: return launch_static_np<DT, 7, WIDE>(c, info);
    case 8: return launch_static_np<DT, 8, WIDE>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ar
