// ar_tma.cuh -- the rank-specialised all-reduce (P = NP <= 8) as a TMA
// bulk-copy pipeline, for calls limited to a few SMs (AR_OPT_MAX_BLOCKS).
//
// The load/store-unit kernel needs most of the GPU to reach full HBM
// bandwidth: a block keeps about 64 KiB in flight, ~70 GB/s at most.  When the
// all-reduce shares the GPU with computation (the DDP overlap of "NCCL,
// NIXL, and Distributed GPU Communication", its overlap checklist), it gets
// a few dozen SMs, so each SM must keep far more bytes in flight.  One block
// per SM runs a pipeline over shared memory:
//   producer (one thread)  bulk-copies (cp.async.bulk) the NP ranks' tiles
//                          of kTile bytes into stage s, completing on
//                          full[s].  A ring tile inside one chunk c is
//                          loaded rotated -- slot k holds rank (c + k) mod NP
//                          -- so the fold below is chunk c's ring order with
//                          no per-element choice; the chunk is tracked as the
//                          tile offset advances (no division per tile, which
//                          would slow the single issuing thread).  The
//                          stage's order (rotation / tree, or "per element"
//                          for a tile that straddles a boundary) goes
//                          to order[s], published by the barrier arrival;
//   consumer warps         warp w takes whole tiles w, w + CW, ...: waits on
//                          full[s], folds each 16-byte column of the NP
//                          slots in registers, narrows, writes the output
//                          tile, releases the inputs on empty[s], and its
//                          lane 0 bulk-stores the output tile to all NP
//                          receive buffers (one bulk group per tile).  A
//                          stage's previous tile belonged to the same warp
//                          (CW divides the stage count), so that lane's own
//                          bulk-group wait guards the output tile's reuse.
// The reduce-scatter variant (SCATTER, ring only) is the same pipeline: shard
// s is ring chunk s, and the output tile goes to its shard's owner only (a
// tile that straddles a shard boundary is stored segment by segment).
// Every mbarrier wait is bounded: on its limit the thread records
// AR_ERR_TIMEOUT and stops; the producer then waits (bounded) for the loads
// it issued and each storing lane for its bulk stores, so no copy is in
// flight into or out of shared memory when the block exits.  No barrier
// spans warps after the start, so a warp that stops cannot block another.
#pragma once

#include <atomic>

#include "../../include/ar.h"
#include "ar_static.cuh"

namespace ar {

namespace tma {

// Pipeline shape per mode (measured, 8 ranks on 48 / 64 SMs): the all-reduce
// (P tiles in, P out) runs best with 6 KiB tiles in 4 stages and 2 consumer
// warps for fp32 / int32, 4 for bf16, whose fold widens and re-packs 8 lanes
// per column; the reduce-scatter (P in, 1 out) with 8 KiB tiles in 3 stages
// and 3 warps.  2 KiB tiles halve either rate, whatever the stage count.
template <bool SCATTER, int DT>
struct Shape {
  static constexpr int kTile = SCATTER ? 8192 : 6144;  // bytes per rank; multiples of 16
  static constexpr int kStages = SCATTER ? 3 : 4;
  static constexpr int kConsumerWarps = SCATTER ? 3 : DT == kBF16 ? 4 : 2;  // divides kStages
  static constexpr int kThreads = 32 + 32 * kConsumerWarps;
  static_assert(kStages % kConsumerWarps == 0, "a stage's tiles must stay with one warp");
};

template <int NP, bool SCATTER, int DT>
constexpr size_t smem_bytes() {
  return (size_t)Shape<SCATTER, DT>::kStages * (NP + 1) * Shape<SCATTER, DT>::kTile;
}

__device__ __forceinline__ uint32_t saddr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(b)) : "memory");
}
// True once the phase of the given parity has completed; false after `limit` polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, uint32_t limit) {
  for (uint32_t i = 0; i < limit; ++i) {
    uint32_t done;
    asm volatile(
        "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
        : "=r"(done)
        : "r"(saddr(b)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(saddr(dst)), "l"(src), "r"(bytes), "r"(saddr(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(saddr(src)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all but the newest N bulk groups have finished reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

template <int NP>
struct Params {
  const char* send[NP];
  char* recv[NP];
  uint64_t bytes;   // whole 16-byte vectors per rank, in bytes
  uint64_t ntiles;  // ceil(bytes / tile)
  uint64_t split;   // ring: vectors per chunk; tree: first vector of tree 1
  float scale;
  int do_scale;
  int tail;         // elements of the trailing partial vector
  int* status;
  uint32_t spin_limit;  // polls of one mbarrier phase before AR_ERR_TIMEOUT
  int skip_produce;     // test hook: the producer issues no copies, so every wait runs out
};

// order[s]: ring -- the rotation c (slot k = rank (c + k) mod NP); tree --
// which tree (0 / 1); kPerElement -- natural slot order, choose per column
constexpr int kPerElement = -1;

template <int NP, int DT, int OP, int ALGO>
__device__ __forceinline__ uint4 fold_column(const uint4 (&r)[NP], int order, uint64_t v, uint64_t split,
                                             float scale, bool do_scale) {
  if (order == kPerElement) return narrow<DT>(reduce_vec<NP, DT, OP, ALGO>(r, v, split), scale, do_scale);
  if constexpr (ALGO == kRing) {
    return narrow<DT>(ring_from<NP, DT, OP, 0>(r), scale, do_scale);  // slots already rotated
  } else {
    if (order == 0) return narrow<DT>(tree_node<NP, DT, OP, 0, tree_root(NP)>(r), scale, do_scale);
    return narrow<DT>(tree_node<NP, DT, OP, 1, tree_root(NP)>(r), scale, do_scale);
  }
}

template <int NP, int DT, int OP, int ALGO, bool SCATTER = false>
__global__ void __launch_bounds__(Shape<SCATTER, DT>::kThreads, 1) allreduce_kernel(const __grid_constant__ Params<NP> p) {
  pdl_enter();
  constexpr int kTile = Shape<SCATTER, DT>::kTile;
  constexpr int kStages = Shape<SCATTER, DT>::kStages;
  constexpr int kConsumerWarps = Shape<SCATTER, DT>::kConsumerWarps;
  extern __shared__ __align__(128) char smem[];
  char* const in = smem;                                  // [stage][slot][kTile]
  char* const out = smem + (size_t)kStages * NP * kTile;  // [stage][kTile]
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages];
  __shared__ int order[kStages];
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const uint64_t mine = p.ntiles > blockIdx.x ? (p.ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const uint64_t stride = (uint64_t)gridDim.x * kTile;
  const uint64_t bytes = p.bytes;

  if (tid < 32) {
    if (tid == 0) {  // producer
      const uint64_t cbytes = p.split * 16;  // ring: chunk; tree: first byte of tree 1
      uint64_t off = (uint64_t)blockIdx.x * kTile;
      int c = ALGO == kRing && cbytes > 0 ? (int)(off / cbytes) : 0;  // once per block
      uint64_t boundary = ALGO == kRing ? (uint64_t)(c + 1) * cbytes : cbytes;
      uint64_t issued = 0;  // tiles [0, issued) have their loads in flight or landed
      for (uint64_t i = 0; i < mine; ++i, off += stride) {
        const int s = (int)(i % kStages);
        if (i >= (uint64_t)kStages &&
            !mbar_wait(&empty[s], (uint32_t)((i / kStages - 1) & 1), p.spin_limit)) {
          atomicExch(p.status, (int)AR_ERR_TIMEOUT);
          break;
        }
        const uint32_t len = (uint32_t)(bytes - off < (uint64_t)kTile ? bytes - off : (uint64_t)kTile);
        int ord;
        if constexpr (ALGO == kRing) {
          while (off >= boundary) {  // a few steps at most per tile
            ++c;
            boundary += cbytes;
          }
          ord = off + len <= boundary ? c : kPerElement;
        } else {
          ord = off + len <= boundary ? 0 : off >= boundary ? 1 : kPerElement;
        }
        if (p.skip_produce) continue;
        order[s] = ord;  // published to the consumers by the arrival below
        mbar_expect_tx(&full[s], len * NP);
        const int rot = ALGO == kRing && ord != kPerElement ? ord : 0;
#pragma unroll
        for (int k = 0; k < NP; ++k) {
          int src = k + rot;
          if (src >= NP) src -= NP;
          bulk_load(in + ((size_t)s * NP + k) * kTile, p.send[src] + off, len, &full[s]);
        }
        issued = i + 1;
      }
      // the last load issued into each stage must have landed before the block exits
      for (uint64_t k = issued > (uint64_t)kStages ? issued - kStages : 0; k < issued; ++k)
        mbar_wait(&full[k % kStages], (uint32_t)((k / kStages) & 1), p.spin_limit);
    }
    return;
  }

  const int w = (tid >> 5) - 1, lane = tid & 31;
  for (uint64_t i = (uint64_t)w; i < mine; i += kConsumerWarps) {
    const int s = (int)(i % kStages);
    if (!mbar_wait(&full[s], (uint32_t)((i / kStages) & 1), p.spin_limit)) {
      atomicExch(p.status, (int)AR_ERR_TIMEOUT);
      break;
    }
    const uint64_t off = (blockIdx.x + i * gridDim.x) * (uint64_t)kTile;
    const uint32_t len = (uint32_t)(bytes - off < (uint64_t)kTile ? bytes - off : (uint64_t)kTile);
    const int ord = order[s];
    // this warp's bulk stores from out[s], kStages tiles back, have read it
    if (lane == 0) bulk_wait_read<kStages / kConsumerWarps - 1>();
    __syncwarp();
    const char* tin = in + (size_t)s * NP * kTile;
    char* tout = out + (size_t)s * kTile;
    for (uint32_t b = (uint32_t)lane * 16; b < len; b += 32 * 16) {
      uint4 r[NP];
#pragma unroll
      for (int k = 0; k < NP; ++k) r[k] = *reinterpret_cast<const uint4*>(tin + (size_t)k * kTile + b);
      *reinterpret_cast<uint4*>(tout + b) =
          fold_column<NP, DT, OP, ALGO>(r, ord, (off + b) / 16, p.split, p.scale, p.do_scale != 0);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // results visible to the bulk stores
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&empty[s]);  // the input slots are free
      if constexpr (SCATTER) {
        const uint64_t sb = p.split * 16;  // shard bytes
        if (ord != kPerElement) {
          bulk_store(p.recv[ord] + (off - (uint64_t)ord * sb), tout, len);
        } else {  // the tile crosses shard boundaries: one store per shard segment
          for (uint64_t pos = off; pos < off + len;) {
            const uint64_t c = pos / sb;
            const uint64_t end = (c + 1) * sb < off + len ? (c + 1) * sb : off + len;
            bulk_store(p.recv[c] + (pos - c * sb), tout + (pos - off), (uint32_t)(end - pos));
            pos = end;
          }
        }
      } else {
#pragma unroll
        for (int k = 0; k < NP; ++k) bulk_store(p.recv[k] + off, tout, len);
      }
      bulk_commit();
    }
  }
  if (lane == 0) {
    bulk_wait_all();
    // the trailing partial vector, element by element in the same order
    if (!SCATTER && p.tail != 0 && blockIdx.x == 0 && w == 0) {
      const uint64_t n = p.bytes / 16;
      uint4 r[NP];
#pragma unroll
      for (int k = 0; k < NP; ++k) r[k] = load_partial<DT>(reinterpret_cast<const uint4*>(p.send[k]) + n, p.tail);
      const uint4 o = narrow<DT>(reduce_vec<NP, DT, OP, ALGO>(r, n, p.split), p.scale, p.do_scale != 0);
#pragma unroll
      for (int k = 0; k < NP; ++k) store_partial<DT>(reinterpret_cast<uint4*>(p.recv[k]) + n, o, p.tail);
    }
  }
}

template <int DT, int NP, int OP, int ALGO, bool SCATTER = false>
cudaError_t launch_one(const Call& c, LaunchInfo* info) {
  auto kernel = allreduce_kernel<NP, DT, OP, ALGO, SCATTER>;
  constexpr int kTile = Shape<SCATTER, DT>::kTile;
  constexpr size_t kSmem = smem_bytes<NP, SCATTER, DT>();
  Params<NP> p;
  for (int k = 0; k < NP; ++k) {
    p.send[k] = static_cast<const char*>(c.send[k]);
    p.recv[k] = static_cast<char*>(c.recv[k]);
  }
  const uint64_t V = (uint64_t)vec_elems(DT);
  p.bytes = (c.count / V) * 16;
  p.ntiles = (p.bytes + kTile - 1) / kTile;
  p.tail = (int)(c.count % V);
  p.split = ALGO == kRing ? ring_chunk_vectors(c.count, NP, DT) : tree_split_vectors(c.count, DT);
  if constexpr (SCATTER) {  // shards of whole vectors: shard s is chunk s
    if (c.shard % V != 0 || c.count != (size_t)NP * c.shard) return cudaErrorInvalidValue;
    p.split = c.shard / V;
    p.tail = 0;
  }
  p.scale = c.scale;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  p.status = c.status;
  p.spin_limit = c.spin_limit;
  p.skip_produce = c.skip_produce;
  // the shared-memory opt-in is a per-device attribute: set it once on each device
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  uint64_t grid = (uint64_t)(c.max_blocks > 0 ? c.max_blocks : c.sms);
  if (grid > (uint64_t)c.sms) grid = (uint64_t)c.sms;  // one block per SM
  if (grid > p.ntiles) grid = p.ntiles;
  if (grid < 1) grid = 1;
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(Shape<SCATTER, DT>::kThreads), kSmem, c.stream, use_pdl(c), p);
  info->kernel = SCATTER ? "tma_reduce_scatter" : ALGO == kRing ? "tma_ring" : "tma_tree";
  info->grid = (int)grid;
  info->block = Shape<SCATTER, DT>::kThreads;
  info->smem = kSmem;
  return cudaGetLastError();
}

template <int DT, int NP>
cudaError_t launch_np(const Call& c, LaunchInfo* info) {
  if (c.shard != 0) {  // reduce-scatter
    switch (c.op) {
      case kSum: return launch_one<DT, NP, kSum, kRing, true>(c, info);
      case kMin: return launch_one<DT, NP, kMin, kRing, true>(c, info);
      case kMax: return launch_one<DT, NP, kMax, kRing, true>(c, info);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (c.op * 4 + c.algo) {
    case kSum * 4 + kRing: return launch_one<DT, NP, kSum, kRing>(c, info);
    case kSum * 4 + kTree: return launch_one<DT, NP, kSum, kTree>(c, info);
    case kMin * 4 + kRing: return launch_one<DT, NP, kMin, kRing>(c, info);
    case kMin * 4 + kTree: return launch_one<DT, NP, kMin, kTree>(c, info);
    case kMax * 4 + kRing: return launch_one<DT, NP, kMax, kRing>(c, info);
    case kMax * 4 + kTree: return launch_one<DT, NP, kMax, kTree>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT>
cudaError_t launch_dt(const Call& c, LaunchInfo* info) {
  switch (c.P) {
    case 1: return launch_np<DT, 1>(c, info);
    case 2: return launch_np<DT, 2>(c, info);
    case 3: return launch_np<DT, 3>(c, info);
    case 4: return launch_np<DT, 4>(c, info);
    case 5: return launch_np<DT, 5>(c, info);
    case 6: return launch_np<DT, 6>(c, info);
    case 7: return launch_np<DT, 7>(c, info);
    case 8: return launch_np<DT, 8>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tma

}  // namespace ar
