// ar_generic.cuh -- ring-order and tree-order all-reduce for any rank count up
// to AR_MAX_RANKS (used above the rank-specialised kernels' limit), templated
// on the block width: 64 threads (ar_generic.cu) for calls with the whole
// GPU, 768 threads, one block per SM (ar_generic_wide.cu), for calls capped to
// a few SMs (AR_OPT_MAX_BLOCKS), where small blocks left each SM with too few
// copies in flight (2.5 TB/s for 72 ranks on 48 SMs in 128-thread blocks).
//
// With many ranks the P input vectors of a column no longer fit in registers,
// and the fold order needs a dynamic rank index.  Each thread owns one column
// (one 16-byte vector of every rank) and streams it through a small ring of
// shared-memory slots in exactly the order the fold consumes it: the ring's
// rotated rank sequence, or the tree's preorder leaf sequence.  W
// asynchronous copies are kept in flight (cp.async, one commit group per
// copy); before each value is used the thread waits until its copy has landed
// (wait_group W-1: all but the W-1 newest groups done), reads it, and refills
// the slot freed one step earlier with the copy W pushes ahead.  The tree
// folds its complete lowbit-4 subtrees in registers and keeps only the nodes
// above them on a small stack.  Shared memory per thread is (W+1) x 16
// bytes whatever P is, so occupancy stays high at P = 72 or 256.  Threads
// never touch each other's slots, so there is no barrier in the main loop.
#pragma once

#include <atomic>

#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

#ifndef AR_GENERIC_WINDOW
#define AR_GENERIC_WINDOW 24
#endif
#ifndef AR_GENERIC_THREADS
#define AR_GENERIC_THREADS 64
#endif

// With the whole GPU: 64-thread blocks, 24 copies in flight per thread (25
// slots, 25.6 KiB per block, 8 blocks per SM).  The same copies in flight per
// SM as 128 threads x 16 but shorter chains per column, so the last wave
// drains sooner: 72 x 4 / 16 MiB int32 ring 92.7 / 350.0 us against
// 94.1 / 353.6 (back to back).  Under a cap: 768 threads, 16 in flight
// (17 x 768 x 16 B = 204 KiB of slots, one block per SM).
constexpr int kWindow = AR_GENERIC_WINDOW;    // copies in flight per thread, whole GPU
constexpr int kThreads = AR_GENERIC_THREADS;  // block width with the whole GPU
constexpr int kWideThreads = 768;             // block width under a cap
constexpr int kWideWindow = 16;               // copies in flight per thread under a cap
template <int THREADS>
__host__ __device__ constexpr int window_of() { return THREADS == kWideThreads ? kWideWindow : kWindow; }
template <int THREADS>
__host__ __device__ constexpr int slots_of() { return window_of<THREADS>() + 1; }  // one spare slot between read and refill
constexpr int kStackDepth = 16;               // >= tree height + 1 for P <= AR_MAX_RANKS

struct GenericParams {
  const uint4* send[AR_MAX_RANKS];
  uint4* recv[AR_MAX_RANKS];
  const int16_t* push;  // device: tree 0's then tree 1's ranks in preorder (P each)
  int P;
  int Q;                // hierarchical: ranks per group (P = G * Q)
  uint64_t count;       // elements per rank (hierarchical sub-chunk lengths)
  uint64_t nfull;
  uint64_t split;  // ring: vectors per chunk; tree: first vector of tree 1
  float scale;
  int do_scale;
  int tail;
};

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The tree's nodes carry labels 1..P; a node of lowbit b has the left
// subtree v-b+1..v-1 and the right subtree v+1..min(v+b-1, P), and its value
// is ((own (+) left) (+) right), its inputs pushed own first (preorder).  A
// subtree that the rank count does not truncate ("complete", 2b - 1 nodes)
// has a shape that depends on b alone.

// Complete subtree of lowbit B <= 4, expanded at compile time (registers only).
template <int B, int DT, int OP, class Next>
__device__ __forceinline__ Acc<DT> small_subtree(Next& next) {
  Acc<DT> acc = next();
  if constexpr (B > 1) {
    fold<DT, OP>(acc, small_subtree<B / 2, DT, OP>(next));
    fold<DT, OP>(acc, small_subtree<B / 2, DT, OP>(next));
  }
  return acc;
}

// Complete subtree of lowbit b (a power of two): b <= 4 directly; above, as
// b/4 blocks of lowbit 4 in order, with the lg = log2(b) - 2 ancestors of
// the current block on a small stack.  Before block i the ancestors whose
// subtree starts there are pushed (lg of them for i = 0, ctz(i) after);
// after it the block's value folds upward: into its parent's partial if it
// is a left child (bit 0 of i clear), else completing the parent, which then
// folds into the grandparent by bit 1, and so on.  Stack traffic is one
// entry per 8 inputs.
template <int DT, int OP, class Next>
__device__ __forceinline__ Acc<DT> complete_subtree(int b, Next& next) {
  if (b == 1) return small_subtree<1, DT, OP>(next);
  if (b == 2) return small_subtree<2, DT, OP>(next);
  if (b == 4) return small_subtree<4, DT, OP>(next);
  Acc<DT> up[kStackDepth];
  const int lg = __ffs(b) - 3;
  int sp = 0;
  Acc<DT> top;
  for (int i = 0; i < b / 4; ++i) {
    for (int k = i == 0 ? lg : __ffs(i) - 1; k > 0; --k) up[sp++] = next();
    top = small_subtree<4, DT, OP>(next);
    for (int bits = i;; bits >>= 1) {
      Acc<DT> parent = up[sp - 1];
      fold<DT, OP>(parent, top);
      if ((bits & 1) == 0) {  // a left child: the parent waits for its right
        up[sp - 1] = parent;
        break;
      }
      top = parent;
      if (--sp == 0) break;   // the subtree's root is complete
    }
  }
  return top;
}

// Folds the column in the algorithm's order; next() yields the widened
// input of the next rank in the push sequence.  The hierarchical order folds
// each group's Q values, then the G partials.  The tree is walked along its
// right spine from the root (the largest power of two <= P), the only part
// the rank count truncates: at a spine node v of lowbit b either the whole
// subtree fits (v + b - 1 <= P) and is one complete subtree, or the node's
// partial (own (+) its complete left subtree) is kept and the walk moves to
// the right child v + h (h the largest power of two <= P - v, below b); the
// partials then fold bottom-up.
template <int DT, int OP, int ALGO, class Next>
__device__ __forceinline__ Acc<DT> fold_sequence(int P, int Q, Next& next) {
  if constexpr (ALGO == kRing) {
    Acc<DT> acc = next();
    for (int k = 1; k < P; ++k) fold<DT, OP>(acc, next());
    return acc;
  } else if constexpr (ALGO == kHier) {
    Acc<DT> total;
    for (int j = 0; j < P; j += Q) {
      Acc<DT> part = next();
      for (int i = 1; i < Q; ++i) fold<DT, OP>(part, next());
      if (j == 0) total = part;
      else fold<DT, OP>(total, part);
    }
    return total;
  } else {
    Acc<DT> spine[kStackDepth];  // partials of the spine nodes above
    int depth = 0;
    int v = 1;
    while (v * 2 <= P) v *= 2;
    int b = v;
    Acc<DT> val;
    for (;;) {
      if (v + b - 1 <= P) {
        val = complete_subtree<DT, OP>(b, next);
        break;
      }
      Acc<DT> own = next();
      fold<DT, OP>(own, complete_subtree<DT, OP>(b / 2, next));
      int h = b / 2;
      while (h >= 1 && v + h > P) h /= 2;
      if (h < 1) {  // no right child
        val = own;
        break;
      }
      spine[depth++] = own;
      v += h;
      b = h;
    }
    while (depth > 0) {
      Acc<DT> parent = spine[--depth];
      fold<DT, OP>(parent, val);
      val = parent;
    }
    return val;
  }
}

// The ranks of a column in push order, one at a time.
template <int ALGO>
struct RankCursor {
  int a, b;               // ring: rank; tree: index; hier: local index, group index
  int P, Q, G, a0, b0;    // hier: start local index a0 (chunk c1 mod Q), group b0 (c2)
  const int16_t* push;    // tree leaf order
  __device__ __forceinline__ int next() {
    if constexpr (ALGO == kRing) {
      const int r = a;
      a = a + 1 == P ? 0 : a + 1;
      return r;
    } else if constexpr (ALGO == kTree) {
      return push[a++];
    } else {
      const int r = b * Q + a;
      a = a + 1 == Q ? 0 : a + 1;
      if (a == a0) b = b + 1 == G ? 0 : b + 1;   // a group's Q ranks are done
      return r;
    }
  }
};

// The cursor of column v, and (ring) its chunk index = the chunk's start rank.
template <int DT, int ALGO>
__device__ __forceinline__ RankCursor<ALGO> column_cursor(const GenericParams& p, uint64_t v,
                                                          const int16_t (*s_push)[AR_MAX_RANKS], int& first) {
  RankCursor<ALGO> cur;
  cur.P = p.P;
  first = ALGO == kRing ? (int)(v / p.split) : 0;
  if constexpr (ALGO == kRing) {
    cur.a = first;
  } else if constexpr (ALGO == kTree) {
    cur.push = s_push[v >= p.split ? 1 : 0];
    cur.a = 0;
  } else {
    // hierarchical: intra-group chunk c1 (split = its length in vectors), then
    // sub-chunk c2 of that chunk across the G groups
    const uint64_t V = 16 / Lanes<DT>::kBytes;
    const uint64_t c1 = v / p.split;
    const uint64_t lo = c1 * p.split * V;
    const uint64_t hi = lo + p.split * V < p.count ? lo + p.split * V : p.count;
    const int G = p.P / p.Q;
    const uint64_t L2v = ((hi - lo + G - 1) / G + V - 1) / V;
    const uint64_t c2 = (v - c1 * p.split) / L2v;
    cur.Q = p.Q;
    cur.G = G;
    cur.a0 = cur.a = (int)(c1 % (uint64_t)p.Q);
    cur.b0 = cur.b = (int)c2;
  }
  return cur;
}

// SCATTER (ring only): reduce-scatter -- chunk c is shard c and its result
// goes only to rank c's receive buffer, at the shard-relative position.
// Under a cap a thread walks several columns (grid-stride); the first W
// copies of its next column are issued before the current column's P stores,
// so the SM's loads do not stall behind a burst of stores.  All slots are free
// by then: every copy has landed and every slot value has been folded.
template <int DT, int OP, int ALGO, bool SCATTER, int THREADS>
__global__ void __launch_bounds__(THREADS) generic_allreduce_kernel(const __grid_constant__ GenericParams p) {
  constexpr int kWin = window_of<THREADS>();
  constexpr int kSlots = slots_of<THREADS>();
  extern __shared__ uint4 slots[];                // [kSlots][THREADS]
  __shared__ const uint4* s_send[AR_MAX_RANKS];
  __shared__ uint4* s_recv[AR_MAX_RANKS];
  __shared__ int16_t s_push[2][AR_MAX_RANKS];   // tree leaf (push) sequences
  pdl_enter();
  const int P = p.P;
  const int tid = threadIdx.x;
  for (int r = tid; r < P; r += THREADS) {
    s_send[r] = p.send[r];
    s_recv[r] = p.recv[r];
    if constexpr (ALGO == kTree) {
      s_push[0][r] = p.push[r];
      s_push[1][r] = p.push[P + r];
    }
  }
  __syncthreads();

  const uint64_t n = p.nfull;
  const uint64_t columns = n + (p.tail ? 1 : 0);
  const uint64_t stride = (uint64_t)gridDim.x * THREADS;
  const uint32_t base = (uint32_t)__cvta_generic_to_shared(&slots[tid]);
  constexpr uint32_t kSlotStride = THREADS * 16;
  // the first kWin copies of column v, into slots 0 .. kWin-1
  auto prologue = [&](uint64_t v, RankCursor<ALGO>& cur) {
  #pragma unroll
    for (int k = 0; k < kWin; ++k) {
      if (k < P) cp_async16(base + k * kSlotStride, s_send[cur.next()] + v);
      cp_async_commit();
    }
  };

  uint64_t v = (uint64_t)blockIdx.x * THREADS + tid;
  int first = 0;
  RankCursor<ALGO> cur{};
  if (v < columns) {
    cur = column_cursor<DT, ALGO>(p, v, s_push, first);
    if (v < n) prologue(v, cur);
  }
  for (; v < columns; v += stride) {
    const uint64_t vn = v + stride;
    int first_n = 0;
    RankCursor<ALGO> cur_n = cur;
    if (v < n) {
      int j = 0;          // values consumed
      int rd = 0;         // slot of value j
      int wr = kWin;      // slot for value j + kWin
      auto next = [&]() -> Acc<DT> {
        cp_async_wait<kWin - 1>();  // value j has landed
        const uint4 raw = slots[rd * THREADS + tid];
        const int k = j + kWin;
        if (k < P) cp_async16(base + wr * kSlotStride, s_send[cur.next()] + v);
        cp_async_commit();
        ++j;
        rd = rd + 1 == kSlots ? 0 : rd + 1;
        wr = wr + 1 == kSlots ? 0 : wr + 1;
        return widen<DT>(raw);
      };
      const Acc<DT> acc = fold_sequence<DT, OP, ALGO>(P, p.Q, next);
      cp_async_wait<0>();
      const uint4 o = narrow<DT>(acc, p.scale, p.do_scale != 0);
      if (vn < columns) {
        cur_n = column_cursor<DT, ALGO>(p, vn, s_push, first_n);
        if (vn < n) prologue(vn, cur_n);
      }
      if constexpr (SCATTER) {
        st_stream(s_recv[first] + (v - (uint64_t)first * p.split), o);
      } else {
        for (int r = 0; r < P; ++r) st_stream(s_recv[r] + v, o);
      }
    } else {
      // the trailing partial vector (the last column): element-wise loads, same order
      auto next = [&]() -> Acc<DT> { return widen<DT>(load_partial<DT>(s_send[cur.next()] + n, p.tail)); };
      const Acc<DT> acc = fold_sequence<DT, OP, ALGO>(P, p.Q, next);
      const uint4 o = narrow<DT>(acc, p.scale, p.do_scale != 0);
      for (int r = 0; r < P; ++r) store_partial<DT>(s_recv[r] + n, o, p.tail);
    }
    cur = cur_n;
    first = first_n;
  }
}

// Dynamic shared memory of THREADS slots rings; above 48 KiB the kernel must
// opt in, once per device.
template <class K>
cudaError_t opt_in_smem(K kernel, size_t smem, std::atomic<uint64_t>& configured) {
  if (smem <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (configured.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess) configured.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Grid: one block per THREADS columns; under a cap at most max_blocks blocks
// (grid-stride), and for the wide width also at most one per SM.
template <int THREADS>
uint64_t generic_grid(uint64_t columns, const Call& c) {
  uint64_t grid = (columns + THREADS - 1) / THREADS;
  if (c.max_blocks > 0 && grid > (uint64_t)c.max_blocks) grid = (uint64_t)c.max_blocks;
  if (THREADS != kThreads && grid > (uint64_t)c.sms) grid = (uint64_t)c.sms;
  return grid < 1 ? 1 : grid;
}

template <int DT, int OP, int ALGO, int THREADS>
cudaError_t launch_generic_one(const Call& c, LaunchInfo* info) {
  auto kernel = generic_allreduce_kernel<DT, OP, ALGO, false, THREADS>;
  GenericParams p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = static_cast<const uint4*>(c.send[r]);
    p.recv[r] = static_cast<uint4*>(c.recv[r]);
  }
  p.push = c.tree_push;
  p.P = c.P;
  p.Q = c.group;
  p.count = c.count;
  const uint64_t V = (uint64_t)vec_elems(DT);
  p.nfull = c.count / V;
  p.tail = (int)(c.count % V);
  if (ALGO == kHier && (c.group < 1 || c.P % c.group != 0)) return cudaErrorInvalidValue;
  p.split = ALGO == kRing   ? ring_chunk_vectors(c.count, c.P, DT)
            : ALGO == kHier ? ring_chunk_vectors(c.count, c.group, DT)  // intra-group chunk
                            : tree_split_vectors(c.count, DT);
  p.scale = c.scale;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  if (ALGO == kTree && c.tree_push == nullptr) return cudaErrorInvalidValue;
  const uint64_t columns = p.nfull + (p.tail ? 1 : 0);
  const uint64_t grid = generic_grid<THREADS>(columns, c);
  if (grid > 0x7fffffffull) return cudaErrorInvalidValue;
  constexpr size_t kSmem = sizeof(uint4) * slots_of<THREADS>() * THREADS;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = opt_in_smem(kernel, kSmem, configured);
  if (e != cudaSuccess) return e;
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(THREADS), kSmem, c.stream, use_pdl(c), p);
  const bool wide = THREADS != kThreads;
  info->kernel = ALGO == kRing ? (wide ? "wide_pipelined_ring" : "pipelined_ring")
                 : ALGO == kHier ? (wide ? "wide_pipelined_hier" : "pipelined_hier")
                                 : (wide ? "wide_pipelined_tree" : "pipelined_tree");
  info->grid = (int)grid;
  info->block = THREADS;
  info->smem = kSmem;
  return cudaGetLastError();
}

template <int DT, int OP, int THREADS>
cudaError_t launch_generic_algo(const Call& c, LaunchInfo* info) {
  if (c.algo == kRing) return launch_generic_one<DT, OP, kRing, THREADS>(c, info);
  if (c.algo == kTree) return launch_generic_one<DT, OP, kTree, THREADS>(c, info);
  if (c.algo == kHier) return launch_generic_one<DT, OP, kHier, THREADS>(c, info);
  return cudaErrorInvalidValue;
}

template <int DT, int THREADS>
cudaError_t launch_generic_op(const Call& c, LaunchInfo* info) {
  switch (c.op) {
    case kSum: return launch_generic_algo<DT, kSum, THREADS>(c, info);
    case kMin: return launch_generic_algo<DT, kMin, THREADS>(c, info);
    case kMax: return launch_generic_algo<DT, kMax, THREADS>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT, int OP, int THREADS>
cudaError_t launch_scatter_one(const Call& c, LaunchInfo* info) {
  auto kernel = generic_allreduce_kernel<DT, OP, kRing, true, THREADS>;
  GenericParams p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = static_cast<const uint4*>(c.send[r]);
    p.recv[r] = static_cast<uint4*>(c.recv[r]);
  }
  p.push = nullptr;
  p.P = c.P;
  p.Q = c.P;
  p.count = c.count;
  const uint64_t V = (uint64_t)vec_elems(DT);
  if (c.shard % V != 0) return cudaErrorInvalidValue;  // whole vectors per shard only
  p.nfull = c.count / V;
  p.tail = 0;
  p.split = c.shard / V;
  p.scale = c.scale;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  const uint64_t grid = generic_grid<THREADS>(p.nfull, c);
  if (grid > 0x7fffffffull) return cudaErrorInvalidValue;
  constexpr size_t kSmem = sizeof(uint4) * slots_of<THREADS>() * THREADS;
  static std::atomic<uint64_t> configured{0};
  cudaError_t e = opt_in_smem(kernel, kSmem, configured);
  if (e != cudaSuccess) return e;
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(THREADS), kSmem, c.stream, use_pdl(c), p);
  info->kernel = THREADS != kThreads ? "wide_pipelined_reduce_scatter" : "pipelined_reduce_scatter";
  info->grid = (int)grid;
  info->block = THREADS;
  info->smem = kSmem;
  return cudaGetLastError();
}

template <int DT, int THREADS>
cudaError_t launch_scatter_op(const Call& c, LaunchInfo* info) {
  switch (c.op) {
    case kSum: return launch_scatter_one<DT, kSum, THREADS>(c, info);
    case kMin: return launch_scatter_one<DT, kMin, THREADS>(c, info);
    case kMax: return launch_scatter_one<DT, kMax, THREADS>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int THREADS>
cudaError_t generic_dispatch(const Call& c, LaunchInfo* info) {
  switch (c.dtype) {
    case kF32: return launch_generic_op<kF32, THREADS>(c, info);
    case kBF16: return launch_generic_op<kBF16, THREADS>(c, info);
    case kI32: return launch_generic_op<kI32, THREADS>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int THREADS>
cudaError_t scatter_dispatch(const Call& c, LaunchInfo* info) {
  switch (c.dtype) {
    case kF32: return launch_scatter_op<kF32, THREADS>(c, info);
    case kBF16: return launch_scatter_op<kBF16, THREADS>(c, info);
    case kI32: return launch_scatter_op<kI32, THREADS>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

}  // namespace ar
