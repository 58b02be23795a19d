// ar_generic.cu -- ring-order and tree-order all-reduce for any rank count up
// to AR_MAX_RANKS (used above the rank-specialised kernels' limit).
//
// With many ranks the NP input vectors of one element group no longer fit in
// registers, and the fold order needs a dynamic rank index.  So each thread
// stages its column -- one 16-byte vector from every rank -- in shared memory
// with asynchronous copies (all P copies in flight at once), waits for its own
// copies only, folds from shared memory (ring: rotated start; tree: a
// postorder program evaluated on a small stack) and stores the result to all
// P receive buffers.  Threads never read each other's slots, so no barrier is
// needed.
#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

constexpr int kStackDepth = 16;  // >= tree height + 1 for P <= AR_MAX_RANKS

struct GenericParams {
  const uint4* send[AR_MAX_RANKS];
  uint4* recv[AR_MAX_RANKS];
  const int16_t* prog;  // tree 0 program, then tree 1 program
  int prog_len;
  int P;
  uint64_t nfull;
  uint64_t split;  // ring: vectors per chunk; tree: first vector of tree 1
  float scale;
  int do_scale;
  int tail;
};

__device__ __forceinline__ void cp_async16(uint32_t smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem), "l"(gmem) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

template <int DT, int OP, int ALGO, int T>
__device__ __forceinline__ Acc<DT> fold_staged(const uint4* stage, int tid, const GenericParams& p,
                                               uint64_t v) {
  const int P = p.P;
  if constexpr (ALGO == kRing) {
    int r = (int)(v / p.split);
    Acc<DT> acc = widen<DT>(stage[r * T + tid]);
    for (int k = 1; k < P; ++k) {
      r = (r + 1 == P) ? 0 : r + 1;
      fold<DT, OP>(acc, widen<DT>(stage[r * T + tid]));
    }
    return acc;
  } else {
    const int16_t* prog = p.prog + (v < p.split ? 0 : p.prog_len);
    Acc<DT> stack[kStackDepth];
    int sp = 0;
    for (int i = 0; i < p.prog_len; ++i) {
      const int op = __ldg(prog + i);
      if (op >= 0) {
        stack[sp++] = widen<DT>(stage[op * T + tid]);
      } else {
        --sp;
        fold<DT, OP>(stack[sp - 1], stack[sp]);
      }
    }
    return stack[0];
  }
}

template <int DT, int OP, int ALGO, int T>
__global__ void __launch_bounds__(T) generic_allreduce_kernel(const __grid_constant__ GenericParams p) {
  extern __shared__ uint4 stage[];  // [P][T]
  const int tid = threadIdx.x;
  const int P = p.P;
  const uint32_t slot = (uint32_t)__cvta_generic_to_shared(stage + tid);
  const uint64_t n = p.nfull;
  for (uint64_t v = (uint64_t)blockIdx.x * T + tid; v < n; v += (uint64_t)gridDim.x * T) {
    for (int r = 0; r < P; ++r) cp_async16(slot + (uint32_t)(r * T * 16), p.send[r] + v);
    cp_async_wait_all();
    const uint4 o =
        narrow<DT>(fold_staged<DT, OP, ALGO, T>(stage, tid, p, v), p.scale, p.do_scale != 0);
    for (int r = 0; r < P; ++r) st_stream(p.recv[r] + v, o);
  }
  if (p.tail != 0 && blockIdx.x == 0 && tid == 0) {
    for (int r = 0; r < P; ++r) stage[r * T] = load_partial<DT>(p.send[r] + n, p.tail);
    const uint4 o =
        narrow<DT>(fold_staged<DT, OP, ALGO, T>(stage, 0, p, n), p.scale, p.do_scale != 0);
    for (int r = 0; r < P; ++r) store_partial<DT>(p.recv[r] + n, o, p.tail);
  }
}

template <int DT, int OP, int ALGO, int T>
cudaError_t launch_generic_one(const Call& c, LaunchInfo* info) {
  auto kernel = generic_allreduce_kernel<DT, OP, ALGO, T>;
  GenericParams p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = static_cast<const uint4*>(c.send[r]);
    p.recv[r] = static_cast<uint4*>(c.recv[r]);
  }
  p.prog = c.tree_prog;
  p.prog_len = c.prog_len;
  p.P = c.P;
  const uint64_t V = (uint64_t)vec_elems(DT);
  p.nfull = c.count / V;
  p.tail = (int)(c.count % V);
  p.split = ALGO == kRing ? ring_chunk_vectors(c.count, c.P, DT) : tree_split_vectors(c.count, DT);
  p.scale = c.scale;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  const size_t smem = (size_t)c.P * T * sizeof(uint4);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int blocks_per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks_per_sm, kernel, T, smem);
  if (e != cudaSuccess) return e;
  if (blocks_per_sm < 1) blocks_per_sm = 1;
  const uint64_t need = (p.nfull + T - 1) / T;
  const uint64_t cap = (uint64_t)c.sms * (uint64_t)blocks_per_sm;
  const int grid = (int)(need < 1 ? 1 : (need < cap ? need : cap));
  kernel<<<grid, T, smem, c.stream>>>(p);
  info->kernel = ALGO == kRing ? "staged_ring" : "staged_tree";
  info->grid = grid;
  info->block = T;
  info->smem = smem;
  return cudaGetLastError();
}

template <int DT, int OP, int ALGO>
cudaError_t launch_generic_t(const Call& c, LaunchInfo* info) {
  // 64 threads keep P * 64 * 16 bytes <= 128 KiB up to P = 128; beyond that 32.
  if (c.P <= 128) return launch_generic_one<DT, OP, ALGO, 64>(c, info);
  return launch_generic_one<DT, OP, ALGO, 32>(c, info);
}

template <int DT, int OP>
cudaError_t launch_generic_algo(const Call& c, LaunchInfo* info) {
  if (c.algo == kRing) return launch_generic_t<DT, OP, kRing>(c, info);
  if (c.algo == kTree) return launch_generic_t<DT, OP, kTree>(c, info);
  return cudaErrorInvalidValue;
}

template <int DT>
cudaError_t launch_generic_op(const Call& c, LaunchInfo* info) {
  switch (c.op) {
    case kSum: return launch_generic_algo<DT, kSum>(c, info);
    case kMin: return launch_generic_algo<DT, kMin>(c, info);
    case kMax: return launch_generic_algo<DT, kMax>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_generic(const Call& c, LaunchInfo* info) {
  switch (c.dtype) {
    case kF32: return launch_generic_op<kF32>(c, info);
    case kBF16: return launch_generic_op<kBF16>(c, info);
    case kI32: return launch_generic_op<kI32>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ar
