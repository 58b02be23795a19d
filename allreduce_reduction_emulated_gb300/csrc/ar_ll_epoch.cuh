// ar_ll_epoch.cuh -- the LL / LL128 per-call epoch, kept on the device.
//
// The LL protocols tag each staged word with the call's epoch.  The epoch
// lives on the device, so a call carries no host state and can be captured
// in a CUDA graph and replayed: state[0] is the last epoch used (0: none
// since the staging area was last cleared, and 0 is never a live flag),
// state[1] counts the blocks of the running call that have read it.
#pragma once

#include "ar_device.cuh"

namespace ar {

__device__ __forceinline__ uint32_t ld_relaxed_u32(const unsigned int* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u32(unsigned int* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

constexpr uint32_t kLLEpochWrap = 0xffffffffu;  // the last 32-bit epoch

// Every block reads the last epoch before doing anything; this call uses
// the next one.
__device__ __forceinline__ uint32_t ll_epoch_begin(const unsigned int* state) {
  __shared__ uint32_t s_epoch;
  if (threadIdx.x == 0) s_epoch = ld_relaxed_u32(state) + 1u;
  __syncthreads();
  return s_epoch;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_u32(unsigned int* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Called by ONE thread of each block, any time after ll_epoch_begin.  The
// count-in is one acquire-release read-modify-write: its release half orders
// the block's read of state[0] (made before the barrier in ll_epoch_begin,
// which this thread has passed) before the increment, and the block that
// completes the count acquires every earlier increment, so all blocks' reads
// happen before its publication of the epoch, which follows in program order.
// (A full fence before a relaxed add gives the same order and measured about
// 0.6 us longer per call.)  The publication need not wait for the other blocks
// to finish: every block has read the old value, and the next call starts only
// after this kernel ends.  The wrap epoch is counted in ll_epoch_end instead.
__device__ __forceinline__ void ll_epoch_arrive(unsigned int* state, uint32_t epoch) {
  if (epoch == kLLEpochWrap) return;
  if (atom_add_acq_rel_u32(&state[1], 1u) == gridDim.x - 1) {
    st_relaxed_u32(&state[1], 0u);
    st_relaxed_u32(&state[0], epoch);
  }
}

// Called by every thread of every block once the block is done with the
// staging area; it does work only for the wrap epoch.  When the last 32-bit
// value has been used, the last block to finish clears the whole staging
// area (`words` 8-byte words) and then resets the epoch to 0, so that
// numbering can restart at 1 without old words matching.
__device__ __forceinline__ void ll_epoch_end(unsigned int* state, uint32_t epoch,
                                             unsigned long long* staging, uint64_t words) {
  if (epoch != kLLEpochWrap) return;  // counted in by ll_epoch_arrive
  __shared__ int s_last;
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    s_last = atomicAdd(&state[1], 1u) == gridDim.x - 1;
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (uint64_t i = threadIdx.x; i < words; i += blockDim.x) st_relaxed_u64(staging + i, 0ull);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    st_relaxed_u32(&state[1], 0u);
    st_relaxed_u32(&state[0], 0u);
  }
}

}  // namespace ar
