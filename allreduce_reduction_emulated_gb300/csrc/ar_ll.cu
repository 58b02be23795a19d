// ar_ll.cu -- the LL (low-latency) small-message all-reduce.
//
// "Demystifying NVSHMEM" (the collectives paragraph): for small messages the
// LL protocol packs the data and its arrival flag into one atomic write, so a
// receiver needs no separate flag, fence or barrier.  Emulated here inside one
// kernel: block group g plays rank g.
//   produce  rank g's buffer is cut into 4-byte payload words; word w is
//            written to rank g's staging slot as one 8-byte word
//            {low: payload, high: flag = this call's epoch};
//   reduce   group g then owns ring chunk g (the ring's reduce-scatter): for
//            each word of the chunk it polls the P ranks' staged words until
//            their flags equal the epoch, folds the payloads in ring order
//            (x_g, x_{g+1}, ...) -- so LL == RING bit for bit -- and writes
//            the result straight into all P receive buffers (the all-gather).
// A new epoch per call means the staging area is never cleared between calls;
// the epoch is kept on the device (ll_epoch_begin / ll_epoch_arrive /
// ll_epoch_end), so a call can be captured in a CUDA graph.  All blocks must be resident at once (a
// reducer waits for other blocks), so the kernel is launched cooperatively;
// every flag wait is bounded, and on its limit the thread records
// AR_ERR_TIMEOUT in the status word and stops reducing.
#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_ll_epoch.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

constexpr int kLLThreads = 256;
constexpr int kLLBatch = 8;  // staged words polled together (loads in flight)

template <int MAXP>
struct LLParams {
  const void* send[MAXP];
  void* recv[MAXP];
  unsigned long long* staging;
  uint64_t stride;       // staged words per rank slot
  int* status;
  uint64_t nbytes;       // bytes per rank
  uint64_t nwords;       // 4-byte payload words per rank
  uint64_t chunk_words;  // words per ring chunk
  unsigned int* epoch_state;
  uint64_t stage_words;  // whole staging area (P slots), cleared on epoch wrap
  uint32_t spin_limit;
  int P;
  int bpr;               // blocks per rank group
  int skip_produce;
  int do_scale;
  float scale;
};

// One payload word: a single fp32 / int32 element or a pair of bf16 elements.
template <int DT> struct Word {
  static constexpr int N = DT == kBF16 ? 2 : 1;
  typename Lanes<DT>::T v[N];
};

template <int DT>
__device__ __forceinline__ Word<DT> widen_word(uint32_t w) {
  Word<DT> a;
  if constexpr (DT == kF32) a.v[0] = __uint_as_float(w);
  else if constexpr (DT == kBF16) { a.v[0] = bf16_lo(w); a.v[1] = bf16_hi(w); }
  else a.v[0] = (int32_t)w;
  return a;
}

template <int DT, int OP>
__device__ __forceinline__ void fold_word(Word<DT>& acc, const Word<DT>& x) {
#pragma unroll
  for (int i = 0; i < Word<DT>::N; ++i) acc.v[i] = combine<DT, OP>(acc.v[i], x.v[i]);
}

template <int DT>
__device__ __forceinline__ uint32_t narrow_word(Word<DT> a, float scale, bool do_scale) {
  if constexpr (DT == kI32) {
    return (uint32_t)a.v[0];
  } else {
    if (do_scale) {
#pragma unroll
      for (int i = 0; i < Word<DT>::N; ++i) a.v[i] = __fmul_rn(a.v[i], scale);
    }
    if constexpr (DT == kF32) return __float_as_uint(a.v[0]);
    else return pack_bf16x2(a.v[0], a.v[1]);
  }
}

// Word w of a rank buffer; only an odd bf16 count leaves a 2-byte last word.
__device__ __forceinline__ uint32_t load_payload(const void* buf, uint64_t w, uint64_t nbytes) {
  if (4 * w + 4 <= nbytes) return static_cast<const uint32_t*>(buf)[w];
  return static_cast<const uint16_t*>(buf)[2 * w];
}

__device__ __forceinline__ void store_payload(void* buf, uint64_t w, uint64_t nbytes, uint32_t v) {
  if (4 * w + 4 <= nbytes) static_cast<uint32_t*>(buf)[w] = v;
  else static_cast<uint16_t*>(buf)[2 * w] = (uint16_t)v;
}

// Reduces ring chunk g in ring order and writes it to every rank; returns
// early (status AR_ERR_TIMEOUT) if a flag wait runs out.
template <int MAXP, int DT, int OP>
__device__ __forceinline__ void ll_reduce_chunk(const LLParams<MAXP>& p, int g, uint64_t lt, uint64_t nt,
                                                uint32_t epoch) {
  const int P = p.P;
  const uint64_t w0 = (uint64_t)g * p.chunk_words;
  uint64_t w1 = w0 + p.chunk_words;
  if (w1 > p.nwords) w1 = p.nwords;
  for (uint64_t w = w0 + lt; w < w1; w += nt) {
    Word<DT> acc;
    for (int k0 = 0; k0 < P; k0 += kLLBatch) {
      unsigned long long x[kLLBatch];
#pragma unroll
      for (int j = 0; j < kLLBatch; ++j) {
        const int k = k0 + j;
        if (k < P) {
          int r = g + k;
          if (r >= P) r -= P;
          x[j] = ld_relaxed_u64(p.staging + (uint64_t)r * p.stride + w);
        }
      }
#pragma unroll
      for (int j = 0; j < kLLBatch; ++j) {
        const int k = k0 + j;
        if (k >= P) break;
        if ((uint32_t)(x[j] >> 32) != epoch) {
          int r = g + k;
          if (r >= P) r -= P;
          const unsigned long long* src = p.staging + (uint64_t)r * p.stride + w;
          uint32_t spins = 0;
          do {
            if (++spins > p.spin_limit) {
              atomicExch(p.status, (int)AR_ERR_TIMEOUT);
              return;
            }
            x[j] = ld_relaxed_u64(src);
          } while ((uint32_t)(x[j] >> 32) != epoch);
        }
        const Word<DT> xw = widen_word<DT>((uint32_t)x[j]);
        if (k == 0) acc = xw;
        else fold_word<DT, OP>(acc, xw);
      }
    }
    const uint32_t out = narrow_word<DT>(acc, p.scale, p.do_scale != 0);
    for (int r = 0; r < P; ++r) store_payload(p.recv[r], w, p.nbytes, out);
  }
}

template <int MAXP, int DT, int OP>
__global__ void __launch_bounds__(kLLThreads) ll_allreduce_kernel(const __grid_constant__ LLParams<MAXP> p) {
  const int g = blockIdx.x / p.bpr;
  const uint64_t lt = (uint64_t)(blockIdx.x % p.bpr) * kLLThreads + threadIdx.x;
  const uint64_t nt = (uint64_t)p.bpr * kLLThreads;
  // the first payload word is loaded while thread 0 reads the epoch
  const bool first = !p.skip_produce && lt < p.nwords;
  const uint32_t w0 = first ? load_payload(p.send[g], lt, p.nbytes) : 0u;
  const uint32_t epoch = ll_epoch_begin(p.epoch_state);
  const unsigned long long tag = (unsigned long long)epoch << 32;

  // produce: stage rank g's payload words with this call's flag
  if (!p.skip_produce) {
    unsigned long long* slot = p.staging + (uint64_t)g * p.stride;
    if (first) st_relaxed_u64(slot + lt, tag | w0);
    for (uint64_t w = lt + nt; w < p.nwords; w += nt)
      st_relaxed_u64(slot + w, tag | load_payload(p.send[g], w, p.nbytes));
  }
  // counted in by the block's last thread, off the reducers' path: with
  // chunks of fewer than 256 words (up to 8 KiB per rank at P = 8) it has
  // nothing to reduce
  if (threadIdx.x == kLLThreads - 1) ll_epoch_arrive(p.epoch_state, epoch);
  ll_reduce_chunk<MAXP, DT, OP>(p, g, lt, nt, epoch);
  ll_epoch_end(p.epoch_state, epoch, p.staging, p.stage_words);
}

template <int MAXP, int DT, int OP>
cudaError_t launch_ll_one(const Call& c, LaunchInfo* info) {
  auto kernel = ll_allreduce_kernel<MAXP, DT, OP>;
  LLParams<MAXP> p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = c.send[r];
    p.recv[r] = c.recv[r];
  }
  p.staging = c.staging;
  p.stride = c.stage_stride;
  p.status = c.status;
  p.nbytes = c.count * elem_bytes(DT);
  p.nwords = (p.nbytes + 3) / 4;
  p.chunk_words = ring_chunk_vectors(c.count, c.P, DT) * 4;  // 16-byte vectors = 4 words
  p.epoch_state = c.epoch_state;
  p.stage_words = c.stage_words;
  p.spin_limit = c.spin_limit;
  p.P = c.P;
  p.skip_produce = c.skip_produce;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  p.scale = c.scale;
  static const int blocks_per_sm = [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kLLThreads, 0) != cudaSuccess) b = 0;
    return b;
  }();
  const int resident = blocks_per_sm * c.sms;
  if (c.P > resident) return cudaErrorCooperativeLaunchTooLarge;
  uint64_t bpr = (p.nwords + kLLThreads - 1) / kLLThreads;
  const uint64_t bpr_cap = (uint64_t)(resident / c.P);
  if (bpr > bpr_cap) bpr = bpr_cap;
  if (bpr < 1) bpr = 1;
  p.bpr = (int)bpr;
  const int grid = c.P * p.bpr;
  void* args[] = {&p};
  cudaError_t e = cudaLaunchCooperativeKernel((const void*)kernel, dim3(grid), dim3(kLLThreads), args,
                                              0, c.stream);
  info->kernel = "ll";
  info->grid = grid;
  info->block = kLLThreads;
  info->smem = 0;
  return e;
}

template <int MAXP, int DT>
cudaError_t launch_ll_op(const Call& c, LaunchInfo* info) {
  switch (c.op) {
    case kSum: return launch_ll_one<MAXP, DT, kSum>(c, info);
    case kMin: return launch_ll_one<MAXP, DT, kMin>(c, info);
    case kMax: return launch_ll_one<MAXP, DT, kMax>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int MAXP>
cudaError_t launch_ll_dt(const Call& c, LaunchInfo* info) {
  switch (c.dtype) {
    case kF32: return launch_ll_op<MAXP, kF32>(c, info);
    case kBF16: return launch_ll_op<MAXP, kBF16>(c, info);
    case kI32: return launch_ll_op<MAXP, kI32>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_ll(const Call& c, LaunchInfo* info) {
  // small parameter block for the common rank counts keeps the launch cheap
  if (c.P <= 8) return launch_ll_dt<8>(c, info);
  return launch_ll_dt<AR_MAX_RANKS>(c, info);
}

}  // namespace ar
