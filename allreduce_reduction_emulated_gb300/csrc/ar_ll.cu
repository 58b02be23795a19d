// ar_ll.cu -- the LL (low-latency) small-message all-reduce.
//
// "Demystifying NVSHMEM" (the collectives paragraph): for small messages the
// LL protocol packs the data and its arrival flag into one atomic write, so a
// receiver needs no separate flag, fence or barrier.  Emulated here with the
// P ranks' producers and receivers as threads of one block per slice of the
// message: block b owns words [b * S, (b + 1) * S) of every rank (S = the
// slice, 32 words for 8 ranks);
//   produce  the block's threads play the P ranks: rank r's 4-byte payload
//            word w is written to rank r's staging slot as one 8-byte word
//            {low: payload, high: flag = this call's epoch};
//   reduce   thread t then receives word w = b * S + t: it polls the P
//            ranks' staged words until their flags equal the epoch, folds the
//            payloads in the ring order of w's chunk (x_c, x_{c+1}, ... for
//            ring chunk c) -- so LL == RING bit for bit -- and writes the
//            result straight into all P receive buffers (the all-gather).
// No block waits for another block, so the kernel needs no cooperative launch
// and its grid is as wide as the message; the only extra cost over the ring
// kernel is the staged word's round trip through L2.  (A layout in which a
// block group played each rank and reduced its ring chunk from other blocks'
// staged words measured 8.3 us at 4 KiB per rank against 6.3 us for this one.)
// A new epoch per call means the staging area is never cleared between calls;
// the epoch is kept on the device (ll_epoch_begin / ll_epoch_arrive /
// ll_epoch_end), so a call can be captured in a CUDA graph.  Every flag wait
// is bounded, and on its limit the thread records AR_ERR_TIMEOUT in the
// status word and stops reducing.
#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_ll_epoch.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

constexpr int kLLThreads = 256;   // threads that stage and receive words
constexpr int kLLBlock = kLLThreads + 32;  // + one warp that counts the block into the epoch
constexpr int kLLBatch = 8;       // staged words polled together (loads in flight)
constexpr int kLLMinSlice = 32;   // words per block when P >= 8 (one staged word per thread)

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
  int slice_words;       // words of every rank per block
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

// Thread t of the block receives word w = base + t (t < nb): it polls the P
// ranks' staged words in the ring order of w's chunk, folds them and writes
// the result to every rank; it returns early (status AR_ERR_TIMEOUT) if a
// flag wait runs out.
template <int MAXP, int DT, int OP>
__device__ __forceinline__ void ll_reduce_slice(const LLParams<MAXP>& p, uint64_t base, uint32_t nb,
                                                uint32_t epoch) {
  const int P = p.P;
  for (uint32_t t = threadIdx.x; t < nb; t += kLLThreads) {
    const uint64_t w = base + t;
    const int g = (int)(w / p.chunk_words);  // ring chunk: folded from rank g
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
__global__ void __launch_bounds__(kLLBlock) ll_allreduce_kernel(const __grid_constant__ LLParams<MAXP> p) {
  pdl_enter();
  const bool worker = threadIdx.x < kLLThreads;
  const uint64_t base = (uint64_t)blockIdx.x * (uint64_t)p.slice_words;
  const uint64_t left = p.nwords - base;
  const uint32_t nb = left < (uint64_t)p.slice_words ? (uint32_t)left : (uint32_t)p.slice_words;
  const uint32_t nstage = (uint32_t)p.P * nb;  // staged words of this block: P ranks x nb
  // staged word i is rank i / nb's word base + i % nb (consecutive threads read
  // consecutive words of one rank); the first is loaded while thread 0 reads
  // the epoch
  const bool first = !p.skip_produce && worker && threadIdx.x < nstage;
  const uint32_t r0 = first ? threadIdx.x / nb : 0u;
  const uint64_t w0 = base + (threadIdx.x - r0 * nb);
  const uint32_t v0 = first ? load_payload(p.send[r0], w0, p.nbytes) : 0u;
  const uint32_t epoch = ll_epoch_begin(p.epoch_state);
  const unsigned long long tag = (unsigned long long)epoch << 32;

  // the extra warp counts the block in at once (ll_epoch_arrive: any time after
  // ll_epoch_begin), so its fence and atomic overlap the staging and polling
  if (threadIdx.x == kLLThreads) ll_epoch_arrive(p.epoch_state, epoch);
  // produce: stage the P ranks' payload words of this slice with this call's flag
  if (!p.skip_produce && worker) {
    if (first) st_relaxed_u64(p.staging + (uint64_t)r0 * p.stride + w0, tag | v0);
    // more than 8 ranks: further words, their loads issued four at a time
    for (uint32_t i0 = threadIdx.x + kLLThreads; i0 < nstage; i0 += 4 * kLLThreads) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t i = i0 + (uint32_t)u * kLLThreads;
        if (i < nstage) {
          const uint32_t r = i / nb;
          v[u] = load_payload(p.send[r], base + (i - r * nb), p.nbytes);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t i = i0 + (uint32_t)u * kLLThreads;
        if (i < nstage) {
          const uint32_t r = i / nb;
          st_relaxed_u64(p.staging + (uint64_t)r * p.stride + base + (i - r * nb), tag | v[u]);
        }
      }
    }
  }
  if (worker) ll_reduce_slice<MAXP, DT, OP>(p, base, nb, epoch);
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
  // one staged word per thread for P <= 8 (slices of 256 / P words, at least
  // 32), widened so that the grid fits in one wave of resident blocks
  static const int blocks_per_sm = [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kLLBlock, 0) != cudaSuccess) b = 1;
    return b > 0 ? b : 1;
  }();
  const uint64_t wave = (uint64_t)blocks_per_sm * (uint64_t)(c.sms > 0 ? c.sms : 1);
  uint64_t slice = (uint64_t)(kLLThreads / (c.P < 1 ? 1 : c.P));
  if (slice < (uint64_t)kLLMinSlice) slice = kLLMinSlice;
  const uint64_t per_wave = (p.nwords + wave - 1) / wave;
  if (slice < per_wave) slice = per_wave;
  if (slice > 0x7fffffffull) return cudaErrorInvalidValue;
  p.slice_words = (int)slice;
  const uint64_t grid = (p.nwords + slice - 1) / slice;
  if (grid == 0 || grid > 0x7fffffffull) return cudaErrorInvalidValue;
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(kLLBlock), 0, c.stream, use_pdl(c), p);
  const cudaError_t e = cudaGetLastError();
  info->kernel = "ll";
  info->grid = (int)grid;
  info->block = kLLBlock;
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
