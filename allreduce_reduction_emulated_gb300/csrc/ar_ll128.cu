// ar_ll128.cu -- the LL128 medium-message all-reduce.
//
// "Demystifying NVSHMEM" (the collectives paragraph) names LL128 next to LL:
// data and arrival flag travel together, here in 128-byte lines of 16 words
// of 8 bytes -- 15 payload words (120 bytes) and one flag word (this call's
// epoch) -- so 94% of the staged bytes are payload against LL's 50%.
// Whole-line atomicity of a 128-byte store is not a guarantee of the PTX
// memory model, so the line is published explicitly: the lanes of a warp
// write the payload words, fence, synchronise, and one lane stores the flag
// word with release semantics; a reader acquires the flag and only then reads
// the payload.  Emulated like LL, one block per slice of the message: block b
// owns lines [b * S, (b + 1) * S) of every rank (S = the slice, 4 lines for 8
// ranks); its warps play the P ranks and stage those lines, then its threads
// receive the slice's payload words -- each acquires the flag of its word's
// line in every rank's slot, reads the word and folds the P values in ring
// order (so LL128 == RING bit for bit) -- and write the result into every
// rank's receive buffer.  No block waits for another block.
// The epoch is kept on the device as for LL, so calls can be captured in a
// CUDA graph.  Every flag wait is bounded; on its limit a thread records
// AR_ERR_TIMEOUT and stops reducing.
#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_ll_epoch.cuh"
#include "ar_launch.h"

namespace ar {

namespace {

constexpr int kThreads = 256;      // threads that stage and receive lines
constexpr int kBlock = kThreads + 32;  // + one warp that counts the block into the epoch
constexpr int kLineWords = 16;     // 8-byte words per 128-byte line
constexpr int kPayloadWords = 15;  // the 16th word is the flag
constexpr int kBatch = 8;          // ranks polled together
constexpr int kWarpLines = 4;      // lines a warp stages at once (8 lanes per line)
constexpr int kRoundLines = kThreads / 32 * kWarpLines;  // lines a block stages at once

template <int MAXP>
struct LL128Params {
  const void* send[MAXP];
  void* recv[MAXP];
  unsigned long long* staging;  // P slots of `stride` 8-byte words (whole lines)
  uint64_t stride;
  int* status;
  uint64_t nbytes;       // bytes per rank
  uint64_t nwords;       // 8-byte payload words per rank
  uint64_t nlines;       // lines per rank
  uint64_t chunk_words;  // payload words per ring chunk (16-byte chunks: even)
  unsigned int* epoch_state;
  uint64_t stage_words;  // whole staging area (P slots), cleared on epoch wrap
  uint32_t spin_limit;
  int P;
  int slice_lines;       // lines of every rank per block
  int skip_produce;
  int do_scale;
  float scale;
};

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// 8-byte payload word w of a rank buffer (zero beyond nbytes).
__device__ __forceinline__ unsigned long long load_word8(const void* buf, uint64_t w, uint64_t nbytes) {
  if (8 * w + 8 <= nbytes) return static_cast<const unsigned long long*>(buf)[w];
  unsigned long long v = 0;
  const uint16_t* h = static_cast<const uint16_t*>(buf);
  for (uint64_t b = 8 * w; b < nbytes; b += 2) v |= (unsigned long long)h[b / 2] << (8 * (b - 8 * w));
  return v;
}

__device__ __forceinline__ void store_word8(void* buf, uint64_t w, uint64_t nbytes, unsigned long long v) {
  if (8 * w + 8 <= nbytes) {
    static_cast<unsigned long long*>(buf)[w] = v;
    return;
  }
  uint16_t* h = static_cast<uint16_t*>(buf);
  for (uint64_t b = 8 * w; b < nbytes; b += 2) h[b / 2] = (uint16_t)(v >> (8 * (b - 8 * w)));
}

// An 8-byte payload word holds 2 fp32 / int32 or 4 bf16 values.
template <int DT> struct Word8 {
  static constexpr int N = DT == kBF16 ? 4 : 2;
  typename Lanes<DT>::T v[N];
};

template <int DT>
__device__ __forceinline__ Word8<DT> widen8(unsigned long long x) {
  Word8<DT> a;
  const uint32_t lo = (uint32_t)x, hi = (uint32_t)(x >> 32);
  if constexpr (DT == kF32) {
    a.v[0] = __uint_as_float(lo);
    a.v[1] = __uint_as_float(hi);
  } else if constexpr (DT == kBF16) {
    a.v[0] = bf16_lo(lo); a.v[1] = bf16_hi(lo); a.v[2] = bf16_lo(hi); a.v[3] = bf16_hi(hi);
  } else {
    a.v[0] = (int32_t)lo;
    a.v[1] = (int32_t)hi;
  }
  return a;
}

template <int DT, int OP>
__device__ __forceinline__ void fold8(Word8<DT>& acc, const Word8<DT>& x) {
#pragma unroll
  for (int i = 0; i < Word8<DT>::N; ++i) acc.v[i] = combine<DT, OP>(acc.v[i], x.v[i]);
}

template <int DT>
__device__ __forceinline__ unsigned long long narrow8(Word8<DT> a, float scale, bool do_scale) {
  if constexpr (DT == kI32) {
    return (unsigned long long)(uint32_t)a.v[0] | ((unsigned long long)(uint32_t)a.v[1] << 32);
  } else {
    if (do_scale) {
#pragma unroll
      for (int i = 0; i < Word8<DT>::N; ++i) a.v[i] = __fmul_rn(a.v[i], scale);
    }
    if constexpr (DT == kF32)
      return (unsigned long long)__float_as_uint(a.v[0]) | ((unsigned long long)__float_as_uint(a.v[1]) << 32);
    else
      return (unsigned long long)pack_bf16x2(a.v[0], a.v[1]) |
             ((unsigned long long)pack_bf16x2(a.v[2], a.v[3]) << 32);
  }
}

// Receives the payload words of lines [l0, l0 + nl) of every rank, one word
// per thread per step: acquires the flag of the word's line in each rank's
// slot, reads the word, folds in ring order and writes the result to every
// rank; returns early (status AR_ERR_TIMEOUT) if a flag wait runs out.
template <int MAXP, int DT, int OP>
__device__ __forceinline__ void ll128_reduce_slice(const LL128Params<MAXP>& p, uint64_t l0, uint32_t nl,
                                                   unsigned long long flag) {
  const int P = p.P;
  const uint64_t wa = l0 * kPayloadWords;
  uint64_t wb = wa + (uint64_t)nl * kPayloadWords;
  if (wb > p.nwords) wb = p.nwords;
  for (uint64_t w = wa + threadIdx.x; w < wb; w += kThreads) {
    const int g = (int)(w / p.chunk_words);  // ring chunk: folded from rank g
    const uint64_t line = w / kPayloadWords;
    const uint64_t off = line * kLineWords + (w - line * kPayloadWords);
    Word8<DT> acc;
    for (int k0 = 0; k0 < P; k0 += kBatch) {
      unsigned long long f[kBatch];
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int k = k0 + j;
        if (k < P) {
          int r = g + k;
          if (r >= P) r -= P;
          f[j] = ld_acquire_u64(p.staging + (uint64_t)r * p.stride + line * kLineWords + kPayloadWords);
        }
      }
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const int k = k0 + j;
        if (k >= P) break;
        int r = g + k;
        if (r >= P) r -= P;
        const unsigned long long* fl = p.staging + (uint64_t)r * p.stride + line * kLineWords + kPayloadWords;
        uint32_t spins = 0;
        while (f[j] != flag) {
          if (++spins > p.spin_limit) {
            atomicExch(p.status, (int)AR_ERR_TIMEOUT);
            return;
          }
          f[j] = ld_acquire_u64(fl);
        }
        const Word8<DT> x = widen8<DT>(ld_relaxed_u64(p.staging + (uint64_t)r * p.stride + off));
        if (k == 0) acc = x;
        else fold8<DT, OP>(acc, x);
      }
    }
    const unsigned long long out = narrow8<DT>(acc, p.scale, p.do_scale != 0);
    for (int r = 0; r < P; ++r) store_word8(p.recv[r], w, p.nbytes, out);
  }
}

template <int MAXP, int DT, int OP>
__global__ void __launch_bounds__(kBlock) ll128_allreduce_kernel(const __grid_constant__ LL128Params<MAXP> p) {
  pdl_enter();
  const bool worker = threadIdx.x < kThreads;
  const int lane = threadIdx.x & 31;
  const int part = lane & 7;  // 16-byte part of a line
  const uint64_t l0 = (uint64_t)blockIdx.x * (uint64_t)p.slice_lines;
  const uint64_t left = p.nlines - l0;
  const uint32_t nl = left < (uint64_t)p.slice_lines ? (uint32_t)left : (uint32_t)p.slice_lines;
  const uint32_t nstage = (uint32_t)p.P * nl;  // lines this block stages: P ranks x nl
  // block line i is rank i / nl's line l0 + i % nl; a warp stages 4 lines at a
  // time, 8 lanes (16 bytes each) per line.  The first round's payload words
  // are loaded while thread 0 reads the epoch.
  const uint32_t i0 = (threadIdx.x >> 5) * kWarpLines + (uint32_t)(lane >> 3);
  unsigned long long a = 0, b = 0;
  const bool live0 = !p.skip_produce && worker && i0 < nstage;
  if (live0) {
    const uint32_t r = i0 / nl;
    const uint64_t w = (l0 + (i0 - r * nl)) * kPayloadWords + 2 * part;
    a = w < p.nwords ? load_word8(p.send[r], w, p.nbytes) : 0ull;
    b = part < 7 && w + 1 < p.nwords ? load_word8(p.send[r], w + 1, p.nbytes) : 0ull;
  }
  const uint32_t epoch = ll_epoch_begin(p.epoch_state);
  const unsigned long long flag = (unsigned long long)epoch;

  // the extra warp counts the block in at once (ll_epoch_arrive: any time after
  // ll_epoch_begin), so its fence and atomic overlap the staging and polling
  if (threadIdx.x == kThreads) ll_epoch_arrive(p.epoch_state, epoch);
  // produce: each line's payload words, then (after a fence and the warp
  // barrier) its flag word stored with release by the line's lane 7 -- a
  // reader that acquires the flag sees the whole line
  if (!p.skip_produce && worker) {
    for (uint32_t i = i0; i - (uint32_t)(lane >> 3) < nstage; i += kRoundLines) {
      const bool live = i < nstage;
      const uint32_t r = live ? i / nl : 0u;
      const uint64_t line = l0 + (i - r * nl);
      unsigned long long* slot = p.staging + (uint64_t)r * p.stride + line * kLineWords;
      if (live) {
        if (i != i0) {
          const uint64_t w = line * kPayloadWords + 2 * part;
          a = w < p.nwords ? load_word8(p.send[r], w, p.nbytes) : 0ull;
          b = part < 7 && w + 1 < p.nwords ? load_word8(p.send[r], w + 1, p.nbytes) : 0ull;
        }
        slot[2 * part] = a;
        if (part < 7) slot[2 * part + 1] = b;
      }
      __threadfence();  // each lane's payload words before the warp barrier ...
      __syncwarp();
      if (live && part == 7) st_release_u64(slot + kPayloadWords, flag);  // ... and the flag after it
    }
  }

  if (worker) ll128_reduce_slice<MAXP, DT, OP>(p, l0, nl, flag);
  ll_epoch_end(p.epoch_state, epoch, p.staging, p.stage_words);
}

template <int MAXP, int DT, int OP>
cudaError_t launch_one(const Call& c, LaunchInfo* info) {
  auto kernel = ll128_allreduce_kernel<MAXP, DT, OP>;
  LL128Params<MAXP> p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = c.send[r];
    p.recv[r] = c.recv[r];
  }
  p.staging = c.staging;
  p.stride = c.stage_stride;
  p.status = c.status;
  p.nbytes = c.count * elem_bytes(DT);
  p.nwords = (p.nbytes + 7) / 8;
  p.nlines = (p.nwords + kPayloadWords - 1) / kPayloadWords;
  p.chunk_words = ring_chunk_vectors(c.count, c.P, DT) * 2;  // 16-byte vectors = 2 words
  p.epoch_state = c.epoch_state;
  p.stage_words = c.stage_words;
  p.spin_limit = c.spin_limit;
  p.P = c.P;
  p.skip_produce = c.skip_produce;
  p.do_scale = (DT != kI32 && c.scale != 1.0f) ? 1 : 0;
  p.scale = c.scale;
  if (p.nlines * kLineWords > p.stride) return cudaErrorInvalidValue;
  // the 8 warps stage 32 lines at once: 4 lines of each of 8 ranks, more for
  // fewer ranks; slices widened so that the grid fits in one wave of resident
  // blocks (a second, nearly empty wave doubled the time at 512 KiB per rank)
  static const int blocks_per_sm = [&] {
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, kBlock, 0) != cudaSuccess) b = 1;
    return b > 0 ? b : 1;
  }();
  const uint64_t wave = (uint64_t)blocks_per_sm * (uint64_t)(c.sms > 0 ? c.sms : 1);
  uint64_t slice = (uint64_t)(kRoundLines / (c.P < 1 ? 1 : c.P));
  if (slice < (uint64_t)kWarpLines) slice = kWarpLines;
  const uint64_t per_wave = (p.nlines + wave - 1) / wave;
  if (slice < per_wave) slice = per_wave;
  if (slice > 0x7fffffffull) return cudaErrorInvalidValue;
  p.slice_lines = (int)slice;
  const uint64_t grid = (p.nlines + slice - 1) / slice;
  if (grid == 0 || grid > 0x7fffffffull) return cudaErrorInvalidValue;
  (void)launch_kernel(kernel, dim3((unsigned)grid), dim3(kBlock), 0, c.stream, use_pdl(c), p);
  const cudaError_t e = cudaGetLastError();
  info->kernel = "ll128";
  info->grid = (int)grid;
  info->block = kBlock;
  info->smem = 0;
  return e;
}

template <int MAXP, int DT>
cudaError_t launch_op(const Call& c, LaunchInfo* info) {
  switch (c.op) {
    case kSum: return launch_one<MAXP, DT, kSum>(c, info);
    case kMin: return launch_one<MAXP, DT, kMin>(c, info);
    case kMax: return launch_one<MAXP, DT, kMax>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

template <int MAXP>
cudaError_t launch_dt(const Call& c, LaunchInfo* info) {
  switch (c.dtype) {
    case kF32: return launch_op<MAXP, kF32>(c, info);
    case kBF16: return launch_op<MAXP, kBF16>(c, info);
    case kI32: return launch_op<MAXP, kI32>(c, info);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Staged 8-byte words per rank for an LL128 limit of `bytes` per rank.
size_t ll128_stage_words(size_t bytes) {
  const size_t words = (bytes + 7) / 8;
  const size_t lines = (words + kPayloadWords - 1) / kPayloadWords;
  return lines * kLineWords;
}

cudaError_t launch_ll128(const Call& c, LaunchInfo* info) {
  if (c.P <= 8) return launch_dt<8>(c, info);
  return launch_dt<AR_MAX_RANKS>(c, info);
}

}  // namespace ar
