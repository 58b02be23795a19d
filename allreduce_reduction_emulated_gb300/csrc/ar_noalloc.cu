// ar_noalloc.cu -- an LL all-reduce for callers that cannot allocate device
// memory (declared in include/ar.h as ar_allreduce_ll_noalloc).
//
// Some callers must not call cudaMalloc: code whose device memory is owned by a
// framework's pool (a library allocation would bypass that pool's accounting
// and limits), code that runs in a latency-critical loop where cudaMalloc /
// cudaFree may synchronize the device, and code that may not allocate once it
// has started.  A communicator (ar_init) allocates its LL staging area, so
// this entry point instead keeps the staging area and the status word in one
// fixed-size array compiled into the library: every GPU that loads the
// library holds that array (about 1 MiB) until the process exits.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Each call stages its words under a fresh epoch, kept in the same
// array on the device, so stale words never match; when the 32-bit epoch runs
// out the kernel clears the staging words once.  The status word starts at
// zero (module load) and is cleared whenever it is read.  Calls that overlap on the GPU (for example on two streams)
// race on the array and must not be issued.
#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>
#include <algorithm>

#include "../../include/ar.h"
#include "ar_launch.h"

namespace {

constexpr size_t kStride = AR_NOALLOC_MAX_BYTES / 4 + 4;  // 8-byte words per rank slot
constexpr size_t kSlotsOffset = 32;  // word 0: the status; word 1: the epoch state
constexpr size_t kScratchWords = kSlotsOffset + (size_t)AR_NOALLOC_MAX_RANKS * kStride;
constexpr uint32_t kSpinLimit = 1u << 22;                  // ~1 s of polls, then AR_ERR_TIMEOUT
constexpr int kMaxDevices = 64;

}  // namespace

static __device__ __align__(256) unsigned long long g_noalloc_scratch[kScratchWords];

namespace {

struct DeviceState {
  std::mutex mu;
  std::atomic<bool> ready{false};
  unsigned long long* base = nullptr;  // device address of g_noalloc_scratch
  int sms = 0;
};

DeviceState g_state[kMaxDevices];

// Per device, with that device current: the array's device address.  (In
// host code the symbol names a host-side stand-in, not device memory.)  A
// lookup that fails leaves the device not ready, and the next call tries
// again.
cudaError_t set_up(DeviceState& s, int dev) {
  if (s.ready.load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(s.mu);
  if (s.ready.load(std::memory_order_relaxed)) return cudaSuccess;
  unsigned long long* base = nullptr;
  int sms = 0;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&base), g_noalloc_scratch);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return e;
  }
  s.base = base;
  s.sms = sms;
  s.ready.store(true, std::memory_order_release);
  return cudaSuccess;
}

bool bad_overlap(const void* const* send, void* const* recv, int P, size_t bytes) {
  std::vector<uintptr_t> starts;
  for (int r = 0; r < P; ++r) {
    starts.push_back((uintptr_t)send[r]);
    starts.push_back((uintptr_t)recv[r]);
  }
  std::sort(starts.begin(), starts.end());
  for (size_t i = 1; i < starts.size(); ++i)
    if (starts[i] != starts[i - 1] && starts[i] - starts[i - 1] < bytes) return true;
  return false;
}

}  // namespace

extern "C" ar_status_t ar_allreduce_ll_noalloc(int nranks, const void* const* sendbufs,
                                               void* const* recvbufs, size_t count, ar_dtype_t dtype,
                                               ar_op_t op, float scale, void* stream,
                                               int* device_status) {
  if (nranks < 1) return AR_ERR_INVALID_ARG;
  if (dtype != AR_FLOAT32 && dtype != AR_BFLOAT16 && dtype != AR_INT32) return AR_ERR_INVALID_ARG;
  if (op != AR_SUM && op != AR_MIN && op != AR_MAX) return AR_ERR_INVALID_ARG;
  if (!(scale == scale)) return AR_ERR_INVALID_ARG;
  if (scale != 1.0f && (dtype == AR_INT32 || op != AR_SUM)) return AR_ERR_UNSUPPORTED;
  const size_t esize = ar::elem_bytes(dtype);
  // beyond the fixed array: too many ranks or too many bytes per rank
  if (nranks > AR_NOALLOC_MAX_RANKS || count > AR_NOALLOC_MAX_BYTES / esize) return AR_ERR_UNSUPPORTED;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return AR_ERR_UNSUPPORTED;
  DeviceState& s = g_state[dev];
  if (set_up(s, dev) != cudaSuccess) return AR_ERR_CUDA;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);

  if (count > 0) {
    if (!sendbufs || !recvbufs) return AR_ERR_INVALID_ARG;
    for (int r = 0; r < nranks; ++r) {
      if (!sendbufs[r] || !recvbufs[r]) return AR_ERR_INVALID_ARG;
      if (((uintptr_t)sendbufs[r] | (uintptr_t)recvbufs[r]) & 15u) return AR_ERR_INVALID_ARG;
    }
    if (bad_overlap(sendbufs, recvbufs, nranks, count * esize)) return AR_ERR_INVALID_ARG;

    ar::Call c;
    c.P = nranks;
    c.send = sendbufs;
    c.recv = recvbufs;
    c.count = count;
    c.dtype = dtype;
    c.op = op;
    c.algo = 1;  // the ring order, which the LL protocol follows
    c.scale = scale;
    c.stream = st;
    c.sms = s.sms;
    c.tree_push = nullptr;
    c.staging = s.base + kSlotsOffset;
    c.stage_stride = kStride;
    c.status = reinterpret_cast<int*>(s.base);
    c.spin_limit = kSpinLimit;
    c.skip_produce = 0;
    c.max_blocks = 0;
    c.group = 1;
    c.shard = 0;
    c.epoch_state = reinterpret_cast<unsigned int*>(s.base + 1);
    c.stage_words = (size_t)AR_NOALLOC_MAX_RANKS * kStride;  // every slot, whatever P
    ar::LaunchInfo info;
    cudaError_t e = ar::launch_ll(c, &info);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return AR_ERR_CUDA;
    }
  }

  if (device_status) {
    // optional, synchronous: wait for the stream, then read and clear the status word
    int h = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess ||
        cudaMemcpy(&h, s.base, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(s.base, 0, sizeof(int)) != cudaSuccess) {
      cudaGetLastError();
      return AR_ERR_CUDA;
    }
    *device_status = h;
  }
  return AR_SUCCESS;
}
