// ar_api.cu -- the C ABI of libar.so (declared in include/ar.h): communicator
// lifetime, argument checks, algorithm selection and kernel dispatch.
// Host code only; the kernels live in ar_static_*.cu and ar_tma_*.cu (P <= 8,
// on the whole GPU and on a few SMs), ar_generic.cu (any P), ar_ll.cu,
// ar_ll128.cu, ar_collectives.cu and ar_tma_gather.cu.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "../../include/ar.h"
#include "ar_device.cuh"
#include "ar_launch.h"

struct ar_comm {
  int P = 0;
  int device = 0;
  int sms = 0;
  // LL staging: P slots of `stage_stride` 8-byte words (one word per 4 payload bytes)
  unsigned long long* staging = nullptr;
  size_t stage_stride = 0;
  size_t ll_capacity_bytes = 0;  // per rank, fixed at ar_init
  size_t ll_max_bytes = 0;       // current AUTO threshold / LL limit (<= capacity)
  uint32_t spin_limit = 0;
  int skip_produce = 0;
  int debug = 0;
  // device control block (kControlInts ints): [0] the ar_status_t word,
  // [2..3] LL epoch state, [4..5] LL128 epoch state ({last epoch, blocks counted in})
  int* status = nullptr;
  int16_t* tree_push = nullptr;  // device: tree 0's then tree 1's ranks in preorder (P each)
  // LL128 staging: P slots of `ll128_stride` 8-byte words (128-byte lines)
  unsigned long long* staging128 = nullptr;
  size_t ll128_stride = 0;
  size_t ll128_capacity_bytes = 0;
  size_t ll128_max_bytes = 0;
  int hier_group = 8;            // AR_ALGO_HIER: ranks per group
  // ar_tune: fastest algorithm per power-of-two size bucket, used by AUTO
  // when auto_tuned is set
  ar_algo_t tuned[AR_TUNE_BUCKETS] = {};
  int tuned_valid = 0;
  int auto_tuned = 0;
  int max_blocks = 0;            // AR_OPT_MAX_BLOCKS (0 = no cap)
  // AR_OPT_CAPPED_KERNEL: kernel for P <= 8 ring / tree all-reduces and
  // reduce-scatters capped below the SM count (0 = the wide load/store shape,
  // 1 = the TMA pipeline; initial value from AR_CAPPED_KERNEL=wide|tma)
  int capped_tma = 0;
};

namespace {

constexpr int kControlInts = 8;
constexpr int kLLEpoch = 2, kLL128Epoch = 4;
constexpr size_t kDefaultLLBytes = 65536;
constexpr uint32_t kDefaultSpinLimit = 1u << 22;  // ~1 s of L2 polls at worst
constexpr size_t kMaxLLBytes = 1u << 20;
constexpr size_t kDefaultLL128Bytes = 1u << 20;
constexpr size_t kMaxLL128Bytes = 16u << 20;

long long env_ll(const char* name, long long dflt) {
  const char* s = std::getenv(name);
  if (!s || !*s) return dflt;
  char* end = nullptr;
  long long v = std::strtoll(s, &end, 0);
  return (end && *end == 0) ? v : dflt;
}

bool valid_dtype(int d) { return d == AR_FLOAT32 || d == AR_BFLOAT16 || d == AR_INT32; }
bool valid_op(int o) { return o == AR_SUM || o == AR_MIN || o == AR_MAX; }
bool valid_algo(int a) {
  return a == AR_ALGO_AUTO || a == AR_ALGO_RING || a == AR_ALGO_TREE || a == AR_ALGO_LL ||
         a == AR_ALGO_HIER || a == AR_ALGO_LL128;
}

// Ranks of tree t in the order its fold consumes them: own rank, then the
// left subtree, then the right subtree (preorder), for ((own (+) left) (+) right).
void emit_preorder(int v, int P, int t, std::vector<int16_t>& out) {
  out.push_back((int16_t)ar::tree_owner(v, P, t));
  const int l = ar::tree_left(v), r = ar::tree_right(v, P);
  if (l) emit_preorder(l, P, t, out);
  if (r) emit_preorder(r, P, t, out);
}

// One NVTX range per collective call, around its launch, in a domain of its
// own (so a caller's default-domain ranges and filters are unaffected).
// Header-only NVTX: a no-op unless a profiler is attached.
nvtxDomainHandle_t nvtx_domain() {
  static const nvtxDomainHandle_t d = nvtxDomainCreateA("allreduce_emulated");
  return d;
}

struct Range {
  explicit Range(const char* name) {
    nvtxEventAttributes_t a = {};
    a.version = NVTX_VERSION;
    a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
    a.messageType = NVTX_MESSAGE_TYPE_ASCII;
    a.message.ascii = name;
    nvtxDomainRangePushEx(nvtx_domain(), &a);
  }
  ~Range() { nvtxDomainRangePop(nvtx_domain()); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

const char* allreduce_range(ar_algo_t a) {
  return a == AR_ALGO_RING   ? "ar_allreduce ring"
         : a == AR_ALGO_TREE ? "ar_allreduce tree"
         : a == AR_ALGO_LL   ? "ar_allreduce ll"
         : a == AR_ALGO_LL128 ? "ar_allreduce ll128"
                             : "ar_allreduce hier";
}

const char* dtype_name(int d) { return d == AR_FLOAT32 ? "f32" : d == AR_BFLOAT16 ? "bf16" : "i32"; }
const char* op_name(int o) { return o == AR_SUM ? "sum" : o == AR_MIN ? "min" : "max"; }
const char* algo_name(int a) {
  return a == AR_ALGO_RING   ? "ring"
         : a == AR_ALGO_TREE ? "tree"
         : a == AR_ALGO_LL   ? "ll"
         : a == AR_ALGO_HIER ? "hier"
         : a == AR_ALGO_LL128 ? "ll128"
                             : "auto";
}

void release(ar_comm* c) {
  if (!c) return;
  if (c->staging) cudaFree(c->staging);
  if (c->staging128) cudaFree(c->staging128);
  if (c->status) cudaFree(c->status);
  if (c->tree_push) cudaFree(c->tree_push);
  delete c;
}

// Bucket i of the tuning table covers per-rank sizes (2^(i+2), 2^(i+3)] bytes.
int tune_bucket(size_t bytes) {
  int i = 0;
  size_t top = 8;
  while (top < bytes && i < AR_TUNE_BUCKETS - 1) {
    top <<= 1;
    ++i;
  }
  return i;
}

ar_algo_t resolve(const ar_comm* c, size_t count, ar_dtype_t dtype, ar_algo_t algo) {
  if (algo != AR_ALGO_AUTO) return algo;
  const size_t bytes = count * ar::elem_bytes(dtype);
  if (c->auto_tuned && c->tuned_valid) {
    ar_algo_t a = c->tuned[tune_bucket(bytes)];
    if (a == AR_ALGO_LL && bytes > c->ll_max_bytes) a = AR_ALGO_RING;
    if (a == AR_ALGO_LL128 && bytes > c->ll128_max_bytes) a = AR_ALGO_RING;
    return a;
  }
  return bytes <= c->ll_max_bytes ? AR_ALGO_LL : AR_ALGO_RING;
}

// Rejects buffers that overlap without starting at the same address.  All 2P
// buffers have the same length, so equal starts mean identical buffers, which
// the kernels allow (each element is read before it is written, by the thread
// that writes it, or -- for LL -- before its flag is published).
bool overlapping(const void* const* send, void* const* recv, int P, size_t bytes) {
  std::vector<uintptr_t> starts;
  starts.reserve(2 * (size_t)P);
  for (int r = 0; r < P; ++r) {
    starts.push_back((uintptr_t)send[r]);
    starts.push_back((uintptr_t)recv[r]);
  }
  std::sort(starts.begin(), starts.end());
  for (size_t i = 1; i < starts.size(); ++i)
    if (starts[i] != starts[i - 1] && starts[i] - starts[i - 1] < bytes) return true;
  return false;
}

// Reduce-scatter / all-gather layouts: the P big buffers hold P * shard
// elements, the P small ones shard elements.  Two buffers may share memory
// only when they are identical or in the in-place layout, where rank r's
// small buffer sits at element offset r * shard inside rank r's big buffer.
bool bad_shard_layout(const void* const* big, const void* const* small, int P, size_t shard_bytes) {
  struct Span {
    uintptr_t lo, hi;
    int rank;
    bool is_big;
  };
  std::vector<Span> v;
  v.reserve(2 * (size_t)P);
  for (int r = 0; r < P; ++r) {
    v.push_back({(uintptr_t)big[r], (uintptr_t)big[r] + (uintptr_t)P * shard_bytes, r, true});
    v.push_back({(uintptr_t)small[r], (uintptr_t)small[r] + shard_bytes, r, false});
  }
  std::sort(v.begin(), v.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
  for (size_t i = 0; i < v.size(); ++i) {
    for (size_t j = i + 1; j < v.size() && v[j].lo < v[i].hi; ++j) {
      const Span& a = v[i];
      const Span& b = v[j];
      if (a.lo == b.lo && a.hi == b.hi) continue;  // identical buffers
      const Span& bg = a.is_big ? a : b;
      const Span& sm = a.is_big ? b : a;
      if (bg.is_big && !sm.is_big && bg.rank == sm.rank &&
          sm.lo == bg.lo + (uintptr_t)sm.rank * shard_bytes)
        continue;  // in place
      return true;
    }
  }
  return false;
}

// Pointers need element alignment; *vec is set when every pointer and the
// shard size are whole 16-byte units (the vector kernels' condition).
ar_status_t check_collective(ar_comm_t c, const void* const* a, const void* const* b, ar_dtype_t dtype,
                             size_t shard, bool* vec) {
  if (!valid_dtype(dtype)) return AR_ERR_INVALID_ARG;
  if (shard == 0) return AR_SUCCESS;
  if (!a || !b) return AR_ERR_INVALID_ARG;
  const size_t es = ar::elem_bytes(dtype);
  if (shard > ((size_t)1 << 62) / es / (size_t)c->P) return AR_ERR_INVALID_ARG;
  uintptr_t bits = (uintptr_t)(shard * es);
  for (int r = 0; r < c->P; ++r) {
    if (!a[r] || !b[r]) return AR_ERR_INVALID_ARG;
    if (((uintptr_t)a[r] | (uintptr_t)b[r]) & (es - 1)) return AR_ERR_INVALID_ARG;
    bits |= (uintptr_t)a[r] | (uintptr_t)b[r];
  }
  *vec = (bits & 15u) == 0;
  if (bad_shard_layout(a, b, c->P, shard * es)) return AR_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return dev == c->device ? AR_SUCCESS : AR_ERR_INVALID_ARG;
}

ar::Call base_call(ar_comm_t c, void* stream) {
  ar::Call call;
  call.P = c->P;
  call.stream = static_cast<cudaStream_t>(stream);
  call.sms = c->sms;
  call.tree_push = c->tree_push;
  call.staging = c->staging;
  call.stage_stride = c->stage_stride;
  call.status = c->status;
  call.spin_limit = c->spin_limit;
  call.skip_produce = c->skip_produce;
  call.epoch_state = nullptr;
  call.stage_words = 0;
  call.shard = 0;
  call.group = c->hier_group;
  call.max_blocks = c->max_blocks;
  call.algo = ar::kRing;
  call.scale = 1.0f;
  call.op = AR_SUM;
  return call;
}

}  // namespace

extern "C" {

const char* ar_get_error_string(ar_status_t s) {
  switch (s) {
    case AR_SUCCESS: return "success";
    case AR_ERR_INVALID_ARG: return "invalid argument";
    case AR_ERR_CUDA: return "CUDA runtime error";
    case AR_ERR_UNSUPPORTED: return "unsupported argument combination";
    case AR_ERR_TIMEOUT: return "device-side wait timed out (LL flag or TMA barrier)";
    case AR_ERR_OOM: return "out of device memory";
    default: return "unknown status";
  }
}

ar_status_t ar_init(int nranks, ar_comm_t* out) {
  if (!out) return AR_ERR_INVALID_ARG;
  *out = nullptr;
  if (nranks < 1 || nranks > AR_MAX_RANKS) return AR_ERR_INVALID_ARG;
  ar_comm* c = new (std::nothrow) ar_comm();
  if (!c) return AR_ERR_OOM;
  c->P = nranks;
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) {
    cudaGetLastError();
    delete c;
    return AR_ERR_CUDA;
  }
  long long ll = env_ll("AR_LL_MAX_BYTES", (long long)kDefaultLLBytes);
  if (ll < 16) ll = 16;
  if (ll > (long long)kMaxLLBytes) ll = (long long)kMaxLLBytes;
  c->ll_capacity_bytes = (size_t)ll;
  c->ll_max_bytes = (size_t)ll;
  long long spin = env_ll("AR_LL_SPIN_LIMIT", (long long)kDefaultSpinLimit);
  c->spin_limit = (uint32_t)std::min<long long>(std::max<long long>(spin, 1), 0xffffffffll);
  c->debug = (int)env_ll("AR_DEBUG", 0);
  {
    const char* k = std::getenv("AR_CAPPED_KERNEL");
    c->capped_tma = (k && std::strcmp(k, "tma") == 0) ? 1 : 0;
  }

  c->stage_stride = (c->ll_capacity_bytes + 3) / 4 + 4;
  const size_t stage_bytes = (size_t)nranks * c->stage_stride * sizeof(unsigned long long);
  long long ll128 = env_ll("AR_LL128_MAX_BYTES", (long long)kDefaultLL128Bytes);
  if (ll128 < 16) ll128 = 16;
  if (ll128 > (long long)kMaxLL128Bytes) ll128 = (long long)kMaxLL128Bytes;
  c->ll128_capacity_bytes = (size_t)ll128;
  c->ll128_max_bytes = (size_t)ll128;
  c->ll128_stride = ar::ll128_stage_words(c->ll128_capacity_bytes);
  const size_t stage128_bytes = (size_t)nranks * c->ll128_stride * sizeof(unsigned long long);
  std::vector<int16_t> push;
  for (int t = 0; t < 2; ++t) emit_preorder(ar::tree_root(nranks), nranks, t, push);
  if (push.size() != 2 * (size_t)nranks) {  // every rank once per tree
    delete c;
    return AR_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaMalloc(&c->staging, stage_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&c->staging128, stage128_bytes);
  if (e == cudaSuccess) e = cudaMemset(c->staging128, 0, stage128_bytes);
  if (e == cudaSuccess) e = cudaMalloc(&c->status, kControlInts * sizeof(int));
  if (e == cudaSuccess) e = cudaMalloc(&c->tree_push, push.size() * sizeof(int16_t));
  if (e == cudaSuccess) e = cudaMemset(c->staging, 0, stage_bytes);
  if (e == cudaSuccess) e = cudaMemset(c->status, 0, kControlInts * sizeof(int));
  if (e == cudaSuccess)
    e = cudaMemcpy(c->tree_push, push.data(), push.size() * sizeof(int16_t), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) {
    cudaGetLastError();
    release(c);
    return e == cudaErrorMemoryAllocation ? AR_ERR_OOM : AR_ERR_CUDA;
  }
  *out = c;
  return AR_SUCCESS;
}

ar_status_t ar_destroy(ar_comm_t c) {
  if (!c) return AR_SUCCESS;
  cudaError_t e = cudaDeviceSynchronize();
  release(c);
  return e == cudaSuccess ? AR_SUCCESS : AR_ERR_CUDA;
}

ar_status_t ar_get_status(ar_comm_t c) {
  if (!c) return AR_ERR_INVALID_ARG;
  int h = 0;
  if (cudaMemcpy(&h, c->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess ||
      cudaMemset(c->status, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return (ar_status_t)h;
}

ar_status_t ar_select_algo(ar_comm_t c, size_t count, ar_dtype_t dtype, ar_algo_t algo,
                           ar_algo_t* chosen) {
  if (!c || !chosen || !valid_dtype(dtype) || !valid_algo(algo)) return AR_ERR_INVALID_ARG;
  *chosen = resolve(c, count, dtype, algo);
  return AR_SUCCESS;
}

ar_status_t ar_set_option(ar_comm_t c, ar_option_t option, long long value) {
  if (!c) return AR_ERR_INVALID_ARG;
  switch (option) {
    case AR_OPT_LL_MAX_BYTES:
      if (value < 16 || (size_t)value > c->ll_capacity_bytes) return AR_ERR_INVALID_ARG;
      c->ll_max_bytes = (size_t)value;
      return AR_SUCCESS;
    case AR_OPT_LL_SPIN_LIMIT:
      if (value < 1 || value > 0xffffffffll) return AR_ERR_INVALID_ARG;
      c->spin_limit = (uint32_t)value;
      return AR_SUCCESS;
    case AR_OPT_DEBUG:
      c->debug = value != 0;
      return AR_SUCCESS;
    case AR_OPT_LL_SKIP_PRODUCER:
      c->skip_produce = value != 0;
      return AR_SUCCESS;
    case AR_OPT_LL128_MAX_BYTES:
      if (value < 16 || (size_t)value > c->ll128_capacity_bytes) return AR_ERR_INVALID_ARG;
      c->ll128_max_bytes = (size_t)value;
      return AR_SUCCESS;
    case AR_OPT_AUTO_TUNED:
      if (value != 0 && !c->tuned_valid) return AR_ERR_INVALID_ARG;  // run ar_tune first
      c->auto_tuned = value != 0;
      return AR_SUCCESS;
    case AR_OPT_MAX_BLOCKS:
      if (value < 0 || value > 0x7fffffffll) return AR_ERR_INVALID_ARG;
      c->max_blocks = (int)value;
      return AR_SUCCESS;
    case AR_OPT_CAPPED_KERNEL:
      if (value != AR_CAPPED_WIDE && value != AR_CAPPED_TMA) return AR_ERR_INVALID_ARG;
      c->capped_tma = value == AR_CAPPED_TMA;
      return AR_SUCCESS;
    case AR_OPT_HIER_GROUP:
      if (value < 1 || value > c->P || c->P % value != 0) return AR_ERR_INVALID_ARG;
      c->hier_group = (int)value;
      return AR_SUCCESS;
    case AR_OPT_LL_EPOCH: {
      if (value < 0 || value >= 0xffffffffll) return AR_ERR_INVALID_ARG;  // see ll_epoch_begin
      const unsigned int st[2] = {(unsigned int)value, 0u};
      if (cudaMemcpy(c->status + kLLEpoch, st, sizeof(st), cudaMemcpyHostToDevice) != cudaSuccess ||
          cudaMemcpy(c->status + kLL128Epoch, st, sizeof(st), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaGetLastError();
        return AR_ERR_CUDA;
      }
      return AR_SUCCESS;
    }
    default:
      return AR_ERR_INVALID_ARG;
  }
}

ar_status_t ar_allreduce(ar_comm_t c, const void* const* sendbufs, void* const* recvbufs,
                         size_t count, ar_dtype_t dtype, ar_op_t op, ar_algo_t algo, float scale,
                         void* stream) {
  if (!c || !valid_dtype(dtype) || !valid_op(op) || !valid_algo(algo)) return AR_ERR_INVALID_ARG;
  if (scale != 1.0f && (dtype == AR_INT32 || op != AR_SUM)) return AR_ERR_UNSUPPORTED;
  if (!(scale == scale)) return AR_ERR_INVALID_ARG;  // NaN scale
  if (count == 0) return AR_SUCCESS;
  if (!sendbufs || !recvbufs) return AR_ERR_INVALID_ARG;
  const size_t esize = ar::elem_bytes(dtype);
  if (count > ((size_t)1 << 62) / esize) return AR_ERR_INVALID_ARG;
  const int P = c->P;
  for (int r = 0; r < P; ++r) {
    if (!sendbufs[r] || !recvbufs[r]) return AR_ERR_INVALID_ARG;
    if (((uintptr_t)sendbufs[r] | (uintptr_t)recvbufs[r]) & 15u) return AR_ERR_INVALID_ARG;
  }
  if (overlapping(sendbufs, recvbufs, P, count * esize)) return AR_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (dev != c->device) return AR_ERR_INVALID_ARG;

  ar_algo_t chosen = resolve(c, count, dtype, algo);
  if (chosen == AR_ALGO_LL && count * esize > c->ll_max_bytes) return AR_ERR_UNSUPPORTED;
  if (chosen == AR_ALGO_LL128 && count * esize > c->ll128_max_bytes) return AR_ERR_UNSUPPORTED;
  if (chosen == AR_ALGO_HIER && P % c->hier_group != 0) return AR_ERR_UNSUPPORTED;

  ar::Call call;
  call.P = P;
  call.send = sendbufs;
  call.recv = recvbufs;
  call.count = count;
  call.dtype = dtype;
  call.op = op;
  call.algo = chosen == AR_ALGO_TREE ? ar::kTree : chosen == AR_ALGO_HIER ? ar::kHier : ar::kRing;
  call.group = c->hier_group;
  call.max_blocks = c->max_blocks;
  call.scale = scale;
  call.stream = static_cast<cudaStream_t>(stream);
  call.sms = c->sms;
  call.tree_push = c->tree_push;
  call.staging = c->staging;
  call.stage_stride = c->stage_stride;
  call.status = c->status;
  call.spin_limit = c->spin_limit;
  call.skip_produce = c->skip_produce;
  call.epoch_state = nullptr;
  call.stage_words = 0;
  call.shard = 0;

  Range range(allreduce_range(chosen));
  ar::LaunchInfo info;
  cudaError_t e;
  if (chosen == AR_ALGO_LL) {
    call.epoch_state = reinterpret_cast<unsigned int*>(c->status + kLLEpoch);
    call.stage_words = (size_t)P * c->stage_stride;
    e = ar::launch_ll(call, &info);
  } else if (chosen == AR_ALGO_LL128) {
    call.staging = c->staging128;
    call.stage_stride = c->ll128_stride;
    call.epoch_state = reinterpret_cast<unsigned int*>(c->status + kLL128Epoch);
    call.stage_words = (size_t)P * c->ll128_stride;
    e = ar::launch_ll128(call, &info);
  } else if (chosen == AR_ALGO_HIER) {
    e = ar::launch_generic(call, &info);
  } else if (P <= ar::kMaxStaticRanks && c->max_blocks > 0 && c->max_blocks < c->sms && !c->capped_tma) {
    // capped to fewer SMs than the GPU has: 1024-thread blocks, one per SM,
    // keep twice the bytes in flight per SM of the 256-thread shape
    e = dtype == AR_FLOAT32    ? ar::launch_wide_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_wide_bf16(call, &info)
                               : ar::launch_wide_i32(call, &info);
  } else if (P <= ar::kMaxStaticRanks && c->max_blocks > 0 && c->max_blocks < c->sms &&
             count * esize / ar::kTmaTileBytes >= (size_t)c->max_blocks) {
    // (AR_CAPPED_KERNEL=tma) capped, with at least a tile per block: the TMA pipeline
    e = dtype == AR_FLOAT32    ? ar::launch_tma_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_tma_bf16(call, &info)
                               : ar::launch_tma_i32(call, &info);
  } else if (P <= ar::kMaxStaticRanks) {
    e = dtype == AR_FLOAT32    ? ar::launch_static_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_static_bf16(call, &info)
                               : ar::launch_static_i32(call, &info);
  } else {
    e = ar::launch_generic(call, &info);
  }
  if (c->debug) {
    std::fprintf(stderr,
                 "[ar] P=%d count=%zu dtype=%s op=%s algo=%s->%s kernel=%s grid=%d block=%d "
                 "smem=%zu bytes/rank=%zu status=%s\n",
                 P, count, dtype_name(dtype), op_name(op), algo_name(algo), algo_name(chosen),
                 info.kernel, info.grid, info.block, info.smem, count * esize,
                 cudaGetErrorString(e));
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return AR_SUCCESS;
}

ar_status_t ar_reduce_scatter(ar_comm_t c, const void* const* sendbufs, void* const* recvbufs,
                              size_t recvcount, ar_dtype_t dtype, ar_op_t op, float scale,
                              void* stream) {
  if (!c || !valid_op(op)) return AR_ERR_INVALID_ARG;
  if (!(scale == scale)) return AR_ERR_INVALID_ARG;
  if (scale != 1.0f && (dtype == AR_INT32 || op != AR_SUM)) return AR_ERR_UNSUPPORTED;
  bool vec = false;
  ar_status_t st = check_collective(c, sendbufs, (const void* const*)recvbufs, dtype, recvcount, &vec);
  if (st != AR_SUCCESS || recvcount == 0) return st;
  ar::Call call = base_call(c, stream);
  call.send = sendbufs;
  call.recv = recvbufs;
  call.count = (size_t)c->P * recvcount;
  call.shard = recvcount;
  call.dtype = dtype;
  call.op = op;
  call.scale = scale;
  Range range("ar_reduce_scatter");
  ar::LaunchInfo info;
  cudaError_t e;
  if (!vec) {
    e = ar::launch_reduce_scatter_elem(call, &info);
  } else if (c->P <= ar::kMaxStaticRanks && c->max_blocks > 0 && c->max_blocks < c->sms && !c->capped_tma) {
    // capped to fewer SMs than the GPU has: the wide shape, shard-owner stores
    e = dtype == AR_FLOAT32    ? ar::launch_wide_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_wide_bf16(call, &info)
                               : ar::launch_wide_i32(call, &info);
  } else if (c->P <= ar::kMaxStaticRanks && c->max_blocks > 0 && c->max_blocks < c->sms &&
             call.count * ar::elem_bytes(dtype) / ar::kTmaTileBytes >= (size_t)c->max_blocks) {
    // (AR_CAPPED_KERNEL=tma) the TMA pipeline, shard-owner stores
    e = dtype == AR_FLOAT32    ? ar::launch_tma_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_tma_bf16(call, &info)
                               : ar::launch_tma_i32(call, &info);
  } else if (c->P <= ar::kMaxStaticRanks) {  // rank-specialised, shard-owner stores
    e = dtype == AR_FLOAT32    ? ar::launch_static_f32(call, &info)
        : dtype == AR_BFLOAT16 ? ar::launch_static_bf16(call, &info)
                               : ar::launch_static_i32(call, &info);
  } else {
    e = ar::launch_reduce_scatter_vec(call, &info);
  }
  if (c->debug)
    std::fprintf(stderr, "[ar] reduce_scatter P=%d recvcount=%zu dtype=%s op=%s kernel=%s grid=%d status=%s\n",
                 c->P, recvcount, dtype_name(dtype), op_name(op), info.kernel, info.grid,
                 cudaGetErrorString(e));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return AR_SUCCESS;
}

ar_status_t ar_all_gather(ar_comm_t c, const void* const* sendbufs, void* const* recvbufs,
                          size_t sendcount, ar_dtype_t dtype, void* stream) {
  if (!c) return AR_ERR_INVALID_ARG;
  bool vec = false;
  ar_status_t st = check_collective(c, (const void* const*)recvbufs, sendbufs, dtype, sendcount, &vec);
  if (st != AR_SUCCESS || sendcount == 0) return st;
  ar::Call call = base_call(c, stream);
  call.send = sendbufs;
  call.recv = recvbufs;
  call.count = (size_t)c->P * sendcount;
  call.shard = sendcount;
  call.dtype = dtype;
  call.algo = vec ? 1 : 0;  // 1: 16-byte vector copy
  Range range("ar_all_gather");
  ar::LaunchInfo info;
  cudaError_t e;
  if (vec && c->max_blocks > 0 && c->max_blocks < c->sms &&
      call.count * ar::elem_bytes(dtype) / ar::kTmaGatherTileBytes >= (size_t)c->max_blocks) {
    // capped to fewer SMs than the GPU has, with at least a tile per block
    e = ar::launch_all_gather_tma(call, &info);
  } else {
    e = ar::launch_all_gather(call, &info);
  }
  if (c->debug)
    std::fprintf(stderr, "[ar] all_gather P=%d sendcount=%zu dtype=%s kernel=%s grid=%d status=%s\n",
                 c->P, sendcount, dtype_name(dtype), info.kernel, info.grid, cudaGetErrorString(e));
  if (e != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  return AR_SUCCESS;
}

ar_status_t ar_tune(ar_comm_t c, ar_algo_t* table, int table_len) {
  if (!c || table_len < 0 || (table_len > 0 && !table)) return AR_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return AR_ERR_CUDA;
  }
  if (dev != c->device) return AR_ERR_INVALID_ARG;
  const int P = c->P;
  const size_t top = (size_t)8 << (AR_TUNE_BUCKETS - 1);  // largest tuned size per rank
  std::vector<void*> bufs(2 * (size_t)P, nullptr);
  cudaStream_t s = nullptr;
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  ar_status_t st = AR_SUCCESS;
  cudaError_t e = cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreate(&e0);
  if (e == cudaSuccess) e = cudaEventCreate(&e1);
  for (size_t i = 0; e == cudaSuccess && i < bufs.size(); ++i) {
    e = cudaMalloc(&bufs[i], top);
    if (e == cudaSuccess) e = cudaMemset(bufs[i], 0, top);
  }
  const int saved_auto = c->auto_tuned;
  c->auto_tuned = 0;
  ar_algo_t result[AR_TUNE_BUCKETS];
  const ar_algo_t candidates[] = {AR_ALGO_RING, AR_ALGO_TREE, AR_ALGO_LL, AR_ALGO_LL128};
  constexpr int kReps = 20;
  for (int b = 0; e == cudaSuccess && st == AR_SUCCESS && b < AR_TUNE_BUCKETS; ++b) {
    const size_t count = ((size_t)8 << b) / 4;  // fp32 elements per rank
    float best = 0.f;
    result[b] = AR_ALGO_RING;
    for (ar_algo_t a : candidates) {
      if (a == AR_ALGO_LL && count * 4 > c->ll_max_bytes) continue;
      if (a == AR_ALGO_LL128 && count * 4 > c->ll128_max_bytes) continue;
      for (int k = 0; k < 2 && st == AR_SUCCESS; ++k)
        st = ar_allreduce(c, bufs.data(), bufs.data() + P, count, AR_FLOAT32, AR_SUM, a, 1.0f, s);
      if (st == AR_SUCCESS) e = cudaEventRecord(e0, s);
      for (int k = 0; k < kReps && st == AR_SUCCESS && e == cudaSuccess; ++k)
        st = ar_allreduce(c, bufs.data(), bufs.data() + P, count, AR_FLOAT32, AR_SUM, a, 1.0f, s);
      if (st != AR_SUCCESS || e != cudaSuccess) break;
      e = cudaEventRecord(e1, s);
      if (e == cudaSuccess) e = cudaEventSynchronize(e1);
      float ms = 0.f;
      if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, e0, e1);
      if (e != cudaSuccess) break;
      if (best == 0.f || ms < best) {
        best = ms;
        result[b] = a;
      }
    }
  }
  if (e == cudaSuccess && st == AR_SUCCESS) {
    ar_status_t dst = ar_get_status(c);  // a timed-out LL wait would void the timings
    if (dst != AR_SUCCESS) st = dst;
  }
  for (void* p : bufs)
    if (p) cudaFree(p);
  if (e0) cudaEventDestroy(e0);
  if (e1) cudaEventDestroy(e1);
  if (s) cudaStreamDestroy(s);
  if (e != cudaSuccess) {
    cudaGetLastError();
    st = e == cudaErrorMemoryAllocation ? AR_ERR_OOM : AR_ERR_CUDA;
  }
  if (st != AR_SUCCESS) {
    c->auto_tuned = saved_auto;
    return st;
  }
  for (int b = 0; b < AR_TUNE_BUCKETS; ++b) c->tuned[b] = result[b];
  for (int b = 0; b < table_len && b < AR_TUNE_BUCKETS; ++b) table[b] = result[b];
  c->tuned_valid = 1;
  c->auto_tuned = 1;
  if (c->debug) {
    std::fprintf(stderr, "[ar] tune P=%d:", P);
    for (int b = 0; b < AR_TUNE_BUCKETS; ++b) std::fprintf(stderr, " %zuB=%s", (size_t)8 << b, algo_name(result[b]));
    std::fprintf(stderr, "\n");
  }
  return AR_SUCCESS;
}

}  // extern "C"
