// ar_tma_gather.cu -- the all-gather ("NCCL, NIXL, and Distributed GPU
// Communication", section "All-gather") as a TMA bulk-copy pipeline, for calls
// capped to fewer SMs than the GPU has (AR_OPT_MAX_BLOCKS), any rank count.
//
// An all-gather has nothing to fold, so one thread per block drives it: for
// each tile of a source shard it waits for the tile's bulk load into a
// shared-memory stage (mbarrier, bounded), bulk-stores it to all P receive
// buffers (one bulk group per tile), then refills the stage freed one tile
// earlier -- once that tile's stores have read it -- with the tile kStages - 1
// ahead.  One block per SM (its stages take most of the shared memory).  On a
// wait limit the thread records AR_ERR_TIMEOUT, waits (bounded) for the loads
// it issued and for its stores, and leaves, so no copy is in flight into or
// out of shared memory when the block exits.
#include "ar_tma.cuh"

namespace ar {

namespace {

constexpr int kGatherTile = (int)kTmaGatherTileBytes;  // bytes per stage (one shard's tile)
constexpr int kGatherStages = 6;
constexpr size_t kGatherSmem = (size_t)kGatherTile * kGatherStages;

struct GatherParams {
  const char* send[AR_MAX_RANKS];
  char* recv[AR_MAX_RANKS];
  int P;
  uint64_t shard;            // bytes per shard (a multiple of 16)
  uint64_t tiles_per_shard;  // ceil(shard / kGatherTile)
  int* status;
  uint32_t spin_limit;
  int skip_produce;          // test hook: no loads are issued, so every wait runs out
};

__global__ void __launch_bounds__(32, 1) all_gather_tma_kernel(const __grid_constant__ GatherParams p) {
  pdl_enter();
  extern __shared__ __align__(128) char smem[];
  __shared__ __align__(8) uint64_t full[kGatherStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kGatherStages; ++s) tma::mbar_init(&full[s], 1);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const uint64_t ntiles = (uint64_t)p.P * p.tiles_per_shard;
  const uint64_t mine = ntiles > blockIdx.x ? (ntiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  auto load = [&](uint64_t j) -> bool {  // tile j of this block into stage j % kGatherStages
    if (j >= mine || p.skip_produce) return false;
    const uint64_t t = blockIdx.x + j * gridDim.x;
    const int s = (int)(t / p.tiles_per_shard);
    const uint64_t off = (t - (uint64_t)s * p.tiles_per_shard) * kGatherTile;
    const uint32_t len = (uint32_t)(p.shard - off < (uint64_t)kGatherTile ? p.shard - off : (uint64_t)kGatherTile);
    uint64_t* bar = &full[j % kGatherStages];
    tma::mbar_expect_tx(bar, len);
    tma::bulk_load(smem + (size_t)(j % kGatherStages) * kGatherTile, p.send[s] + off, len, bar);
    return true;
  };
  uint64_t issued = 0;  // loads of tiles [0, issued) were issued
  for (uint64_t j = 0; j + 1 < kGatherStages; ++j)
    if (load(j)) issued = j + 1;
  uint64_t j = 0;
  for (; j < mine; ++j) {
    if (!tma::mbar_wait(&full[j % kGatherStages], (uint32_t)((j / kGatherStages) & 1), p.spin_limit)) {
      atomicExch(p.status, (int)AR_ERR_TIMEOUT);
      break;
    }
    const uint64_t t = blockIdx.x + j * gridDim.x;
    const int s = (int)(t / p.tiles_per_shard);
    const uint64_t off = (t - (uint64_t)s * p.tiles_per_shard) * kGatherTile;
    const uint32_t len = (uint32_t)(p.shard - off < (uint64_t)kGatherTile ? p.shard - off : (uint64_t)kGatherTile);
    const char* src = smem + (size_t)(j % kGatherStages) * kGatherTile;
    const uint64_t dst = (uint64_t)s * p.shard + off;
    for (int r = 0; r < p.P; ++r) tma::bulk_store(p.recv[r] + dst, src, len);
    tma::bulk_commit();
    // the stage of tile j - 1 is refilled with tile j + kGatherStages - 1
    // once its stores have read it
    tma::bulk_wait_read<1>();
    if (load(j + kGatherStages - 1)) issued = j + kGatherStages;
  }
  tma::bulk_wait_all();
  // after a timeout at tile j, loads issued for tiles [j, issued) -- at most
  // one per stage -- may still be landing
  for (uint64_t k = j; k < issued; ++k)
    tma::mbar_wait(&full[k % kGatherStages], (uint32_t)((k / kGatherStages) & 1), p.spin_limit);
}

}  // namespace

cudaError_t launch_all_gather_tma(const Call& c, LaunchInfo* info) {
  GatherParams p;
  for (int r = 0; r < c.P; ++r) {
    p.send[r] = static_cast<const char*>(c.send[r]);
    p.recv[r] = static_cast<char*>(c.recv[r]);
  }
  const size_t es = elem_bytes(c.dtype);
  p.P = c.P;
  p.shard = (uint64_t)c.shard * es;
  if (p.shard % 16 != 0) return cudaErrorInvalidValue;
  p.tiles_per_shard = (p.shard + kGatherTile - 1) / kGatherTile;
  p.status = c.status;
  p.spin_limit = c.spin_limit;
  p.skip_produce = c.skip_produce;
  static std::atomic<uint64_t> configured{0};  // the shared-memory opt-in is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || !(configured.load(std::memory_order_acquire) & bit)) {
    e = cudaFuncSetAttribute(all_gather_tma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGatherSmem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const uint64_t ntiles = (uint64_t)c.P * p.tiles_per_shard;
  uint64_t grid = (uint64_t)(c.max_blocks > 0 ? c.max_blocks : c.sms);
  if (grid > (uint64_t)c.sms) grid = (uint64_t)c.sms;
  if (grid > ntiles) grid = ntiles;
  if (grid < 1) grid = 1;
  (void)launch_kernel(all_gather_tma_kernel, dim3((unsigned)grid), dim3(32), kGatherSmem, c.stream, use_pdl(c), p);
  info->kernel = "tma_all_gather";
  info->grid = (int)grid;
  info->block = 32;
  info->smem = kGatherSmem;
  return cudaGetLastError();
}

}  // namespace ar
