// zq_reduce.cu -- launch unit for the quantized-reduce kernels built for two
// CTAs an SM (one instantiation per input and output code format), the
// allocation-free variant's shard table, and the reader of the reduce
// kernels' device error words. Launches of at most kFewShards shards go to
// the three-CTA instantiations of zq_reduce_few.cu.
#include <cstddef>
#include <mutex>

#include "zq_reduce_launch.h"

namespace zq {

cudaError_t launch_reduce(const ReduceArgs &a, int fin, int fout, cudaStream_t st) {
  if (a.nshards <= kFewShards) return launch_reduce_few(a, fin, fout, st);
  return go_r_io<2>(a, fin, fout, st);
}

cudaError_t launch_reduce_hop(const HopArgs &a, int fin, int fout, cudaStream_t st) {
  if (a.nshards <= kFewShards) return launch_reduce_hop_few(a, fin, fout, st);
  return go_r_io<2>(a, fin, fout, st);
}

// ---------------------------------------------------------------------------
// The allocation-free variant for many shards. The shard pointer table lives
// in this file-scope device array (16 KiB, held by every GPU that loads the
// library until the process exits). Its name in host code is only a host-side
// stand-in: the kernels get the device address, looked up with
// cudaGetSymbolAddress while the device is current, on the first call in each
// CUDA context (the address is cached per device together with the context it
// belongs to, so a new primary context after cudaDeviceReset is looked up
// again). Every call overwrites the first nshards entries of both lists with
// stream-ordered copies, and the kernel reads no other entry, so nothing
// needs clearing. All calls share the table: calls whose work overlaps on the
// GPU (different streams, not ordered) race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) ShardTable g_shard_table;

namespace {
constexpr int kMaxTableDevices = 64;
struct TableSlot {
  void *ctx;
  ShardTable *ptr;
};
TableSlot g_table[kMaxTableDevices] = {};
std::mutex g_table_mutex;

// The current CUDA context (driver handle), through the runtime's driver
// entry point (the library does not link the driver library itself).
void *current_context() {
  using GetCtx = int (*)(void **);
  static GetCtx fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<GetCtx>(p);
  }();
  void *ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

cudaError_t table_address(ShardTable **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxTableDevices) return cudaErrorInvalidDevice;
  void *ctx = current_context();
  std::lock_guard<std::mutex> lock(g_table_mutex);
  TableSlot &slot = g_table[dev];
  if (!slot.ptr || slot.ctx != ctx) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_shard_table);
    if (e != cudaSuccess) return e;
    slot.ptr = static_cast<ShardTable *>(p);
    slot.ctx = ctx;
  }
  *out = slot.ptr;
  return cudaSuccess;
}
}  // namespace

cudaError_t launch_reduce_static(const void *const *codes, const float *const *scales,
                                 const TableReduceArgs &args, int fin, int fout,
                                 cudaStream_t st) {
  if (args.nshards < 1 || args.nshards > kStaticMaxShards) return cudaErrorInvalidValue;
  ShardTable *tab = nullptr;
  cudaError_t e = table_address(&tab);
  if (e != cudaSuccess) return e;
  const size_t bytes = size_t(args.nshards) * sizeof(void *);
  char *base = reinterpret_cast<char *>(tab);  // device address: arithmetic only
  e = cudaMemcpyAsync(base + offsetof(ShardTable, codes), codes, bytes, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyAsync(base + offsetof(ShardTable, scales), scales, bytes, cudaMemcpyHostToDevice,
                      st);
  if (e != cudaSuccess) return e;
  TableReduceArgs a = args;
  a.tab = tab;
  return go_r_io<2>(a, fin, fout, st);
}

// ---------------------------------------------------------------------------
// Wait self-test: one CTA of two warps waits on an mbarrier that nothing
// arrives on, with the reduce kernels' bounded waits (warp 0 the consumers'
// warp-wide wait, lane 0 of warp 1 the producer's single-thread wait) and a
// short limit. Both waits run out, record the timeout in this unit's device
// error word (the one the reduce kernels of this unit use) and return.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(64) wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_addr(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_init_fence();
  }
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (w == 0) {
    if (!mbar_wait_warp(b, 0u, limit_ns) && lane == 0) atomicOr(&g_dev_error, kDevErrWaitTimeout);
  } else if (lane == 0) {
    if (!mbar_wait_thread(b, 0u, limit_ns)) atomicOr(&g_dev_error, kDevErrWaitTimeout);
  }
}

cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st) {
  wait_selftest_kernel<<<1, 64, 0, st>>>(limit_ns);
  return cudaGetLastError();
}

unsigned take_reduce_device_error() {
  return take_unit_error_word() | take_reduce_few_device_error();
}

}  // namespace zq
