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
// stand-in: the kernels get the device address, looked up once per device
// with cudaGetSymbolAddress while that device is current (on the device's
// first call). Every call overwrites the first nshards entries of both lists
// with stream-ordered copies, and the kernel reads no other entry, so nothing
// needs clearing. All calls share the table: calls whose work overlaps on the
// GPU (different streams, not ordered) race on it.
// ---------------------------------------------------------------------------
static __device__ __align__(256) ShardTable g_shard_table;

namespace {
constexpr int kMaxTableDevices = 64;
ShardTable *g_table_ptr[kMaxTableDevices] = {nullptr};
std::mutex g_table_mutex;

cudaError_t table_address(ShardTable **out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxTableDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_table_mutex);
  if (!g_table_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_shard_table);
    if (e != cudaSuccess) return e;
    g_table_ptr[dev] = static_cast<ShardTable *>(p);
  }
  *out = g_table_ptr[dev];
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

unsigned take_reduce_device_error() {
  return take_unit_error_word() | take_reduce_few_device_error();
}

}  // namespace zq
