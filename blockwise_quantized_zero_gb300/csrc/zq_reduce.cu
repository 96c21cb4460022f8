// zq_reduce.cu -- launch unit for the quantized-reduce kernels (one
// instantiation per input and output code format), and the reader of the
// reduce kernels' device error word.
#include <cstddef>
#include <mutex>

#include "zq_host.h"

namespace zq {

// Elements of all the problems of one launch.
static int64_t launch_elements(const ReduceArgs &a) { return a.n; }
static int64_t launch_elements(const TableReduceArgs &a) { return a.n; }
static int64_t launch_elements(const HopArgs &a) {
  return ((a.n + kTile * kRedConsumers - 1) / (kTile * kRedConsumers)) * kTile * kRedConsumers *
         a.nprob;
}

// Persistent grid of CTAs of eight consumer warps and one producer warp: one
// CTA per CTA tile (8192 elements), at most one wave.
template <int FIN, int FOUT, typename A> static cudaError_t go_r(const A &a, cudaStream_t st) {
  constexpr auto K = reduce_kernel<FIN, FOUT, A>;
  constexpr int kSmem = RedGeom<FIN>::kSmem;
  const int occ = ctas_per_sm<K, kSmem, kRedThreads>();
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t span = int64_t(kRedConsumers) * kTile;
  const int64_t ctas = (launch_elements(a) + span - 1) / span;
  const int64_t cap = int64_t(device_sm_count()) * occ;
  const unsigned grid = static_cast<unsigned>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
  return launch_pdl_threads(K, grid, kRedThreads, kSmem, st, a);
}

template <int FIN, typename A> static cudaError_t go_r_o(const A &a, int fout, cudaStream_t st) {
  switch (fout) {
    case F_INT2: return go_r<FIN, F_INT2>(a, st);
    case F_INT4: return go_r<FIN, F_INT4>(a, st);
    case F_INT6: return go_r<FIN, F_INT6>(a, st);
    case F_INT8: return go_r<FIN, F_INT8>(a, st);
    case F_E4M3: return go_r<FIN, F_E4M3>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <typename A> static cudaError_t go_r_io(const A &a, int fin, int fout, cudaStream_t st) {
  switch (fin) {
    case F_INT2: return go_r_o<F_INT2>(a, fout, st);
    case F_INT4: return go_r_o<F_INT4>(a, fout, st);
    case F_INT6: return go_r_o<F_INT6>(a, fout, st);
    case F_INT8: return go_r_o<F_INT8>(a, fout, st);
    case F_E4M3: return go_r_o<F_E4M3>(a, fout, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce(const ReduceArgs &a, int fin, int fout, cudaStream_t st) {
  return go_r_io(a, fin, fout, st);
}

cudaError_t launch_reduce_hop(const HopArgs &a, int fin, int fout, cudaStream_t st) {
  return go_r_io(a, fin, fout, st);
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
  return go_r_io(a, fin, fout, st);
}

unsigned take_reduce_device_error() {
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof v) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  if (v != 0) {
    const unsigned zero = 0;
    (void)cudaMemcpyToSymbol(g_dev_error, &zero, sizeof zero);
  }
  return v;
}

}  // namespace zq
