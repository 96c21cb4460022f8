// zq_reduce.cu -- launch unit for the quantized-reduce kernels (one
// instantiation per input and output code format), and the reader of the
// reduce kernels' device error word.
#include "zq_host.h"

namespace zq {

// Persistent grid of CTAs of eight consumer warps and one producer warp: one
// CTA per CTA tile (8192 elements), at most one wave.
template <int FIN, int FOUT> static cudaError_t go_r(const ReduceArgs &a, cudaStream_t st) {
  constexpr auto K = reduce_kernel<FIN, FOUT>;
  constexpr int kSmem = RedGeom<FIN>::kSmem;
  const int occ = ctas_per_sm<K, kSmem, kRedThreads>();
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t span = int64_t(kRedConsumers) * kTile;
  const int64_t ctas = (a.n + span - 1) / span;
  const int64_t cap = int64_t(device_sm_count()) * occ;
  const unsigned grid = static_cast<unsigned>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
  return launch_pdl_threads(K, grid, kRedThreads, kSmem, st, a);
}

template <int FIN> static cudaError_t go_r_o(const ReduceArgs &a, int fout, cudaStream_t st) {
  switch (fout) {
    case F_INT2: return go_r<FIN, F_INT2>(a, st);
    case F_INT4: return go_r<FIN, F_INT4>(a, st);
    case F_INT6: return go_r<FIN, F_INT6>(a, st);
    case F_INT8: return go_r<FIN, F_INT8>(a, st);
    case F_E4M3: return go_r<FIN, F_E4M3>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_reduce(const ReduceArgs &a, int fin, int fout, cudaStream_t st) {
  switch (fin) {
    case F_INT2: return go_r_o<F_INT2>(a, fout, st);
    case F_INT4: return go_r_o<F_INT4>(a, fout, st);
    case F_INT6: return go_r_o<F_INT6>(a, fout, st);
    case F_INT8: return go_r_o<F_INT8>(a, fout, st);
    case F_E4M3: return go_r_o<F_E4M3>(a, fout, st);
    default: return cudaErrorInvalidValue;
  }
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
