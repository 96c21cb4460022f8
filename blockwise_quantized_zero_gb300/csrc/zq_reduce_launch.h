// zq_reduce_launch.h -- grid sizing and format dispatch of the reduce
// kernels, shared by the launch units that instantiate them for two CTAs an
// SM (zq_reduce.cu) and for three (zq_reduce_few.cu, launches of at most
// kFewShards shards).
#pragma once

#include "zq_host.h"

namespace zq {

// Elements of all the problems of one launch.
static inline int64_t launch_elements(const ReduceArgs &a) { return a.n; }
static inline int64_t launch_elements(const TableReduceArgs &a) { return a.n; }
static inline int64_t launch_elements(const HopArgs &a) {
  return ((a.n + kTile * kRedConsumers - 1) / (kTile * kRedConsumers)) * kTile * kRedConsumers *
         a.nprob;
}

// Persistent grid of CTAs of eight consumer warps and one producer warp: one
// CTA per CTA tile (8192 elements), at most one wave.
template <int OCC, int FIN, int FOUT, typename A>
static cudaError_t go_r(const A &a, cudaStream_t st) {
  constexpr auto K = reduce_kernel<FIN, FOUT, A, OCC>;
  constexpr int kSmem = RedGeom<FIN, OCC>::kSmem;
  const int occ = ctas_per_sm<K, kSmem, kRedThreads>();
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int64_t span = int64_t(kRedConsumers) * kTile;
  const int64_t ctas = (launch_elements(a) + span - 1) / span;
  const int64_t cap = int64_t(device_sm_count()) * occ;
  const unsigned grid = static_cast<unsigned>(ctas < 1 ? 1 : (ctas < cap ? ctas : cap));
  return launch_pdl_threads(K, grid, kRedThreads, kSmem, st, a);
}

template <int OCC, int FIN, typename A>
static cudaError_t go_r_o(const A &a, int fout, cudaStream_t st) {
  switch (fout) {
    case F_INT2: return go_r<OCC, FIN, F_INT2>(a, st);
    case F_INT4: return go_r<OCC, FIN, F_INT4>(a, st);
    case F_INT6: return go_r<OCC, FIN, F_INT6>(a, st);
    case F_INT8: return go_r<OCC, FIN, F_INT8>(a, st);
    case F_E4M3: return go_r<OCC, FIN, F_E4M3>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int OCC, typename A>
static cudaError_t go_r_io(const A &a, int fin, int fout, cudaStream_t st) {
  switch (fin) {
    case F_INT2: return go_r_o<OCC, F_INT2>(a, fout, st);
    case F_INT4: return go_r_o<OCC, F_INT4>(a, fout, st);
    case F_INT6: return go_r_o<OCC, F_INT6>(a, fout, st);
    case F_INT8: return go_r_o<OCC, F_INT8>(a, fout, st);
    case F_E4M3: return go_r_o<OCC, F_E4M3>(a, fout, st);
    default: return cudaErrorInvalidValue;
  }
}

// Read and clear the device error word of the including launch unit.
static inline unsigned take_unit_error_word() {
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
