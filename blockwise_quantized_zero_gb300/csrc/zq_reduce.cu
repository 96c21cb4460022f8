// zq_reduce.cu -- launch unit for the quantized-reduce kernels (one
// instantiation per input and output code format).
#include "zq_host.h"

namespace zq {

template <int FIN, int FOUT, int KU> static cudaError_t go_r_u(const ReduceArgs &a, cudaStream_t st) {
  constexpr auto K = reduce_kernel<FIN, FOUT, KU>;
  // grid_for counts 1024-element tiles; a KU = 1 tile is half of one
  return launch_pdl(K, grid_for<K>(a.n * (2 / KU)), st, a);
}

template <int FIN, int FOUT> static cudaError_t go_r(const ReduceArgs &a, cudaStream_t st) {
  return go_r_u<FIN, FOUT, 2>(a, st);
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

}  // namespace zq
