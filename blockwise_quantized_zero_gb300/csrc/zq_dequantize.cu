// zq_dequantize.cu -- launch unit for the dequantize kernels.
#include "zq_host.h"

namespace zq {

template <int FMT, int DT>
static cudaError_t go_d(const void *codes, const float *scales, int64_t n, int64_t G, void *dst,
                        cudaStream_t st, bool wide) {
  constexpr auto K = dequantize_kernel<FMT, DT>;
  return launch_pdl(K, grid_for<K>(n), 0, st, static_cast<const uint8_t *>(codes), scales, dst, n,
                    log2_block(G), wide ? 1 : 0);
}

template <int FMT>
static cudaError_t go_d_t(const void *codes, const float *scales, int64_t n, int64_t G, void *dst,
                          int dt, cudaStream_t st, bool wide) {
  switch (dt) {
    case DT_F32: return go_d<FMT, DT_F32>(codes, scales, n, G, dst, st, wide);
    case DT_F16: return go_d<FMT, DT_F16>(codes, scales, n, G, dst, st, wide);
    case DT_BF16: return go_d<FMT, DT_BF16>(codes, scales, n, G, dst, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dequantize(const void *codes, const float *scales, int64_t n, int fmt,
                              int64_t G, void *dst, int dt, cudaStream_t st, bool wide) {
  switch (fmt) {
    case F_INT2: return go_d_t<F_INT2>(codes, scales, n, G, dst, dt, st, wide);
    case F_INT4: return go_d_t<F_INT4>(codes, scales, n, G, dst, dt, st, wide);
    case F_INT6: return go_d_t<F_INT6>(codes, scales, n, G, dst, dt, st, wide);
    case F_INT8: return go_d_t<F_INT8>(codes, scales, n, G, dst, dt, st, wide);
    case F_E4M3: return go_d_t<F_E4M3>(codes, scales, n, G, dst, dt, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
