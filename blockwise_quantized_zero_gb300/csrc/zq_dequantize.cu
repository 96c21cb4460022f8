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

template <int FMT, int DT>
static cudaError_t go_dm(const DequantMultiArgs &a, cudaStream_t st) {
  constexpr auto K = dequantize_multi_kernel<FMT, DT>;
  const int64_t full = a.tile0[a.count];
  int64_t need = (full + kWarps - 1) / kWarps;
  const int64_t tails = (a.count + kWarps - 1) / kWarps;
  if (need < tails) need = tails;
  const int64_t cap = int64_t(device_sm_count()) * ctas_per_sm<K>();
  const unsigned grid = unsigned(need < 1 ? 1 : (need < cap ? need : cap));
  return launch_pdl(K, grid, 0, st, a);
}

template <int FMT>
static cudaError_t go_dm_t(const DequantMultiArgs &a, int dt, cudaStream_t st) {
  switch (dt) {
    case DT_F32: return go_dm<FMT, DT_F32>(a, st);
    case DT_F16: return go_dm<FMT, DT_F16>(a, st);
    case DT_BF16: return go_dm<FMT, DT_BF16>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dequantize_multi(const DequantMultiArgs &a, int fmt, int dt, cudaStream_t st) {
  switch (fmt) {
    case F_INT2: return go_dm_t<F_INT2>(a, dt, st);
    case F_INT4: return go_dm_t<F_INT4>(a, dt, st);
    case F_INT6: return go_dm_t<F_INT6>(a, dt, st);
    case F_INT8: return go_dm_t<F_INT8>(a, dt, st);
    case F_E4M3: return go_dm_t<F_E4M3>(a, dt, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
