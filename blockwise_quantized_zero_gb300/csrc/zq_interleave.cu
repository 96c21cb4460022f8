// zq_interleave.cu -- launch unit for the quantize and dequantize kernels in
// the metadata-interleaved record layout (integer codes; every element type
// and block size is a separate quantize instantiation, G is a run-time
// argument of dequantize).
#include "zq_host.h"

namespace zq {

template <int DT, int FMT, int G>
static cudaError_t go_qi(const void *src, int64_t n, void *rec, cudaStream_t st, bool wide) {
  constexpr auto K = quantize_kernel<DT, FMT, G, true>;
  return launch_pdl(K, grid_for<K>(n, kQuantizeTilesPerWarp), 0, st, src, static_cast<uint8_t *>(rec),
                    static_cast<float *>(nullptr), n, wide ? 1 : 0, SliceRemap{1, 1, 0});
}

template <int DT, int FMT>
static cudaError_t go_qi_g(const void *src, int64_t n, int64_t G, void *rec, cudaStream_t st,
                           bool wide) {
  switch (G) {
    case 32: return go_qi<DT, FMT, 32>(src, n, rec, st, wide);
    case 64: return go_qi<DT, FMT, 64>(src, n, rec, st, wide);
    case 128: return go_qi<DT, FMT, 128>(src, n, rec, st, wide);
    case 256: return go_qi<DT, FMT, 256>(src, n, rec, st, wide);
    case 512: return go_qi<DT, FMT, 512>(src, n, rec, st, wide);
    case 1024: return go_qi<DT, FMT, 1024>(src, n, rec, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT>
static cudaError_t go_qi_f(const void *src, int64_t n, int fmt, int64_t G, void *rec,
                           cudaStream_t st, bool wide) {
  switch (fmt) {
    case F_INT2: return go_qi_g<DT, F_INT2>(src, n, G, rec, st, wide);
    case F_INT4: return go_qi_g<DT, F_INT4>(src, n, G, rec, st, wide);
    case F_INT6: return go_qi_g<DT, F_INT6>(src, n, G, rec, st, wide);
    case F_INT8: return go_qi_g<DT, F_INT8>(src, n, G, rec, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize_interleaved(const void *src, int dt, int64_t n, int fmt, int64_t G,
                                        void *rec, cudaStream_t st, bool wide) {
  switch (dt) {
    case DT_F32: return go_qi_f<DT_F32>(src, n, fmt, G, rec, st, wide);
    case DT_F16: return go_qi_f<DT_F16>(src, n, fmt, G, rec, st, wide);
    case DT_BF16: return go_qi_f<DT_BF16>(src, n, fmt, G, rec, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

template <int FMT, int DT>
static cudaError_t go_di(const void *rec, int64_t n, int64_t G, void *dst, cudaStream_t st,
                         bool wide) {
  constexpr auto K = dequantize_kernel<FMT, DT, true>;
  return launch_pdl(K, grid_for<K>(n), 0, st, static_cast<const uint8_t *>(rec),
                    static_cast<const float *>(nullptr), dst, n, log2_block(G), wide ? 1 : 0);
}

template <int FMT>
static cudaError_t go_di_t(const void *rec, int64_t n, int64_t G, void *dst, int dt,
                           cudaStream_t st, bool wide) {
  switch (dt) {
    case DT_F32: return go_di<FMT, DT_F32>(rec, n, G, dst, st, wide);
    case DT_F16: return go_di<FMT, DT_F16>(rec, n, G, dst, st, wide);
    case DT_BF16: return go_di<FMT, DT_BF16>(rec, n, G, dst, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_dequantize_interleaved(const void *rec, int64_t n, int fmt, int64_t G, void *dst,
                                          int dt, cudaStream_t st, bool wide) {
  switch (fmt) {
    case F_INT2: return go_di_t<F_INT2>(rec, n, G, dst, dt, st, wide);
    case F_INT4: return go_di_t<F_INT4>(rec, n, G, dst, dt, st, wide);
    case F_INT6: return go_di_t<F_INT6>(rec, n, G, dst, dt, st, wide);
    case F_INT8: return go_di_t<F_INT8>(rec, n, G, dst, dt, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
