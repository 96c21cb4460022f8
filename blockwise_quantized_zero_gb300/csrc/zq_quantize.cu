// zq_quantize.cu -- launch unit for the quantize kernels (every element type,
// code format and block size is a separate instantiation).
#include "zq_host.h"

namespace zq {

template <int DT, int FMT, int G>
static cudaError_t go_q(const void *src, int64_t n, void *codes, float *scales, cudaStream_t st,
                        bool wide, const SliceRemap &rm) {
  constexpr auto K = quantize_kernel<DT, FMT, G>;
  return launch_pdl(K, grid_for<K>(n, kQuantizeTilesPerWarp), 0, st, src, static_cast<uint8_t *>(codes), scales, n,
                    wide ? 1 : 0, rm);
}

template <int DT, int FMT>
static cudaError_t go_q_g(const void *src, int64_t n, int64_t G, void *codes, float *scales,
                          cudaStream_t st, bool wide, const SliceRemap &rm) {
  switch (G) {
    case 32: return go_q<DT, FMT, 32>(src, n, codes, scales, st, wide, rm);
    case 64: return go_q<DT, FMT, 64>(src, n, codes, scales, st, wide, rm);
    case 128: return go_q<DT, FMT, 128>(src, n, codes, scales, st, wide, rm);
    case 256: return go_q<DT, FMT, 256>(src, n, codes, scales, st, wide, rm);
    case 512: return go_q<DT, FMT, 512>(src, n, codes, scales, st, wide, rm);
    case 1024: return go_q<DT, FMT, 1024>(src, n, codes, scales, st, wide, rm);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT>
static cudaError_t go_q_f(const void *src, int64_t n, int fmt, int64_t G, void *codes,
                          float *scales, cudaStream_t st, bool wide, const SliceRemap &rm) {
  switch (fmt) {
    case F_INT2: return go_q_g<DT, F_INT2>(src, n, G, codes, scales, st, wide, rm);
    case F_INT4: return go_q_g<DT, F_INT4>(src, n, G, codes, scales, st, wide, rm);
    case F_INT6: return go_q_g<DT, F_INT6>(src, n, G, codes, scales, st, wide, rm);
    case F_INT8: return go_q_g<DT, F_INT8>(src, n, G, codes, scales, st, wide, rm);
    case F_E4M3: return go_q_g<DT, F_E4M3>(src, n, G, codes, scales, st, wide, rm);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize(const void *src, int dt, int64_t n, int fmt, int64_t G, void *codes,
                            float *scales, cudaStream_t st, bool wide, const SliceRemap &rm) {
  switch (dt) {
    case DT_F32: return go_q_f<DT_F32>(src, n, fmt, G, codes, scales, st, wide, rm);
    case DT_F16: return go_q_f<DT_F16>(src, n, fmt, G, codes, scales, st, wide, rm);
    case DT_BF16: return go_q_f<DT_BF16>(src, n, fmt, G, codes, scales, st, wide, rm);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
