// zq_fp8.cu -- launch unit for the in-place FP8 accumulate kernels.
#include "zq_host.h"

namespace zq {

template <int DT, int G>
static cudaError_t go_a(void *codes, float *scales, const void *grad, int64_t n, cudaStream_t st,
                        bool wide) {
  constexpr auto K = fp8_accumulate_kernel<DT, G>;
  return launch_pdl(K, grid_for<K>(n), 0, st, static_cast<uint8_t *>(codes), scales, grad, n,
                    wide ? 1 : 0, 1.0f);
}

template <int DT>
static cudaError_t go_a_g(void *codes, float *scales, const void *grad, int64_t n, int64_t G,
                          cudaStream_t st, bool wide) {
  switch (G) {
    case 32: return go_a<DT, 32>(codes, scales, grad, n, st, wide);
    case 64: return go_a<DT, 64>(codes, scales, grad, n, st, wide);
    case 128: return go_a<DT, 128>(codes, scales, grad, n, st, wide);
    case 256: return go_a<DT, 256>(codes, scales, grad, n, st, wide);
    case 512: return go_a<DT, 512>(codes, scales, grad, n, st, wide);
    case 1024: return go_a<DT, 1024>(codes, scales, grad, n, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_fp8_accumulate(void *codes, float *scales, const void *grad, int dt, int64_t n,
                                  int64_t G, cudaStream_t st, bool wide) {
  switch (dt) {
    case DT_F32: return go_a_g<DT_F32>(codes, scales, grad, n, G, st, wide);
    case DT_F16: return go_a_g<DT_F16>(codes, scales, grad, n, G, st, wide);
    case DT_BF16: return go_a_g<DT_BF16>(codes, scales, grad, n, G, st, wide);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
