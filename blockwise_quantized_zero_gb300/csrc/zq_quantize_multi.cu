// zq_quantize_multi.cu -- launch unit for the multi-tensor quantize kernels
// (one instantiation per element type, code format and block size).
#include "zq_host.h"

namespace zq {

template <int DT, int FMT, int G>
static cudaError_t go_qm(const MultiArgs &a, cudaStream_t st) {
  constexpr auto K = quantize_multi_kernel<DT, FMT, G>;
  // one persistent wave; no more CTAs than the tiles need (two tiles a warp,
  // as for one tensor, and at least one warp per tensor's tail)
  const int64_t full = a.tile0[a.count];
  const int64_t per_cta = int64_t(kWarps) * kQuantizeTilesPerWarp;
  int64_t need = (full + per_cta - 1) / per_cta;
  const int64_t tails = (a.count + kWarps - 1) / kWarps;
  if (need < tails) need = tails;
  const int64_t cap = int64_t(device_sm_count()) * ctas_per_sm<K>();
  const unsigned grid = unsigned(need < 1 ? 1 : (need < cap ? need : cap));
  return launch_pdl(K, grid, 0, st, a);
}

template <int DT, int FMT>
static cudaError_t go_qm_g(const MultiArgs &a, int64_t G, cudaStream_t st) {
  switch (G) {
    case 32: return go_qm<DT, FMT, 32>(a, st);
    case 64: return go_qm<DT, FMT, 64>(a, st);
    case 128: return go_qm<DT, FMT, 128>(a, st);
    case 256: return go_qm<DT, FMT, 256>(a, st);
    case 512: return go_qm<DT, FMT, 512>(a, st);
    case 1024: return go_qm<DT, FMT, 1024>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

template <int DT>
static cudaError_t go_qm_f(const MultiArgs &a, int fmt, int64_t G, cudaStream_t st) {
  switch (fmt) {
    case F_INT2: return go_qm_g<DT, F_INT2>(a, G, st);
    case F_INT4: return go_qm_g<DT, F_INT4>(a, G, st);
    case F_INT6: return go_qm_g<DT, F_INT6>(a, G, st);
    case F_INT8: return go_qm_g<DT, F_INT8>(a, G, st);
    case F_E4M3: return go_qm_g<DT, F_E4M3>(a, G, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_quantize_multi(const MultiArgs &a, int dt, int fmt, int64_t G, cudaStream_t st) {
  switch (dt) {
    case DT_F32: return go_qm_f<DT_F32>(a, fmt, G, st);
    case DT_F16: return go_qm_f<DT_F16>(a, fmt, G, st);
    case DT_BF16: return go_qm_f<DT_BF16>(a, fmt, G, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace zq
