// zq_host.h -- host-side launch plumbing shared by the libzq launch units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "zq_kernels.cuh"

namespace zq {

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Resident CTAs per SM for one kernel instantiation with SMEM bytes of
// dynamic shared memory (computed once; a kernel that needs more than the
// default 48 KB is granted it first). 0 if the kernel cannot be made to fit.
template <auto Kernel, int SMEM = 0, int THREADS = kThreads> int ctas_per_sm() {
  static const int v = [] {
    if (SMEM > 48 * 1024 &&
        cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
            cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    int b = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, Kernel, THREADS, SMEM) != cudaSuccess ||
        b < 1) {
      (void)cudaGetLastError();
      b = SMEM > 0 ? 0 : 1;
    }
    return b;
  }();
  return v;
}

// Persistent grid: enough CTAs for every warp tile (or for every group of
// tiles_per_warp tiles), at most one wave.
template <auto Kernel, int SMEM = 0> unsigned grid_for(int64_t n, int tiles_per_warp = 1) {
  const int64_t tiles = (n + kTile - 1) / kTile;
  const int64_t per_cta = int64_t(kThreads / 32) * tiles_per_warp;
  const int64_t ctas = (tiles + per_cta - 1) / per_cta;
  const int64_t cap = int64_t(device_sm_count()) * ctas_per_sm<Kernel, SMEM>();
  const int64_t g = ctas < cap ? ctas : cap;
  return static_cast<unsigned>(g > 0 ? g : 1);
}

// Launch with programmatic dependent launch allowed: the kernel may be
// scheduled while the previous kernel on the stream drains; every kernel of
// this library waits for its predecessor (griddepcontrol.wait) before it
// touches global memory, so stream order and memory visibility are those of
// an ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_threads(void (*kernel)(KArgs...), unsigned grid, unsigned threads,
                               size_t smem, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, size_t smem, cudaStream_t st,
                       Args... args) {
  return launch_pdl_threads(kernel, grid, kThreads, smem, st, args...);
}

// Quantize grids give every warp at least two tiles, so that the load of a
// warp's next tile overlaps the current tile's arithmetic even for small
// tensors (measured: 1 Mi-element calls, eight in flight, 4105 -> 4500 GB/s;
// four tiles a warp left too few CTAs, 3178 GB/s). Large tensors are capped
// at one wave either way.
constexpr int kQuantizeTilesPerWarp = 2;

// Launchers (one translation unit each). They return the launch status.
cudaError_t launch_quantize(const void *src, int dt, int64_t n, int fmt, int64_t G, void *codes,
                            float *scales, cudaStream_t st, bool wide,
                            const SliceRemap &rm = SliceRemap{1, 1, 0});
// One launch over up to kMultiMax tensors (same type, format and block size).
cudaError_t launch_quantize_multi(const MultiArgs &a, int dt, int fmt, int64_t G, cudaStream_t st);
cudaError_t launch_dequantize_multi(const DequantMultiArgs &a, int fmt, int dt, cudaStream_t st);
cudaError_t launch_dequantize(const void *codes, const float *scales, int64_t n, int fmt,
                              int64_t G, void *dst, int dt, cudaStream_t st, bool wide);
// The metadata-interleaved record layout (integer codes).
cudaError_t launch_quantize_interleaved(const void *src, int dt, int64_t n, int fmt, int64_t G,
                                        void *rec, cudaStream_t st, bool wide);
cudaError_t launch_dequantize_interleaved(const void *rec, int64_t n, int fmt, int64_t G, void *dst,
                                          int dt, cudaStream_t st, bool wide);
cudaError_t launch_reduce(const ReduceArgs &a, int fin, int fout, cudaStream_t st);
// All P reduces of one hop of the two-hop reduce in one launch.
cudaError_t launch_reduce_hop(const HopArgs &a, int fin, int fout, cudaStream_t st);
// The same reduce with up to kStaticMaxShards shards whose pointers (host
// arrays) are copied into a static device table on the stream.
cudaError_t launch_reduce_static(const void *const *codes, const float *const *scales,
                                 const TableReduceArgs &args, int fin, int fout, cudaStream_t st);
// The same two launches with the kernels built for three CTAs an SM (at most
// kFewShards shards).
cudaError_t launch_reduce_few(const ReduceArgs &a, int fin, int fout, cudaStream_t st);
cudaError_t launch_reduce_hop_few(const HopArgs &a, int fin, int fout, cudaStream_t st);
// The bounded-wait self-test (a wait that nothing completes, limit_ns long).
cudaError_t launch_wait_selftest(uint64_t limit_ns, cudaStream_t st);
// Reads and clears the device error words of the launch units.
unsigned take_reduce_device_error();
unsigned take_reduce_few_device_error();

// The dequant-fused GEMM (tcgen05): y = x * bf16(dequantize(codes, scales))^T.
cudaError_t launch_gemm_dequant(const void *x, int64_t M, int64_t K, const void *codes,
                                const float *scales, int fmt, int64_t G, int64_t N, void *y,
                                int out_dt, cudaStream_t st);
void gemm_tile_shape(int64_t M, int64_t N, int64_t K, int &bm, int &bn, int &split);
unsigned take_gemm_device_error();

cudaError_t launch_fp8_accumulate(void *codes, float *scales, const void *grad, int dt, int64_t n,
                                  int64_t G, cudaStream_t st, bool wide);

inline int log2_block(int64_t G) {
  int l = 0;
  while ((int64_t(1) << l) < G) ++l;
  return l;
}

}  // namespace zq
