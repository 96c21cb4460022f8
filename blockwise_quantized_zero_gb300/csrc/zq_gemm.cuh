// zq_gemm.cuh -- dequantization fused into the GEMM that consumes quantized
// weights (AGoQ, section "C. Kernel Fusion": the quantize/dequantize
// arithmetic runs on the CUDA cores and the GEMM on the tensor cores; ZeRO++
// qwZ: a layer computes with the dequantized gathered weights):
//
//     y[m][n] = sum_k x[m][k] * W_hat[n][k],   W_hat = bf16(fl32(q * s)),
//
// x: M x K bf16 activations (row-major); W: the N x K weight matrix held as
// the library's blockwise codes and fp32 scales of its flattened row-major
// form (blocks of G along each row); y: M x N, fp32 or bf16 (one rounding of
// the fp32 accumulator).
//
// One persistent CTA per SM walks output tiles of BM x BN (BM = 128 or 256:
// one or two 128-row MMAs per step on the same weight operand); each k-block
// is 64 deep. Problems with too few tiles split K over thread-block clusters
// instead (below). The tile and the split come from a cost model on the
// host (gemm_tile_shape). Launches use programmatic dependent launch: the
// set-up runs before griddepcontrol.wait, every global access after it.
// Warp roles (22 warps):
//   warp 0      one lane issues the tiled bulk copies (TMA) of the activation
//               tile (BM x 64 bf16, 128-byte swizzled) and of the packed code
//               tile (BN rows x 64 codes) into a stage of shared memory;
//   warp 1      allocates the tensor memory and one lane issues the
//               tcgen05.mma steps (128 x BN x 16 for each 128-row half of
//               the tile, bf16 in, fp32 accumulated in tensor memory) once a
//               stage's activations and dequantized weights are ready; two
//               accumulators alternate between tiles when they fit;
//   warps 2-17  dequantize the stage's codes: 16 codes and their block scale
//               per task, fl32(q * s) rounded to bf16, written into the
//               weight operand's 128-byte-swizzled K-major layout; a row's
//               block scale is loaded once per block, a k-block ahead, by one
//               of the row's four threads and shared by a warp shuffle;
//   warps 18-21 read a finished accumulator from tensor memory (each warp its
//               32 lanes = 32 rows of each half) and store the rows of y.
// Stage buffers are recycled through mbarriers (full: copies landed; ready:
// weights dequantized; empty: the MMAs that read the stage completed; and per
// accumulator full / empty). Every wait is bounded in time and also gives up
// when another role has given up; a wait that runs out sets the device error
// word and the CTA drains its copies and MMAs, frees its tensor memory and
// returns.
#pragma once

#include <cuda.h>

#include "zq_host.h"
#include "zq_tc.cuh"

namespace zq {

constexpr int kGemmMmaM = 128;       // rows of one MMA (and of one TMEM accumulator)
constexpr int kGemmBK = 64;          // k-block depth: 64 bf16 = one 128-byte swizzle row
constexpr int kGemmDequantWarps = 16;
constexpr int kGemmDqThreads = kGemmDequantWarps * 32;
constexpr int kGemmEpiWarps = 4;
constexpr int kGemmWarps = 2 + kGemmDequantWarps + kGemmEpiWarps;
constexpr int kGemmThreads = kGemmWarps * 32;
constexpr int kGemmSmemBudget = 220 * 1024;

// Split-K for problems with too few output tiles to fill the GPU (few
// tokens): a cluster of CS CTAs (2, 4 or 8) shares one 128-row output tile,
// CTA r taking k-blocks [r KB / CS, (r+1) KB / CS). After its last MMA each
// CTA copies its accumulator to shared memory; after a cluster barrier, CTA r
// sums rows [r 128 / CS, (r+1) 128 / CS) of the CS partial tiles, read through
// distributed shared memory in rank order (a fixed order: the result does not
// depend on timing), and stores them; a second cluster barrier keeps every
// CTA resident until its partial sums have been read.
constexpr int kGemmMaxSplit = 8;

// Output tile BM x BN: BM / 128 MMAs of 128 rows per 16-deep step share the
// dequantized weight operand (the dequantization work per flop is 1 / 2BM).
template <int FMT, int BN, int BM> struct GemmGeom {
  static constexpr int kBits = Fmt<FMT>::kBits;
  static constexpr int kHalves = BM / kGemmMmaM;                // MMAs per step
  static constexpr int kABytes = BM * kGemmBK * 2;              // activation tile
  static constexpr int kBBytes = BN * kGemmBK * 2;              // dequantized weight tile
  static constexpr int kCodeRow = kGemmBK * kBits / 8;          // code bytes of one weight row
  static constexpr int kCBytes = BN * kCodeRow;                 // packed code tile
  // The copy ring (activations + codes) and the ring of dequantized weight
  // operands are separate, so that the copies run several k-blocks ahead
  // while only two weight operands are held.
  static constexpr int kStage = ((kABytes + kCBytes + 1023) / 1024) * 1024;
  static constexpr int kBRing = 2;
  // 16-code tasks per dequantizing thread per k-block
  static constexpr int kTasks = BN * (kGemmBK / 16);
  static constexpr int kTasksPerThread = (kTasks + kGemmDqThreads - 1) / kGemmDqThreads;
  static constexpr int kStagesFit = (kGemmSmemBudget - 2048 - kBRing * kBBytes) / kStage;
  static constexpr int kStages = kStagesFit > 6 ? 6 : kStagesFit;
  static constexpr int kBOff = kStages * kStage;                // 1024-aligned
  static constexpr int kBarOff = kBOff + kBRing * kBBytes;
  // Accumulators: one per tile of kHalves * BN fp32 columns; two alternate
  // between tiles when they fit in the 512 columns of tensor memory.
  static constexpr int kAccCols = kHalves * BN;
  static constexpr int kAccs = 2 * kAccCols <= 512 ? 2 : 1;
  static constexpr uint32_t kTmemCols = uint32_t(kAccs * kAccCols);
  // full, empty per copy stage; ready, free per weight operand; full, empty
  // per accumulator; drain; then the tmem slot and the abort flag
  static constexpr int kNumBars = 2 * kStages + 2 * kBRing + 2 * kAccs + 1;
  static constexpr int kSmem = 1024 + kBarOff + kNumBars * 8 + 16;
  // Split-K (one output tile per cluster): each CTA's fp32 partial sums, rows
  // of BN + 4 words (the padding spreads one row per lane over the banks),
  // reuse the stage and weight-operand memory once the MMAs are done.
  static constexpr int kPartStride = BN + 4;
  static constexpr int kPartBytes = kGemmMmaM * kPartStride * 4;
  static constexpr uint32_t kTxBytes = kABytes + kCBytes;
  static_assert(BM == 128 || BM == 256, "tile rows");
  static_assert(kStages >= 2, "at least two stages");
  static_assert(kGemmDqThreads % 4 == 0, "a thread keeps one 16-code column of its rows");
  static_assert(kCodeRow % 16 == 0, "TMA boxes are whole 16-byte units");
  static_assert(BN == 64 || BN == 128 || BN == 256, "MMA N");
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocation");
  static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

struct GemmArgs {
  const float *scales;
  void *y;
  int64_t M, N, K;
  int log2G;
  int tiles_m, tiles_n;
};

// Output tile t -> (m block, n block): groups of up to 16 m blocks walk the n
// blocks together, so the CTAs running at one time share activation rows and
// weight tiles in L2.
__device__ __forceinline__ void gemm_tile(int t, int tiles_m, int tiles_n, int &mb, int &nb) {
  constexpr int kGroup = 16;
  const int per_group = kGroup * tiles_n;
  const int g = t / per_group, rem = t - g * per_group;
  const int gm = min(kGroup, tiles_m - g * kGroup);
  mb = g * kGroup + rem % gm;
  nb = rem / gm;
}

// Bounded wait of one thread; gives up early once another role has.
__device__ __forceinline__ bool gemm_wait_thread(uint32_t bar, uint32_t parity,
                                                 volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 30); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_ns() - t0 > kWaitLimitNs) break;
  }
  *abort = 1;
  atomicOr(&g_dev_error, kDevErrWaitTimeout);
  return false;
}

// Warp-uniform bounded wait (every lane of the warp calls it).
__device__ __forceinline__ bool gemm_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort) {
  if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 0; i < (1u << 30); ++i) {
    if (__all_sync(kFull, mbar_try_wait(bar, parity))) return true;
    if (__any_sync(kFull, *abort != 0)) return false;
    if (__any_sync(kFull, global_ns() - t0 > kWaitLimitNs)) break;
  }
  if ((threadIdx.x & 31) == 0) {
    *abort = 1;
    atomicOr(&g_dev_error, kDevErrWaitTimeout);
  }
  __syncwarp();
  return false;
}

}  // namespace zq
