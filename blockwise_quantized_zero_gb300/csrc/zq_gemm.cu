// zq_gemm.cu -- launch unit of the dequant-fused GEMM (kernel design in
// zq_gemm.cuh): y = x * bf16(dequantize(W))^T on the tcgen05 tensor cores.
#include <cstring>
#include <mutex>

#include "zq_gemm.cuh"

namespace zq {

// SPLIT: launched in clusters of CS CTAs (split-K, one output tile per
// cluster); otherwise persistent, one CTA per SM.
template <int FMT, int BN, int BM, int OUT, bool SPLIT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    gemm_dequant_kernel(const __grid_constant__ CUtensorMap tm_x,
                        const __grid_constant__ CUtensorMap tm_codes, const GemmArgs a) {
  using GG = GemmGeom<FMT, BN, BM>;
  static_assert(!SPLIT || BM == kGemmMmaM, "split-K tiles have one 128-row half");
  static_assert(!SPLIT || GG::kPartBytes <= GG::kBarOff, "partial sums fit the stage memory");
  constexpr int S = GG::kStages, NB = GG::kBRing, NACC = GG::kAccs, H = GG::kHalves;
  constexpr int BITS = GG::kBits;
  extern __shared__ uint8_t gemm_smem_raw[];
  const uint32_t raw = smem_addr(gemm_smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 1024-byte aligned (128-byte swizzle atoms)
  uint8_t *gbase = gemm_smem_raw + (base - raw);
  const uint32_t bar0 = base + GG::kBarOff;
  // copy stage s: full (copies landed), empty (MMAs and dequantizers done with it)
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  // weight operand b: ready (dequantized), free (the MMAs that read it completed)
  auto bready = [&](int b) { return bar0 + 8u * (2 * S + b); };
  auto bfree = [&](int b) { return bar0 + 8u * (2 * S + NB + b); };
  // accumulator c: full (last MMA of the tile completed), empty (read out)
  auto acc_full = [&](int c) { return bar0 + 8u * (2 * S + 2 * NB + c); };
  auto acc_empty = [&](int c) { return bar0 + 8u * (2 * S + 2 * NB + NACC + c); };
  const uint32_t drain = bar0 + 8u * (2 * S + 2 * NB + 2 * NACC);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gbase + GG::kBarOff + 8 * GG::kNumBars);
  volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
  auto sA = [&](int s) { return base + uint32_t(s) * GG::kStage; };
  auto sC = [&](int s) { return base + uint32_t(s) * GG::kStage + GG::kABytes; };
  auto sB = [&](int b) { return base + GG::kBOff + uint32_t(b) * GG::kBBytes; };
  const uint8_t *gC0 = gbase + GG::kABytes;  // generic pointer to stage 0's codes

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntiles = a.tiles_m * a.tiles_n;
  const int KB = int(a.K / kGemmBK);
  // Work of this CTA: tiles t0, t0 + tstep, ... and k-blocks [kb0, kb1) of each.
  const int cs = SPLIT ? int(tc::cluster_size()) : 1;
  const int rank = SPLIT ? int(tc::cluster_rank()) : 0;
  const int t0 = SPLIT ? int(blockIdx.x) / cs : int(blockIdx.x);
  const int tstep = SPLIT ? ntiles : int(gridDim.x);
  const int kb0 = int(int64_t(rank) * KB / cs), kb1 = int(int64_t(rank + 1) * KB / cs);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1 + kGemmDequantWarps);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(bready(b), kGemmDequantWarps);
      mbar_init(bfree(b), 1);
    }
    for (int c = 0; c < NACC; ++c) {
      mbar_init(acc_full(c), 1);
      mbar_init(acc_empty(c), kGemmEpiWarps);
    }
    mbar_init(drain, 1);
    *abort = 0;
    mbar_init_fence();
  }
  if (w == 1) {
    tc::tmem_alloc(smem_addr(tmem_slot), GG::kTmemCols);
    tc::tmem_relinquish();
  }
  if (w == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tm_x);
    tc::tma_prefetch_desc(&tm_codes);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // Programmatic dependent launch: the set-up above may overlap the previous
  // grid's last CTAs; no global memory is read or written before it has
  // completed (griddepcontrol.wait), and the next grid may be scheduled.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  if (w == 0) {
    // ---------------- producer: one lane issues the tiled copies ----------------
    if (lane == 0) {
      uint32_t u = 0;
      bool ok = true;
      for (int t = t0; t < ntiles && ok; t += tstep) {
        int mb, nb;
        gemm_tile(t, a.tiles_m, a.tiles_n, mb, nb);
        for (int kb = kb0; kb < kb1; ++kb, ++u) {
          const int s = int(u % S);
          const uint32_t r = u / S;
          if (r >= 1 && !gemm_wait_thread(empty(s), (r - 1) & 1u, abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full(s), GG::kTxBytes);
          tc::tma_load_2d(sA(s), &tm_x, kb * kGemmBK, mb * BM, full(s));
          tc::tma_load_2d(sC(s), &tm_codes, kb * GG::kCodeRow, nb * BN, full(s));
        }
      }
      if (!ok) {  // copies in flight land before the CTA's memory is released
        const uint32_t first = u > uint32_t(S) ? u - S : 0u;
        for (uint32_t v = first; v < u; ++v) (void)mbar_wait_thread(full(int(v % S)), (v / S) & 1u);
      }
    }
    __syncwarp();
  } else if (w == 1) {
    // ---------------- MMA issuer: one lane ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kGemmMmaM, BN);
      uint32_t u = 0;
      int i = 0;
      bool ok = true, issued = false;
      for (int t = t0; t < ntiles && ok; t += tstep, ++i) {
        const int ab = i % NACC;
        const uint32_t ra = uint32_t(i / NACC);
        if (ra >= 1 && !gemm_wait_thread(acc_empty(ab), (ra - 1) & 1u, abort)) break;
        tc::fence_after_sync();
        const uint32_t d = tmem + uint32_t(ab * GG::kAccCols);
        for (int kb = kb0; kb < kb1; ++kb, ++u) {
          const int s = int(u % S), b = int(u % NB);
          if (!gemm_wait_thread(full(s), (u / S) & 1u, abort) ||
              !gemm_wait_thread(bready(b), (u / NB) & 1u, abort)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
          const uint64_t bd = tc::smem_desc_sw128(sB(b));
#pragma unroll
          for (int h = 0; h < H; ++h) {  // the 128-row halves share the weight operand
            const uint64_t ad = tc::smem_desc_sw128(sA(s) + uint32_t(h * kGemmMmaM * 128));
#pragma unroll
            for (int k4 = 0; k4 < kGemmBK / 16; ++k4)  // +32 bytes along K per step
              tc::mma_bf16(d + uint32_t(h * BN), ad + 2u * k4, bd + 2u * k4, idesc,
                           (kb != kb0 || k4 != 0) ? 1u : 0u);
          }
          tc::mma_commit(empty(s));
          tc::mma_commit(bfree(b));
          issued = true;
        }
        if (ok) tc::mma_commit(acc_full(ab));
      }
      if (issued) {  // every MMA has completed before the tensor memory is released
        tc::mma_commit(drain);
        (void)mbar_wait_thread(drain, 0u);
      }
    }
    __syncwarp();
  } else if (w < 2 + kGemmDequantWarps) {
    // ---------------- dequantize: codes -> bf16 weight operand ----------------
    // Thread dt owns the tasks i = 0 .. T-1: weight-tile row r0 + i * kRowStep
    // (r0 = dt / 4), 16-code column c16 = dt % 4. Rows of one thread differ by
    // a multiple of 8, so their swizzled chunk positions are the same and all
    // shared-memory offsets are per-thread constants. The four threads of a
    // row are adjacent lanes; the block scale of a row's 16-code run is loaded
    // by one of them (c16 = 0, and c16 = 2 for G = 32, where a k-block holds
    // two blocks), only when the k-block starts a new block (every G / 64
    // k-blocks), one k-block ahead, and passed to the others by a shuffle.
    constexpr int T = GG::kTasksPerThread;
    constexpr int kRowStep = kGemmDqThreads / 4;
    constexpr int CB = GG::kCodeRow;
    const int dt = (w - 2) * 32 + lane, c16 = dt & 3, r0 = dt >> 2;
    const uint32_t b_off0 = uint32_t(r0) * 128u + ((uint32_t(2 * c16) ^ uint32_t(r0 & 7)) << 4);
    const uint32_t b_off1 = uint32_t(r0) * 128u + ((uint32_t(2 * c16 + 1) ^ uint32_t(r0 & 7)) << 4);
    const int c_off = r0 * CB + c16 * (16 * BITS / 8);
    const int lg = a.log2G;
    const bool owner = lg == 5 ? (c16 & 1) == 0 : c16 == 0;
    const int src = lg == 5 ? (lane & ~1) : (lane & ~3);
    const int kpp = lg <= 6 ? 1 : 1 << (lg - 6);  // k-blocks per block
    // Cursor one k-block ahead of the dequantization: tile f_t, k-block f_kb,
    // each task's element index at k = 0.
    int f_t = t0, f_kb = kb0;
    int64_t f_e[T];
    auto f_tile = [&]() {
      if (f_t < ntiles) {
        int mb, nb;
        gemm_tile(f_t, a.tiles_m, a.tiles_n, mb, nb);
#pragma unroll
        for (int i = 0; i < T; ++i)
          f_e[i] = (int64_t(nb) * BN + r0 + i * kRowStep) * a.K + c16 * 16;
      }
    };
    auto f_next = [&]() {
      if (++f_kb == kb1) {
        f_kb = kb0;
        f_t += tstep;
        f_tile();
      }
    };
    float cur[T], nxt[T];
    f_tile();
#pragma unroll
    for (int i = 0; i < T; ++i) {
      cur[i] = 0.0f;
      nxt[i] = 0.0f;
      if (owner && dt + i * kGemmDqThreads < GG::kTasks && f_t < ntiles)
        cur[i] = ld_nc_f32(a.scales + ((f_e[i] + int64_t(kb0) * kGemmBK) >> lg));
    }
    f_next();
    uint32_t u = 0;
    bool ok = true;
    for (int t = t0; t < ntiles && ok; t += tstep) {
      for (int kb = kb0; kb < kb1; ++kb, ++u) {
        const int s = int(u % S), b = int(u % NB);
        const bool fresh = f_t < ntiles && f_kb % kpp == 0;  // the next k-block starts a block
        if (fresh && owner) {
#pragma unroll
          for (int i = 0; i < T; ++i)
            if (dt + i * kGemmDqThreads < GG::kTasks)
              nxt[i] = ld_nc_f32(a.scales + ((f_e[i] + int64_t(f_kb) * kGemmBK) >> lg));
        }
        if (!gemm_wait_warp(full(s), (u / S) & 1u, abort) ||
            (u >= uint32_t(NB) && !gemm_wait_warp(bfree(b), (u / NB - 1) & 1u, abort))) {
          ok = false;
          break;
        }
        const uint8_t *cs = gC0 + size_t(s) * GG::kStage + c_off;
        const uint32_t bb = sB(b);
#pragma unroll
        for (int i = 0; i < T; ++i) {
          const float sc = __shfl_sync(kFull, cur[i], src);
          if (dt + i * kGemmDqThreads < GG::kTasks) {
            uint32_t wv[Fmt<FMT>::kWords16];
            load_codes16_smem<BITS>(cs + i * kRowStep * CB, wv);
            float y[kVec];
            dequant16<FMT>(wv, sc, y);
            uint32_t p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              __nv_bfloat162 h = __floats2bfloat162_rn(y[2 * q], y[2 * q + 1]);
              p[q] = *reinterpret_cast<uint32_t *>(&h);
            }
            const uint32_t rb = bb + uint32_t(i * kRowStep * 128);
            tc::st_shared_v4(rb + b_off0, p[0], p[1], p[2], p[3]);
            tc::st_shared_v4(rb + b_off1, p[4], p[5], p[6], p[7]);
          }
        }
        fence_proxy_async_smem();  // the tensor cores read these bytes through the async proxy
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bready(b));
          mbar_arrive(empty(s));  // this warp is done with the stage's codes
        }
        if (fresh) {
#pragma unroll
          for (int i = 0; i < T; ++i) cur[i] = nxt[i];
        }
        f_next();
      }
    }
  } else {
    // ---------------- epilogue: tensor memory -> y ----------------
    const int q = w & 3;  // this warp may read TMEM lanes [32q, 32q + 32)
    if constexpr (SPLIT) {
      // one tile: copy the partial sums (row 32q + lane) to shared memory
      if (t0 < ntiles && gemm_wait_warp(acc_full(0), 0u, abort)) {
        tc::fence_after_sync();
        const uint32_t row = base + uint32_t((q * 32 + lane) * GG::kPartStride * 4);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tc::tmem_ld32(tmem + (uint32_t(q * 32) << 16) + uint32_t(c), v);
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            tc::st_shared_v4(row + uint32_t((c + k) * 4), v[k], v[k + 1], v[k + 2], v[k + 3]);
        }
      }
      tc::fence_before_sync();
    }
    int i = 0;
    for (int t = t0; t < ntiles && !SPLIT; t += tstep, ++i) {
      int mb, nb;
      gemm_tile(t, a.tiles_m, a.tiles_n, mb, nb);
      const int ab = i % NACC;
      if (!gemm_wait_warp(acc_full(ab), uint32_t(i / NACC) & 1u, abort)) break;
      tc::fence_after_sync();
#pragma unroll 1
      for (int h = 0; h < H; ++h) {
        const int64_t m = int64_t(mb) * BM + h * kGemmMmaM + q * 32 + lane;
        const uint32_t taddr =
            tmem + (uint32_t(q * 32) << 16) + uint32_t(ab * GG::kAccCols + h * BN);
#pragma unroll 1
        for (int c = 0; c < BN; c += 32) {
          uint32_t v[32];
          tc::tmem_ld32(taddr + uint32_t(c), v);
          if (m < a.M) {
            const int64_t off = m * a.N + int64_t(nb) * BN + c;
            if constexpr (OUT == DT_F32) {
              uint32_t *dst = static_cast<uint32_t *>(a.y) + off;
#pragma unroll
              for (int k = 0; k < 32; k += 4) st_v4(dst + k, v[k], v[k + 1], v[k + 2], v[k + 3]);
            } else {
              uint32_t hb[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                __nv_bfloat162 b2 = __floats2bfloat162_rn(__uint_as_float(v[2 * k]),
                                                          __uint_as_float(v[2 * k + 1]));
                hb[k] = *reinterpret_cast<uint32_t *>(&b2);
              }
              uint16_t *dst = static_cast<uint16_t *>(a.y) + off;
#pragma unroll
              for (int k = 0; k < 16; k += 4) st_v4(dst + 2 * k, hb[k], hb[k + 1], hb[k + 2], hb[k + 3]);
            }
          }
        }
      }
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(ab));
    }
  }

  if constexpr (SPLIT) {
    tc::cluster_sync();  // every CTA's partial sums are in its shared memory
    if (w >= 2 + kGemmDequantWarps && t0 < ntiles) {
      // rows [rank * 128 / cs, (rank + 1) * 128 / cs) of the tile: the sum of
      // the cs partial tiles in rank order, 4 columns a lane
      int mb, nb;
      gemm_tile(t0, a.tiles_m, a.tiles_n, mb, nb);
      const int rows = kGemmMmaM / cs, ew = w - (2 + kGemmDequantWarps);
      for (int r = rank * rows + ew; r < (rank + 1) * rows; r += kGemmEpiWarps) {
        const int64_t m = int64_t(mb) * BM + r;
        if (m >= a.M) break;
        for (int c = lane * 4; c < BN; c += 128) {
          const uint32_t off = base + uint32_t((r * GG::kPartStride + c) * 4);
          float x0, x1, x2, x3;
          tc::ld_cluster_v4(tc::peer_addr(off, 0), x0, x1, x2, x3);
          for (int p = 1; p < cs; ++p) {
            float y0, y1, y2, y3;
            tc::ld_cluster_v4(tc::peer_addr(off, uint32_t(p)), y0, y1, y2, y3);
            x0 = __fadd_rn(x0, y0);
            x1 = __fadd_rn(x1, y1);
            x2 = __fadd_rn(x2, y2);
            x3 = __fadd_rn(x3, y3);
          }
          const int64_t o = m * a.N + int64_t(nb) * BN + c;
          if constexpr (OUT == DT_F32) {
            st_v4(static_cast<uint32_t *>(a.y) + o, __float_as_uint(x0), __float_as_uint(x1),
                  __float_as_uint(x2), __float_as_uint(x3));
          } else {
            __nv_bfloat162 h0 = __floats2bfloat162_rn(x0, x1), h1 = __floats2bfloat162_rn(x2, x3);
            uint2 *dst = reinterpret_cast<uint2 *>(static_cast<uint16_t *>(a.y) + o);
            *dst = make_uint2(*reinterpret_cast<uint32_t *>(&h0), *reinterpret_cast<uint32_t *>(&h1));
          }
        }
      }
    }
    tc::cluster_sync();  // no CTA leaves while its partial sums may still be read
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (w == 1) tc::tmem_dealloc(tmem, GG::kTmemCols);
}

// ---------------------------------------------------------------------------
// Host side: tensor maps (through the runtime's driver entry point, so the
// library does not link the driver library), tile width, launch.
// ---------------------------------------------------------------------------
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                 const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                 const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encode_tiled() {
  static EncodeTiled fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
      (void)cudaGetLastError();
      p = nullptr;
    }
    return reinterpret_cast<EncodeTiled>(p);
  }();
  return fn;
}

// 2-D map of a row-major matrix of `rows` x `cols` elements (dtype, elem
// bytes), row pitch `pitch` bytes, copied in boxes of box_rows x box_cols.
cudaError_t make_map(CUtensorMap *m, CUtensorMapDataType dt, const void *ptr, uint64_t rows,
                     uint64_t cols, uint64_t pitch, uint32_t box_rows, uint32_t box_cols,
                     CUtensorMapSwizzle sw) {
  EncodeTiled enc = encode_tiled();
  if (!enc) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {pitch};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int FMT, int BN, int BM, int OUT, bool SPLIT = false>
cudaError_t go_gemm(const void *x, const void *codes, const GemmArgs &a, int split,
                    cudaStream_t st) {
  using GG = GemmGeom<FMT, BN, BM>;
  constexpr auto K = gemm_dequant_kernel<FMT, BN, BM, OUT, SPLIT>;
  static const cudaError_t attr =
      cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, GG::kSmem);
  if (attr != cudaSuccess) return attr;
  CUtensorMap tx, tcd;
  std::memset(&tx, 0, sizeof tx);
  std::memset(&tcd, 0, sizeof tcd);
  cudaError_t e = make_map(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, uint64_t(a.M), uint64_t(a.K),
                           uint64_t(a.K) * 2u, BM, kGemmBK, CU_TENSOR_MAP_SWIZZLE_128B);
  if (e != cudaSuccess) return e;
  const uint64_t code_pitch = uint64_t(a.K) * GG::kBits / 8u;
  e = make_map(&tcd, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, uint64_t(a.N), code_pitch, code_pitch,
               BN, GG::kCodeRow, CU_TENSOR_MAP_SWIZZLE_NONE);
  if (e != cudaSuccess) return e;
  const int tiles = a.tiles_m * a.tiles_n;
  if constexpr (SPLIT) {  // one cluster of `split` CTAs per output tile
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(unsigned(tiles * split));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = GG::kSmem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, K, tx, tcd, a);
    return e != cudaSuccess ? e : cudaGetLastError();
  } else {
    (void)split;
    const int grid = tiles < device_sm_count() ? tiles : device_sm_count();
    e = launch_pdl_threads(K, unsigned(grid), unsigned(kGemmThreads), size_t(GG::kSmem), st, tx,
                           tcd, a);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
}

// The tile shapes built: 256 x 256 and 256 x 128 for problems with enough
// rows, 128 x 128 and 128 x 64 otherwise.
template <int FMT, int OUT>
cudaError_t go_gemm_shape(const void *x, const void *codes, const GemmArgs &a, int bm, int bn,
                          int split, cudaStream_t st) {
  if (split > 1) {
    if (bm == 128 && bn == 256) return go_gemm<FMT, 256, 128, OUT, true>(x, codes, a, split, st);
    if (bm == 128 && bn == 128) return go_gemm<FMT, 128, 128, OUT, true>(x, codes, a, split, st);
    return cudaErrorInvalidValue;
  }
  if (bm == 256 && bn == 256) return go_gemm<FMT, 256, 256, OUT>(x, codes, a, 1, st);
  if (bm == 256 && bn == 128) return go_gemm<FMT, 128, 256, OUT>(x, codes, a, 1, st);
  if (bm == 128 && bn == 128) return go_gemm<FMT, 128, 128, OUT>(x, codes, a, 1, st);
  if (bm == 128 && bn == 64) return go_gemm<FMT, 64, 128, OUT>(x, codes, a, 1, st);
  return cudaErrorInvalidValue;
}

template <int OUT>
cudaError_t go_gemm_fmt(const void *x, const void *codes, const GemmArgs &a, int fmt, int bm,
                        int bn, int split, cudaStream_t st) {
  switch (fmt) {
    case F_INT2: return go_gemm_shape<F_INT2, OUT>(x, codes, a, bm, bn, split, st);
    case F_INT4: return go_gemm_shape<F_INT4, OUT>(x, codes, a, bm, bn, split, st);
    case F_INT6: return go_gemm_shape<F_INT6, OUT>(x, codes, a, bm, bn, split, st);
    case F_INT8: return go_gemm_shape<F_INT8, OUT>(x, codes, a, bm, bn, split, st);
    case F_E4M3: return go_gemm_shape<F_E4M3, OUT>(x, codes, a, bm, bn, split, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// CTAs of split-K clusters of `cs` CTAs that can be resident at once
// (clusters are placed within GPU processing clusters, so fewer than one per
// SM in general), from the occupancy query of a representative kernel (all
// split kernels take one CTA an SM); cached per device.
namespace {
std::mutex g_cluster_mutex;
int g_cluster_ctas[64][4];  // [device][log2 cs]

int split_ctas_per_wave(int cs) {
  const int sms = device_sm_count();
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    (void)cudaGetLastError();
    return sms / cs * cs;
  }
  const int li = cs == 2 ? 1 : cs == 4 ? 2 : 3;
  std::lock_guard<std::mutex> lock(g_cluster_mutex);
  if (g_cluster_ctas[dev][li] == 0) {
    constexpr auto K = gemm_dequant_kernel<F_INT8, 256, 128, DT_BF16, true>;
    using GG = GemmGeom<F_INT8, 256, 128>;
    int n = 0;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = unsigned(cs);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(cs * sms));
    cfg.blockDim = dim3(kGemmThreads);
    cfg.dynamicSmemBytes = GG::kSmem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(K, cudaFuncAttributeMaxDynamicSharedMemorySize, GG::kSmem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n, K, &cfg) != cudaSuccess || n < 1) {
      (void)cudaGetLastError();
      n = sms / cs;
    }
    g_cluster_ctas[dev][li] = n * cs;
  }
  return g_cluster_ctas[dev][li];
}
}  // namespace

// Tile shape and split, from a cost model: each candidate, unsplit
// (persistent CTAs, 256 x 256, 256 x 128, 128 x 128 or 128 x 64) or, for
// problems of at most 512 rows, split-K over clusters of 2, 4 or 8 CTAs
// (128 x 256 or 128 x 128 tiles, at least 4 k-blocks a CTA), is given the
// time waves x (k-blocks a CTA x time a k-block) + fixed time, with the
// times measured on GB300 (microseconds a 64-deep k-block: 256 x 256 0.885,
// 256 x 128 0.60, 128 x 256 0.664, 128 x 128 0.49, 128 x 64 0.42; fixed: 3
// unsplit, 11 a split CTA, which adds the partial-tile exchange), and the
// fastest is taken. Waves: tiles / SMs rounded up for the persistent
// kernels; for clusters, the CTAs over those resident at once.
void gemm_tile_shape(int64_t M, int64_t N, int64_t K, int &bm, int &bn, int &split) {
  const int64_t sms = device_sm_count();
  const double kb = double(K / kGemmBK);
  struct Unsplit { int bm, bn; double t; };
  const Unsplit us[4] = {{256, 256, 0.885}, {256, 128, 0.60}, {128, 128, 0.49}, {128, 64, 0.42}};
  double best = 1e300;
  bm = 128;
  bn = 64;
  split = 1;
  for (const auto &u : us) {
    if (N % u.bn != 0) continue;
    const int64_t tiles = (M + u.bm - 1) / u.bm * (N / u.bn);
    const double t = double((tiles + sms - 1) / sms) * (kb * u.t) + 3.0;
    if (t < best) {
      best = t;
      bm = u.bm;
      bn = u.bn;
    }
  }
  if (M > 512) return;
  struct Split { int bn; double t; };
  const Split sp[2] = {{256, 0.664}, {128, 0.49}};
  for (const auto &c : sp) {
    if (N % c.bn != 0) continue;
    const int64_t tiles = (M + 127) / 128 * (N / c.bn);
    for (int cs = 2; cs <= kGemmMaxSplit; cs *= 2) {
      if (kb < 4.0 * cs) continue;
      const int64_t wave = split_ctas_per_wave(cs);
      const double t = double((tiles * cs + wave - 1) / wave) * (kb / cs * c.t + 11.0);
      if (t < best) {
        best = t;
        bm = 128;
        bn = c.bn;
        split = cs;
      }
    }
  }
}

cudaError_t launch_gemm_dequant(const void *x, int64_t M, int64_t K, const void *codes,
                                const float *scales, int fmt, int64_t G, int64_t N, void *y,
                                int out_dt, cudaStream_t st) {
  int bm = 128, bn = 64, split = 1;
  gemm_tile_shape(M, N, K, bm, bn, split);
  GemmArgs a;
  a.scales = scales;
  a.y = y;
  a.M = M;
  a.N = N;
  a.K = K;
  a.log2G = log2_block(G);
  a.tiles_m = int((M + bm - 1) / bm);
  a.tiles_n = int(N / bn);
  if (out_dt == DT_F32) return go_gemm_fmt<DT_F32>(x, codes, a, fmt, bm, bn, split, st);
  if (out_dt == DT_BF16) return go_gemm_fmt<DT_BF16>(x, codes, a, fmt, bm, bn, split, st);
  return cudaErrorInvalidValue;
}

unsigned take_gemm_device_error() {
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
