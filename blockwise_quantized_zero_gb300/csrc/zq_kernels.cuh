// zq_kernels.cuh -- the libzq kernels (sm_103a): quantize, dequantize,
// quantized reduce and in-place FP8 accumulate.
//
// Work decomposition (all four kernels): a persistent grid of 256-thread CTAs
// strides over "warp tiles" of 1024 consecutive elements. Lane l of a warp
// owns the 16-element runs [e0 + j*512 + 16*l, +16) for j = 0, 1, so every
// warp-wide load and store instruction touches one contiguous span (512 B of
// bf16 per 256-bit load; 2*b bytes of codes per lane). Because G divides
// 1024 and a tile starts at a multiple of 1024, a tile holds whole blocks: a
// block of G <= 512 elements is G/16 adjacent lanes of one j, a block of 1024
// is the whole tile. The block absmax is a shuffle tree over those lanes.
// A tile that runs past n (at most one per call) is processed by a slower
// warp-cooperative tail routine that handles a partial last block.
#pragma once

#include "zq_device.cuh"

namespace zq {

constexpr int kThreads = 256;
constexpr int kU = 2;                      // 16-element runs per lane per tile
constexpr int kTile = 32 * kVec * kU;      // 1024 elements per warp tile
constexpr int kRun = 32 * kVec;            // 512 elements per warp-wide run

// ---------------------------------------------------------------------------
// Layouts of the quantized form. Planar: the codes are one LSB-first bit
// stream and the block scales a separate fp32 array. Interleaved (Aquavit's
// metadata interleaving): one byte stream of block records, record k = block
// k's fp32 scale followed by its codes (G*b/8 bytes), so the record stride
// 4 + G*b/8 is a multiple of 4 bytes but not of 8; integer codes only. The
// quantize and dequantize kernels take the layout as a template flag IL.
// ---------------------------------------------------------------------------
__host__ __device__ constexpr int log2_of(int G) { return G <= 1 ? 0 : 1 + log2_of(G / 2); }

template <int B> __device__ __forceinline__ int64_t il_stride(int lg) {
  return 4 + ((int64_t(B) << lg) >> 3);
}

// Byte offset of the code bits of element e, e the first element of a
// 16-element run or of a block (blocks of 2^lg elements).
template <bool IL, int B> __device__ __forceinline__ int64_t code_off(int64_t e, int lg) {
  if constexpr (IL) {
    const int64_t k = e >> lg;
    return k * il_stride<B>(lg) + 4 + (((e - (k << lg)) * B) >> 3);
  } else {
    return e * B / 8;
  }
}

template <bool IL, int B>
__device__ __forceinline__ void put_codes16(uint8_t *p, const uint32_t (&w)[B / 2]) {
  if constexpr (IL) store_codes16_a4<B>(p, w);
  else store_codes16<B>(p, w);
}

// Store the scale of block k (blocks of 2^lg elements).
template <bool IL, int B>
__device__ __forceinline__ void put_scale(uint8_t *codes, float *scales, int64_t k, int lg,
                                          float s) {
  if constexpr (IL) *reinterpret_cast<float *>(codes + k * il_stride<B>(lg)) = s;
  else scales[k] = s;
}

// Programmatic dependent launch: wait until the previous grid on the stream
// has completed and its writes are visible, then let the next grid be
// scheduled. Every kernel calls this before its first global memory load or
// store (only an L2 prefetch hint may come earlier: see WarpCursor).
__device__ __forceinline__ void pdl_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

struct WarpCursor {
  int lane;
  int64_t warp, nwarps;
  __device__ __forceinline__ WarpCursor() {
    pdl_enter();
    lane = threadIdx.x & 31;
    warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  }
  // The same, first asking L2 for the warp's first input tile (tile_bytes at
  // in + warp * tile_bytes, if the warp has a tile): a prefetch is only a
  // hint, so it may be issued before the previous grid has finished (a
  // write of that grid to the same bytes still reaches L2 after it).
  __device__ __forceinline__ WarpCursor(const void *in, int64_t tile_bytes, int64_t ntiles) {
    lane = threadIdx.x & 31;
    warp = (int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    if (in && warp < ntiles) {
      const char *p = static_cast<const char *>(in) + warp * tile_bytes;
      for (int64_t o = int64_t(lane) * 128; o < tile_bytes; o += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + o));
    }
    pdl_enter();
  }
  // The partial last tile (if any) goes to the warp that would take tile
  // n / kTile in the grid-stride order.
  __device__ __forceinline__ bool owns_tail(int64_t n) const {
    return (n % kTile) != 0 && warp == (n / kTile) % nwarps;
  }
};

// ===========================================================================
// Quantize
// ===========================================================================
// Tensor-slice reordering of the output tiles (qgZ): the tensor is P = A*L
// chunks of tpc tiles, and chunk c = a*L + l is written at slice position
// l*A + a (the transpose of the A x L chunk grid). tpc == 0: no reordering.
struct SliceRemap {
  int A, L;
  int64_t tpc;
  __device__ __forceinline__ int64_t out_tile(int64_t t) const {
    if (tpc == 0) return t;
    const uint32_t c = uint32_t(t / tpc), cl = c % uint32_t(L);
    return (int64_t(cl) * A + c / uint32_t(L)) * tpc + (t - int64_t(c) * tpc);
  }
  __device__ __forceinline__ int64_t in_tile(int64_t o) const {
    if (tpc == 0) return o;
    const uint32_t p = uint32_t(o / tpc), pa = p % uint32_t(A);
    return (int64_t(pa) * L + p / uint32_t(A)) * tpc + (o - int64_t(p) * tpc);
  }
};

// Block scales of one tile. Lane l computes the scale (block_scale: the
// division-free remainder-corrected quotient, bit-identical to the IEEE
// division absmax / qmax) and its reciprocal for block l of the tile (there are 1024 / G <= 32 blocks),
// stores it, and the values are shuffled back to the lanes of each block.
// m[j] is the lane's block absmax for run j (already reduced over the block).
template <int FMT, int G, bool IL>
__device__ __forceinline__ void tile_scales(const float (&m)[kU], float (&s)[kU], float (&r)[kU],
                                            uint8_t *__restrict__ codes,
                                            float *__restrict__ scales, int64_t e0, int lane) {
  constexpr int B = Fmt<FMT>::kBits, LG = log2_of(G);
  if constexpr (G == kTile) {
    const float sb = block_scale<FMT>(fmaxf(m[0], m[1])), rb = safe_rcp(sb);
    s[0] = s[1] = sb;
    r[0] = r[1] = rb;
    if (lane == 0) put_scale<IL, B>(codes, scales, e0 / G, LG, sb);
  } else {
    constexpr int L = G / kVec;          // lanes per block
    constexpr int PER_RUN = kRun / G;    // blocks per run
    constexpr int NB = kTile / G;        // blocks per tile
    // gather: lane l holds the absmax of block l
    const int src = (lane % PER_RUN) * L;
    const float g0 = __shfl_sync(kFull, m[0], src), g1 = __shfl_sync(kFull, m[1], src);
    const float mb = (lane < PER_RUN) ? g0 : g1;
    const float sb = block_scale<FMT>(mb), rb = safe_rcp(sb);
    if (lane < NB) put_scale<IL, B>(codes, scales, e0 / G + lane, LG, sb);
    // scatter: the lanes of block (j, lane / L) fetch its scale
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int owner = j * PER_RUN + lane / L;
      s[j] = __shfl_sync(kFull, sb, owner);
      r[j] = __shfl_sync(kFull, rb, owner);
    }
  }
}

// Runs (16 elements of one lane) that the fast path could not decide are not
// fixed in place, where one flagged lane would hold up its whole warp: they go
// to a per-warp queue in shared memory (start index, block scale and, for
// 16-bit sources, the run's raw words), and the warp fixes them 32 at a time,
// one run per lane, as soon as 32 are queued; the last partial batch is fixed
// when the warp runs out of tiles. A tile adds at most 64 runs to fewer than
// 32 pending ones, so 96 entries suffice.
constexpr int kQueue = 96;
constexpr int kWarps = kThreads / 32;
template <int DT> constexpr bool kStash = (DT != DT_F32);

template <int DT> struct FixQueue {
  int64_t e[kWarps][kQueue];
  float s[kWarps][kQueue];
  uint32_t raw[kStash<DT> ? kWarps : 1][kStash<DT> ? kQueue : 1][kRawWords<DT>];
};

// Fix the queued runs [first, first + count) of warp w: lane i takes entry
// first + i, recomputes its 16 codes with the exact resolution of the
// flagged elements, and overwrites the fast-path code words.
template <int DT, int FMT, int G, bool IL>
__device__ __noinline__ void quantize_flush(FixQueue<DT> &fq, int w, int first, int count,
                                            const void *__restrict__ src,
                                            uint8_t *__restrict__ codes, int lane, bool wide,
                                            const SliceRemap rm) {
  constexpr int B = Fmt<FMT>::kBits, W = Fmt<FMT>::kWords16;
  __syncwarp();  // queue entries and fast-path codes of all lanes are visible
  for (int base = 0; base < count; base += 32) {
    const int i = base + lane;
    if (i < count) {
      const int slot = first + i;
      const int64_t e = fq.e[w][slot];
      const float s = fq.s[w][slot];
      uint32_t raw[kRawWords<DT>];
      if constexpr (kStash<DT>) {
#pragma unroll
        for (int k = 0; k < kRawWords<DT>; ++k) raw[k] = fq.raw[w][slot][k];
      } else {  // e is the output position; the source is read at the input one
        load16_raw<DT>(src, rm.in_tile(e / kTile) * kTile + e % kTile, raw, wide);
      }
      float x[kVec];
      widen16<DT>(raw, x);
      const float r = safe_rcp(s);
      uint8_t *cp = codes + code_off<IL, B>(e, log2_of(G));
      uint32_t wd[W];
      const bool normal = (FMT == F_E4M3) ? scale_is_normal(s) : (s == 0.0f || scale_is_normal(s));
      if (normal && FMT != F_E4M3) {
        quant16_fix<FMT>(x, s, r, 1u, wd);  // recomputes the run; needs no old words
      } else if (normal) {
        ld_v4(cp, wd[0], wd[1], wd[2], wd[3]);  // E4M3: 16 code bytes
        quant16_fix<FMT>(x, s, r, 1u, wd);
      } else {
        quant16_exact<FMT>(x, s, wd);
      }
      put_codes16<IL, B>(cp, wd);
    }
  }
  __syncwarp();
}

template <int DT, int FMT, int G, bool IL>
__device__ __forceinline__ void quantize_tile(const uint32_t (&raw)[kU][kRawWords<DT>],
                                              uint8_t *__restrict__ codes,
                                              float *__restrict__ scales, int64_t e0, int lane,
                                              FixQueue<DT> &fq, int w, int &count) {
  constexpr int B = Fmt<FMT>::kBits, W = Fmt<FMT>::kWords16;
  float x[kU][kVec];
  float m[kU];
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    widen16<DT>(raw[j], x[j]);
    m[j] = absmax16_raw<DT>(raw[j], x[j]);
  }
  if constexpr (G <= kRun) {
#pragma unroll
    for (int j = 0; j < kU; ++j) m[j] = group_max<G / kVec>(m[j]);
  } else {
    m[0] = m[1] = warp_max(fmaxf(m[0], m[1]));
  }
  float s[kU], r[kU];
  tile_scales<FMT, G, IL>(m, s, r, codes, scales, e0, lane);

#pragma unroll
  for (int j = 0; j < kU; ++j) {
    uint32_t wd[W];
    const int64_t e = e0 + j * kRun + lane * kVec;
    const uint32_t flagged = quant16_try_fast<FMT>(x[j], s[j], r[j], wd);
    put_codes16<IL, B>(codes + code_off<IL, B>(e, log2_of(G)), wd);
    const unsigned ballot = __ballot_sync(kFull, flagged != 0u);
    if (ballot) {
      if (flagged) {
        const int slot = count + __popc(ballot & ((1u << lane) - 1u));
        fq.e[w][slot] = e;
        fq.s[w][slot] = s[j];
        if constexpr (kStash<DT>) {
#pragma unroll
          for (int k = 0; k < kRawWords<DT>; ++k) fq.raw[w][slot][k] = raw[j][k];
        }
      }
      count += __popc(ballot);
    }
  }
}

// Exact, warp-cooperative quantization of elements [e0, n) (fewer than one
// tile; e0 is a multiple of G). Each lane builds whole 32-bit code words.
template <int DT, int FMT, int G, bool IL>
__device__ __noinline__ void quantize_tail(const void *__restrict__ src,
                                           uint8_t *__restrict__ codes,
                                           float *__restrict__ scales, int64_t e0, int64_t n,
                                           int lane) {
  constexpr int B = Fmt<FMT>::kBits;
  for (int64_t lo = e0; lo < n; lo += G) {
    uint32_t *cw = reinterpret_cast<uint32_t *>(codes + code_off<IL, B>(lo, log2_of(G)));
    const int64_t hi = (lo + G < n) ? lo + G : n;
    float m = 0.0f;
    for (int64_t i = lo + lane; i < hi; i += 32) m = fmaxf(m, fabsf(load1_f32<DT>(src, i)));
    const float s = block_scale<FMT>(warp_max(m));
    if (lane == 0) put_scale<IL, B>(codes, scales, lo / G, log2_of(G), s);
    const int64_t len = hi - lo, nwords = (len * B + 31) / 32;
    for (int64_t wi = lane; wi < nwords; wi += 32) {
      const int64_t bit0 = wi * 32;
      const int64_t first = bit0 / B;
      const int64_t last = ((bit0 + 32 + B - 1) / B < len) ? (bit0 + 32 + B - 1) / B : len;
      uint32_t word = 0;
      for (int64_t e = first; e < last; ++e) {
        const uint32_t c = code1_exact<FMT>(load1_f32<DT>(src, lo + e), s);
        const int sh = static_cast<int>(e * B - bit0);
        word |= (sh >= 0) ? (c << sh) : (c >> (-sh));
      }
      cw[wi] = word;
    }
  }
}

template <int DT, int FMT, int G, bool IL = false>
__global__ void __launch_bounds__(kThreads, 3) quantize_kernel(const void *__restrict__ src,
                                                            uint8_t *__restrict__ codes,
                                                            float *__restrict__ scales,
                                                            int64_t n, int wide,
                                                            const SliceRemap rm) {
  static_assert(!IL || FMT != F_E4M3, "the interleaved layout holds integer codes");
  const WarpCursor c(src, int64_t(kTile) * (DT == DT_F32 ? 4 : 2), n / kTile);
  const int64_t nfull = n / kTile;
  const bool wd = wide != 0;
  __shared__ FixQueue<DT> fq;
  const int w = threadIdx.x >> 5;
  int count = 0;  // warp-uniform
  // Software pipeline: the loads of tile t + nwarps are in flight while
  // tile t is quantized.
  uint32_t raw[kU][kRawWords<DT>];
  int64_t t = c.warp;
  if (t < nfull) {
#pragma unroll
    for (int j = 0; j < kU; ++j) load16_raw<DT>(src, t * kTile + j * kRun + c.lane * kVec, raw[j], wd);
  }
  for (; t < nfull; t += c.nwarps) {
    uint32_t cur[kU][kRawWords<DT>];
#pragma unroll
    for (int j = 0; j < kU; ++j)
#pragma unroll
      for (int k = 0; k < kRawWords<DT>; ++k) cur[j][k] = raw[j][k];
    const int64_t tn = t + c.nwarps;
    if (tn < nfull) {
#pragma unroll
      for (int j = 0; j < kU; ++j)
        load16_raw<DT>(src, tn * kTile + j * kRun + c.lane * kVec, raw[j], wd);
    }
    quantize_tile<DT, FMT, G, IL>(cur, codes, scales, rm.out_tile(t) * kTile, c.lane, fq, w, count);
    while (count >= 32) {  // fix full batches right away, newest first
      count -= 32;
      quantize_flush<DT, FMT, G, IL>(fq, w, count, 32, src, codes, c.lane, wd, rm);
    }
  }
  if (count) quantize_flush<DT, FMT, G, IL>(fq, w, 0, count, src, codes, c.lane, wd, rm);
  if (c.owns_tail(n)) quantize_tail<DT, FMT, G, IL>(src, codes, scales, nfull * kTile, n, c.lane);
}

// ---------------------------------------------------------------------------
// Multi-tensor quantize: one launch over a list of tensors (same element
// type, format and block size). The full tiles of all tensors are numbered
// consecutively (tensor k owns tiles [tile0[k], tile0[k+1])) and walked in
// the same grid-stride order as one large tensor, so the warps stream one
// narrow window of memory at a time. A queued fix-up run also records its
// tensor, so the queue is flushed in full batches as in quantize_kernel.
// Each tensor's partial last tile goes to warp k % nwarps.
// ---------------------------------------------------------------------------
constexpr int kMultiMax = 256;  // tensors per launch (the list travels in the kernel parameters)

struct MultiArgs {
  const void *src[kMultiMax];
  uint8_t *codes[kMultiMax];
  float *scales[kMultiMax];
  int64_t n[kMultiMax];
  int64_t tile0[kMultiMax + 1];  // prefix sums of full tiles
  int count;
  int wide;
};

// Fix the queued runs [first, first + count) of warp w, each in its own
// tensor (quantize_flush with per-entry source and code pointers).
template <int DT, int FMT, int G>
__device__ __noinline__ void quantize_flush_multi(FixQueue<DT> &fq, const int16_t (&fk)[kQueue],
                                                  int w, int first, int count, const MultiArgs &a,
                                                  int lane, bool wide) {
  constexpr int B = Fmt<FMT>::kBits, W = Fmt<FMT>::kWords16;
  __syncwarp();
  for (int base = 0; base < count; base += 32) {
    const int i = base + lane;
    if (i < count) {
      const int slot = first + i;
      const int64_t e = fq.e[w][slot];
      const float s = fq.s[w][slot];
      const int k = fk[slot];
      uint32_t raw[kRawWords<DT>];
      if constexpr (kStash<DT>) {
#pragma unroll
        for (int q = 0; q < kRawWords<DT>; ++q) raw[q] = fq.raw[w][slot][q];
      } else {
        load16_raw<DT>(a.src[k], e, raw, wide);
      }
      float x[kVec];
      widen16<DT>(raw, x);
      const float r = safe_rcp(s);
      uint8_t *cp = a.codes[k] + code_off<false, B>(e, log2_of(G));
      uint32_t wd[W];
      const bool normal = (FMT == F_E4M3) ? scale_is_normal(s) : (s == 0.0f || scale_is_normal(s));
      if (normal && FMT != F_E4M3) {
        quant16_fix<FMT>(x, s, r, 1u, wd);
      } else if (normal) {
        ld_v4(cp, wd[0], wd[1], wd[2], wd[3]);
        quant16_fix<FMT>(x, s, r, 1u, wd);
      } else {
        quant16_exact<FMT>(x, s, wd);
      }
      put_codes16<false, B>(cp, wd);
    }
  }
  __syncwarp();
}

template <int DT, int FMT, int G>
__global__ void __launch_bounds__(kThreads, 3) quantize_multi_kernel(const __grid_constant__ MultiArgs a) {
  const WarpCursor c;
  const bool wd = a.wide != 0;
  const int64_t total = a.tile0[a.count];
  __shared__ FixQueue<DT> fq;
  __shared__ int16_t fqk[kWarps][kQueue];  // tensor of each queued run
  const int w = threadIdx.x >> 5;
  int count = 0;  // warp-uniform
  uint32_t raw[kU][kRawWords<DT>];
  int k = 0, kn = 0;  // tensors of the current and the next tile (they only grow)
  auto load_tile = [&](int64_t t, int kk) {
    const int64_t e0 = (t - a.tile0[kk]) * kTile;
#pragma unroll
    for (int j = 0; j < kU; ++j) load16_raw<DT>(a.src[kk], e0 + j * kRun + c.lane * kVec, raw[j], wd);
  };
  if (c.warp < total) {
    while (c.warp >= a.tile0[kn + 1]) ++kn;
    load_tile(c.warp, kn);
  }
  for (int64_t t = c.warp; t < total; t += c.nwarps) {
    uint32_t cur[kU][kRawWords<DT>];
#pragma unroll
    for (int j = 0; j < kU; ++j)
#pragma unroll
      for (int q = 0; q < kRawWords<DT>; ++q) cur[j][q] = raw[j][q];
    k = kn;
    const int64_t tn = t + c.nwarps;
    if (tn < total) {
      while (tn >= a.tile0[kn + 1]) ++kn;
      load_tile(tn, kn);
    }
    const int c0 = count;
    quantize_tile<DT, FMT, G, false>(cur, a.codes[k], a.scales[k], (t - a.tile0[k]) * kTile,
                                     c.lane, fq, w, count);
    for (int i = c0 + c.lane; i < count; i += 32) fqk[w][i] = int16_t(k);
    while (count >= 32) {  // fix full batches right away, newest first
      count -= 32;
      quantize_flush_multi<DT, FMT, G>(fq, fqk[w], w, count, 32, a, c.lane, wd);
    }
  }
  if (count) quantize_flush_multi<DT, FMT, G>(fq, fqk[w], w, 0, count, a, c.lane, wd);
  for (int kk = int(c.warp); kk < a.count; kk += int(c.nwarps)) {
    if (a.n[kk] % kTile)
      quantize_tail<DT, FMT, G, false>(a.src[kk], a.codes[kk], a.scales[kk],
                                       (a.n[kk] / kTile) * kTile, a.n[kk], c.lane);
  }
}

// ===========================================================================
// Dequantize
// ===========================================================================
// Tiles in flight per warp: 6 for codes of up to 4 bits, 4 for wider codes
// (whose larger register slots would otherwise cost occupancy).
template <int FMT> constexpr int kDequantAhead = Fmt<FMT>::kBits <= 4 ? 6 : 4;

template <int FMT, int DT, bool IL = false>
__global__ void __launch_bounds__(kThreads) dequantize_kernel(const uint8_t *__restrict__ codes,
                                                              const float *__restrict__ scales,
                                                              void *__restrict__ dst, int64_t n,
                                                              int log2G, int wide) {
  constexpr int B = Fmt<FMT>::kBits, W = Fmt<FMT>::kWords16;
  static_assert(!IL || FMT != F_E4M3, "the interleaved layout holds integer codes");
  const WarpCursor c(IL ? nullptr : codes, int64_t(kTile) * B / 8, n / kTile);
  const int64_t nfull = n / kTile;
  const bool wd = wide != 0;
  // Software pipeline: the codes and scales of the warp's next PF tiles are
  // in flight (a ring of register slots) while tile t is decoded and
  // stored; the loads are small, so several are needed to cover the latency.
  constexpr int PF = kDequantAhead<FMT>;
  uint32_t w[PF][kU][W];
  float s[PF][kU];
  auto load = [&](int64_t tile, uint32_t (&wd_)[kU][W], float (&sd_)[kU]) {
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t e = tile * kTile + j * kRun + c.lane * kVec;
      if constexpr (IL) {  // the run's record: scale, then codes
        const int64_t k = e >> log2G;
        const uint8_t *rec = codes + k * il_stride<B>(log2G);
        load_codes16_a4<B>(rec + 4 + (((e - (k << log2G)) * B) >> 3), wd_[j]);
        sd_[j] = ld_nc_f32(reinterpret_cast<const float *>(rec));
      } else {
        load_codes16<B>(codes + e * B / 8, wd_[j]);
        sd_[j] = ld_nc_f32(scales + (e >> log2G));
      }
    }
  };
#pragma unroll
  for (int k = 0; k < PF; ++k)
    if (c.warp + k * c.nwarps < nfull) load(c.warp + k * c.nwarps, w[k], s[k]);
  for (int64_t t = c.warp; t < nfull;) {
#pragma unroll
    for (int k = 0; k < PF; ++k) {  // slot k holds tile t
      if (t < nfull) {
        uint32_t wc[kU][W];
        float sc[kU];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          sc[j] = s[k][j];
#pragma unroll
          for (int q = 0; q < W; ++q) wc[j][q] = w[k][j][q];
        }
        const int64_t tn = t + PF * c.nwarps;
        if (tn < nfull) load(tn, w[k], s[k]);
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          float y[kVec];
          dequant16<FMT>(wc[j], sc[j], y);
          store16<DT>(dst, t * kTile + j * kRun + c.lane * kVec, y, wd);
        }
        t += c.nwarps;
      }
    }
  }
  if (c.owns_tail(n)) {
    for (int64_t i = nfull * kTile + c.lane; i < n; i += 32) {
      if constexpr (IL) {
        const int64_t k = i >> log2G;
        const uint8_t *rec = codes + k * il_stride<B>(log2G);
        store1<DT>(dst, i, dequant1<FMT>(rec + 4, i - (k << log2G),
                                         *reinterpret_cast<const float *>(rec)));
      } else {
        store1<DT>(dst, i, dequant1<FMT>(codes, i, scales[i >> log2G]));
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Multi-tensor dequantize: the dequantize kernel over a list of tensors (same
// format, block size and output type), their full tiles numbered
// consecutively and walked in grid-stride order with the same ring of tiles
// in flight; each ring slot remembers its tile's tensor. Each tensor's
// partial last tile goes to warp k % nwarps.
// ---------------------------------------------------------------------------
struct DequantMultiArgs {
  const uint8_t *codes[kMultiMax];
  const float *scales[kMultiMax];
  void *dst[kMultiMax];
  int64_t n[kMultiMax];
  int64_t tile0[kMultiMax + 1];  // prefix sums of full tiles
  int count;
  int log2G;
  int wide;
};

template <int FMT, int DT>
__global__ void __launch_bounds__(kThreads) dequantize_multi_kernel(
    const __grid_constant__ DequantMultiArgs a) {
  constexpr int B = Fmt<FMT>::kBits, W = Fmt<FMT>::kWords16;
  const WarpCursor c;
  const int64_t total = a.tile0[a.count];
  const bool wd = a.wide != 0;
  const int lg = a.log2G;
  constexpr int PF = kDequantAhead<FMT>;
  uint32_t w[PF][kU][W];
  float s[PF][kU];
  int ks[PF];
  int kl = 0;  // tensor of the last tile loaded (tiles are loaded in increasing order)
  auto load = [&](int64_t tile, uint32_t (&wd_)[kU][W], float (&sd_)[kU], int &k_) {
    while (tile >= a.tile0[kl + 1]) ++kl;
    k_ = kl;
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t e = (tile - a.tile0[kl]) * kTile + j * kRun + c.lane * kVec;
      load_codes16<B>(a.codes[kl] + e * B / 8, wd_[j]);
      sd_[j] = ld_nc_f32(a.scales[kl] + (e >> lg));
    }
  };
#pragma unroll
  for (int k = 0; k < PF; ++k) {
    ks[k] = 0;
    if (c.warp + k * c.nwarps < total) load(c.warp + k * c.nwarps, w[k], s[k], ks[k]);
  }
  for (int64_t t = c.warp; t < total;) {
#pragma unroll
    for (int k = 0; k < PF; ++k) {  // slot k holds tile t
      if (t < total) {
        uint32_t wc[kU][W];
        float sc[kU];
        const int kt = ks[k];
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          sc[j] = s[k][j];
#pragma unroll
          for (int q = 0; q < W; ++q) wc[j][q] = w[k][j][q];
        }
        const int64_t tn = t + PF * c.nwarps;
        if (tn < total) load(tn, w[k], s[k], ks[k]);
        const int64_t e0 = (t - a.tile0[kt]) * kTile;
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          float y[kVec];
          dequant16<FMT>(wc[j], sc[j], y);
          store16<DT>(a.dst[kt], e0 + j * kRun + c.lane * kVec, y, wd);
        }
        t += c.nwarps;
      }
    }
  }
  for (int kk = int(c.warp); kk < a.count; kk += int(c.nwarps)) {
    for (int64_t i = (a.n[kk] / kTile) * kTile + c.lane; i < a.n[kk]; i += 32)
      store1<DT>(a.dst[kk], i, dequant1<FMT>(a.codes[kk], i, a.scales[kk][i >> lg]));
  }
}

// ===========================================================================
// Quantized reduce: acc = +0; acc = fl(acc + fl(D(shard r))) for r in order;
// then requantize acc with (FOUT, Gout).
// ===========================================================================
constexpr int kMaxShards = 64;

struct ReduceArgs {
  const uint8_t *codes[kMaxShards];
  const float *scales[kMaxShards];
  uint8_t *out_codes;
  float *out_scales;
  float *sum_out;
  int64_t n;
  int nshards;
  int log2Gin;
  int log2Gout;
  int wide;
  float one;  // 1.0f, passed at run time (see accumulate16)
  // one problem per launch
  __device__ int problems() const { return 1; }
  __device__ const uint8_t *shard_codes(int, int r) const { return codes[r]; }
  __device__ const float *shard_scales(int, int r) const { return scales[r]; }
  __device__ uint8_t *out_codes_of(int) const { return out_codes; }
  __device__ float *out_scales_of(int) const { return out_scales; }
  __device__ float *sum_out_of(int) const { return sum_out; }
};

// The same arguments with the shard pointers in a device-memory table instead
// of the kernel parameters (up to kStaticMaxShards shards).
constexpr int kStaticMaxShards = 1024;
struct ShardTable {
  const uint8_t *codes[kStaticMaxShards];
  const float *scales[kStaticMaxShards];
};
struct TableReduceArgs {
  const ShardTable *tab;
  uint8_t *out_codes;
  float *out_scales;
  float *sum_out;
  int64_t n;
  int nshards;
  int log2Gin;
  int log2Gout;
  int wide;
  float one;
  __device__ int problems() const { return 1; }
  __device__ const uint8_t *shard_codes(int, int r) const { return tab->codes[r]; }
  __device__ const float *shard_scales(int, int r) const { return tab->scales[r]; }
  __device__ uint8_t *out_codes_of(int) const { return out_codes; }
  __device__ float *out_scales_of(int) const { return out_scales; }
  __device__ float *sum_out_of(int) const { return sum_out; }
};

// One hop of qgZ's two-hop reduce: P problems of equal length in one launch
// (P = A*L <= kMaxShards GPUs). Problem p = a*L + l is GPU p's reduce. Hop 1:
// shard r is part l (offset l*part elements, part = A*m) of GPU a*L + r's
// input. Hop 2: shard r is chunk a (offset a*part, part = m) of GPU r*L + l's
// hop-1 result.
struct HopArgs {
  const uint8_t *in_codes[kMaxShards];  // per GPU
  const float *in_scales[kMaxShards];
  uint8_t *out_codes[kMaxShards];       // per problem
  float *out_scales[kMaxShards];
  float *sums[kMaxShards];              // entries may be null
  int64_t n;                            // elements per problem
  int64_t part;
  int nprob, nshards, log2Gin, log2Gout, wide;
  float one;
  int hop, A, L, bits_in;
  __device__ int problems() const { return nprob; }
  __device__ int gpu_of(int p, int r) const { return hop == 1 ? (p / L) * L + r : r * L + p % L; }
  __device__ int64_t off_of(int p) const {
    return (hop == 1 ? int64_t(p % L) : int64_t(p / L)) * part;
  }
  __device__ const uint8_t *shard_codes(int p, int r) const {
    return in_codes[gpu_of(p, r)] + off_of(p) * bits_in / 8;
  }
  __device__ const float *shard_scales(int p, int r) const {
    return in_scales[gpu_of(p, r)] + (off_of(p) >> log2Gin);
  }
  __device__ uint8_t *out_codes_of(int p) const { return out_codes[p]; }
  __device__ float *out_scales_of(int p) const { return out_scales[p]; }
  __device__ float *sum_out_of(int p) const { return sums[p]; }
};

// One problem of a reduce launch, with the member names the requantization
// and tail routines use.
// (The accessors read the kernel parameters where they are used, so that a
// one-problem launch keeps no copies of its pointers in registers.)
template <typename A> struct RedView {
  const A *a;
  int p;
  __device__ const uint8_t *shard_codes(int r) const { return a->shard_codes(p, r); }
  __device__ const float *shard_scales(int r) const { return a->shard_scales(p, r); }
  __device__ uint8_t *codes_out() const { return a->out_codes_of(p); }
  __device__ float *scales_out() const { return a->out_scales_of(p); }
  __device__ float *sums_out() const { return a->sum_out_of(p); }
  __device__ int64_t n() const { return a->n; }
  __device__ int nshards() const { return a->nshards; }
  __device__ int log2Gin() const { return a->log2Gin; }
  __device__ int log2Gout() const { return a->log2Gout; }
};

template <typename A> __device__ __forceinline__ RedView<A> view_of(const A &a, int p) {
  return RedView<A>{&a, p};
}

// Add shard r's 16 dequantized values into acc: acc = fl(acc + fl(q * s)).
// ptxas contracts a packed mul.rn.f32x2 feeding a packed add.rn.f32x2 into a
// fused multiply-add (even with the explicit .rn and -fmad=false), which
// would skip the rounding of the product. The add is therefore written as a
// packed fma of the rounded product with `one`, a 1.0f that arrives at run
// time: fl(d * 1 + acc) = fl(d + acc) exactly, and since ptxas cannot know
// that `one` is 1, it can neither drop the multiply nor fold the product in.
// FIRST: acc = fl(+0 + d) for the first shard (the sum starts at +0; the
// addend is the constant 0, so the registers need no clearing).
template <int FIN, bool FIRST = false>
__device__ __forceinline__ void accumulate16(float (&acc)[kVec],
                                             const uint32_t (&w)[Fmt<FIN>::kWords16], float s,
                                             float one) {
  float d[kVec];
  dequant16<FIN>(w, s, d);
#pragma unroll
  for (int v = 0; v < kVec; v += 2) {
    if constexpr (FIRST)
      fma2(acc[v], acc[v + 1], d[v], d[v + 1], one, one, 0.0f, 0.0f);
    else
      fma2(acc[v], acc[v + 1], d[v], d[v + 1], one, one, acc[v], acc[v + 1]);
  }
}

// Requantize the sums of one tile of KU runs (KU*512 elements) with block
// size 2^log2Gout (run time). As in quantize: the block absmax is a shuffle
// tree over the G/16 lanes of a block; lane l then computes the scale of
// block l of the tile (block_scale: division-free, bit-identical to the IEEE
// division) and its reciprocal, stores it, and the lanes of each block fetch
// them back with a shuffle.
template <int FOUT, int KU, typename A>
__device__ __forceinline__ void requant_tile(const A &a, float (&acc)[KU][kVec],
                                             int64_t e0, int lane) {
  constexpr int B = Fmt<FOUT>::kBits, W = Fmt<FOUT>::kWords16;
  const int lg = a.log2Gout();                 // 5 .. 10, and G <= KU * 512
  float m[KU], s[KU], r[KU];
#pragma unroll
  for (int j = 0; j < KU; ++j) m[j] = absmax16(acc[j]);
  if (lg - 4 <= 5) {                         // a block lies within one run
    const int L = 1 << (lg - 4);             // lanes per block
#pragma unroll
    for (int j = 0; j < KU; ++j) m[j] = group_max_rt(m[j], L);
    const int per_run = 32 >> (lg - 4);      // blocks per run
    const int src = (lane & (per_run - 1)) << (lg - 4);
    float mb = __shfl_sync(kFull, m[0], src);
    if constexpr (KU == 2) {
      const float m1 = __shfl_sync(kFull, m[1], src);
      mb = (lane < per_run) ? mb : m1;
    }
    const float sb = block_scale<FOUT>(mb), rb = safe_rcp(sb);
    if (lane < per_run * KU) a.scales_out()[(e0 >> lg) + lane] = sb;
#pragma unroll
    for (int j = 0; j < KU; ++j) {
      const int owner = j * per_run + (lane >> (lg - 4));
      s[j] = __shfl_sync(kFull, sb, owner);
      r[j] = __shfl_sync(kFull, rb, owner);
    }
  } else {                                   // G = 1024 = the whole two-run tile
    const float mt = warp_max(KU == 2 ? fmaxf(m[0], m[KU - 1]) : m[0]);
    const float sb = block_scale<FOUT>(mt), rb = safe_rcp(sb);
#pragma unroll
    for (int j = 0; j < KU; ++j) {
      s[j] = sb;
      r[j] = rb;
    }
    if (lane == 0) a.scales_out()[e0 >> lg] = sb;
  }
  uint32_t w[KU][W];
#pragma unroll
  for (int j = 0; j < KU; ++j) {
    const uint32_t flagged = quant16_try_fast<FOUT>(acc[j], s[j], r[j], w[j]);
    if (flagged) quant16_fix<FOUT>(acc[j], s[j], r[j], flagged, w[j]);
  }
#pragma unroll
  for (int j = 0; j < KU; ++j)
    store_codes16<B>(a.codes_out() + (e0 + j * kRun + lane * kVec) * B / 8, w[j]);
}

// Sum over shards of element i (tails).
template <int FIN, typename A> __device__ __forceinline__ float reduce1(const A &a, int64_t i) {
  float acc = 0.0f;
  for (int r = 0; r < a.nshards(); ++r)
    acc = __fadd_rn(acc, dequant1<FIN>(a.shard_codes(r), i, a.shard_scales(r)[i >> a.log2Gin()]));
  return acc;
}

template <int FIN, int FOUT, typename A>
__device__ __noinline__ void reduce_tail(const A &a, int64_t e0, int lane) {
  constexpr int B = Fmt<FOUT>::kBits;
  const int64_t n = a.n(), Gout = int64_t(1) << a.log2Gout();
  uint32_t *cw = reinterpret_cast<uint32_t *>(a.codes_out());
  for (int64_t lo = e0; lo < n; lo += Gout) {
    const int64_t hi = (lo + Gout < n) ? lo + Gout : n;
    float m = 0.0f;
    for (int64_t i = lo + lane; i < hi; i += 32) {
      const float v = reduce1<FIN, A>(a, i);
      if (a.sums_out()) a.sums_out()[i] = v;
      m = fmaxf(m, fabsf(v));
    }
    const float s = block_scale<FOUT>(warp_max(m));
    if (lane == 0) a.scales_out()[lo >> a.log2Gout()] = s;
    const int64_t len = hi - lo, nwords = (len * B + 31) / 32, w0 = lo * B / 32;
    for (int64_t wi = lane; wi < nwords; wi += 32) {
      const int64_t bit0 = wi * 32, first = bit0 / B;
      const int64_t last = ((bit0 + 32 + B - 1) / B < len) ? (bit0 + 32 + B - 1) / B : len;
      uint32_t word = 0;
      for (int64_t e = first; e < last; ++e) {
        const uint32_t c = code1_exact<FOUT>(reduce1<FIN, A>(a, lo + e), s);
        const int sh = static_cast<int>(e * B - bit0);
        word |= (sh >= 0) ? (c << sh) : (c >> (-sh));
      }
      cw[w0 + wi] = word;
    }
  }
}

// Codes of one lane-vector (16 codes, 2*b bytes) from shared memory.
template <int BITS>
__device__ __forceinline__ void load_codes16_smem(const uint8_t *p, uint32_t (&w)[BITS / 2]) {
  if constexpr (BITS == 2) {
    w[0] = *reinterpret_cast<const uint32_t *>(p);
  } else if constexpr (BITS == 4) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    w[0] = v.x;
    w[1] = v.y;
  } else if constexpr (BITS == 6) {  // 12 bytes at a 4-byte aligned offset
    const uint32_t *q = reinterpret_cast<const uint32_t *>(p);
    w[0] = q[0];
    w[1] = q[1];
    w[2] = q[2];
  } else {
    const uint4 v = *reinterpret_cast<const uint4 *>(p);
    w[0] = v.x;
    w[1] = v.y;
    w[2] = v.z;
    w[3] = v.w;
  }
}

// Shared-memory pipeline of the reduce (warp-specialized). A CTA has eight
// consumer warps and one producer warp. A CTA tile is eight consecutive
// 1024-element tiles (one per consumer warp); a unit is one CTA tile of
// kShards consecutive shards. For every shard of a unit the producer brings
// in the codes of the CTA tile with one bulk copy (and its scales with
// another when their byte count is a multiple of 16, i.e. always for
// G_in <= 256 and for whole CTA tiles), into one of kStages stage buffers.
// Each stage has a "full" barrier (armed by the producer with the byte count)
// and an "empty" barrier (one arrival per consumer warp once it has read the
// stage).
constexpr int kRedConsumers = 8;
constexpr int kRedThreads = (kRedConsumers + 1) * 32;

// Stage geometry, per the CTAs an SM holds (OCC, the kernel's launch bound;
// measured on 134M int4 elements). OCC = 2 (up to 96 registers a thread):
// 2-bit codes use four stages of up to 24 KB, wider codes two stages of up
// to 40 KB (8 int4 shards a unit: more shards per unit, fewer unit
// overheads). OCC = 3 (up to 72 registers), for launches of at most
// kFewShards shards, where the requantization after every few shards is
// latency-bound and more warps hide it: three stages of up to 24 KB (2
// shards 168 -> 139 us, 4 shards 133 -> 129 us; 8 shards would lose, 194.5
// -> 217 us).
constexpr int kFewShards = 4;

template <int FIN, int OCC = 2> struct RedGeom {
  static_assert(OCC == 2 || OCC == 3, "reduce geometries exist for 2 and 3 CTAs an SM");
  static constexpr int kCodeBytes = kTile * Fmt<FIN>::kBits / 8;  // one shard, one tile
  static constexpr int kShardBytes =                               // codes + room for G_in = 32
      kRedConsumers * kCodeBytes + kRedConsumers * (kTile / 32) * 4;
  static constexpr int kBudget = (OCC == 3 || Fmt<FIN>::kBits <= 2) ? 24576 : 40960;
  static constexpr int kShards = (kBudget / kShardBytes) > 1 ? kBudget / kShardBytes : 1;
  static constexpr int kScaleOff = kShards * kRedConsumers * kCodeBytes;
  static constexpr int kStage = kShards * kShardBytes;
  static constexpr int kStages = OCC == 3 ? 3 : (Fmt<FIN>::kBits <= 2 ? 4 : 2);
  static constexpr int kBarOff = kStages * kStage;
  static constexpr int kSmem = kBarOff + kStages * 16;  // full + empty barrier per stage
  static_assert(kCodeBytes % 16 == 0 && kStage % 16 == 0, "bulk copies need 16-byte multiples");
};

// Device error word of this translation unit (read by zq_device_status).
static __device__ unsigned int g_dev_error = 0;

template <int FIN, int FOUT, typename A, int OCC = 2>
__global__ void __launch_bounds__(kRedThreads, OCC)
    reduce_kernel(const __grid_constant__ A a) {
  using RG = RedGeom<FIN, OCC>;
  constexpr int BIN = Fmt<FIN>::kBits, WIN = Fmt<FIN>::kWords16, CB = RG::kCodeBytes;
  constexpr int S = RG::kStages;
  extern __shared__ __align__(128) uint8_t red_smem[];
  pdl_enter();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t full0 = smem_addr(red_smem + RG::kBarOff), empty0 = full0 + 8 * S;
  const int64_t nfull = a.n / kTile;                                 // whole 1024-element tiles
  const int64_t nct = (nfull + kRedConsumers - 1) / kRedConsumers;   // CTA tiles per problem
  const int64_t nctall = nct * a.problems();                         // CTA tiles of the launch
  const int nb = (a.nshards + RG::kShards - 1) / RG::kShards;        // units per CTA tile
  const int64_t mytiles =
      blockIdx.x < nctall ? (nctall - 1 - int64_t(blockIdx.x)) / gridDim.x + 1 : 0;
  const int64_t nunits = mytiles * nb;
  const int lgin = a.log2Gin;
  const int nbt = kTile >> lgin;  // input blocks per tile

  if (threadIdx.x == 0) {
#pragma unroll
    for (int st = 0; st < S; ++st) {
      mbar_init(full0 + 8 * st, 1);
      mbar_init(empty0 + 8 * st, kRedConsumers);
    }
    mbar_init_fence();
  }
  __syncthreads();

  if (w == kRedConsumers) {  // producer warp: lane 0 issues every copy
    if (lane != 0) return;
    // cursor of unit u: problem p, its CTA tile ct, shard batch k
    int p = nct > 0 ? int(blockIdx.x / nct) : 0;
    int64_t ct = blockIdx.x - int64_t(p) * nct;
    int k = 0;
    for (int64_t u = 0; u < nunits; ++u) {
      const int st = int(u % S);
      if (u >= S && !mbar_wait_thread(empty0 + 8 * st, uint32_t(u / S - 1) & 1u)) {
        // Timed out: record it, wait (bounded) for the copies in flight, stop.
        atomicOr(&g_dev_error, kDevErrWaitTimeout);
        for (int64_t v = u - S; v < u; ++v)
          (void)mbar_wait_thread(full0 + 8 * int(v % S), uint32_t(v / S) & 1u);
        return;
      }
      const int r0 = k * RG::kShards;
      const int ns = min(RG::kShards, a.nshards - r0);
      const int64_t left = nfull - ct * kRedConsumers;
      const int cnt = int(left < kRedConsumers ? left : kRedConsumers);
      const uint32_t cbytes = uint32_t(cnt) * CB, sbytes = uint32_t(cnt * nbt) * 4u;
      const bool stma = (sbytes % 16u) == 0u;
      const uint32_t full = full0 + 8 * st;
      const uint32_t dst = smem_addr(red_smem + st * RG::kStage);
      fence_proxy_async_smem();
      mbar_arrive_expect_tx(full, uint32_t(ns) * (cbytes + (stma ? sbytes : 0u)));
      for (int q = 0; q < ns; ++q) {
        bulk_g2s(dst + q * kRedConsumers * CB, a.shard_codes(p, r0 + q) + ct * kRedConsumers * CB,
                 cbytes, full);
        if (stma)
          bulk_g2s(dst + RG::kScaleOff + q * kRedConsumers * nbt * 4,
                   a.shard_scales(p, r0 + q) + ct * kRedConsumers * nbt, sbytes, full);
      }
      if (++k == nb) {
        k = 0;
        for (ct += gridDim.x; ct >= nct && p < a.problems(); ct -= nct) ++p;
      }
    }
    return;
  }

  // consumer warp w: tile w of every CTA tile
  float acc[kU][kVec];
  // cursor of unit u: problem p, its CTA tile ct, shard batch k
  int p = nct > 0 ? int(blockIdx.x / nct) : 0;
  int64_t ct = blockIdx.x - int64_t(p) * nct;
  int k = 0;
  RedView<A> v = view_of(a, p < a.problems() ? p : 0);
  for (int64_t u = 0; u < nunits; ++u) {
    const int st = int(u % S);
    if (!mbar_wait_warp(full0 + 8 * st, uint32_t(u / S) & 1u)) {
      if (lane == 0) atomicOr(&g_dev_error, kDevErrWaitTimeout);
      return;
    }
    const int r0 = k * RG::kShards;
    const int ns = min(RG::kShards, a.nshards - r0);
    const int64_t left = nfull - ct * kRedConsumers;
    const int cnt = int(left < kRedConsumers ? left : kRedConsumers);
    const bool stma = ((cnt * nbt * 4) % 16) == 0;
    const int64_t e0 = (ct * kRedConsumers + w) * kTile;
    if (w < cnt) {
      const uint8_t *sb = red_smem + st * RG::kStage;
      // shard q of the unit: codes from the stage, scale from the stage or
      // from global memory (G_in >= 512 at the end of the tensor); the first
      // shard of a tile starts the sum
      auto shard = [&](int q, auto first, auto scales_in_stage) {
        const uint8_t *cq = sb + (q * kRedConsumers + w) * CB;
        const float *sq =
            reinterpret_cast<const float *>(sb + RG::kScaleOff) + (q * kRedConsumers + w) * nbt;
#pragma unroll
        for (int j = 0; j < kU; ++j) {
          const int off = j * kRun + lane * kVec;
          uint32_t wv[WIN];
          load_codes16_smem<BIN>(cq + off * BIN / 8, wv);
          const float s = decltype(scales_in_stage)::value
                              ? sq[off >> lgin]
                              : ld_nc_f32(v.shard_scales(r0 + q) + ((e0 + off) >> lgin));
          accumulate16<FIN, decltype(first)::value>(acc[j], wv, s, a.one);
        }
      };
      using T = std::true_type;
      using F = std::false_type;
      if (stma) {
        if (k == 0) shard(0, T{}, T{}); else shard(0, F{}, T{});
#pragma unroll
        for (int q = 1; q < RG::kShards; ++q)
          if (q < ns) shard(q, F{}, T{});  // shard order is the summation order
      } else {
        if (k == 0) shard(0, T{}, F{}); else shard(0, F{}, F{});
        for (int q = 1; q < ns; ++q) shard(q, F{}, F{});
      }
    }
    __syncwarp();  // every lane has read the stage
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
    if (k == nb - 1 && w < cnt) {  // last unit of the tile
      if (float *so = v.sums_out()) {
#pragma unroll
        for (int j = 0; j < kU; ++j)
          store16<DT_F32>(so, e0 + j * kRun + lane * kVec, acc[j], a.wide != 0);
      }
      requant_tile<FOUT, kU, RedView<A>>(v, acc, e0, lane);
    }
    if (++k == nb) {
      k = 0;
      for (ct += gridDim.x; ct >= nct && p < a.problems(); ct -= nct) ++p;
      v.p = p;
    }
  }
  // the partial last tile (fewer than 1024 elements) of every problem goes to
  // warp 0 of CTA 0
  if ((a.n % kTile) != 0 && blockIdx.x == 0 && w == 0)
    for (int p = 0; p < a.problems(); ++p)
      reduce_tail<FIN, FOUT, RedView<A>>(view_of(a, p), nfull * kTile, lane);
}

// ===========================================================================
// FP8 accumulate, in place: v = fl(fl(e4m3(c) * s) + g); requantize to E4M3.
// Each warp reads and rewrites only its own tile (codes and block scales),
// and every lane reads the old scale before the block-max shuffle that
// precedes the new scale's store, so the in-place update is race free.
// ===========================================================================
template <int DT, int G>
__device__ __forceinline__ void fp8acc_tile(uint8_t *codes, float *scales,
                                            const void *__restrict__ grad, int64_t e0, int lane,
                                            bool wide, float one) {
  float v[kU][kVec];
  uint32_t w[kU][4];
  float sold[kU];
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const int64_t e = e0 + j * kRun + lane * kVec;
    ld_v4(codes + e, w[j][0], w[j][1], w[j][2], w[j][3]);
    sold[j] = scales[e / G];
    load16_f32<DT>(grad, e, v[j], wide);
  }
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    float d[kVec];
    dequant16<F_E4M3>(w[j], sold[j], d);
    // v = fl(d + g) as a packed fma with the run-time 1.0f (see accumulate16)
#pragma unroll
    for (int k = 0; k < kVec; k += 2)
      fma2(v[j][k], v[j][k + 1], d[k], d[k + 1], one, one, v[j][k], v[j][k + 1]);
  }
  float s[kU], r[kU];
  if constexpr (G <= kRun) {
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      s[j] = block_scale<F_E4M3>(group_max<G / kVec>(absmax16(v[j])));
      r[j] = safe_rcp(s[j]);
      if ((lane & (G / kVec - 1)) == 0) scales[(e0 + j * kRun + lane * kVec) / G] = s[j];
    }
  } else {
    const float m = warp_max(fmaxf(absmax16(v[0]), absmax16(v[1])));
    s[0] = s[1] = block_scale<F_E4M3>(m);
    r[0] = r[1] = safe_rcp(s[0]);
    if (lane == 0) scales[e0 / G] = s[0];
  }
#pragma unroll
  for (int j = 0; j < kU; ++j) {
    const uint32_t flagged = quant16_try_fast<F_E4M3>(v[j], s[j], r[j], w[j]);
    if (flagged) quant16_fix<F_E4M3>(v[j], s[j], r[j], flagged, w[j]);
  }
#pragma unroll
  for (int j = 0; j < kU; ++j)
    st_v4(codes + e0 + j * kRun + lane * kVec, w[j][0], w[j][1], w[j][2], w[j][3]);
}

template <int DT, int G>
__device__ __noinline__ void fp8acc_tail(uint8_t *codes, float *scales,
                                         const void *__restrict__ grad, int64_t e0, int64_t n,
                                         int lane) {
  for (int64_t lo = e0; lo < n; lo += G) {
    const int64_t hi = (lo + G < n) ? lo + G : n;
    const float sold = scales[lo / G];
    float m = 0.0f;
    for (int64_t i = lo + lane; i < hi; i += 32)
      m = fmaxf(m, fabsf(__fadd_rn(__fmul_rn(f32_from_e4m3(codes[i]), sold),
                                   load1_f32<DT>(grad, i))));
    const float s = block_scale<F_E4M3>(warp_max(m));
    // every lane has read `sold` and the old codes of its words before any
    // lane writes: the codes of one word are read and written by one lane
    const int64_t len = hi - lo, nwords = (len + 3) / 4;
    uint32_t *cw = reinterpret_cast<uint32_t *>(codes + lo);
    for (int64_t wi = lane; wi < nwords; wi += 32) {
      uint32_t word = 0;
      for (int k = 0; k < 4 && wi * 4 + k < len; ++k) {
        const int64_t i = lo + wi * 4 + k;
        const float vi = __fadd_rn(__fmul_rn(f32_from_e4m3(codes[i]), sold), load1_f32<DT>(grad, i));
        word |= code_e4m3_exact(vi, s) << (8 * k);
      }
      cw[wi] = word;
    }
    __syncwarp();
    if (lane == 0) scales[lo / G] = s;
  }
}

template <int DT, int G>
__global__ void __launch_bounds__(kThreads) fp8_accumulate_kernel(uint8_t *codes, float *scales,
                                                                  const void *__restrict__ grad,
                                                                  int64_t n, int wide, float one) {
  const WarpCursor c;
  const int64_t nfull = n / kTile;
  for (int64_t t = c.warp; t < nfull; t += c.nwarps)
    fp8acc_tile<DT, G>(codes, scales, grad, t * kTile, c.lane, wide != 0, one);
  if (c.owns_tail(n)) fp8acc_tail<DT, G>(codes, scales, grad, nfull * kTile, n, c.lane);
}

}  // namespace zq
