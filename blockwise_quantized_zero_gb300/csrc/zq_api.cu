// zq_api.cu -- the C ABI of libzq (declared in include/zq.h): argument
// validation, aliasing and device-pointer checks, and dispatch to the launch
// units. Every argument error is reported before any work is enqueued.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "zq.h"
#include "zq_host.h"

namespace zq {

namespace {

thread_local int g_last_cuda_error = 0;

constexpr int kMaxDevices = 64;
int g_sm_count[kMaxDevices] = {0};
std::mutex g_sm_mutex;

int bits_of(int fmt) {
  switch (fmt) {
    case ZQ_INT2: return 2;
    case ZQ_INT4: return 4;
    case ZQ_INT6: return 6;
    case ZQ_INT8: return 8;
    case ZQ_E4M3: return 8;
    default: return 0;
  }
}

int elem_bytes(int dt) {
  switch (dt) {
    case ZQ_F32: return 4;
    case ZQ_F16: return 2;
    case ZQ_BF16: return 2;
    default: return 0;
  }
}

bool valid_block(int64_t G) {
  return G == 32 || G == 64 || G == 128 || G == 256 || G == 512 || G == 1024;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned32(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
  Range(const void *p, size_t bytes)
      : lo(reinterpret_cast<uintptr_t>(p)), hi(reinterpret_cast<uintptr_t>(p) + bytes) {}
  bool overlaps(const Range &o) const { return lo < o.hi && o.lo < hi && lo != hi && o.lo != o.hi; }
};

// Device-pointer check: memory of the current device, or managed memory.
// Disabled by setting the environment variable ZQ_CHECK_POINTERS=0.
bool pointer_checks_enabled() {
  static const bool on = [] {
    const char *v = std::getenv("ZQ_CHECK_POINTERS");
    return !(v && v[0] == '0');
  }();
  return on;
}

zq_status check_device_ptr(const void *p) {
  if (!pointer_checks_enabled()) return ZQ_OK;
  cudaPointerAttributes attr;
  std::memset(&attr, 0, sizeof(attr));
  const cudaError_t e = cudaPointerGetAttributes(&attr, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    g_last_cuda_error = static_cast<int>(e);
    return ZQ_ERR_INVALID_ARG;
  }
  if (attr.type == cudaMemoryTypeManaged) return ZQ_OK;
  if (attr.type != cudaMemoryTypeDevice) return ZQ_ERR_INVALID_ARG;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || attr.device != dev) {
    (void)cudaGetLastError();
    return ZQ_ERR_INVALID_ARG;
  }
  return ZQ_OK;
}

// True when some output range overlaps another range (input or output);
// inputs may overlap each other. Sort and sweep: O(n log n).
bool any_output_overlap(std::vector<Range> ins, std::vector<Range> outs) {
  struct Tagged {
    uintptr_t lo, hi;
    bool out;
  };
  std::vector<Tagged> all;
  all.reserve(ins.size() + outs.size());
  for (const Range &r : ins)
    if (r.lo != r.hi) all.push_back({r.lo, r.hi, false});
  for (const Range &r : outs)
    if (r.lo != r.hi) all.push_back({r.lo, r.hi, true});
  std::sort(all.begin(), all.end(), [](const Tagged &x, const Tagged &y) { return x.lo < y.lo; });
  uintptr_t end_all = 0, end_out = 0;
  for (const Tagged &r : all) {
    if (r.lo < (r.out ? end_all : end_out)) return true;
    end_all = std::max(end_all, r.hi);
    if (r.out) end_out = std::max(end_out, r.hi);
  }
  return false;
}

zq_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return ZQ_OK;
  g_last_cuda_error = static_cast<int>(e);
  return ZQ_ERR_CUDA;
}

cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    (void)cudaGetLastError();
    return 148;
  }
  std::lock_guard<std::mutex> lock(g_sm_mutex);
  if (g_sm_count[dev] == 0) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        sms < 1) {
      (void)cudaGetLastError();
      sms = 148;
    }
    g_sm_count[dev] = sms;
  }
  return g_sm_count[dev];
}

// Argument checks shared by the two reduce entry points (they differ only in
// the largest shard count); ZQ_OK with n == 0 means "nothing to do".
static zq_status check_reduce(const void *const *codes, const float *const *scales, int nshards,
                       int max_shards, int64_t n, int format_in, int64_t G_in,
                       const void *out_codes, const float *out_scales, int format_out,
                       int64_t G_out, const float *sum_out) {
  if (!bits_of(format_in) || !bits_of(format_out)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G_in) || !valid_block(G_out) || nshards < 1 || nshards > max_shards)
    return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!codes || !scales || !out_codes || !out_scales) return ZQ_ERR_INVALID_ARG;
  for (int r = 0; r < nshards; ++r)
    if (!codes[r] || !scales[r]) return ZQ_ERR_INVALID_ARG;
  for (int r = 0; r < nshards; ++r)
    if (!aligned16(codes[r]) || !aligned16(scales[r])) return ZQ_ERR_MISALIGNED;
  if (!aligned16(out_codes) || !aligned16(out_scales) || (sum_out && !aligned16(sum_out)))
    return ZQ_ERR_MISALIGNED;
  const Range oc(out_codes, zq_codes_bytes(format_out, n)),
      os(out_scales, size_t(zq_num_blocks(n, G_out)) * 4u),
      sm(sum_out, sum_out ? size_t(n) * 4u : 0u);
  if (oc.overlaps(os) || oc.overlaps(sm) || os.overlaps(sm)) return ZQ_ERR_ALIAS;
  for (int r = 0; r < nshards; ++r) {
    const Range ic(codes[r], zq_codes_bytes(format_in, n)),
        is(scales[r], size_t(zq_num_blocks(n, G_in)) * 4u);
    for (const Range *o : {&oc, &os, &sm})
      if (o->overlaps(ic) || o->overlaps(is)) return ZQ_ERR_ALIAS;
  }
  for (int r = 0; r < nshards; ++r) {
    if (zq_status st = check_device_ptr(codes[r])) return st;
    if (zq_status st = check_device_ptr(scales[r])) return st;
  }
  if (zq_status st = check_device_ptr(out_codes)) return st;
  if (zq_status st = check_device_ptr(out_scales)) return st;
  if (sum_out)
    if (zq_status st = check_device_ptr(sum_out)) return st;
  return ZQ_OK;
}

static_assert(ZQ_STATIC_MAX_SHARDS == kStaticMaxShards, "shard table size");

}  // namespace zq

using namespace zq;

extern "C" {

size_t zq_codes_bytes(int format, int64_t n) {
  const int b = bits_of(format);
  if (b == 0 || n < 0) return 0;
  return static_cast<size_t>((n * b + 31) / 32) * 4u;
}

int64_t zq_num_blocks(int64_t n, int64_t G) {
  if (n < 0 || !valid_block(G)) return 0;
  return (n + G - 1) / G;
}

zq_status zq_wait_selftest(int64_t limit_us, void *stream) {
  if (limit_us < 1 || limit_us > 100000) return ZQ_ERR_INVALID_ARG;
  return from_cuda(launch_wait_selftest(uint64_t(limit_us) * 1000u, as_stream(stream)));
}

const char *zq_status_string(int status) {
  switch (status) {
    case ZQ_OK: return "ok";
    case ZQ_ERR_INVALID_ARG: return "invalid argument";
    case ZQ_ERR_UNSUPPORTED: return "unsupported format or element type";
    case ZQ_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ZQ_ERR_ALIAS: return "output overlaps an input";
    case ZQ_ERR_CUDA: return "CUDA runtime error";
    case ZQ_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

int zq_last_cuda_error(void) { return g_last_cuda_error; }

zq_status zq_device_status(void *stream) {
  const cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(e);
    return ZQ_ERR_CUDA;
  }
  const unsigned err = zq::take_reduce_device_error() | zq::take_gemm_device_error();
  return (err & zq::kDevErrWaitTimeout) ? ZQ_ERR_TIMEOUT : ZQ_OK;
}

zq_status zq_quantize(const void *src, int src_dtype, int64_t n, int format, int64_t G, void *codes,
                      float *scales, void *stream) {
  if (!bits_of(format) || !elem_bytes(src_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!src || !codes || !scales) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(codes) || !aligned16(scales)) return ZQ_ERR_MISALIGNED;
  const Range rs(src, size_t(n) * elem_bytes(src_dtype)), rc(codes, zq_codes_bytes(format, n)),
      rk(scales, size_t(zq_num_blocks(n, G)) * 4u);
  if (rc.overlaps(rs) || rk.overlaps(rs) || rc.overlaps(rk)) return ZQ_ERR_ALIAS;
  for (const void *p : {static_cast<const void *>(src), static_cast<const void *>(codes),
                        static_cast<const void *>(scales)})
    if (zq_status st = check_device_ptr(p)) return st;
  const bool wide = aligned32(src);
  return from_cuda(launch_quantize(src, src_dtype, n, format, G, codes, scales, as_stream(stream),
                                   wide));
}

zq_status zq_quantize_multi(const void *const *src, const int64_t *n, int count, int src_dtype,
                            int format, int64_t G, void *const *codes, float *const *scales,
                            void *stream) {
  if (!bits_of(format) || !elem_bytes(src_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (count < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (count == 0) return ZQ_OK;
  if (!src || !n || !codes || !scales) return ZQ_ERR_INVALID_ARG;
  std::vector<Range> ins, outs;
  bool wide = true;
  for (int k = 0; k < count; ++k) {
    if (n[k] < 0) return ZQ_ERR_INVALID_ARG;
    if (n[k] == 0) continue;
    if (!src[k] || !codes[k] || !scales[k]) return ZQ_ERR_INVALID_ARG;
    if (!aligned16(src[k]) || !aligned16(codes[k]) || !aligned16(scales[k])) return ZQ_ERR_MISALIGNED;
    if (!aligned32(src[k])) wide = false;
    ins.emplace_back(src[k], size_t(n[k]) * elem_bytes(src_dtype));
    outs.emplace_back(codes[k], zq_codes_bytes(format, n[k]));
    outs.emplace_back(scales[k], size_t(zq_num_blocks(n[k], G)) * 4u);
  }
  if (any_output_overlap(std::move(ins), std::move(outs))) return ZQ_ERR_ALIAS;
  for (int k = 0; k < count; ++k) {
    if (n[k] == 0) continue;
    for (const void *p : {src[k], static_cast<const void *>(codes[k]),
                          static_cast<const void *>(scales[k])})
      if (zq_status st = check_device_ptr(p)) return st;
  }
  // launches of up to kMultiMax tensors (empty tensors are left out)
  MultiArgs a;
  std::memset(&a, 0, sizeof(a));
  a.wide = wide ? 1 : 0;
  int m = 0;
  auto flush = [&]() -> zq_status {
    if (m == 0) return ZQ_OK;
    a.count = m;
    const zq_status st = from_cuda(launch_quantize_multi(a, src_dtype, format, G, as_stream(stream)));
    m = 0;
    a.tile0[0] = 0;
    return st;
  };
  a.tile0[0] = 0;
  for (int k = 0; k < count; ++k) {
    if (n[k] == 0) continue;
    a.src[m] = src[k];
    a.codes[m] = static_cast<uint8_t *>(codes[k]);
    a.scales[m] = scales[k];
    a.n[m] = n[k];
    a.tile0[m + 1] = a.tile0[m] + n[k] / kTile;
    if (++m == kMultiMax)
      if (zq_status st = flush()) return st;
  }
  return flush();
}

zq_status zq_dequantize_multi(const void *const *codes, const float *const *scales,
                              const int64_t *n, int count, int format, int64_t G, void *const *dst,
                              int dst_dtype, void *stream) {
  if (!bits_of(format) || !elem_bytes(dst_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (count < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (count == 0) return ZQ_OK;
  if (!codes || !scales || !n || !dst) return ZQ_ERR_INVALID_ARG;
  std::vector<Range> ins, outs;
  bool wide = true;
  for (int k = 0; k < count; ++k) {
    if (n[k] < 0) return ZQ_ERR_INVALID_ARG;
    if (n[k] == 0) continue;
    if (!codes[k] || !scales[k] || !dst[k]) return ZQ_ERR_INVALID_ARG;
    if (!aligned16(codes[k]) || !aligned16(scales[k]) || !aligned16(dst[k])) return ZQ_ERR_MISALIGNED;
    if (!aligned32(dst[k])) wide = false;
    ins.emplace_back(codes[k], zq_codes_bytes(format, n[k]));
    ins.emplace_back(scales[k], size_t(zq_num_blocks(n[k], G)) * 4u);
    outs.emplace_back(dst[k], size_t(n[k]) * elem_bytes(dst_dtype));
  }
  if (any_output_overlap(std::move(ins), std::move(outs))) return ZQ_ERR_ALIAS;
  for (int k = 0; k < count; ++k) {
    if (n[k] == 0) continue;
    for (const void *p : {codes[k], static_cast<const void *>(scales[k]),
                          static_cast<const void *>(dst[k])})
      if (zq_status st = check_device_ptr(p)) return st;
  }
  DequantMultiArgs a;
  std::memset(&a, 0, sizeof(a));
  a.log2G = log2_block(G);
  a.wide = wide ? 1 : 0;
  int m = 0;
  auto flush = [&]() -> zq_status {
    if (m == 0) return ZQ_OK;
    a.count = m;
    const zq_status st = from_cuda(launch_dequantize_multi(a, format, dst_dtype, as_stream(stream)));
    m = 0;
    return st;
  };
  a.tile0[0] = 0;
  for (int k = 0; k < count; ++k) {
    if (n[k] == 0) continue;
    a.codes[m] = static_cast<const uint8_t *>(codes[k]);
    a.scales[m] = scales[k];
    a.dst[m] = dst[k];
    a.n[m] = n[k];
    a.tile0[m + 1] = a.tile0[m] + n[k] / kTile;
    if (++m == kMultiMax)
      if (zq_status st = flush()) return st;
  }
  return flush();
}

zq_status zq_quantize_reordered(const void *src, int src_dtype, int64_t n, int format, int64_t G,
                                int nodes, int gpus_per_node, void *codes, float *scales,
                                void *stream) {
  if (!bits_of(format) || !elem_bytes(src_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (nodes < 1 || gpus_per_node < 1 || nodes * gpus_per_node > ZQ_MAX_SHARDS)
    return ZQ_ERR_INVALID_ARG;
  const int64_t P = int64_t(nodes) * gpus_per_node;
  if (n < 0 || !valid_block(G) || n % (P * 1024) != 0) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!src || !codes || !scales) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(codes) || !aligned16(scales)) return ZQ_ERR_MISALIGNED;
  const Range rs(src, size_t(n) * elem_bytes(src_dtype)), rc(codes, zq_codes_bytes(format, n)),
      rk(scales, size_t(zq_num_blocks(n, G)) * 4u);
  if (rc.overlaps(rs) || rk.overlaps(rs) || rc.overlaps(rk)) return ZQ_ERR_ALIAS;
  for (const void *p : {static_cast<const void *>(src), static_cast<const void *>(codes),
                        static_cast<const void *>(scales)})
    if (zq_status st = check_device_ptr(p)) return st;
  const SliceRemap rm{nodes, gpus_per_node, n / (P * 1024)};
  return from_cuda(launch_quantize(src, src_dtype, n, format, G, codes, scales, as_stream(stream),
                                   aligned32(src), rm));
}

zq_status zq_reduce_two_hop(const void *const *codes, const float *const *scales, int nodes,
                            int gpus_per_node, int64_t n, int format_in, int64_t G_in,
                            void *const *mid_codes, float *const *mid_scales, int format_mid,
                            int64_t G_mid, void *const *out_codes, float *const *out_scales,
                            int format_out, int64_t G_out, float *const *sums, void *stream) {
  if (!bits_of(format_in) || !bits_of(format_mid) || !bits_of(format_out))
    return ZQ_ERR_UNSUPPORTED;
  if (nodes < 1 || gpus_per_node < 1 || nodes * gpus_per_node > ZQ_MAX_SHARDS)
    return ZQ_ERR_INVALID_ARG;
  const int A = nodes, L = gpus_per_node, P = A * L;
  // chunks of a multiple of 4096 elements keep every per-shard code and scale
  // slice 16-byte aligned (the reduce kernel reads them with bulk copies)
  if (n < 0 || !valid_block(G_in) || !valid_block(G_mid) || !valid_block(G_out) ||
      n % (int64_t(P) * 4096) != 0)
    return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!codes || !scales || !mid_codes || !mid_scales || !out_codes || !out_scales)
    return ZQ_ERR_INVALID_ARG;
  const int64_t m = n / P;
  const int bin = bits_of(format_in), bmid = bits_of(format_mid);
  // every buffer: present, 16-byte aligned, on this device, and no output
  // (hop-1 result, final codes, scales, sums) overlapping any other buffer
  std::vector<Range> inputs, outputs;
  for (int g = 0; g < P; ++g) {
    if (!codes[g] || !scales[g] || !mid_codes[g] || !mid_scales[g] || !out_codes[g] ||
        !out_scales[g] || (sums && !sums[g]))
      return ZQ_ERR_INVALID_ARG;
    const void *all[7] = {codes[g], scales[g], mid_codes[g], mid_scales[g], out_codes[g],
                          out_scales[g], sums ? sums[g] : nullptr};
    for (const void *p : all)
      if (p && !aligned16(p)) return ZQ_ERR_MISALIGNED;
    inputs.emplace_back(codes[g], zq_codes_bytes(format_in, n));
    inputs.emplace_back(scales[g], size_t(zq_num_blocks(n, G_in)) * 4u);
    outputs.emplace_back(mid_codes[g], zq_codes_bytes(format_mid, int64_t(A) * m));
    outputs.emplace_back(mid_scales[g], size_t(zq_num_blocks(int64_t(A) * m, G_mid)) * 4u);
    outputs.emplace_back(out_codes[g], zq_codes_bytes(format_out, m));
    outputs.emplace_back(out_scales[g], size_t(zq_num_blocks(m, G_out)) * 4u);
    if (sums) outputs.emplace_back(sums[g], size_t(m) * 4u);
  }
  for (size_t i = 0; i < outputs.size(); ++i) {
    for (const Range &r : inputs)
      if (outputs[i].overlaps(r)) return ZQ_ERR_ALIAS;
    for (size_t j = i + 1; j < outputs.size(); ++j)
      if (outputs[i].overlaps(outputs[j])) return ZQ_ERR_ALIAS;
  }
  for (int g = 0; g < P; ++g) {
    const void *all[7] = {codes[g], scales[g], mid_codes[g], mid_scales[g], out_codes[g],
                          out_scales[g], sums ? sums[g] : nullptr};
    for (const void *p : all)
      if (p)
        if (zq_status st = check_device_ptr(p)) return st;
  }
  const cudaStream_t st = as_stream(stream);
  // every shard slice the hops read starts 16-byte aligned (n is a multiple of
  // 4096 * P); checked again here because the kernels read them with bulk copies
  for (int g = 0; g < P; ++g)
    for (int64_t off : {int64_t(0), m, int64_t(A) * m}) {
      if (!aligned16(static_cast<const uint8_t *>(codes[g]) + off * bin / 8) ||
          !aligned16(scales[g] + off / G_in) ||
          !aligned16(static_cast<const uint8_t *>(mid_codes[g]) + off * bmid / 8) ||
          !aligned16(mid_scales[g] + off / G_mid))
        return ZQ_ERR_MISALIGNED;
    }
  HopArgs h;
  // hop 1: GPU (node x, local l) sums part l (A*m elements) of the GPUs of node x
  std::memset(&h, 0, sizeof(h));
  for (int g = 0; g < P; ++g) {
    h.in_codes[g] = static_cast<const uint8_t *>(codes[g]);
    h.in_scales[g] = scales[g];
    h.out_codes[g] = static_cast<uint8_t *>(mid_codes[g]);
    h.out_scales[g] = mid_scales[g];
  }
  h.n = int64_t(A) * m;
  h.part = int64_t(A) * m;
  h.nprob = P;
  h.nshards = L;
  h.log2Gin = log2_block(G_in);
  h.log2Gout = log2_block(G_mid);
  h.wide = 1;
  h.one = 1.0f;
  h.hop = 1;
  h.A = A;
  h.L = L;
  h.bits_in = bin;
  if (zq_status s2 = from_cuda(launch_reduce_hop(h, format_in, format_mid, st))) return s2;
  // hop 2: GPU (node x, local l) sums chunk x of the hop-1 results of GPUs (*, l)
  std::memset(&h, 0, sizeof(h));
  bool wide = true;
  for (int g = 0; g < P; ++g) {
    h.in_codes[g] = static_cast<const uint8_t *>(mid_codes[g]);
    h.in_scales[g] = mid_scales[g];
    h.out_codes[g] = static_cast<uint8_t *>(out_codes[g]);
    h.out_scales[g] = out_scales[g];
    h.sums[g] = sums ? sums[g] : nullptr;
    if (sums && !aligned32(sums[g])) wide = false;
  }
  h.n = m;
  h.part = m;
  h.nprob = P;
  h.nshards = A;
  h.log2Gin = log2_block(G_mid);
  h.log2Gout = log2_block(G_out);
  h.wide = wide ? 1 : 0;
  h.one = 1.0f;
  h.hop = 2;
  h.A = A;
  h.L = L;
  h.bits_in = bmid;
  if (zq_status s2 = from_cuda(launch_reduce_hop(h, format_mid, format_out, st))) return s2;
  return ZQ_OK;
}

size_t zq_interleaved_bytes(int format, int64_t n, int64_t G) {
  if (format == ZQ_E4M3 || !bits_of(format) || n < 0 || !valid_block(G)) return 0;
  return zq_codes_bytes(format, n) + size_t(zq_num_blocks(n, G)) * 4u;
}

zq_status zq_quantize_interleaved(const void *src, int src_dtype, int64_t n, int format, int64_t G,
                                  void *records, void *stream) {
  if (format == ZQ_E4M3 || !bits_of(format) || !elem_bytes(src_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!src || !records) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(src) || !aligned16(records)) return ZQ_ERR_MISALIGNED;
  const Range rs(src, size_t(n) * elem_bytes(src_dtype)),
      rr(records, zq_interleaved_bytes(format, n, G));
  if (rr.overlaps(rs)) return ZQ_ERR_ALIAS;
  for (const void *p : {src, static_cast<const void *>(records)})
    if (zq_status st = check_device_ptr(p)) return st;
  return from_cuda(launch_quantize_interleaved(src, src_dtype, n, format, G, records,
                                               as_stream(stream), aligned32(src)));
}

zq_status zq_dequantize_interleaved(const void *records, int64_t n, int format, int64_t G,
                                    void *dst, int dst_dtype, void *stream) {
  if (format == ZQ_E4M3 || !bits_of(format) || !elem_bytes(dst_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!records || !dst) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(records) || !aligned16(dst)) return ZQ_ERR_MISALIGNED;
  const Range rd(dst, size_t(n) * elem_bytes(dst_dtype)),
      rr(records, zq_interleaved_bytes(format, n, G));
  if (rd.overlaps(rr)) return ZQ_ERR_ALIAS;
  for (const void *p : {records, static_cast<const void *>(dst)})
    if (zq_status st = check_device_ptr(p)) return st;
  return from_cuda(launch_dequantize_interleaved(records, n, format, G, dst, dst_dtype,
                                                 as_stream(stream), aligned32(dst)));
}

zq_status zq_aquavit_schedule(int64_t t, int64_t T, double a, double c, int *format, int64_t *G,
                              double *target, double *width) {
  if (!format || !G || T < 1 || t < 0 || t > T || !(a > 0.0) || !(c >= 0.0) || !std::isfinite(a) ||
      !std::isfinite(c))
    return ZQ_ERR_INVALID_ARG;
  const double want = 8.0 - 6.0 / (a + c * double(t) / double(T));
  // The 18 available widths in increasing order (b = 2, 4, 6; G = 1024 .. 32);
  // scanning upwards with a strict comparison keeps the narrower pair on a tie.
  int best_b = 0;
  int64_t best_G = 0;
  double best_w = 0.0, best_d = 0.0;
  for (int b = 2; b <= 6; b += 2)
    for (int64_t g = 1024; g >= 32; g /= 2) {
      const double w = double(b) + 32.0 / double(g), d = std::fabs(w - want);
      if (best_b == 0 || d < best_d) {
        best_b = b;
        best_G = g;
        best_w = w;
        best_d = d;
      }
    }
  *format = best_b;  // ZQ_INT2 / ZQ_INT4 / ZQ_INT6 are the bit counts
  *G = best_G;
  if (target) *target = want;
  if (width) *width = best_w;
  return ZQ_OK;
}

zq_status zq_dequantize(const void *codes, const float *scales, int64_t n, int format, int64_t G,
                        void *dst, int dst_dtype, void *stream) {
  if (!bits_of(format) || !elem_bytes(dst_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!codes || !scales || !dst) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(codes) || !aligned16(scales) || !aligned16(dst)) return ZQ_ERR_MISALIGNED;
  const Range rd(dst, size_t(n) * elem_bytes(dst_dtype)), rc(codes, zq_codes_bytes(format, n)),
      rk(scales, size_t(zq_num_blocks(n, G)) * 4u);
  if (rd.overlaps(rc) || rd.overlaps(rk)) return ZQ_ERR_ALIAS;
  for (const void *p : {static_cast<const void *>(codes), static_cast<const void *>(scales),
                        static_cast<const void *>(dst)})
    if (zq_status st = check_device_ptr(p)) return st;
  const bool wide = aligned32(dst);
  return from_cuda(launch_dequantize(codes, scales, n, format, G, dst, dst_dtype,
                                     as_stream(stream), wide));
}


zq_status zq_reduce_quantized(const void *const *codes, const float *const *scales, int nshards,
                              int64_t n, int format_in, int64_t G_in, void *out_codes,
                              float *out_scales, int format_out, int64_t G_out, float *sum_out,
                              void *stream) {
  if (zq_status st = check_reduce(codes, scales, nshards, ZQ_MAX_SHARDS, n, format_in, G_in,
                                  out_codes, out_scales, format_out, G_out, sum_out))
    return st;
  if (n == 0) return ZQ_OK;

  ReduceArgs a;
  std::memset(&a, 0, sizeof(a));
  for (int r = 0; r < nshards; ++r) {
    a.codes[r] = static_cast<const uint8_t *>(codes[r]);
    a.scales[r] = scales[r];
  }
  a.out_codes = static_cast<uint8_t *>(out_codes);
  a.out_scales = out_scales;
  a.sum_out = sum_out;
  a.n = n;
  a.nshards = nshards;
  a.log2Gin = log2_block(G_in);
  a.log2Gout = log2_block(G_out);
  a.wide = (!sum_out || aligned32(sum_out)) ? 1 : 0;
  a.one = 1.0f;
  return from_cuda(launch_reduce(a, format_in, format_out, as_stream(stream)));
}

zq_status zq_reduce_ring(const void *const *codes, const float *const *scales, int nshards,
                         int64_t n, int format, int64_t G, void *const *partial_codes,
                         float *const *partial_scales, void *out_codes, float *out_scales,
                         int format_out, int64_t G_out, float *sum_out, void *stream) {
  // partial buffers are used from three shards on; their argument checks come
  // first, the device-pointer checks after the shared reduce checks
  const bool chain = nshards > 2 && nshards <= ZQ_MAX_SHARDS && n > 0 && bits_of(format) &&
                     bits_of(format_out) && valid_block(G) && valid_block(G_out);
  if (chain) {
    if (!codes || !scales || !out_codes || !out_scales) return ZQ_ERR_INVALID_ARG;
    for (int r = 0; r < nshards; ++r)
      if (!codes[r] || !scales[r]) return ZQ_ERR_INVALID_ARG;
    if (!partial_codes || !partial_scales) return ZQ_ERR_INVALID_ARG;
    std::vector<Range> held;  // every buffer the chain reads or writes
    for (int r = 0; r < nshards; ++r) {
      held.emplace_back(codes[r], zq_codes_bytes(format, n));
      held.emplace_back(scales[r], size_t(zq_num_blocks(n, G)) * 4u);
    }
    held.emplace_back(out_codes, zq_codes_bytes(format_out, n));
    held.emplace_back(out_scales, size_t(zq_num_blocks(n, G_out)) * 4u);
    held.emplace_back(sum_out, sum_out ? size_t(n) * 4u : 0u);
    for (int k = 0; k < 2; ++k) {
      if (!partial_codes[k] || !partial_scales[k]) return ZQ_ERR_INVALID_ARG;
      if (!aligned16(partial_codes[k]) || !aligned16(partial_scales[k])) return ZQ_ERR_MISALIGNED;
      const Range pc(partial_codes[k], zq_codes_bytes(format, n)),
          ps(partial_scales[k], size_t(zq_num_blocks(n, G)) * 4u);
      for (const Range &h : held)
        if (h.overlaps(pc) || h.overlaps(ps)) return ZQ_ERR_ALIAS;
      if (pc.overlaps(ps)) return ZQ_ERR_ALIAS;
      held.push_back(pc);
      held.push_back(ps);
    }
  }
  if (zq_status st = check_reduce(codes, scales, nshards, ZQ_MAX_SHARDS, n, format, G, out_codes,
                                  out_scales, format_out, G_out, sum_out))
    return st;
  if (n == 0) return ZQ_OK;
  if (chain)
    for (int k = 0; k < 2; ++k) {
      if (zq_status st = check_device_ptr(partial_codes[k])) return st;
      if (zq_status st = check_device_ptr(partial_scales[k])) return st;
    }
  // hop r: the shard-ordered reduce of [partial, shard r], requantized into
  // the ring format (partial buffer r % 2) or, at the last hop, the output
  ReduceArgs a;
  std::memset(&a, 0, sizeof(a));
  a.n = n;
  a.log2Gin = log2_block(G);
  a.one = 1.0f;
  if (nshards == 1) {
    a.codes[0] = static_cast<const uint8_t *>(codes[0]);
    a.scales[0] = scales[0];
    a.nshards = 1;
    a.out_codes = static_cast<uint8_t *>(out_codes);
    a.out_scales = out_scales;
    a.sum_out = sum_out;
    a.log2Gout = log2_block(G_out);
    a.wide = (!sum_out || aligned32(sum_out)) ? 1 : 0;
    return from_cuda(launch_reduce(a, format, format_out, as_stream(stream)));
  }
  const uint8_t *pcodes = static_cast<const uint8_t *>(codes[0]);
  const float *pscales = scales[0];
  a.nshards = 2;
  for (int r = 1; r < nshards; ++r) {
    const bool last = r == nshards - 1;
    a.codes[0] = pcodes;
    a.scales[0] = pscales;
    a.codes[1] = static_cast<const uint8_t *>(codes[r]);
    a.scales[1] = scales[r];
    a.out_codes = static_cast<uint8_t *>(last ? out_codes : partial_codes[r % 2]);
    a.out_scales = last ? out_scales : partial_scales[r % 2];
    a.sum_out = last ? sum_out : nullptr;
    a.log2Gout = log2_block(last ? G_out : G);
    a.wide = (!a.sum_out || aligned32(a.sum_out)) ? 1 : 0;
    if (zq_status st = from_cuda(launch_reduce(a, format, last ? format_out : format,
                                               as_stream(stream))))
      return st;
    pcodes = a.out_codes;
    pscales = a.out_scales;
  }
  return ZQ_OK;
}

zq_status zq_reduce_quantized_static(const void *const *codes, const float *const *scales,
                                     int nshards, int64_t n, int format_in, int64_t G_in,
                                     void *out_codes, float *out_scales, int format_out,
                                     int64_t G_out, float *sum_out, void *stream) {
  if (zq_status st = check_reduce(codes, scales, nshards, ZQ_STATIC_MAX_SHARDS, n, format_in,
                                  G_in, out_codes, out_scales, format_out, G_out, sum_out))
    return st;
  if (n == 0) return ZQ_OK;
  // The table is filled by copies from the caller's host arrays, which a
  // captured graph would replay from memory the caller has since reused:
  // refuse while the stream is being captured, with nothing enqueued.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaError_t e = cudaStreamIsCapturing(as_stream(stream), &cap)) return from_cuda(e);
  if (cap != cudaStreamCaptureStatusNone) return ZQ_ERR_INVALID_ARG;

  TableReduceArgs a;
  std::memset(&a, 0, sizeof(a));
  a.out_codes = static_cast<uint8_t *>(out_codes);
  a.out_scales = out_scales;
  a.sum_out = sum_out;
  a.n = n;
  a.nshards = nshards;
  a.log2Gin = log2_block(G_in);
  a.log2Gout = log2_block(G_out);
  a.wide = (!sum_out || aligned32(sum_out)) ? 1 : 0;
  a.one = 1.0f;
  return from_cuda(launch_reduce_static(codes, scales, a, format_in, format_out,
                                        as_stream(stream)));
}

zq_status zq_gemm_dequant(const void *x, int64_t M, int64_t K, const void *w_codes,
                          const float *w_scales, int format, int64_t G, int64_t N, void *y,
                          int y_dtype, void *stream) {
  if (!bits_of(format) || (y_dtype != ZQ_F32 && y_dtype != ZQ_BF16)) return ZQ_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return ZQ_OK;
  if (K == 0 || K % 64 != 0 || K % G != 0 || N % 64 != 0 || M > (int64_t(1) << 31) ||
      N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
    return ZQ_ERR_INVALID_ARG;
  if (((M + 127) / 128) * (N / 64) >= (int64_t(1) << 31)) return ZQ_ERR_INVALID_ARG;
  if (!x || !w_codes || !w_scales || !y) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_codes) || !aligned16(w_scales) || !aligned16(y))
    return ZQ_ERR_MISALIGNED;
  const Range rx(x, size_t(M) * size_t(K) * 2u), rc(w_codes, zq_codes_bytes(format, N * K)),
      rs(w_scales, size_t(zq_num_blocks(N * K, G)) * 4u),
      ry(y, size_t(M) * size_t(N) * (y_dtype == ZQ_F32 ? 4u : 2u));
  if (ry.overlaps(rx) || ry.overlaps(rc) || ry.overlaps(rs)) return ZQ_ERR_ALIAS;
  for (const void *p : {x, w_codes, static_cast<const void *>(w_scales), static_cast<const void *>(y)})
    if (zq_status st = check_device_ptr(p)) return st;
  return from_cuda(launch_gemm_dequant(x, M, K, w_codes, w_scales, format, G, N, y, y_dtype,
                                       as_stream(stream)));
}

zq_status zq_gemm_plan(int64_t M, int64_t N, int64_t K, int *bm, int *bn, int *split) {
  if (!bm || !bn || !split || M < 0 || N <= 0 || K <= 0 || N % 64 != 0 || K % 64 != 0)
    return ZQ_ERR_INVALID_ARG;
  int a = 128, b = 64, c = 1;
  gemm_tile_shape(M, N, K, a, b, c);
  *bm = a;
  *bn = b;
  *split = c;
  return ZQ_OK;
}

zq_status zq_fp8_accumulate(void *main_codes, float *main_scales, const void *grad, int grad_dtype,
                            int64_t n, int64_t G, void *stream) {
  if (!elem_bytes(grad_dtype)) return ZQ_ERR_UNSUPPORTED;
  if (n < 0 || !valid_block(G)) return ZQ_ERR_INVALID_ARG;
  if (n == 0) return ZQ_OK;
  if (!main_codes || !main_scales || !grad) return ZQ_ERR_INVALID_ARG;
  if (!aligned16(main_codes) || !aligned16(main_scales) || !aligned16(grad))
    return ZQ_ERR_MISALIGNED;
  const Range rc(main_codes, zq_codes_bytes(ZQ_E4M3, n)),
      rs(main_scales, size_t(zq_num_blocks(n, G)) * 4u),
      rg(grad, size_t(n) * elem_bytes(grad_dtype));
  if (rc.overlaps(rs) || rg.overlaps(rc) || rg.overlaps(rs)) return ZQ_ERR_ALIAS;
  for (const void *p : {static_cast<const void *>(main_codes),
                        static_cast<const void *>(main_scales), grad})
    if (zq_status st = check_device_ptr(p)) return st;
  const bool wide = aligned32(grad);
  return from_cuda(launch_fp8_accumulate(main_codes, main_scales, grad, grad_dtype, n, G,
                                         as_stream(stream), wide));
}

}  // extern "C"
