/*
 * zq.h -- C ABI of libzq: blockwise quantize / pack / dequantize /
 * quantized-reduce / FP8-accumulate kernels for one GB300 GPU (sm_103a).
 *
 * The operations follow these pages:
 *  [ZeRO++]  "Quantized LLM Training at Scale with ZeRO++" -- section "Blockwise
 *            weight quantization cuts forward-gather traffic in half" (qwZ:
 *            weights split into blocks, 8-bit codes with a scale per block) and
 *            section "QGZ keeps reductions in full precision while sending
 *            quantized gradients" (qgZ: 4/8-bit gradients dequantized, summed in
 *            full precision, requantized once);
 *  [Aquavit] "Aquavit: Ascending Quantization for Communication-Efficient
 *            Vast-Scale Distributed Training" (review) -- granularity
 *            modulation, Eq. 6 / Table 1: b in {2,4,6,8}, 32 bits of metadata
 *            per G-element block, bpw = b + 32/G;
 *  [AGoQ]    "AGoQ: Activation and Gradient Quantization for Memory-Efficient
 *            Distributed Training of LLMs" -- section 2.B (QuanGrad): "Local
 *            Accumulation" and the "Local Reduce" step of the precision-
 *            preserved all-reduce.
 *
 * ----------------------------------------------------------------------------
 * Data layout (identical for every call)
 * ----------------------------------------------------------------------------
 *  - A tensor is a flat array of n elements; blocks are G consecutive elements
 *    (G in {32, 64, 128, 256, 512, 1024}); the last block may be partial.
 *  - scales: one fp32 per block, nb = ceil(n / G) of them, in block order,
 *    scale = absmax(block) / qmax with qmax = 2^(b-1) - 1 (1, 7, 31, 127), or
 *    absmax / 448 for E4M3. A block whose scale is 0 has all-zero codes.
 *  - codes: integer code q = clamp(rint(x / scale), -qmax, qmax) (IEEE binary32
 *    division, ties to even) stored as b-bit two's complement; code i occupies
 *    bits [i*b, i*b + b) of a little-endian stream of 32-bit words (LSB first;
 *    6-bit codes straddle words). E4M3 codes are one byte each, the nearest
 *    E4M3 value of x / scale (ties to even, saturating at +-448). The stream
 *    is zq_codes_bytes(format, n) bytes long; unused trailing bits are zero.
 *  - Dequantized value: fl32(q * scale) (or fl32(e4m3(q) * scale)), then one
 *    round-to-nearest-even to the output type.
 *
 * ----------------------------------------------------------------------------
 * Conventions
 * ----------------------------------------------------------------------------
 *  - Every data pointer is a DEVICE pointer (memory the GPU can address, e.g.
 *    from cudaMalloc or a torch CUDA tensor), 16-byte aligned, owned by the
 *    caller. The library allocates nothing, and no compute call waits for the
 *    GPU: work is enqueued on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and the call returns. Two calls may block the host:
 *    zq_device_status synchronizes the stream by design, and
 *    zq_reduce_quantized_static copies the caller's host pointer arrays with
 *    cudaMemcpyAsync, which for pageable host memory returns only once the
 *    bytes are staged. Pointer arrays (shards) are HOST arrays, read during
 *    the call only.
 *  - Outputs are complete once the enqueued work has finished AND
 *    zq_device_status has returned ZQ_OK for it: a reduce whose bounded
 *    device-side wait ran out leaves its outputs undefined (see
 *    zq_device_status).
 *  - Argument errors return synchronously with no work enqueued. A failed
 *    launch returns ZQ_ERR_CUDA; zq_last_cuda_error() then gives the CUDA
 *    runtime error code (per host thread). Errors that occur later on the
 *    device surface through the usual CUDA stream error reporting.
 *  - Outputs must not overlap inputs (ZQ_ERR_ALIAS), except the documented
 *    in-place update of zq_fp8_accumulate.
 *  - NaN and infinite inputs are outside the contract.
 *  - n = 0 is valid and enqueues nothing.
 *  - The calls are thread-safe: they keep no state between calls except
 *    per-device launch parameters computed on first use.
 */
#ifndef ZQ_H
#define ZQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum zq_status {
    ZQ_OK = 0,
    ZQ_ERR_INVALID_ARG = 1, /* null pointer, n < 0, bad block size, bad shard count */
    ZQ_ERR_UNSUPPORTED = 2, /* unknown format or element type */
    ZQ_ERR_MISALIGNED = 3,  /* a data pointer is not 16-byte aligned */
    ZQ_ERR_ALIAS = 4,       /* an output overlaps an input */
    ZQ_ERR_CUDA = 5,        /* the CUDA runtime reported an error (see zq_last_cuda_error) */
    ZQ_ERR_TIMEOUT = 6      /* a bounded device-side wait ran out (see zq_device_status) */
} zq_status;

/* Element types of uncompressed tensors. */
typedef enum zq_dtype { ZQ_F32 = 0, ZQ_F16 = 1, ZQ_BF16 = 2 } zq_dtype;

/* Code formats: the value is the integer bit width, except E4M3. */
typedef enum zq_format {
    ZQ_INT2 = 2,
    ZQ_INT4 = 4,
    ZQ_INT6 = 6,
    ZQ_INT8 = 8,
    ZQ_E4M3 = 0x48
} zq_format;

/* Largest shard count accepted by zq_reduce_quantized. */
#define ZQ_MAX_SHARDS 64

/* Largest shard count accepted by zq_reduce_quantized_static. */
#define ZQ_STATIC_MAX_SHARDS 1024

/* Bytes of the packed code stream for n elements: ceil(n * bits / 32) * 4.
 * With n a multiple of G this is n * b / 8 ([Aquavit] Eq. 6 without the
 * metadata term). Returns 0 for an unknown format or n < 0. Host only. */
size_t zq_codes_bytes(int format, int64_t n);

/* Number of blocks, ceil(n / G); 0 for an invalid G or n < 0. Host only. */
int64_t zq_num_blocks(int64_t n, int64_t G);

/*
 * zq_quantize -- blockwise symmetric quantization ([ZeRO++] qwZ section;
 * [Aquavit] Eq. 6 for b in {2,4,6,8}; [AGoQ] 2.B for E4M3).
 *   src      device, n elements of src_dtype (ZQ_F32 / ZQ_F16 / ZQ_BF16)
 *   format   ZQ_INT2 / ZQ_INT4 / ZQ_INT6 / ZQ_INT8 / ZQ_E4M3
 *   G        block size, a power of two in [32, 1024]
 *   codes    device, zq_codes_bytes(format, n) bytes, written in full
 *   scales   device, zq_num_blocks(n, G) floats, written in full
 * Results are bit-identical to the definition in the layout section above.
 */
zq_status zq_quantize(const void *src, int src_dtype, int64_t n, int format, int64_t G, void *codes,
                      float *scales, void *stream);

/*
 * zq_quantize_multi -- zq_quantize of `count` tensors in as few launches as
 * possible (one per 256 tensors): the results are exactly those of `count`
 * separate zq_quantize calls, but a list of small tensors (a layer's weights,
 * many buffers of a few MB each) streams at the rate of one large tensor
 * instead of paying a launch and a partly filled grid per tensor. A library
 * entry point with no counterpart on the pages; the tensor list is copied into
 * the kernel parameters, so nothing is allocated.
 *   src, n, codes, scales  HOST arrays of `count` entries: tensor k has n[k]
 *             elements at src[k] (device) and writes codes[k], scales[k]
 *             (device) as zq_quantize(src[k], ..., n[k], ...) would; n[k] = 0
 *             is allowed (its pointers are then ignored)
 *   src_dtype, format, G   shared by all tensors
 * Errors as zq_quantize, checked for every tensor before anything is
 * enqueued; no output may overlap any input or any other output.
 */
zq_status zq_quantize_multi(const void *const *src, const int64_t *n, int count, int src_dtype,
                            int format, int64_t G, void *const *codes, float *const *scales,
                            void *stream);

/*
 * zq_dequantize_multi -- zq_dequantize of `count` tensors in as few launches
 * as possible (one per 256 tensors), with the same results as `count`
 * separate calls (a library entry point with no counterpart on the pages;
 * nothing is allocated).
 *   codes, scales, n, dst  HOST arrays of `count` entries: tensor k's n[k]
 *             codes and scales (device, zq_quantize's layout) and its output
 *             dst[k] (device, n[k] elements of dst_dtype); n[k] = 0 allowed
 *   format, G, dst_dtype   shared by all tensors
 * Errors as zq_dequantize, checked for every tensor before anything is
 * enqueued; no output may overlap any input or any other output.
 */
zq_status zq_dequantize_multi(const void *const *codes, const float *const *scales,
                              const int64_t *n, int count, int format, int64_t G, void *const *dst,
                              int dst_dtype, void *stream);

/*
 * zq_dequantize -- inverse of zq_quantize ([ZeRO++] qwZ: dequantize after the
 * gather; qgZ: dequantize before the full-precision reduction).
 *   codes, scales  device, as written by zq_quantize(format, G)
 *   dst            device, n elements of dst_dtype, written in full
 */
zq_status zq_dequantize(const void *codes, const float *scales, int64_t n, int format, int64_t G,
                        void *dst, int dst_dtype, void *stream);

/*
 * zq_reduce_quantized -- quantized gradient reduce ([ZeRO++] qgZ section:
 * dequantize, reduce in full precision, requantize once; [AGoQ] 2.B "Local
 * Reduce": FP8 shards dequantized to FP32, summed, requantized to FP8).
 * For every element i:  acc = +0.0f;  for r = 0 .. nshards-1 in order:
 * acc = fl32(acc + fl32(D(shard r, i)));  then acc is quantized with
 * (format_out, G_out) exactly as zq_quantize would. The sum is not averaged.
 *   codes[r], scales[r]  device pointers held in HOST arrays of nshards
 *                        entries; shard r in (format_in, G_in) layout
 *   nshards              1 .. ZQ_MAX_SHARDS
 *   out_codes, out_scales  device, (format_out, G_out) layout
 *   sum_out              device, n floats (the fp32 sums), or NULL
 * Results are bit-identical to the definition (the shard order is kept).
 */
zq_status zq_reduce_quantized(const void *const *codes, const float *const *scales, int nshards,
                              int64_t n, int format_in, int64_t G_in, void *out_codes,
                              float *out_scales, int format_out, int64_t G_out, float *sum_out,
                              void *stream);

/*
 * zq_reduce_quantized_static -- zq_reduce_quantized for more shards than fit
 * in kernel parameters (up to ZQ_STATIC_MAX_SHARDS = 1024), without allocating
 * anything. There is no counterpart on the pages: this is a library entry point
 * for callers that cannot allocate device memory themselves or let a library do
 * it -- e.g. code whose device memory is entirely owned by another allocator (a
 * framework's caching allocator that has reserved most of HBM, where a stray
 * cudaMalloc can fail or fragment the pool), or a runtime that forbids
 * allocation on its hot path. The shard pointer table that a many-shard reduce
 * needs in device memory lives in a static 16 KiB device array that every GPU
 * which loads the library holds until the process exits.
 * Arguments, results and errors are those of zq_reduce_quantized, except:
 *   nshards   1 .. ZQ_STATIC_MAX_SHARDS; a larger count returns
 *             ZQ_ERR_INVALID_ARG with nothing enqueued.
 *   codes[r], scales[r]  HOST arrays, copied into the device table on `stream`
 *             (stream-ordered copies from host memory) during the call; for
 *             pageable host memory the call returns once they are staged.
 *   stream    must not be capturing: the copies read the caller's host arrays,
 *             which a replayed graph would read again after the caller has
 *             reused them. A call on a capturing stream returns
 *             ZQ_ERR_INVALID_ARG with nothing enqueued (and leaves the
 *             capture intact).
 * The first call in each CUDA context on a device looks up the table's device
 * address with cudaGetSymbolAddress (with that device current) and caches it
 * with the context handle; a new context (e.g. after cudaDeviceReset) is
 * looked up again. All calls share the one table: calls whose work overlaps
 * on the GPU (e.g. on two streams that are not ordered) race on it and must not
 * be issued; calls on one stream are ordered and safe. It calls no cudaMalloc,
 * cudaFree or other allocating routine.
 */
zq_status zq_reduce_quantized_static(const void *const *codes, const float *const *scales,
                                     int nshards, int64_t n, int format_in, int64_t G_in,
                                     void *out_codes, float *out_scales, int format_out,
                                     int64_t G_out, float *sum_out, void *stream);

/*
 * zq_quantize_reordered -- zq_quantize fused with qgZ's tensor-slice
 * reordering ([ZeRO++] sections "Tensor-slice reordering fixes incorrect
 * gradient placement" and "The implementation combines kernel fusion with
 * communication overlap": the reordering is fused into the quantization).
 * The n elements are P = nodes * gpus_per_node chunks of n / P elements;
 * chunk c (the chunk GPU c owns after the reduce-scatter, c = a *
 * gpus_per_node + l for GPU l of node a) is quantized on its own and its codes
 * and scales are stored at slice position l * nodes + a (the transpose of the
 * nodes x gpus_per_node grid of chunks), so that part l of the output holds,
 * node by node, the chunks that GPU l of every node will own.
 *   nodes, gpus_per_node  >= 1, product <= ZQ_MAX_SHARDS
 *   n                     a multiple of 1024 * nodes * gpus_per_node
 * Other arguments, layout and errors as zq_quantize. With one node or one
 * GPU per node the result equals zq_quantize's.
 */
zq_status zq_quantize_reordered(const void *src, int src_dtype, int64_t n, int format, int64_t G,
                                int nodes, int gpus_per_node, void *codes, float *scales,
                                void *stream);

/*
 * zq_reduce_two_hop -- qgZ's two-hop quantized reduce ([ZeRO++] sections "Two-
 * hop communication prevents QGZ traffic from multiplying across GPUs" and
 * "The implementation combines kernel fusion with communication overlap"),
 * with the P = nodes * gpus_per_node GPUs simulated as buffers on this GPU.
 * GPU g = a * gpus_per_node + l holds codes[g], scales[g]: n elements in the
 * layout of zq_quantize_reordered (format_in, G_in). With m = n / P:
 *   hop 1 (intra-node; the dequantize + reduce fused with the requantization
 *     for the inter-node step): mid[g] = requantize(format_mid, G_mid) of the
 *     shard-ordered fp32 sum over l2 = 0..gpus_per_node-1 of part l (the
 *     nodes * m elements at offset l * nodes * m) of GPU a * gpus_per_node + l2;
 *   hop 2 (inter-node): out[g] = requantize(format_out, G_out) of the
 *     node-ordered fp32 sum over a2 = 0..nodes-1 of chunk a (the m elements at
 *     offset a * m) of mid[a2 * gpus_per_node + l]; sums[g] (optional) receives
 *     those fp32 sums. out[g] is the reduced chunk g.
 * Each sum is exactly zq_reduce_quantized's (+0.0f, then one binary32 add per
 * term in the order given); the hop-1 results pass through format_mid, as the
 * pages' protocol sends them. Two reduce launches (one per hop, each over all
 * P GPUs' problems) are enqueued on `stream`.
 *   all pointer arrays   HOST arrays of P device pointers; mid_codes[g] holds
 *                        zq_codes_bytes(format_mid, nodes * m) bytes and
 *                        mid_scales[g] zq_num_blocks(nodes * m, G_mid) floats;
 *                        out_codes[g] / out_scales[g] / sums[g]: m elements
 *   sums                 NULL, or an array of P device pointers
 *   n                    a multiple of 4096 * P (keeps every slice 16-byte aligned)
 * Errors as zq_reduce_quantized; no output may overlap any input or output.
 */
zq_status zq_reduce_two_hop(const void *const *codes, const float *const *scales, int nodes,
                            int gpus_per_node, int64_t n, int format_in, int64_t G_in,
                            void *const *mid_codes, float *const *mid_scales, int format_mid,
                            int64_t G_mid, void *const *out_codes, float *const *out_scales,
                            int format_out, int64_t G_out, float *const *sums, void *stream);

/*
 * zq_reduce_ring -- the ring reduce-scatter's sequential hops for one chunk,
 * the scheme qgZ replaces ([ZeRO++] "QGZ keeps reductions in full precision
 * while sending quantized gradients": in the ring, every hop dequantizes,
 * adds and requantizes). Built for the accuracy comparison with
 * zq_reduce_quantized (one requantization). With partial_0 = shard 0:
 *   hop r = 1 .. nshards-1:  acc = fl32(D(partial_{r-1}) + D(shard r))
 *     (zq_reduce_quantized over the two terms [partial, shard r]);
 *     partial_r = requantize(format, G) of acc into partial buffer r % 2,
 *     except at the last hop, which requantizes to (format_out, G_out) into
 *     out and writes acc to sum_out (optional).
 *   One shard: out = requantize(format_out, G_out) of D(shard 0).
 * The partial sums travel in the shards' own format (format, G).
 *   partial_codes, partial_scales  HOST arrays of 2 device pointers, each
 *       zq_codes_bytes(format, n) bytes / zq_num_blocks(n, G) floats; used
 *       (and required) only for nshards >= 3; no overlap with anything else
 * Other arguments and errors as zq_reduce_quantized (format_in = format).
 * nshards - 1 reduce launches (one for one shard) are enqueued on `stream`.
 */
zq_status zq_reduce_ring(const void *const *codes, const float *const *scales, int nshards,
                         int64_t n, int format, int64_t G, void *const *partial_codes,
                         float *const *partial_scales, void *out_codes, float *out_scales,
                         int format_out, int64_t G_out, float *sum_out, void *stream);

/*
 * zq_interleaved_bytes -- bytes of the metadata-interleaved record stream of
 * n elements ([Aquavit] summary of the implementation, "metadata
 * interleaving", and Eq. 6): one record per G-element block, the block's
 * fp32 scale (4 bytes, little endian) followed by its packed codes (the
 * LSB-first b-bit stream of zq_quantize restricted to the block: G*b/8
 * bytes, or the code bits of a partial last block padded to whole 32-bit
 * words). No padding between records, so the stream has exactly
 * zq_codes_bytes(format, n) + 4 * zq_num_blocks(n, G) bytes and the width
 * stays b + 32/G bits per element. Integer formats only: returns 0 for
 * ZQ_E4M3, an unknown format or an invalid G.
 */
size_t zq_interleaved_bytes(int format, int64_t n, int64_t G);

/*
 * zq_quantize_interleaved -- zq_quantize writing the interleaved record
 * stream instead of separate codes and scales. The codes and scales are
 * exactly zq_quantize's, regrouped.
 *   records  device, zq_interleaved_bytes(format, n, G) bytes, 16-byte aligned,
 *            must not overlap src
 *   format   ZQ_INT2, ZQ_INT4, ZQ_INT6 or ZQ_INT8 (ZQ_E4M3: ZQ_ERR_UNSUPPORTED)
 * Other arguments and errors as zq_quantize.
 */
zq_status zq_quantize_interleaved(const void *src, int src_dtype, int64_t n, int format, int64_t G,
                                  void *records, void *stream);

/*
 * zq_dequantize_interleaved -- zq_dequantize reading an interleaved record
 * stream: y = fl32(q * s) with s the record's scale, then one RNE rounding to
 * dst_dtype. Same results as zq_dequantize of the planar form.
 *   records  device, zq_interleaved_bytes(format, n, G) bytes, 16-byte aligned
 *   dst      device, n elements of dst_dtype; must not overlap records
 * Other arguments and errors as zq_dequantize (integer formats only).
 */
zq_status zq_dequantize_interleaved(const void *records, int64_t n, int format, int64_t G,
                                    void *dst, int dst_dtype, void *stream);

/*
 * zq_aquavit_schedule -- [Aquavit]'s ascending width schedule (summary and
 * Section 5.1): the target width at step t of T is
 *   bpw(t) = 8 - 6 / (a + c * t / T)       ((a, c) = (0.9, 5) on the pages),
 * and the step uses the available pair (b in {2, 4, 6}, G in {32, ..., 1024};
 * the pages' range 2.03 to 7.00 bits per element) whose b + 32/G is nearest
 * to bpw(t), ties to the narrower pair. (The pages give no rule from width to
 * pair; this nearest-width reading is the library's.) Host-only arithmetic.
 *   t, T          0 <= t <= T, T >= 1
 *   a, c          a > 0, c >= 0
 *   format, G     out: ZQ_INT2 / ZQ_INT4 / ZQ_INT6 and the block size
 *   target, width out (either may be NULL): bpw(t) and b + 32/G of the pair
 * Returns ZQ_ERR_INVALID_ARG for arguments outside these ranges or NULL
 * format / G.
 */
zq_status zq_aquavit_schedule(int64_t t, int64_t T, double a, double c, int *format, int64_t *G,
                              double *target, double *width);

/*
 * zq_fp8_accumulate -- in-place FP8 gradient accumulation ([AGoQ] 2.B "Local
 * Accumulation", with the addition in fp32):
 *   v_i = fl32(fl32(e4m3(c_i) * s_block) + g_i), then the block is requantized
 *   to E4M3 with a new scale absmax(v)/448, overwriting codes and scales.
 *   main_codes   device, n E4M3 bytes (zq_codes_bytes(ZQ_E4M3, n) bytes), in place
 *   main_scales  device, zq_num_blocks(n, G) floats, in place
 *   grad         device, n elements of grad_dtype; must not overlap the main gradient
 * A main gradient of all-zero codes and zero scales is the empty accumulator.
 */
zq_status zq_fp8_accumulate(void *main_codes, float *main_scales, const void *grad, int grad_dtype,
                            int64_t n, int64_t G, void *stream);

/*
 * zq_gemm_dequant -- the dequantization fused into the GEMM that consumes the
 * quantized weights ([AGoQ] section "C. Kernel Fusion": quantization and
 * dequantization fused with the adjacent GEMMs, their arithmetic on the CUDA
 * cores and the GEMM on the tensor cores; [ZeRO++] qwZ: the layer computes
 * with the dequantized gathered weights):
 *     y[m][n] = sum over k of x[m][k] * W_hat[n][k],
 *     W_hat[n][k] = bf16(fl32(q * s))  -- exactly zq_dequantize's bf16 output
 *                                         for element n*K + k of W,
 * accumulated in fp32 on the tensor cores (tcgen05, bf16 operands; the order
 * of the fp32 additions is the hardware's), then stored as fp32 or rounded
 * once to bf16. The bf16 weight matrix is never written to memory. Problems
 * with few rows may split K over a cluster of 2, 4 or 8 CTAs (zq_gemm_plan);
 * their partial tiles are added in a fixed order, so the result does not
 * depend on timing either way.
 *   x          device, M x K bf16, row-major (K-major)
 *   w_codes,   device, the zq_quantize output (format, G) of the N x K weight
 *   w_scales   matrix flattened row-major: zq_codes_bytes(format, N*K) bytes
 *              and zq_num_blocks(N*K, G) floats; G must divide K, so every
 *              block lies within one row
 *   y          device, M x N of y_dtype (ZQ_F32 or ZQ_BF16), row-major,
 *              written in full; must not overlap x, w_codes or w_scales
 *   M          >= 0 (any; rows past M in the last tile are not stored)
 *   N, K       multiples of 64 (N, K, M <= 2^31)
 * Errors: ZQ_ERR_UNSUPPORTED for an unknown format or y_dtype;
 * ZQ_ERR_INVALID_ARG for sizes outside these rules; ZQ_ERR_MISALIGNED /
 * ZQ_ERR_ALIAS as elsewhere. M = 0 or N = 0 enqueues nothing. The kernel's
 * pipeline waits are bounded (zq_device_status reports one that ran out).
 */
zq_status zq_gemm_dequant(const void *x, int64_t M, int64_t K, const void *w_codes,
                          const float *w_scales, int format, int64_t G, int64_t N, void *y,
                          int y_dtype, void *stream);

/*
 * zq_gemm_plan -- the output tile zq_gemm_dequant uses for an M x N x K
 * problem on the current device: *bm x *bn rows x columns, and *split CTAs
 * (one cluster) sharing each tile's K range (1: no split). Host only; it
 * queries the device's SM count and cluster occupancy once.
 * Errors: ZQ_ERR_INVALID_ARG for null outputs or sizes zq_gemm_dequant
 * refuses (M < 0, N or K not a positive multiple of 64).
 */
zq_status zq_gemm_plan(int64_t M, int64_t N, int64_t K, int *bm, int *bn, int *split);

/*
 * zq_device_status -- errors the kernels found on the device. The reduce
 * kernels and the dequant-fused GEMM stream tiles into shared memory with
 * bulk asynchronous copies and wait for them with a time limit (2 s); a wait
 * that runs out stops that warp's work (its outputs are then incomplete) and
 * sets a device error word instead of hanging the GPU. This call waits for `stream` to finish
 * (cudaStreamSynchronize), reads and clears the error words of all kernels,
 * and returns ZQ_ERR_TIMEOUT if any wait ran out since the last call,
 * ZQ_ERR_CUDA if the stream reported a CUDA error, and ZQ_OK otherwise.
 * (A library-side check with no counterpart on the pages.)
 */
zq_status zq_device_status(void *stream);

/*
 * zq_wait_selftest -- exercises the bounded device-side waits that
 * zq_device_status reports (a library-side check with no counterpart on the
 * pages). Enqueues one small kernel that waits, with the reduce kernels' own
 * wait routines (the warp-wide wait of their consumer warps and the single-
 * thread wait of their producer lane), on a shared-memory barrier that nothing
 * completes, for limit_us microseconds each; both waits run out, set the
 * timeout bit of the device error word and return. The next
 * zq_device_status(stream) therefore returns ZQ_ERR_TIMEOUT (and clears the
 * word); no output buffer is involved, and the CUDA context stays usable.
 *   limit_us  1 .. 100000 (at most 0.1 s); otherwise ZQ_ERR_INVALID_ARG
 */
zq_status zq_wait_selftest(int64_t limit_us, void *stream);

/* Static description of a status code. */
const char *zq_status_string(int status);

/* CUDA runtime error code (cudaError_t) behind the last ZQ_ERR_CUDA returned
 * on the calling host thread; 0 if none. */
int zq_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZQ_H */
