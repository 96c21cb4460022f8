/*
 * zq_oracle.c -- the oracle for the blockwise quantize / pack / dequantize /
 * quantized-reduce / FP8-accumulate path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE. This is a plain, slow, single-threaded
 * restatement of what the path computes, written so that it can be checked
 * against the pages by eye. Only the test suite, the package smoke check and
 * the benchmark's CPU-baseline leg may load it. It shares no source, header,
 * table or helper with the CUDA library, and it never calls it.
 *
 * What the pages fix (titles and sections of the source pages):
 *  [ZeRO++]  "Quantized LLM Training at Scale with ZeRO++", section "Blockwise
 *            weight quantization cuts forward-gather traffic in half": weights
 *            are split into blocks and each block is quantized to 8 bits with
 *            its own scale.  Section "QGZ keeps reductions in full precision
 *            while sending quantized gradients": 4- or 8-bit gradients are
 *            dequantized and summed in full precision, then requantized once.
 *  [Aquavit] "Aquavit: Ascending Quantization for Communication-Efficient
 *            Vast-Scale Distributed Training" (review), summary item on
 *            granularity modulation and the glossary entry (Eq. 6, Table 1):
 *            b stays in {2,4,6,8}, each G-element block carries 32 bits of
 *            metadata, so the effective width is b + 32/G bits per element.
 *  [AGoQ]    "AGoQ: Activation and Gradient Quantization for Memory-Efficient
 *            Distributed Training of LLMs", section 2.B (QuanGrad), "Local
 *            Accumulation" (dequantize the FP8 main gradient, add the new
 *            gradient, requantize) and "Precision-Preserved All-Reduce", step
 *            2 "Local Reduce" (dequantize to FP32, sum, requantize to FP8).
 *
 * Readings taken where the pages are silent (each one is a choice):
 *  R1  symmetric codes with one fp32 scale per block and no zero point
 *      (the 32 metadata bits of [Aquavit] are that scale);
 *  R2  scale = absmax / (2^(b-1) - 1) for integer codes and absmax / 448 for
 *      E4M3 (448 is the largest finite E4M3 value);
 *  R3  every rounding is IEEE round-to-nearest, ties-to-even: the division,
 *      the rounding to an integer code and every format conversion;
 *  R4  x / s is one IEEE binary32 division; no fused multiply-add anywhere
 *      (this file must be compiled with -ffp-contract=off);
 *  R5  integer codes are b-bit two's complement in [-qmax, qmax], packed
 *      LSB-first into a bit stream (bit j of the stream is bit j%8 of byte
 *      j/8, i.e. a little-endian stream of 32-bit words); the stream is zero
 *      padded to a multiple of 4 bytes; E4M3 codes are one byte each; scales
 *      are a separate fp32 array in block order;
 *  R6  blocks are G consecutive elements of the flattened tensor; the last
 *      block may be partial;
 *  R7  the reduce is a plain sum (no division by the shard count) taken in
 *      shard index order and starting from +0.0f;
 *  R8  the FP8 accumulate adds in fp32: v = fl(fl(D8(c) * s) + g);
 *  R9  a block whose scale is zero (all-zero block, or a scale that
 *      underflows to zero) gets all-zero code bits.
 *  R10 qgZ's hierarchy ([ZeRO++] sections "Two-hop communication prevents
 *      QGZ traffic from multiplying across GPUs" and "Tensor-slice
 *      reordering fixes incorrect gradient placement"): P = A*L GPUs, A
 *      nodes of L GPUs, GPU g = a*L + l; every gradient is split into P equal
 *      chunks and chunk c is the one GPU c owns after the reduce-scatter.
 *      The reordering is the transpose of the A x L chunk grid: chunk
 *      c = a*L + l is stored at slice position l*A + a, so that part l
 *      (positions l*A .. l*A+A-1) holds, node by node, the chunks that local
 *      GPU l of every node will own. (The pages show an example swap, not a
 *      rule; this is the permutation that makes the two hops below deliver
 *      chunk g to GPU g.)
 *  R11 hop 1 (intra-node, the fused "dequantization and reduction with
 *      inter-node quantization"): GPU (a, l) sums part l of GPUs
 *      (a, 0), ..., (a, L-1) in that order and requantizes it; hop 2
 *      (inter-node): GPU (a, l) sums the a-th chunk of the hop-1 results of
 *      GPUs (0, l), ..., (A-1, l) in that order and requantizes it. Each hop
 *      is one reduce as in R7.
 *  R12 the chunk size n / P is a multiple of 1024 elements, so every chunk
 *      is whole blocks and whole code words.
 *  R13 [Aquavit]'s metadata interleaving (named in the summary of its
 *      implementation, section 5.2-5.3; the layout itself is not described):
 *      one byte stream of block records, record k = block k's fp32 scale (4
 *      bytes, little endian) followed by block k's codes as their own bit
 *      stream (R5) -- G*b/8 bytes for a whole block, the code bits of a
 *      partial last block zero padded to whole 32-bit words. No padding
 *      between records, so the stream is exactly as long as the planar codes
 *      plus scales and the width stays b + 32/G bits per element. Integer
 *      codes only (the b in {2,4,6,8} of granularity modulation).
 *  R14 [Aquavit]'s ascending schedule (summary, Section 5.1): at step t of T
 *      the target width is bpw(t) = 8 - 6/(a + c*t/T), (a, c) = (0.9, 5) by
 *      default. The pages give the range of widths used, 2.03 (b = 2,
 *      G = 1024) to 7.00 (b = 6, G = 32), and no rule that maps a width to a
 *      (b, G) pair; the reading taken: the pair with b in {2,4,6} and G in
 *      {32,...,1024} whose b + 32/G is nearest to bpw(t), ties to the
 *      narrower. (The pages' mean of 5.79 bits over 1000 steps is not met by
 *      this or by the continuous schedule, whose mean is 5.74.)
 *  R15 the ring reduce-scatter that qgZ replaces ([ZeRO++] "QGZ keeps
 *      reductions in full precision while sending quantized gradients":
 *      every hop dequantizes, adds and requantizes): the partial sum of a
 *      chunk travels in the gradients' own format (b, G); hop r (r = 1 ..
 *      N-1) computes acc = fl(D(partial) + D(shard r)) -- the reduce of R7
 *      over the two terms [partial, shard r] -- and requantizes it; the
 *      first partial is shard 0 itself; the last hop keeps acc (the fp32
 *      result) and requantizes it to the output format.
 *  R16 the dequantization fused into the GEMM that consumes the gathered
 *      weights ([AGoQ] section "C. Kernel Fusion": quantization and
 *      dequantization fused with the adjacent GEMMs, the quantize/dequantize
 *      arithmetic on the CUDA cores and the GEMM on the tensor cores; [ZeRO++]
 *      qwZ: the weights a layer uses are the dequantized gathered ones):
 *      the weight matrix W (N x K, row-major) is held as the codes and scales
 *      of its flattened form, blocks of G along each row (K a multiple of G);
 *      the GEMM's weight operand is that matrix dequantized and rounded to
 *      bf16 exactly as the dequantize with a bf16 output does,
 *      W_hat = bf16(fl32(q * s)); the product is y = x W_hat^T for bf16
 *      activations x (M x K, row-major), summed in full precision. The
 *      oracle gives the exact sum (every product of two bf16 values is exact
 *      in binary64, and binary64 accumulation of K terms errs by at most
 *      K 2^-53 of the sum of magnitudes, far below any fp32 accumulation),
 *      together with that sum of magnitudes, from which a caller derives the
 *      error bound of an fp32 accumulation in any order.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* Element types and code formats. The numbering is an interface convention
 * that the tests pass through; it is spelled out again here on purpose. */
#define ORC_F32 0
#define ORC_F16 1
#define ORC_BF16 2

#define ORC_INT2 2
#define ORC_INT4 4
#define ORC_INT6 6
#define ORC_INT8 8
#define ORC_E4M3 0x48

#define ORC_OK 0
#define ORC_BAD (-1)

/* ------------------------------------------------------------------------ */
/* Format helpers                                                           */
/* ------------------------------------------------------------------------ */

/* Bits per code, or 0 for an unknown format. */
static int code_bits(int fmt)
{
    switch (fmt) {
    case ORC_INT2: return 2;
    case ORC_INT4: return 4;
    case ORC_INT6: return 6;
    case ORC_INT8: return 8;
    case ORC_E4M3: return 8;
    default: return 0;
    }
}

/* Largest integer code magnitude, 2^(b-1) - 1 (reading R2). */
static int int_qmax(int fmt) { return (1 << (code_bits(fmt) - 1)) - 1; }

static int valid_block(int64_t G)
{
    return G == 32 || G == 64 || G == 128 || G == 256 || G == 512 || G == 1024;
}

static int elem_size(int dtype)
{
    return dtype == ORC_F32 ? 4 : (dtype == ORC_F16 || dtype == ORC_BF16) ? 2 : 0;
}

/* Bytes of the packed code stream: ceil(n*b/32) 32-bit words (reading R5). */
int64_t orc_codes_bytes(int fmt, int64_t n)
{
    int b = code_bits(fmt);
    if (b == 0 || n < 0) return -1;
    return ((n * b + 31) / 32) * 4;
}

/* Number of G-element blocks, ceil(n/G) (reading R6). */
int64_t orc_num_blocks(int64_t n, int64_t G)
{
    if (n < 0 || !valid_block(G)) return -1;
    return (n + G - 1) / G;
}

/* ------------------------------------------------------------------------ */
/* Binary floating-point formats, written from their definitions            */
/* (IEEE 754 binary16 and binary32; bfloat16 = upper half of binary32;      */
/* OCP 8-bit floating point E4M3: bias 7, no infinities, S.1111.111 = NaN,  */
/* largest finite 448).                                                      */
/* ------------------------------------------------------------------------ */

/* Round a finite magnitude a >= 0 (a double holding a binary32 value) to the
 * nearest value of a binary format with p significand bits (hidden bit
 * included) and smallest normal exponent emin, ties to even. Values below
 * 2^emin are rounded to multiples of 2^(emin-p+1) (gradual underflow). No
 * overflow handling: the caller decides what happens above its largest value. */
static double round_to_format(double a, int p, int emin)
{
    int k;
    double quantum, t, r;
    if (a == 0.0) return 0.0;
    (void)frexp(a, &k);           /* a = f * 2^k with f in [0.5, 1) */
    if (k - 1 < emin) k = emin + 1;
    quantum = ldexp(1.0, (k - 1) - (p - 1));
    t = a / quantum;              /* exact: division by a power of two */
    r = nearbyint(t);             /* default mode: nearest, ties to even */
    return r * quantum;           /* exact */
}

/* Exponent e with 2^e <= a < 2^(e+1), for a > 0. */
static int exponent_of(double a)
{
    int k;
    (void)frexp(a, &k);
    return k - 1;
}

static float bits_to_f32(uint32_t u)
{
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static uint32_t f32_to_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
float orc_f16_decode(uint32_t h)
{
    int sign = (h >> 15) & 1, ex = (h >> 10) & 31, fr = h & 1023;
    double v;
    if (ex == 0) v = ldexp((double)fr, -24);
    else if (ex == 31) v = fr ? NAN : INFINITY;
    else v = ldexp(1024.0 + fr, ex - 25);
    return (float)(sign ? -v : v);
}

uint32_t orc_f16_encode(float x)
{
    uint32_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs((double)x), r;
    int e;
    if (isnan(x)) return 0x7E00u;
    if (isinf(x)) return sign | 0x7C00u;
    r = round_to_format(a, 11, -14);
    if (r > 65504.0) return sign | 0x7C00u;          /* overflow to infinity */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) return sign | (uint32_t)(r / ldexp(1.0, -24));
    e = exponent_of(r);
    return sign | (uint32_t)(e + 15) << 10 | (uint32_t)((r / ldexp(1.0, e) - 1.0) * 1024.0);
}

/* bfloat16 is the upper 16 bits of a binary32 (8 significand bits). */
float orc_bf16_decode(uint32_t h) { return bits_to_f32((h & 0xFFFFu) << 16); }

uint32_t orc_bf16_encode(float x)
{
    uint32_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs((double)x), r;
    if (isnan(x)) return 0x7FC0u;
    if (isinf(x)) return sign | 0x7F80u;
    r = round_to_format(a, 8, -126);
    if (r > ldexp(255.0, 120)) return sign | 0x7F80u; /* above (2-2^-7)*2^127 */
    /* r is a bfloat16 value, so it is exact in binary32; keep the top half. */
    return sign | (f32_to_bits((float)r) >> 16);
}

/* E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits. */
float orc_e4m3_decode(uint32_t c)
{
    int sign = (c >> 7) & 1, ex = (c >> 3) & 15, fr = c & 7;
    double v;
    if (ex == 15 && fr == 7) return NAN;
    if (ex == 0) v = ldexp((double)fr, -9);
    else v = ldexp(8.0 + fr, ex - 10);
    return (float)(sign ? -v : v);
}

/* Round to nearest E4M3, ties to even, saturating to +-448 ("satfinite"). */
uint32_t orc_e4m3_encode(float x)
{
    uint32_t sign = signbit(x) ? 0x80u : 0u;
    double a = fabs((double)x), r;
    int e;
    if (isnan(x)) return 0x7Fu;
    r = isinf(x) ? 448.0 : round_to_format(a, 4, -6);
    if (r > 448.0) r = 448.0;
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -6)) return sign | (uint32_t)(r / ldexp(1.0, -9));
    e = exponent_of(r);
    return sign | (uint32_t)(e + 7) << 3 | (uint32_t)((r / ldexp(1.0, e) - 1.0) * 8.0);
}

/* Element i of a source buffer, widened exactly to binary32. */
static float load_elem(const void *p, int dtype, int64_t i)
{
    if (dtype == ORC_F32) return ((const float *)p)[i];
    if (dtype == ORC_F16) return orc_f16_decode(((const uint16_t *)p)[i]);
    return orc_bf16_decode(((const uint16_t *)p)[i]);
}

/* Store a binary32 value as element i of a destination buffer (one RNE
 * rounding for the 16-bit types). */
static void store_elem(void *p, int dtype, int64_t i, float v)
{
    if (dtype == ORC_F32) ((float *)p)[i] = v;
    else if (dtype == ORC_F16) ((uint16_t *)p)[i] = (uint16_t)orc_f16_encode(v);
    else ((uint16_t *)p)[i] = (uint16_t)orc_bf16_encode(v);
}

/* ------------------------------------------------------------------------ */
/* Bit stream (reading R5)                                                  */
/* ------------------------------------------------------------------------ */

static void put_bits(uint8_t *stream, int64_t pos, int nbits, uint32_t value)
{
    int k;
    for (k = 0; k < nbits; ++k)
        if ((value >> k) & 1u) stream[(pos + k) >> 3] |= (uint8_t)(1u << ((pos + k) & 7));
}

static uint32_t get_bits(const uint8_t *stream, int64_t pos, int nbits)
{
    uint32_t v = 0;
    int k;
    for (k = 0; k < nbits; ++k)
        v |= (uint32_t)((stream[(pos + k) >> 3] >> ((pos + k) & 7)) & 1u) << k;
    return v;
}

/* ------------------------------------------------------------------------ */
/* One block: absmax, scale, codes                                          */
/* ------------------------------------------------------------------------ */

/* Quantize the values v[0..len) of one block into the stream at element
 * offset first; returns the block's scale. [ZeRO++] qwZ section; [Aquavit]
 * Eq. 6; [AGoQ] 2.B for the E4M3 case. */
static float quantize_block(const float *v, int64_t len, int fmt, uint8_t *codes, int64_t first)
{
    int b = code_bits(fmt);
    float m = 0.0f, s;
    int64_t i;

    /* absmax over the block (exact, order free) */
    for (i = 0; i < len; ++i)
        if (fabsf(v[i]) > m) m = fabsf(v[i]);

    /* scale: one IEEE binary32 division (R2, R3) */
    if (fmt == ORC_E4M3) s = m / 448.0f;
    else s = m / (float)int_qmax(fmt);

    for (i = 0; i < len; ++i) {
        uint32_t c;
        if (s == 0.0f) {
            c = 0; /* R9 */
        } else if (fmt == ORC_E4M3) {
            float t = v[i] / s;
            c = orc_e4m3_encode(t);
        } else {
            int qmax = int_qmax(fmt);
            float t = v[i] / s;      /* IEEE division, R4 */
            float q = nearbyintf(t); /* ties to even, R3 */
            if (q > (float)qmax) q = (float)qmax;
            if (q < (float)-qmax) q = (float)-qmax;
            c = (uint32_t)(int32_t)q & ((1u << b) - 1u); /* two's complement */
        }
        put_bits(codes, (first + i) * b, b, c);
    }
    return s;
}

/* Value of code element i: the integer code, or the E4M3 value, times s. */
static float dequant_elem(const uint8_t *codes, float s, int fmt, int64_t i)
{
    int b = code_bits(fmt);
    uint32_t c = get_bits(codes, i * b, b);
    if (fmt == ORC_E4M3) return orc_e4m3_decode(c) * s;
    {
        int32_t q = (int32_t)c;
        if (c & (1u << (b - 1))) q -= (int32_t)(1u << b); /* sign extend */
        return (float)q * s;                                /* one binary32 multiply */
    }
}

/* ------------------------------------------------------------------------ */
/* Public oracle entry points                                               */
/* ------------------------------------------------------------------------ */

/* Each entry point below keeps one block of widened values (G <= 1024) in a
 * local array, so that independent calls may run on several host threads at
 * once (the full-size parity tests split a tensor into whole-block chunks). */

/* Quantize n elements of src (dtype) into packed codes and one scale per
 * block. codes must hold orc_codes_bytes(fmt, n) bytes, scales
 * orc_num_blocks(n, G) floats. */
int orc_quantize(const void *src, int dtype, int64_t n, int fmt, int64_t G, uint8_t *codes,
                 float *scales)
{
    float scratch[1024];
    int64_t k, i, nb;
    if (!code_bits(fmt) || !valid_block(G) || !elem_size(dtype) || n < 0) return ORC_BAD;
    memset(codes, 0, (size_t)orc_codes_bytes(fmt, n));
    nb = orc_num_blocks(n, G);
    for (k = 0; k < nb; ++k) {
        int64_t lo = k * G, len = (n - lo < G) ? n - lo : G;
        for (i = 0; i < len; ++i) scratch[i] = load_elem(src, dtype, lo + i);
        scales[k] = quantize_block(scratch, len, fmt, codes, lo);
    }
    return ORC_OK;
}

/* Dequantize: y = fl32(q * s), then one RNE rounding to dst_dtype. */
int orc_dequantize(const uint8_t *codes, const float *scales, int64_t n, int fmt, int64_t G,
                   void *dst, int dst_dtype)
{
    int64_t i;
    if (!code_bits(fmt) || !valid_block(G) || !elem_size(dst_dtype) || n < 0) return ORC_BAD;
    for (i = 0; i < n; ++i) store_elem(dst, dst_dtype, i, dequant_elem(codes, scales[i / G], fmt, i));
    return ORC_OK;
}

/* Quantized reduce ([ZeRO++] qgZ; [AGoQ] Local Reduce): for every element,
 * acc = +0.0f, then acc = fl(acc + D(shard r)) for r = 0..nshards-1 in
 * order; optionally store acc; then quantize acc with (fmt_out, G_out). */
int orc_reduce(const uint8_t *const *codes, const float *const *scales, int nshards, int64_t n,
               int fmt_in, int64_t G_in, uint8_t *out_codes, float *out_scales, int fmt_out,
               int64_t G_out, float *sum_out)
{
    float scratch[1024];
    int64_t k, i, nb;
    int r;
    if (!code_bits(fmt_in) || !code_bits(fmt_out) || !valid_block(G_in) || !valid_block(G_out) ||
        nshards < 1 || n < 0)
        return ORC_BAD;
    memset(out_codes, 0, (size_t)orc_codes_bytes(fmt_out, n));
    nb = orc_num_blocks(n, G_out);
    for (k = 0; k < nb; ++k) {
        int64_t lo = k * G_out, len = (n - lo < G_out) ? n - lo : G_out;
        for (i = 0; i < len; ++i) {
            float acc = 0.0f;
            for (r = 0; r < nshards; ++r) {
                float d = dequant_elem(codes[r], scales[r][(lo + i) / G_in], fmt_in, lo + i);
                acc = acc + d; /* one binary32 addition per shard, in shard order */
            }
            scratch[i] = acc;
            if (sum_out) sum_out[lo + i] = acc;
        }
        out_scales[k] = quantize_block(scratch, len, fmt_out, out_codes, lo);
    }
    return ORC_OK;
}

/* Slice position of chunk c (reading R10). */
static int64_t slice_position(int64_t c, int A, int L) { return (c % L) * A + c / L; }

static int two_hop_ok(int64_t n, int A, int L)
{
    int64_t P = (int64_t)A * L;
    return A >= 1 && L >= 1 && A <= 64 && L <= 64 && n >= 0 && n % (P * 1024) == 0;
}

/* Quantize with tensor-slice reordering ([ZeRO++] "Tensor-slice reordering
 * fixes incorrect gradient placement", readings R10 and R12): the n elements
 * form P = A*L chunks of m = n/P; chunk c is quantized on its own and its
 * codes and scales are written at slice position (c % L)*A + c/L. */
int orc_quantize_reordered(const void *src, int dtype, int64_t n, int fmt, int64_t G, int A, int L,
                           uint8_t *codes, float *scales)
{
    int64_t P, m, c;
    if (!code_bits(fmt) || !valid_block(G) || !elem_size(dtype) || !two_hop_ok(n, A, L))
        return ORC_BAD;
    P = (int64_t)A * L;
    m = n / P;
    for (c = 0; c < P; ++c) {
        int64_t pos = slice_position(c, A, L);
        int rc = orc_quantize((const char *)src + c * m * elem_size(dtype), dtype, m, fmt, G,
                              codes + pos * m * code_bits(fmt) / 8, scales + pos * m / G);
        if (rc != ORC_OK) return rc;
    }
    return ORC_OK;
}

/* Two-hop quantized reduce (readings R10-R12), all GPUs simulated here.
 * codes[g], scales[g]: GPU g's n elements in the reordered layout (fmt_in,
 * G_in). Hop 1: mid[a*L + l] = requant_(fmt_mid, G_mid)( sum over l2 = 0..L-1
 * of part l of GPU a*L + l2 ), A*m elements. Hop 2: out[a*L + l] =
 * requant_(fmt_out, G_out)( sum over a2 = 0..A-1 of chunk a of mid[a2*L + l] ),
 * m elements: the reduced chunk a*L + l. sums[g] (optional, m floats each)
 * receives hop 2's fp32 sums. */
int orc_reduce_two_hop(const uint8_t *const *codes, const float *const *scales, int A, int L,
                       int64_t n, int fmt_in, int64_t G_in, uint8_t *const *mid_codes,
                       float *const *mid_scales, int fmt_mid, int64_t G_mid,
                       uint8_t *const *out_codes, float *const *out_scales, int fmt_out,
                       int64_t G_out, float *const *sums)
{
    const uint8_t *sc[64];
    const float *ss[64];
    int64_t m;
    int a, l, r, rc;
    if (!code_bits(fmt_in) || !code_bits(fmt_mid) || !code_bits(fmt_out) || !valid_block(G_in) ||
        !valid_block(G_mid) || !valid_block(G_out) || !two_hop_ok(n, A, L))
        return ORC_BAD;
    m = n / ((int64_t)A * L);
    for (a = 0; a < A; ++a)      /* hop 1 */
        for (l = 0; l < L; ++l) {
            int64_t off = (int64_t)l * A * m;
            for (r = 0; r < L; ++r) {
                sc[r] = codes[a * L + r] + off * code_bits(fmt_in) / 8;
                ss[r] = scales[a * L + r] + off / G_in;
            }
            rc = orc_reduce(sc, ss, L, (int64_t)A * m, fmt_in, G_in, mid_codes[a * L + l],
                            mid_scales[a * L + l], fmt_mid, G_mid, 0);
            if (rc != ORC_OK) return rc;
        }
    for (a = 0; a < A; ++a)      /* hop 2 */
        for (l = 0; l < L; ++l) {
            int64_t off = (int64_t)a * m;
            for (r = 0; r < A; ++r) {
                sc[r] = mid_codes[r * L + l] + off * code_bits(fmt_mid) / 8;
                ss[r] = mid_scales[r * L + l] + off / G_mid;
            }
            rc = orc_reduce(sc, ss, A, m, fmt_mid, G_mid, out_codes[a * L + l],
                            out_scales[a * L + l], fmt_out, G_out, sums ? sums[a * L + l] : 0);
            if (rc != ORC_OK) return rc;
        }
    return ORC_OK;
}

/* FP8 gradient accumulation in place ([AGoQ] Local Accumulation, reading R8):
 * v = fl(fl(D8(c) * s) + g), then E4M3 requantization of v with block G. */
int orc_fp8_accumulate(uint8_t *codes, float *scales, const void *grad, int grad_dtype, int64_t n,
                       int64_t G)
{
    float scratch[1024];
    int64_t k, i, nb;
    if (!valid_block(G) || !elem_size(grad_dtype) || n < 0) return ORC_BAD;
    nb = orc_num_blocks(n, G);
    for (k = 0; k < nb; ++k) {
        int64_t lo = k * G, len = (n - lo < G) ? n - lo : G;
        for (i = 0; i < len; ++i) {
            float d = orc_e4m3_decode(codes[lo + i]) * scales[k];
            scratch[i] = d + load_elem(grad, grad_dtype, lo + i);
        }
        /* the block's old code bytes are replaced by the new ones */
        for (i = 0; i < len; ++i) codes[lo + i] = 0;
        scales[k] = quantize_block(scratch, len, ORC_E4M3, codes, lo);
    }
    return ORC_OK;
}

/* Array forms of the codecs (kind = ORC_F16, ORC_BF16 or ORC_E4M3), so that
 * the tests can check every bit pattern without one foreign call per value. */
int orc_encode_n(int kind, const float *x, int64_t n, uint32_t *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) {
        if (kind == ORC_F16) out[i] = orc_f16_encode(x[i]);
        else if (kind == ORC_BF16) out[i] = orc_bf16_encode(x[i]);
        else if (kind == ORC_E4M3) out[i] = orc_e4m3_encode(x[i]);
        else return ORC_BAD;
    }
    return ORC_OK;
}

int orc_decode_n(int kind, const uint32_t *c, int64_t n, float *out)
{
    int64_t i;
    for (i = 0; i < n; ++i) {
        if (kind == ORC_F16) out[i] = orc_f16_decode(c[i]);
        else if (kind == ORC_BF16) out[i] = orc_bf16_decode(c[i]);
        else if (kind == ORC_E4M3) out[i] = orc_e4m3_decode(c[i]);
        else return ORC_BAD;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [Aquavit] metadata interleaving (reading R13)                            */
/* ------------------------------------------------------------------------ */

/* Bytes of the interleaved record stream of n elements, or -1 when the
 * format has no interleaved form. */
int64_t orc_il_bytes(int fmt, int64_t n, int64_t G)
{
    int64_t nb, k, total = 0;
    if (fmt == ORC_E4M3 || !code_bits(fmt) || !valid_block(G) || n < 0) return -1;
    nb = orc_num_blocks(n, G);
    for (k = 0; k < nb; ++k) {
        int64_t len = (n - k * G < G) ? n - k * G : G;
        total += 4 + orc_codes_bytes(fmt, len);
    }
    return total;
}

/* Quantize n elements of src into the record stream rec (orc_il_bytes
 * bytes): each block is quantized exactly as by orc_quantize, its scale
 * written at the start of its record and its codes after it. */
int orc_quantize_interleaved(const void *src, int dtype, int64_t n, int fmt, int64_t G, uint8_t *rec)
{
    float scratch[1024];
    int64_t k, i, nb, pos = 0;
    if (orc_il_bytes(fmt, n, G) < 0 || !elem_size(dtype)) return ORC_BAD;
    memset(rec, 0, (size_t)orc_il_bytes(fmt, n, G));
    nb = orc_num_blocks(n, G);
    for (k = 0; k < nb; ++k) {
        int64_t lo = k * G, len = (n - lo < G) ? n - lo : G;
        uint32_t sb;
        float s;
        for (i = 0; i < len; ++i) scratch[i] = load_elem(src, dtype, lo + i);
        s = quantize_block(scratch, len, fmt, rec + pos + 4, 0);
        sb = f32_to_bits(s);
        for (i = 0; i < 4; ++i) rec[pos + i] = (uint8_t)(sb >> (8 * i));
        pos += 4 + orc_codes_bytes(fmt, len);
    }
    return ORC_OK;
}

/* Dequantize a record stream: y = fl32(q * s) with s read from the record's
 * head, then one RNE rounding to dst_dtype (as orc_dequantize). */
int orc_dequantize_interleaved(const uint8_t *rec, int64_t n, int fmt, int64_t G, void *dst,
                               int dst_dtype)
{
    int64_t k, i, nb, pos = 0;
    if (orc_il_bytes(fmt, n, G) < 0 || !elem_size(dst_dtype)) return ORC_BAD;
    nb = orc_num_blocks(n, G);
    for (k = 0; k < nb; ++k) {
        int64_t lo = k * G, len = (n - lo < G) ? n - lo : G;
        uint32_t sb = 0;
        float s;
        for (i = 0; i < 4; ++i) sb |= (uint32_t)rec[pos + i] << (8 * i);
        s = bits_to_f32(sb);
        for (i = 0; i < len; ++i) store_elem(dst, dst_dtype, lo + i, dequant_elem(rec + pos + 4, s, fmt, i));
        pos += 4 + orc_codes_bytes(fmt, len);
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* [Aquavit] ascending schedule (reading R14)                               */
/* ------------------------------------------------------------------------ */

/* Target width at step t of T: 8 - 6 / (a + c t / T). */
double orc_aquavit_bpw(int64_t t, int64_t T, double a, double c)
{
    return 8.0 - 6.0 / (a + c * (double)t / (double)T);
}

/* The (b, G) pair for a target width: nearest b + 32/G over b in {2,4,6},
 * G in {32,...,1024}, ties to the narrower pair. Returns the pair's width. */
double orc_aquavit_pick(double bpw, int *bits, int64_t *G)
{
    double best = -1.0, bestd = 0.0;
    int b;
    int64_t g;
    for (b = 2; b <= 6; b += 2)
        for (g = 32; g <= 1024; g *= 2) {
            double w = b + 32.0 / (double)g, d = fabs(w - bpw);
            if (best < 0.0 || d < bestd || (d == bestd && w < best)) {
                best = w;
                bestd = d;
                *bits = b;
                *G = g;
            }
        }
    return best;
}

/* ------------------------------------------------------------------------ */
/* Ring reduce-scatter hops (reading R15), for the accuracy comparison      */
/* ------------------------------------------------------------------------ */

/* Reduce N shards (fmt, G) the ring way: partial_0 = shard 0; for r = 1 ..
 * N-1, acc = fl(D(partial_{r-1}) + D(shard r)); partial_r = quantize(acc)
 * with (fmt, G) for r < N-1 and with (fmt_out, G_out) into out for r = N-1,
 * whose acc goes to sum_out (optional). One shard: out = quantize(D(shard 0)).
 * pc[0..1], ps[0..1]: two partial buffers of n elements in (fmt, G). */
int orc_reduce_ring(const uint8_t *const *codes, const float *const *scales, int nshards, int64_t n,
                    int fmt, int64_t G, uint8_t *const *pc, float *const *ps, uint8_t *out_codes,
                    float *out_scales, int fmt_out, int64_t G_out, float *sum_out)
{
    const uint8_t *sc[2];
    const float *ss[2];
    int r, rc;
    if (nshards < 1 || nshards > 64) return ORC_BAD;
    if (nshards == 1)
        return orc_reduce(codes, scales, 1, n, fmt, G, out_codes, out_scales, fmt_out, G_out, sum_out);
    sc[0] = codes[0];
    ss[0] = scales[0];
    for (r = 1; r < nshards; ++r) {
        sc[1] = codes[r];
        ss[1] = scales[r];
        if (r < nshards - 1) {
            rc = orc_reduce(sc, ss, 2, n, fmt, G, pc[r % 2], ps[r % 2], fmt, G, 0);
            sc[0] = pc[r % 2];
            ss[0] = ps[r % 2];
        } else {
            rc = orc_reduce(sc, ss, 2, n, fmt, G, out_codes, out_scales, fmt_out, G_out, sum_out);
        }
        if (rc != ORC_OK) return rc;
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Dequantization fused into the consumer GEMM (reading R16)                */
/* ------------------------------------------------------------------------ */

/* For each of the `count` output positions (rows[i], cols[i]):
 *   y[i]    = sum over k of x[rows[i]][k] * W_hat[cols[i]][k]   (exact, binary64)
 *   absy[i] = sum over k of |x[rows[i]][k] * W_hat[cols[i]][k]|
 * with W_hat[n][k] the bf16 rounding of the dequantized element n*K + k of
 * the flattened weight (codes, scales in (fmt, G) layout). x holds M*K bf16
 * bit patterns. Requires K to be a multiple of G. */
int orc_gemm_dequant(const uint16_t *x, int64_t M, int64_t K, const uint8_t *codes,
                     const float *scales, int fmt, int64_t G, int64_t N, const int64_t *rows,
                     const int64_t *cols, int64_t count, double *y, double *absy)
{
    int64_t i, k;
    if (!code_bits(fmt) || !valid_block(G) || M < 1 || N < 1 || K < 1 || K % G != 0 || count < 0)
        return ORC_BAD;
    for (i = 0; i < count; ++i) {
        int64_t m = rows[i], n = cols[i];
        double acc = 0.0, mag = 0.0;
        if (m < 0 || m >= M || n < 0 || n >= N) return ORC_BAD;
        for (k = 0; k < K; ++k) {
            int64_t e = n * K + k;
            float wf = dequant_elem(codes, scales[e / G], fmt, e);       /* fl32(q * s) */
            double w = (double)orc_bf16_decode(orc_bf16_encode(wf));     /* then bf16 */
            double a = (double)orc_bf16_decode(x[m * K + k]);
            acc += a * w; /* exact product; binary64 sum */
            mag += fabs(a * w);
        }
        y[i] = acc;
        absy[i] = mag;
    }
    return ORC_OK;
}
