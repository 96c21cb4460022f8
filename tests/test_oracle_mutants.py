"""Mutation tests for the oracle's pins.

Each case plants one plausible mistake in a temporary copy of the oracle's C
source (never in the repository file), builds it, and checks that at least one
pin from tests/pins.py fails against the broken build. A mutation that no pin
catches would mean the pins leave that part of the oracle unchecked.
"""
import os
import shutil
import tempfile

import pytest

import oracle as O
import pins

SRC = os.path.join(os.path.dirname(O.__file__), "zq_oracle.c")

# (name, text to find (must occur exactly once), replacement)
MUTANTS = [
    ("round_half_away", "float q = nearbyintf(t); /* ties to even, R3 */", "float q = roundf(t);"),
    ("round_half_up", "float q = nearbyintf(t); /* ties to even, R3 */", "float q = floorf(t + 0.5f);"),
    ("truncate_instead_of_round", "float q = nearbyintf(t); /* ties to even, R3 */", "float q = truncf(t);"),
    ("qmax_off_by_one", "else s = m / (float)int_qmax(fmt);", "else s = m / (float)(int_qmax(fmt) + 1);"),
    ("multiply_by_reciprocal", "float t = v[i] / s;      /* IEEE division, R4 */",
     "float t = v[i] * (1.0f / s);"),
    ("no_clamp", "if (q > (float)qmax) q = (float)qmax;", ""),
    ("e4m3_wrong_max", "if (fmt == ORC_E4M3) s = m / 448.0f;", "if (fmt == ORC_E4M3) s = m / 240.0f;"),
    ("msb_first_packing",
     "if ((value >> k) & 1u) stream[(pos + k) >> 3] |= (uint8_t)(1u << ((pos + k) & 7));",
     "if ((value >> k) & 1u) stream[(pos + k) >> 3] |= (uint8_t)(1u << (7 - ((pos + k) & 7)));"),
    ("no_sign_extension", "if (c & (1u << (b - 1))) q -= (int32_t)(1u << b); /* sign extend */", ""),
    ("wrong_scale_index", "store_elem(dst, dst_dtype, i, dequant_elem(codes, scales[i / G], fmt, i));",
     "store_elem(dst, dst_dtype, i, dequant_elem(codes, scales[(i + 1) / G < (n + G - 1) / G ? (i + 1) / G : i / G], fmt, i));"),
    ("reverse_shard_order", "for (r = 0; r < nshards; ++r) {", "for (r = nshards - 1; r >= 0; --r) {"),
    ("reduce_mean", "acc = acc + d; /* one binary32 addition per shard, in shard order */",
     "acc = acc + d / (float)nshards;"),
    ("reduce_uses_out_block", "scales[r][(lo + i) / G_in]", "scales[r][(lo + i) / G_out]"),
    ("reduce_fma",
     "float d = dequant_elem(codes[r], scales[r][(lo + i) / G_in], fmt_in, lo + i);\n"
     "                acc = acc + d; /* one binary32 addition per shard, in shard order */",
     "acc = fmaf(dequant_elem(codes[r], 1.0f, fmt_in, lo + i), scales[r][(lo + i) / G_in], acc);"),
    ("accumulate_fma", "float d = orc_e4m3_decode(codes[lo + i]) * scales[k];\n"
     "            scratch[i] = d + load_elem(grad, grad_dtype, lo + i);",
     "scratch[i] = fmaf(orc_e4m3_decode(codes[lo + i]), scales[k], load_elem(grad, grad_dtype, lo + i));"),
    ("accumulate_drops_grad", "scratch[i] = d + load_elem(grad, grad_dtype, lo + i);", "scratch[i] = d;"),
    ("accumulate_drops_main", "scratch[i] = d + load_elem(grad, grad_dtype, lo + i);",
     "scratch[i] = load_elem(grad, grad_dtype, lo + i);"),
    ("f16_subnormal_exponent", "if (ex == 0) v = ldexp((double)fr, -24);", "if (ex == 0) v = ldexp((double)fr, -25);"),
    ("round_down_in_formats", "r = nearbyint(t);             /* default mode: nearest, ties to even */",
     "r = floor(t);"),
    ("e4m3_no_saturation", "if (r > 448.0) r = 448.0;", ""),
    ("e4m3_bias_8", "else v = ldexp(8.0 + fr, ex - 10);", "else v = ldexp(8.0 + fr, ex - 11);"),
    ("absmax_without_abs", "if (fabsf(v[i]) > m) m = fabsf(v[i]);", "if (v[i] > m) m = v[i];"),
    ("partial_block_off_by_one",
     "int64_t lo = k * G, len = (n - lo < G) ? n - lo : G;\n"
     "        for (i = 0; i < len; ++i) scratch[i] = load_elem(src, dtype, lo + i);",
     "int64_t lo = k * G, len = (n - lo < G) ? n - lo - 1 : G;\n"
     "        for (i = 0; i < len; ++i) scratch[i] = load_elem(src, dtype, lo + i);"),
    ("codes_not_cleared", "memset(codes, 0, (size_t)orc_codes_bytes(fmt, n));", ""),
    ("reorder_identity", "static int64_t slice_position(int64_t c, int A, int L) { return (c % L) * A + c / L; }",
     "static int64_t slice_position(int64_t c, int A, int L) { (void)A; (void)L; return c; }"),
    ("hop1_wrong_part", "            int64_t off = (int64_t)l * A * m;",
     "            int64_t off = (int64_t)((l + 1) % L) * A * m;"),
    ("hop2_wrong_chunk", "            int64_t off = (int64_t)a * m;",
     "            int64_t off = (int64_t)((a + 1) % A) * m;"),
    ("hop1_reverse_order",
     "                sc[r] = codes[a * L + r] + off * code_bits(fmt_in) / 8;\n"
     "                ss[r] = scales[a * L + r] + off / G_in;",
     "                sc[r] = codes[a * L + (L - 1 - r)] + off * code_bits(fmt_in) / 8;\n"
     "                ss[r] = scales[a * L + (L - 1 - r)] + off / G_in;"),
    ("hop2_reverse_order",
     "                sc[r] = mid_codes[r * L + l] + off * code_bits(fmt_mid) / 8;\n"
     "                ss[r] = mid_scales[r * L + l] + off / G_mid;",
     "                sc[r] = mid_codes[(A - 1 - r) * L + l] + off * code_bits(fmt_mid) / 8;\n"
     "                ss[r] = mid_scales[(A - 1 - r) * L + l] + off / G_mid;"),
    ("hop2_wrong_owner",
     "            rc = orc_reduce(sc, ss, A, m, fmt_mid, G_mid, out_codes[a * L + l],\n"
     "                            out_scales[a * L + l], fmt_out, G_out, sums ? sums[a * L + l] : 0);",
     "            rc = orc_reduce(sc, ss, A, m, fmt_mid, G_mid, out_codes[l * A + a],\n"
     "                            out_scales[l * A + a], fmt_out, G_out, sums ? sums[l * A + a] : 0);"),
    ("il_scale_big_endian", "for (i = 0; i < 4; ++i) rec[pos + i] = (uint8_t)(sb >> (8 * i));",
     "for (i = 0; i < 4; ++i) rec[pos + i] = (uint8_t)(sb >> (8 * (3 - i)));"),
    ("il_codes_before_scale",
     "s = quantize_block(scratch, len, fmt, rec + pos + 4, 0);\n"
     "        sb = f32_to_bits(s);\n"
     "        for (i = 0; i < 4; ++i) rec[pos + i] = (uint8_t)(sb >> (8 * i));",
     "s = quantize_block(scratch, len, fmt, rec + pos, 0);\n"
     "        sb = f32_to_bits(s);\n"
     "        for (i = 0; i < 4; ++i) rec[pos + orc_codes_bytes(fmt, len) + i] = (uint8_t)(sb >> (8 * i));"),
    # (stays inside the buffer: records overlap instead of running past its end)
    ("il_stride_without_scale",
     "        pos += 4 + orc_codes_bytes(fmt, len);\n    }\n    return ORC_OK;\n}\n\n/* Dequantize a record stream",
     "        pos += orc_codes_bytes(fmt, len);\n    }\n    return ORC_OK;\n}\n\n/* Dequantize a record stream"),
    ("il_dequant_reads_codes_as_scale", "for (i = 0; i < 4; ++i) sb |= (uint32_t)rec[pos + i] << (8 * i);",
     "for (i = 0; i < 4; ++i) sb |= (uint32_t)rec[pos + 4 + i] << (8 * i);"),
    ("il_size_without_scales", "total += 4 + orc_codes_bytes(fmt, len);", "total += orc_codes_bytes(fmt, len);"),
    ("schedule_a_c_swapped", "return 8.0 - 6.0 / (a + c * (double)t / (double)T);",
     "return 8.0 - 6.0 / (c + a * (double)t / (double)T);"),
    ("schedule_descending", "return 8.0 - 6.0 / (a + c * (double)t / (double)T);",
     "return 8.0 - 6.0 / (a + c * (double)(T - t) / (double)T);"),
    ("pick_rounds_up", "double w = b + 32.0 / (double)g, d = fabs(w - bpw);",
     "double w = b + 32.0 / (double)g, d = (w >= bpw) ? w - bpw : 1e9;"),
    ("pick_allows_8_bit", "for (b = 2; b <= 6; b += 2)", "for (b = 2; b <= 8; b += 2)"),
    ("ring_is_one_hop", "    if (nshards == 1)\n        return orc_reduce(codes, scales, 1, n,",
     "    if (nshards >= 1)\n        return orc_reduce(codes, scales, nshards, n,"),
    ("ring_reverse_chain",
     "    sc[0] = codes[0];\n    ss[0] = scales[0];\n    for (r = 1; r < nshards; ++r) {\n"
     "        sc[1] = codes[r];\n        ss[1] = scales[r];",
     "    sc[0] = codes[nshards - 1];\n    ss[0] = scales[nshards - 1];\n    for (r = 1; r < nshards; ++r) {\n"
     "        sc[1] = codes[nshards - 1 - r];\n        ss[1] = scales[nshards - 1 - r];"),
    # (same sizes: int8 partials written as E4M3 bytes and read back as int8)
    ("ring_partial_in_another_format",
     "rc = orc_reduce(sc, ss, 2, n, fmt, G, pc[r % 2], ps[r % 2], fmt, G, 0);",
     "rc = orc_reduce(sc, ss, 2, n, fmt, G, pc[r % 2], ps[r % 2], fmt == ORC_INT8 ? ORC_E4M3 : fmt, G, 0);"),
    ("gemm_transposed_weight", "int64_t e = n * K + k;", "int64_t e = k * N + n;"),
    ("gemm_no_bf16_rounding", "double w = (double)orc_bf16_decode(orc_bf16_encode(wf));",
     "double w = (double)wf;"),
    ("gemm_scale_of_row_start", "float wf = dequant_elem(codes, scales[e / G], fmt, e);",
     "float wf = dequant_elem(codes, scales[(n * K) / G], fmt, e);"),
    ("gemm_column_major_activations", "double a = (double)orc_bf16_decode(x[m * K + k]);",
     "double a = (double)orc_bf16_decode(x[k * M + m < M * K ? k * M + m : 0]);"),
    ("gemm_signed_magnitudes", "mag += fabs(a * w);", "mag += a * w;"),
    ("ring_skips_last_hop", "    for (r = 1; r < nshards; ++r) {\n        sc[1] = codes[r];",
     "    for (r = 1; r < nshards - 1; ++r) {\n        sc[1] = codes[r];"),
]


def _first_failure(lib):
    for pin in pins.FAST_PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, IndexError, OverflowError) as e:  # noqa: PERF203
            return pin.__name__, e
    return None


@pytest.fixture(scope="module")
def workdir():
    d = tempfile.mkdtemp(prefix="zq_mutants_")
    yield d
    shutil.rmtree(d, ignore_errors=True)


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(workdir, name, find, repl):
    text = open(SRC).read()
    assert text.count(find) == 1, f"mutation anchor for {name} no longer matches the oracle"
    src = os.path.join(workdir, f"{name}.c")
    with open(src, "w") as f:
        f.write(text.replace(find, repl))
    lib = O.load(O.build(src=src, out=os.path.join(workdir, f"{name}.so")))
    caught = _first_failure(lib)
    assert caught is not None, f"no pin catches the mutation {name}"
