"""Pins for the oracle: checks against what the pages, the format specifications
and the mathematics fix, independent of the oracle's own code.

Each ``pin_*`` takes a loaded oracle library (so that the mutation tests can
run the same checks against deliberately broken builds) and raises
AssertionError on a mismatch. Sizes are kept small so that the whole set runs
in seconds; the exhaustive variants live in the test modules.

Independent routes used here (none of them re-runs the oracle's formula):
  * values printed on the pages (tests/golden/*.json, each with its source);
  * the OCP FP8 and IEEE 754 format definitions, through torch's float8 and
    bfloat16 conversions and numpy's float16 conversion (library routines);
  * exact rational arithmetic (fractions.Fraction) for divisions and roundings;
  * correctly rounded binary32 quotients obtained as binary64 quotients rounded
    to binary32 (double rounding is innocuous for division when the wide
    format has at least 2p+2 bits: S. Figueroa, "When is double rounding
    innocuous?", SIGNUM Newsletter 30(3), 1995);
  * closed forms (power-of-two scales make every product and partial sum
    exact, so fp32 results must equal integer arithmetic);
  * invariants (block independence, idempotence, error bounds).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
INT_FORMATS = (O.INT2, O.INT4, O.INT6, O.INT8)
ALL_FORMATS = INT_FORMATS + (O.E4M3,)
BLOCKS = (32, 64, 128, 256, 512, 1024)


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def qmax(fmt: int) -> int:
    return (1 << (O.BITS[fmt] - 1)) - 1


# ---------------------------------------------------------------------------
# exact helpers (independent of the oracle)
# ---------------------------------------------------------------------------

def rn32(v: Fraction) -> Fraction:
    """Nearest binary32 value to the rational v (ties to even), by exact arithmetic."""
    if v == 0:
        return Fraction(0)
    sign = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 23)
    r = round(a / quantum)  # Fraction rounds half to even
    return sign * r * quantum


def div32(x: np.ndarray, s) -> np.ndarray:
    """Correctly rounded binary32 quotient x/s via a binary64 quotient (Figueroa)."""
    return (np.asarray(x, dtype=np.float64) / np.float64(s)).astype(np.float32)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def torch_bf16_bits(x32: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def torch_e4m3_codes(x32: np.ndarray) -> np.ndarray:
    import torch

    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def unpack_codes(codes: np.ndarray, n: int, bits: int) -> np.ndarray:
    """Signed integer codes from the LSB-first stream, read with numpy's bit unpacking."""
    stream = np.unpackbits(codes, bitorder="little")[: n * bits].reshape(n, bits).astype(np.int64)
    vals = (stream << np.arange(bits)).sum(axis=1)
    return np.where(vals >= (1 << (bits - 1)), vals - (1 << bits), vals)


def rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)


# ---------------------------------------------------------------------------
# sizes and payloads printed on the pages
# ---------------------------------------------------------------------------

def pin_bpw_endpoints(lib):
    """Aquavit Table 1 endpoints: 2-bit/G=1024 -> 2.03 bpw, 6-bit/G=32 -> 7.00 bpw."""
    g = golden("granularity_modulation_bpw.json")
    fmt_of = {2: O.INT2, 4: O.INT4, 6: O.INT6, 8: O.INT8}
    x = rng(1).standard_normal(8192).astype(np.float32)
    for e in g["printed_endpoints"]:
        codes, scales = O.quantize(x, fmt_of[e["bits"]], e["G"], lib=lib)
        bpw = (codes.nbytes + scales.nbytes) * 8 / x.size
        assert f"{bpw:.2f}" == e["bpw_printed"], (e, bpw)


def pin_bpw_formula(lib):
    """Eq. 6 of the Aquavit page, bpw = b + 32/G, for every (b, G) of the sweep."""
    g = golden("granularity_modulation_bpw.json")
    fmt_of = {2: O.INT2, 4: O.INT4, 6: O.INT6, 8: O.INT8}
    n = 4096
    x = rng(2).standard_normal(n).astype(np.float32)
    for b in g["bits"]:
        for G in g["block_sizes"]:
            codes, scales = O.quantize(x, fmt_of[b], G, lib=lib)
            assert Fraction((codes.nbytes + scales.nbytes) * 8, n) == b + Fraction(32, G), (b, G)


def pin_zeropp_payload(lib):
    """ZeRO++: 3M -> 0.75M = 0.5M (int8 weights) + 0 (hpZ) + 0.25M (int4 gradients)."""
    g = golden("zeropp_payload.json")
    n = 1 << 14
    w = rng(3).standard_normal(n).astype(np.float16)
    fp16_bytes = w.nbytes
    c8, _ = O.quantize(w, O.INT8, 256, lib=lib)
    c4, _ = O.quantize(w.astype(np.float32), O.INT4, 128, lib=lib)
    parts = g["parts"]
    assert Fraction(c8.nbytes, fp16_bytes) == Fraction(parts["forward_allgather_int8_weights"])
    assert Fraction(c4.nbytes, fp16_bytes) == Fraction(parts["gradient_reduce_int4"])
    total = Fraction(c8.nbytes + 0 + c4.nbytes, fp16_bytes)
    assert total == Fraction(g["zeropp_total_in_M"]) and g["baseline_collectives_in_M"] == 3.0


def pin_bit_layout(lib):
    """Hand-derived packed bytes for each code width (scale exactly 1)."""
    fmt_of = {2: O.INT2, 4: O.INT4, 6: O.INT6, 8: O.INT8}
    for case in golden("bit_layout.json")["cases"]:
        x = np.array(case["values"], dtype=np.float32)
        codes, scales = O.quantize(x, fmt_of[case["bits"]], 32, lib=lib)
        assert scales[0] == 1.0, case
        assert codes.tobytes().hex() == case["bytes"], (case, codes.tobytes().hex())


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------

def pin_e4m3_points(lib):
    g = golden("e4m3_points.json")
    for e in g["encode"]:
        got = O.encode_array("e4m3", np.array([e["x"]], np.float32), lib=lib)[0]
        assert got == int(e["code"], 16), (e, hex(got))
    for e in g["decode"]:
        got = O.decode_array("e4m3", np.array([int(e["code"], 16)]), lib=lib)[0]
        if e["x"] == "nan":
            assert math.isnan(got), e
        else:
            assert got == e["x"], (e, got)


def pin_e4m3_vs_library(lib, n_random=200_000):
    """All 256 decodes, and encodes of random values, midpoints and their neighbours."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    got = O.decode_array("e4m3", codes.astype(np.uint32), lib=lib)
    assert np.array_equal(np.isnan(ref), np.isnan(got))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok].view(np.uint32), got[ok].view(np.uint32))
    # midpoints between consecutive finite magnitudes, and one binary32 ulp either side
    mags = np.unique(np.abs(ref[ok]).astype(np.float64))
    mids = ((mags[1:] + mags[:-1]) / 2).astype(np.float32)
    around = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)),
                             mags.astype(np.float32)])
    r = rng(4)
    rand = (r.uniform(-1, 1, n_random) * 2.0 ** r.integers(-14, 9, n_random)).astype(np.float32)
    x = np.concatenate([around, -around, rand])
    x = x[np.abs(x) < 464]  # the library maps values at and above 464 to NaN, not to 448
    assert np.array_equal(O.encode_array("e4m3", x, lib=lib), torch_e4m3_codes(x).astype(np.uint32))


def pin_f16_vs_library(lib, n_random=200_000):
    allbits = np.arange(65536, dtype=np.uint32)
    ref = allbits.astype(np.uint16).view(np.float16).astype(np.float32)
    got = O.decode_array("f16", allbits, lib=lib)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan].view(np.uint32), got[~nan].view(np.uint32))
    r = rng(5)
    finite = ref[~nan & np.isfinite(ref)].astype(np.float64)
    mags = np.unique(np.abs(finite))
    mids = ((mags[1:] + mags[:-1]) / 2).astype(np.float32)
    rand = (r.uniform(-1, 1, n_random) * 2.0 ** r.integers(-30, 17, n_random)).astype(np.float32)
    x = np.concatenate([mids, -mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9)), rand])
    assert np.array_equal(O.encode_array("f16", x, lib=lib), x.astype(np.float16).view(np.uint16).astype(np.uint32))


def pin_bf16_vs_library(lib, n_random=200_000):
    import torch

    allbits = np.arange(65536, dtype=np.uint32)
    ref = torch.from_numpy(allbits.astype(np.uint16).view(np.int16)).view(torch.bfloat16).float().numpy()
    got = O.decode_array("bf16", allbits, lib=lib)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan].view(np.uint32), got[~nan].view(np.uint32))
    r = rng(6)
    bits = r.integers(0, 1 << 32, n_random, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) < 3.3e38)]
    # exact ties: the low 16 bits equal to 0x8000
    ties = ((bits & 0xFFFF0000) | 0x8000).view(np.float32)
    ties = ties[np.isfinite(ties) & (np.abs(ties) < 3.3e38)]
    x = np.concatenate([x, ties])
    assert np.array_equal(O.encode_array("bf16", x, lib=lib), torch_bf16_bits(x).astype(np.uint32))


# ---------------------------------------------------------------------------
# quantize: scale, rounding, clamp, packing
# ---------------------------------------------------------------------------

def expected_int_codes(x32: np.ndarray, fmt: int, G: int):
    """Codes and scales of the definition, by an independent route (Figueroa
    quotients, numpy rint, explicit clamp); blocks of G along x32."""
    n = x32.size
    nb = (n + G - 1) // G
    qm = qmax(fmt)
    scales = np.zeros(nb, np.float32)
    q = np.zeros(n, np.int64)
    for k in range(nb):
        blk = x32[k * G:(k + 1) * G]
        m = np.float32(np.max(np.abs(blk))) if blk.size else np.float32(0)
        s = div32(np.array([m]), qm)[0]
        scales[k] = s
        if s == 0:
            continue
        t = div32(blk, s)
        q[k * G:(k + 1) * G] = np.clip(np.rint(t).astype(np.int64), -qm, qm)
    return q, scales


def pin_rounding_exhaustive_16bit(lib, fmt=O.INT4, src="bf16", absmax=1.2265625):
    """Every finite 16-bit value x with |x| <= M placed in blocks led by M:
    codes and scales equal the definition computed by an independent route."""
    G = 32
    allbits = np.arange(65536, dtype=np.uint32)
    M = np.float32(absmax)  # exact in bf16 and fp16
    if src == "bf16":
        vals = bf16_to_f32(allbits)
    else:
        vals = allbits.astype(np.uint16).view(np.float16).astype(np.float32)
    keep = np.isfinite(vals) & (np.abs(vals) <= M)
    test_bits = allbits[keep]
    nblk = (test_bits.size + G - 2) // (G - 1)
    pad = nblk * (G - 1) - test_bits.size
    test_bits = np.concatenate([test_bits, np.zeros(pad, np.uint32)])
    lead_bits = (M.view(np.uint32) >> 16) if src == "bf16" else np.float16(M).view(np.uint16)
    blocks = np.concatenate([np.full((nblk, 1), lead_bits, np.uint32), test_bits.reshape(nblk, G - 1)], axis=1)
    bits16 = blocks.reshape(-1).astype(np.uint16)
    x32 = bf16_to_f32(bits16) if src == "bf16" else bits16.view(np.float16).astype(np.float32)
    dtype = O.BF16 if src == "bf16" else O.F16
    codes, scales = O.quantize(bits16 if src == "bf16" else bits16.view(np.float16), fmt, G, dtype=dtype, lib=lib)
    q_ref, s_ref = expected_int_codes(x32, fmt, G)
    assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32))
    assert np.array_equal(unpack_codes(codes, x32.size, O.BITS[fmt]), q_ref)


def pin_rounding_fractions(lib, n=600):
    """Exact rational check: s = RN32(m/qmax), code = round-half-even(RN32(x/s)), clamped."""
    r = rng(7)
    for fmt in INT_FORMATS:
        x = (r.standard_normal(n) * 0.05).astype(np.float32)
        codes, scales = O.quantize(x, fmt, 32, lib=lib)
        q = unpack_codes(codes, n, O.BITS[fmt])
        qm = qmax(fmt)
        for k in range(n // 32 + (n % 32 > 0)):
            blk = x[k * 32:(k + 1) * 32]
            m = max(Fraction(float(abs(v))) for v in blk)
            s = rn32(m / qm)
            assert Fraction(float(scales[k])) == s
            for i, v in enumerate(blk):
                want = max(-qm, min(qm, round(rn32(Fraction(float(v)) / s))))
                assert q[k * 32 + i] == want, (fmt, k, i, float(v))


def pin_exact_multiples_and_ties(lib):
    """Power-of-two scale: x = k*s gives code k; x = (k+1/2)*s goes to the even neighbour."""
    for fmt in INT_FORMATS:
        qm = qmax(fmt)
        s = 2.0 ** -7
        ks = np.arange(-qm, qm + 1)
        x = np.concatenate([[qm * s], ks * s]).astype(np.float32)
        codes, scales = O.quantize(x, fmt, 32 if x.size <= 32 else 256, lib=lib)
        assert scales[0] == np.float32(s)
        assert np.array_equal(unpack_codes(codes, x.size, O.BITS[fmt])[1:], ks)
        if qm >= 3:
            halves = np.arange(-qm + 1, qm - 1) + 0.5  # k + 1/2 strictly inside the range
            x = np.concatenate([[qm * s], halves * s]).astype(np.float32)
            codes, _ = O.quantize(x, fmt, 256, lib=lib)
            want = np.round(halves).astype(np.int64)  # numpy rounds halves to even
            assert np.array_equal(unpack_codes(codes, x.size, O.BITS[fmt])[1:], want), fmt


def pin_zero_and_tiny_blocks(lib):
    """All-zero block -> scale 0 and zero codes; subnormal scales still give codes in range."""
    for fmt in ALL_FORMATS:
        x = np.zeros(64, np.float32)
        x[32:] = np.float32(1.0)
        codes, scales = O.quantize(x, fmt, 32, lib=lib)
        assert scales[0] == 0.0 and not np.any(codes[: O.BITS[fmt] * 32 // 8])
    # bf16 subnormal inputs: the scale is subnormal, the code must still be the definition's
    tiny_bits = np.array([0x0001, 0x0003, 0x8002, 0x0000, 0x0005] * 7, np.uint16)[:32]
    x32 = bf16_to_f32(tiny_bits)
    for fmt in INT_FORMATS:
        codes, scales = O.quantize(tiny_bits, fmt, 32, dtype=O.BF16, lib=lib)
        q_ref, s_ref = expected_int_codes(x32, fmt, 32)
        assert np.array_equal(scales.view(np.uint32), s_ref.view(np.uint32))
        assert np.array_equal(unpack_codes(codes, 32, O.BITS[fmt]), q_ref), fmt
        assert np.all(np.abs(q_ref) <= qmax(fmt))
    # fp32 subnormals: m = 300 * 2^-149 and qmax = 127 give s = 2 * 2^-149, so
    # m / s = 150 and the clamp to 127 decides the code
    ulp0 = np.float32(2.0 ** -149)
    x = (np.array([300, -300, 299, 255, 254, -256, 3, 0] * 4, np.float64) * 2.0 ** -149).astype(np.float32)
    q_ref, s_ref = expected_int_codes(x, O.INT8, 32)
    assert s_ref[0] == 2 * ulp0 and np.rint(div32(x, s_ref[0])).max() > 127
    codes, scales = O.quantize(x, O.INT8, 32, lib=lib)
    assert scales[0] == s_ref[0]
    assert np.array_equal(unpack_codes(codes, x.size, 8), q_ref)


def pin_e4m3_quantize(lib, n=4096):
    """E4M3 codes: s = RN32(m/448), code = E4M3_RNE_satfinite(RN32(x/s)) via the library encoder."""
    r = rng(8)
    x = (r.standard_normal(n) * 1e-3).astype(np.float32)
    x[::97] *= 40
    for G in (32, 128, 1024):
        codes, scales = O.quantize(x, O.E4M3, G, lib=lib)
        for k in range(n // G):
            blk = x[k * G:(k + 1) * G]
            s = div32(np.array([np.max(np.abs(blk))]), 448)[0]
            assert scales[k] == s
            want = torch_e4m3_codes(div32(blk, s))
            assert np.array_equal(codes[k * G:(k + 1) * G], want), (G, k)


def pin_block_independence(lib):
    """Quantizing a concatenation of whole blocks equals concatenating the pieces;
    a partial last block uses only its own elements."""
    r = rng(9)
    for fmt in ALL_FORMATS:
        for G in (32, 256):
            a = (r.standard_normal(3 * G) * 0.02).astype(np.float32)
            b = (r.standard_normal(G // 2 + 3) * 0.5).astype(np.float32)
            ca, sa = O.quantize(a, fmt, G, lib=lib)
            cb, sb = O.quantize(b, fmt, G, lib=lib)
            cab, sab = O.quantize(np.concatenate([a, b]), fmt, G, lib=lib)
            assert np.array_equal(sab, np.concatenate([sa, sb]))
            bits = O.BITS[fmt]
            na = a.size * bits // 8
            assert np.array_equal(cab[:na], ca[:na])
            nb = (b.size * bits + 7) // 8
            assert np.array_equal(cab[na:na + nb], cb[:nb])
            assert not np.any(cab[na + nb:])  # zero padding


def pin_odd_symmetry(lib):
    """Q(-x) = -Q(x): the scale depends on |x| only and rounding to nearest
    with ties to even is symmetric about zero, so negating a block negates
    every integer code (E4M3: flips every sign bit except of +0 codes) and
    keeps the scale. Half-up rounding or a biased magic constant breaks it
    on the exact half-steps included here."""
    r = rng(51)
    for fmt in ALL_FORMATS:
        for G in (32, 128):
            q = qmax(fmt) if fmt != O.E4M3 else 7
            x = (r.standard_normal(4 * G) * 0.02).astype(np.float32)
            x[:G] = ((np.arange(G) % (2 * q + 1)) - q + 0.5).astype(np.float32)  # half-steps
            x[0] = np.float32(q)  # absmax q: scale 1, so the half-steps are exact ties
            cp, sp = O.quantize(x, fmt, G, lib=lib)
            cn, sn = O.quantize(-x, fmt, G, lib=lib)
            assert np.array_equal(sp.view(np.uint32), sn.view(np.uint32)), (fmt, G)
            if fmt == O.E4M3:
                flip = np.where((cp & 0x7F) != 0, cp ^ 0x80, cp)
                assert np.array_equal(cn, flip), (fmt, G)
            else:
                b = O.BITS[fmt]
                assert np.array_equal(unpack_codes(cn, x.size, b), -unpack_codes(cp, x.size, b)), (fmt, G)


def pin_power_of_two_scaling(lib):
    """Q(2^k x): the block absmax, the scale and every quotient x/s scale by
    2^k exactly (no rounding changes while nothing underflows or overflows),
    so the codes are identical and the scales are 2^k times the originals."""
    r = rng(52)
    for fmt in ALL_FORMATS:
        for G in (64, 1024):
            x = (r.standard_normal(3 * G + 17) * 0.02).astype(np.float32)
            c0, s0 = O.quantize(x, fmt, G, lib=lib)
            for k in (-20, -3, 5, 40):
                ck, sk = O.quantize((x * np.float32(2.0 ** k)).astype(np.float32), fmt, G, lib=lib)
                assert np.array_equal(ck, c0), (fmt, G, k)
                assert np.array_equal(sk, (s0 * np.float32(2.0 ** k)).astype(np.float32)), (fmt, G, k)


def pin_roundtrip_bound(lib):
    """|x - D(Q(x))| <= s * (1/2 + 2^-22 * qmax) for integer codes with fp32 output;
    E4M3: |x - D| <= 2^-4 |x| + 2^-10 s + 2^-23 |x| (half an E4M3 ulp, plus rounding)."""
    r = rng(10)
    n = 8192
    x = np.concatenate([(r.standard_normal(n // 2) * 0.02), r.laplace(0, 1e-4, n // 2)]).astype(np.float32)
    x[::331] *= 50
    for fmt in ALL_FORMATS:
        for G in (32, 1024):
            codes, scales = O.quantize(x, fmt, G, lib=lib)
            y = O.dequantize(codes, scales, n, fmt, G, O.F32, lib=lib)
            s = np.repeat(scales, G)[:n].astype(np.float64)
            err = np.abs(x.astype(np.float64) - y)
            if fmt == O.E4M3:
                bound = 2.0 ** -4 * np.abs(x) + 2.0 ** -10 * s + 2.0 ** -22 * np.abs(x)
            else:
                bound = s * (0.5 + 2.0 ** -22 * qmax(fmt))
            assert np.all(err <= bound), (fmt, G, float(np.max(err / np.maximum(bound, 1e-30))))


def pin_idempotence(lib):
    """Q(D(Q(x))) reproduces the codes; scales move by at most one binary32 ulp."""
    r = rng(11)
    n = 4096
    x = (r.standard_normal(n) * 0.02).astype(np.float32)
    for fmt in ALL_FORMATS:
        for G in (32, 128):
            c1, s1 = O.quantize(x, fmt, G, lib=lib)
            y = O.dequantize(c1, s1, n, fmt, G, O.F32, lib=lib)
            c2, s2 = O.quantize(y, fmt, G, lib=lib)
            assert np.array_equal(c1, c2), (fmt, G)
            ulps = np.abs(s1.view(np.int32).astype(np.int64) - s2.view(np.int32).astype(np.int64))
            assert np.all(ulps <= 1), (fmt, G)


def pin_dequant_values(lib):
    """Dequantized fp32 = code value * scale as a single binary32 product, checked
    with exact rationals; bf16/f16 outputs are one nearest-even rounding of it
    (torch and numpy conversions)."""
    r = rng(12)
    n = 2048
    x = (r.standard_normal(n) * 0.03).astype(np.float32)
    for fmt in ALL_FORMATS:
        G = 64
        codes, scales = O.quantize(x, fmt, G, lib=lib)
        y32 = O.dequantize(codes, scales, n, fmt, G, O.F32, lib=lib)
        if fmt == O.E4M3:
            vals = O.decode_array("e4m3", codes[:n].astype(np.uint32), lib=lib)
            import torch
            vals_lib = torch.from_numpy(codes[:n].copy()).view(torch.float8_e4m3fn).float().numpy()
            assert np.array_equal(vals, vals_lib)
        else:
            vals = unpack_codes(codes, n, O.BITS[fmt]).astype(np.float32)
        for i in range(0, n, 7):
            want = rn32(Fraction(float(vals[i])) * Fraction(float(scales[i // G])))
            assert Fraction(float(y32[i])) == want, (fmt, i)
        ybf = O.dequantize(codes, scales, n, fmt, G, O.BF16, lib=lib)
        assert np.array_equal(ybf, torch_bf16_bits(y32))
        yh = O.dequantize(codes, scales, n, fmt, G, O.F16, lib=lib)
        assert np.array_equal(yh, y32.astype(np.float16).view(np.uint16))


# ---------------------------------------------------------------------------
# reduce
# ---------------------------------------------------------------------------

def _shards(r, N, n, fmt, G, scale=1e-4):
    out = []
    for _ in range(N):
        x = r.laplace(0, scale, n).astype(np.float32)
        out.append(O.quantize(x, fmt, G))
    return out


def pin_reduce_zero_shard_neutral(lib):
    """An all-zero shard (zero codes, zero scales) inserted at any position
    changes nothing: every term it adds is +0, and a binary32 sum that
    starts from +0 is unchanged by adding +0. A mean instead of a sum, or a
    shard read at the wrong index, breaks this."""
    r = rng(53)
    n, G = 2 * 1024 + 77, 128
    shards = _shards(r, 3, n, O.INT4, G)
    zc = np.zeros_like(shards[0][0])
    zs = np.zeros_like(shards[0][1])
    base = O.reduce([c for c, _ in shards], [sc for _, sc in shards], n, O.INT4, G, O.INT8, 64,
                    want_sum=True, lib=lib)
    for pos in range(4):
        cs = [c for c, _ in shards]
        ss = [sc for _, sc in shards]
        cs.insert(pos, zc)
        ss.insert(pos, zs)
        got = O.reduce(cs, ss, n, O.INT4, G, O.INT8, 64, want_sum=True, lib=lib)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1]), pos
        assert np.array_equal(got[2].view(np.uint32), base[2].view(np.uint32)), pos


def pin_reduce_single_shard(lib):
    """N = 1: the reduce is dequantize (fp32) followed by quantize."""
    r = rng(13)
    for fin, Gin, fout, Gout in ((O.INT4, 128, O.INT4, 128), (O.INT4, 128, O.INT8, 256),
                                 (O.E4M3, 128, O.E4M3, 128), (O.INT8, 64, O.INT2, 32)):
        n = 2048 + 64
        (c, s), = _shards(r, 1, n, fin, Gin)
        oc, os_, sm = O.reduce([c], [s], n, fin, Gin, fout, Gout, want_sum=True, lib=lib)
        y = O.dequantize(c, s, n, fin, Gin, O.F32, lib=lib)
        assert np.array_equal(sm.view(np.uint32), y.view(np.uint32))
        c2, s2 = O.quantize(y, fout, Gout, lib=lib)
        assert np.array_equal(oc, c2) and np.array_equal(os_, s2)


def pin_reduce_pow2_exact(lib):
    """Power-of-two scales make every term and partial sum exact: the fp32 sum
    equals the integer sum of codes times the scale."""
    r = rng(14)
    N, n, G = 8, 1024, 128
    fmt = O.INT4
    k = 12
    codes, scales, qs = [], [], []
    for _ in range(N):
        q = r.integers(-7, 8, n)
        q[::G] = 7  # absmax = 7 * 2^-k in every block, so s = 2^-k exactly
        x = (q * 2.0 ** -k).astype(np.float32)
        c, s = O.quantize(x, fmt, G, lib=lib)
        assert np.all(s == np.float32(2.0 ** -k))
        codes.append(c)
        scales.append(s)
        qs.append(q)
    _, _, sm = O.reduce(codes, scales, n, fmt, G, O.INT8, 256, want_sum=True, lib=lib)
    want = np.sum(qs, axis=0) * 2.0 ** -k
    assert np.array_equal(sm.astype(np.float64), want)


def pin_reduce_order(lib):
    """Shard order is the summation order: 1 + 2^-24 + 2^-24 is 1 in fp32 when
    summed left to right, but 1 + 2^-23 when summed right to left."""
    n, G = 32, 32
    vals = [1.0, 2.0 ** -24, 2.0 ** -24]
    codes, scales = [], []
    for v in vals:
        x = np.full(n, np.float32(v))
        c, s = O.quantize(x, O.INT2, G, lib=lib)  # qmax = 1, so s = v and codes = 1
        codes.append(c)
        scales.append(s)
    _, _, sm = O.reduce(codes, scales, n, O.INT2, G, O.INT8, G, want_sum=True, lib=lib)
    assert np.all(sm == np.float32(1.0))
    _, _, sm_rev = O.reduce(codes[::-1], scales[::-1], n, O.INT2, G, O.INT8, G, want_sum=True, lib=lib)
    assert np.all(sm_rev == np.float32(1.0 + 2.0 ** -23))


def pin_reduce_plain_sum_and_bound(lib):
    """The reduce is a sum, not a mean, and stays within the recursive-summation
    bound (N-1) u sum|d_r| of the exact sum (Higham, Accuracy and Stability of
    Numerical Algorithms, 2nd ed., section 4.2)."""
    r = rng(15)
    N, n = 8, 4096
    sh = _shards(r, N, n, O.INT4, 128)
    _, _, sm = O.reduce([c for c, _ in sh], [s for _, s in sh], n, O.INT4, 128, O.INT4, 128,
                        want_sum=True, lib=lib)
    terms = np.array([O.dequantize(c, s, n, O.INT4, 128, O.F32, lib=lib) for c, s in sh], np.float64)
    exact = terms.sum(axis=0)
    bound = (N - 1) * 2.0 ** -24 * np.abs(terms).sum(axis=0) * (1 + 1e-6)
    assert np.all(np.abs(sm - exact) <= bound)
    # two identical shards sum to exactly twice the value
    c, s = sh[0]
    _, _, two = O.reduce([c, c], [s, s], n, O.INT4, 128, O.INT4, 128, want_sum=True, lib=lib)
    assert np.array_equal(two, 2 * terms[0].astype(np.float32))


def pin_reduce_two_roundings(lib):
    """Each term is rounded before it is added: with codes (-3, 3) and scales
    (1, 1 + 2^-23) the definition gives fl(-3 + fl(3 (1 + 2^-23))) = 2^-21,
    while a fused multiply-add would give 3 * 2^-23."""
    n, G = 32, 32
    c0 = np.zeros(n * 8 // 8, np.uint8)
    c0[:] = np.uint8(0xFD)  # int8 code -3
    c1 = np.full(n, 3, np.uint8)
    s0 = np.array([1.0], np.float32)
    s1 = np.array([1.0 + 2.0 ** -23], np.float32)
    _, _, sm = O.reduce([c0, c1], [s0, s1], n, O.INT8, G, O.INT8, G, want_sum=True, lib=lib)
    want = rn32(rn32(Fraction(-3)) + rn32(3 * Fraction(float(s1[0]))))
    assert want == Fraction(2) ** -21
    assert all(Fraction(float(v)) == want for v in sm)


def pin_fp8_reduce_no_overflow(lib):
    """AGoQ's precision-preserved reduce: eight FP8 shards at the E4M3 maximum sum
    to 8 * 448 = 3584 with no saturation, because the result gets its own scale."""
    n, G = 128, 128
    x = np.full(n, np.float32(448.0))
    c, s = O.quantize(x, O.E4M3, G, lib=lib)
    assert s[0] == 1.0 and np.all(c == 0x7E)
    oc, os_, sm = O.reduce([c] * 8, [s] * 8, n, O.E4M3, G, O.E4M3, G, want_sum=True, lib=lib)
    assert np.all(sm == 3584.0) and os_[0] == 8.0 and np.all(oc == 0x7E)
    y = O.dequantize(oc, os_, n, O.E4M3, G, O.F32, lib=lib)
    assert np.all(y == 3584.0)


# ---------------------------------------------------------------------------
# FP8 accumulate
# ---------------------------------------------------------------------------

def pin_fp8_accumulate(lib):
    """Zero main gradient: accumulate(g) == Q8(g). Zero gradient: codes unchanged.
    Four steps stay within the per-step E4M3 rounding of the exact running sum."""
    r = rng(16)
    n, G = 4096, 128
    main_c = np.zeros(n, np.uint8)
    main_s = np.zeros(n // G, np.float32)
    g = torch_bf16_bits((r.standard_normal(n) * 1e-3).astype(np.float32))
    c1, s1 = O.fp8_accumulate(main_c, main_s, g, G, grad_dtype=O.BF16, lib=lib)
    cq, sq = O.quantize(g, O.E4M3, G, dtype=O.BF16, lib=lib)
    assert np.array_equal(c1, cq[:n]) and np.array_equal(s1, sq)
    zero = np.zeros(n, np.uint16)
    c2, s2 = O.fp8_accumulate(c1, s1, zero, G, grad_dtype=O.BF16, lib=lib)
    assert np.array_equal(c2, c1)
    assert np.all(np.abs(s2.view(np.int32).astype(np.int64) - s1.view(np.int32)) <= 1)
    # each step stores D8(c)*s + g rounded once to E4M3 (up to the fp32 roundings)
    c, s = main_c, main_s
    for _ in range(4):
        gi = torch_bf16_bits((r.standard_normal(n) * 1e-3).astype(np.float32))
        prev = O.dequantize(c, s, n, O.E4M3, G, O.F32, lib=lib)
        c, s = O.fp8_accumulate(c, s, gi, G, grad_dtype=O.BF16, lib=lib)
        v = prev.astype(np.float64) + bf16_to_f32(gi)
        now = O.dequantize(c, s, n, O.E4M3, G, O.F32, lib=lib)
        ss = np.repeat(s, G).astype(np.float64)
        assert np.all(np.abs(now - v) <= 2.0 ** -4 * np.abs(v) + 2.0 ** -10 * ss + 2.0 ** -20 * np.abs(v))


def pin_fp8_accumulate_cancellation(lib):
    """Adding the exact negation of the dequantized main gradient (an fp32
    gradient) cancels every element: fl(d + (-d)) = +0, the block absmax is
    0, so every scale is 0 and every code 0x00. The dequantized values d are
    recomputed here from torch's E4M3 decoding and one binary32 product."""
    import torch

    r = rng(54)
    n, G = 4096, 128
    g0 = torch_bf16_bits((r.standard_normal(n) * 1e-3).astype(np.float32))
    c, s = O.fp8_accumulate(np.zeros(n, np.uint8), np.zeros(n // G, np.float32), g0, G,
                            grad_dtype=O.BF16, lib=lib)
    e = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).float().numpy()
    d = (e * np.repeat(s, G)).astype(np.float32)  # one binary32 product each
    c2, s2 = O.fp8_accumulate(c, s, -d, G, grad_dtype=O.F32, lib=lib)
    assert not np.any(c2) and not np.any(s2.view(np.uint32))


def pin_fp8_accumulate_two_roundings(lib):
    """v = fl(fl(D8(c) * s) + g): with D8 = 9/8, s = 1 + 2^-22 and g = -9/8 the
    product rounds to 9/8 + 2^-22, so v = 2^-22 (a fused form gives 9 * 2^-25),
    and the new block scale is RN32(v / 448)."""
    n, G = 128, 128
    codes = np.zeros(n, np.uint8)
    codes[0] = 0x39  # E4M3 1.125
    scales = np.array([1.0 + 2.0 ** -22], np.float32)
    g = np.zeros(n, np.uint16)
    g[0] = torch_bf16_bits(np.array([-1.125], np.float32))[0]
    c, s = O.fp8_accumulate(codes, scales, g, G, grad_dtype=O.BF16, lib=lib)
    v = rn32(rn32(Fraction(9, 8) * Fraction(float(scales[0]))) - Fraction(9, 8))
    assert v == Fraction(2) ** -22
    assert Fraction(float(s[0])) == rn32(v / 448)
    assert c[0] == 0x7E and not np.any(c[1:])


# ---------------------------------------------------------------------------
# qgZ hierarchy: tensor-slice reordering and the two-hop reduce ([ZeRO++]
# sections "Two-hop communication prevents QGZ traffic from multiplying across
# GPUs" and "Tensor-slice reordering fixes incorrect gradient placement").
# ---------------------------------------------------------------------------
_M = 1024  # chunk elements


def pin_reordered_quantize_identity(lib):
    """With one node, or one GPU per node, the reordering is the identity, so
    the reordered quantization equals the plain one byte for byte."""
    for A, L in ((1, 4), (4, 1)):
        x = rng(A * 10 + L).standard_normal(A * L * _M).astype(np.float32)
        for fmt, G in ((O.INT4, 128), (O.INT6, 32), (O.E4M3, 256)):
            c, sc = O.quantize_reordered(x, fmt, G, A, L, lib=lib)
            wc, ws = O.quantize(x, fmt, G, lib=lib)
            assert np.array_equal(c, wc) and np.array_equal(sc.view(np.uint32), ws.view(np.uint32))


def pin_two_hop_ownership(lib):
    """A gradient that is zero except for chunk c* on GPU g* reaches, after the
    two hops, GPU c* (the chunk's owner) and no other GPU: the goal the pages
    give for the reordering."""
    for A, L in ((2, 2), (2, 4), (4, 2), (3, 2)):
        P, n = A * L, A * L * _M
        for g_star, c_star in ((0, P - 1), (P - 1, 0), (1, 2 % P), (P // 2, (P // 2 + 1) % P)):
            xs = [np.zeros(n, np.float32) for _ in range(P)]
            xs[g_star][c_star * _M:(c_star + 1) * _M] = rng(g_star).standard_normal(_M)
            q = [O.quantize_reordered(x, O.INT4, 128, A, L, lib=lib) for x in xs]
            _, out, sums = O.reduce_two_hop([c for c, _ in q], [sc for _, sc in q], A, L, n, O.INT4,
                                            128, O.INT8, 64, O.INT4, 128, want_sum=True, lib=lib)
            for g in range(P):
                nonzero = np.any(out[g][0] != 0) or np.any(out[g][1] != 0) or np.any(sums[g] != 0)
                assert nonzero == (g == c_star), (A, L, g_star, c_star, g)


def pin_two_hop_exact_sums(lib):
    """int8 blocks with absmax 127 * 2^k (scale 2^k, exact), one GPU of each
    node nonzero per block (so the hop-1 sum is that block and requantizing it
    is exact): the final fp32 sums equal the integer sum over all P GPUs."""
    k, G = -9, 32
    for A, L in ((2, 2), (2, 4), (4, 2)):
        P, n = A * L, A * L * _M
        nb = n // G
        ints = []
        for g in range(P):
            r = np.random.default_rng([5, g])
            q = r.integers(-127, 128, n)
            q[::G] = 127 * np.where(r.random(nb) < 0.5, 1, -1)
            active = (np.arange(nb) % L) == (g % L)
            ints.append(np.where(np.repeat(active, G), q, 0).astype(np.int64))
        xs = [(q * 2.0 ** k).astype(np.float32) for q in ints]
        qs = [O.quantize_reordered(x, O.INT8, G, A, L, lib=lib) for x in xs]
        _, out, sums = O.reduce_two_hop([c for c, _ in qs], [sc for _, sc in qs], A, L, n, O.INT8, G,
                                        O.INT8, G, O.INT8, G, want_sum=True, lib=lib)
        total = np.sum(ints, axis=0)
        for g in range(P):
            want = (total[g * _M:(g + 1) * _M] * 2.0 ** k).astype(np.float32)
            assert np.array_equal(sums[g], want), (A, L, g)


def pin_two_hop_order(lib):
    """Each hop sums in GPU order: with values 1, 2^-24, 2^-24 (int2 codes, so
    the scale is the value itself), summing left to right gives 1 and right to
    left 1 + 2^-23. Three nodes of one GPU test hop 2; one node of three GPUs
    tests hop 1 (its sum survives the int2 requantization as the scale)."""
    vals = [1.0, 2.0 ** -24, 2.0 ** -24]
    for A, L in ((3, 1), (1, 3)):
        n = 3 * _M
        q = [O.quantize_reordered(np.full(n, np.float32(v)), O.INT2, 32, A, L, lib=lib) for v in vals]
        _, out, sums = O.reduce_two_hop([c for c, _ in q], [sc for _, sc in q], A, L, n, O.INT2, 32,
                                        O.INT2, 32, O.INT8, 32, want_sum=True, lib=lib)
        for g in range(3):
            assert np.all(sums[g] == np.float32(1.0)), (A, L, g)


# ---------------------------------------------------------------------------
# Aquavit: metadata interleaving and the ascending schedule ([Aquavit] summary
# of the implementation, Section 5.1-5.3; Eq. 6; readings R13 and R14).
# ---------------------------------------------------------------------------

def _pack_lsb_first(q, bits):
    """Two's-complement codes packed LSB first into 32-bit little-endian words
    (an integer bit accumulator, independent of the oracle's bit writer)."""
    acc, nbits = 0, 0
    for v in q:
        acc |= (int(v) & ((1 << bits) - 1)) << nbits
        nbits += bits
    nbytes = -(-nbits // 32) * 4
    return acc.to_bytes(nbytes, "little")


def pin_il_size(lib):
    """The interleaved stream is exactly as long as codes plus scales: b + 32/G
    bits per element (Eq. 6) for whole blocks; E4M3 has no interleaved form."""
    fmt_of = {2: O.INT2, 4: O.INT4, 6: O.INT6, 8: O.INT8}
    for b, fmt in fmt_of.items():
        for G in BLOCKS:
            for nblk in (1, 3, 64):
                n = nblk * G
                assert Fraction(O.il_bytes(fmt, n, G, lib) * 8, n) == b + Fraction(32, G), (b, G, n)
    assert O.il_bytes(O.E4M3, 1024, 128, lib) == -1


def pin_il_hand_records(lib):
    """Two hand-built streams: records are [fp32 scale, little endian][codes]
    with no padding; a partial last block's codes fill whole 32-bit words."""
    import struct

    # int4, G = 32, two blocks: block 0 holds k * 0.5 (absmax 3.5 -> scale 0.5,
    # codes k exactly), block 1 is zero (scale 0, codes 0)
    k = np.array([(i % 15) - 7 for i in range(32)])
    x = np.concatenate([k * 0.5, np.zeros(32)]).astype(np.float32)
    want = struct.pack("<f", 0.5) + _pack_lsb_first(k, 4) + struct.pack("<f", 0.0) + bytes(16)
    got = O.quantize_interleaved(x, O.INT4, 32, lib=lib)
    assert got.tobytes() == want, (got.tobytes().hex(), want.hex())
    # 6-bit, G = 32, 40 elements: block 0 = k * 2^-3 (absmax 31/8 -> scale
    # 1/8), block 1 = 8 elements (absmax 31/4 -> scale 1/4) -> 48 bits of codes
    k0 = np.array([((3 * i) % 63) - 31 for i in range(32)])
    k1 = np.array([31, -31, 1, 0, -1, 5, -6, 2])
    x = np.concatenate([k0 / 8.0, k1 / 4.0]).astype(np.float32)
    want = (struct.pack("<f", 0.125) + _pack_lsb_first(k0, 6) + struct.pack("<f", 0.25)
            + _pack_lsb_first(k1, 6))
    assert len(want) == 4 + 24 + 4 + 8
    got = O.quantize_interleaved(x, O.INT6, 32, lib=lib)
    assert got.tobytes() == want, (got.tobytes().hex(), want.hex())
    y = O.dequantize_interleaved(got, x.size, O.INT6, 32, O.F32, lib=lib)
    assert np.array_equal(y, x)


def pin_il_is_a_regrouping(lib):
    """Record k holds block k's planar scale and codes (the planar codec is
    pinned above); dequantizing the stream gives the planar result."""
    r = rng(31)
    for fmt, G, n in ((O.INT2, 1024, 3 * 1024 + 200), (O.INT4, 128, 1000), (O.INT8, 32, 32 * 7 + 9)):
        x = (r.standard_normal(n) * 0.02).astype(np.float32)
        rec = O.quantize_interleaved(x, fmt, G, lib=lib).tobytes()
        codes, scales = O.quantize(x, fmt, G, lib=lib)
        pos = 0
        for kb in range(-(-n // G)):
            lo, hi = kb * G, min(n, kb * G + G)
            cb = -(-(hi - lo) * O.BITS[fmt] // 32) * 4
            assert rec[pos:pos + 4] == scales[kb:kb + 1].tobytes(), (fmt, G, kb)
            start = lo * O.BITS[fmt] // 8
            assert rec[pos + 4:pos + 4 + cb] == codes.tobytes()[start:start + cb], (fmt, G, kb)
            pos += 4 + cb
        assert pos == len(rec)
        for dt in (O.F32, O.BF16):
            y = O.dequantize_interleaved(np.frombuffer(rec, np.uint8), n, fmt, G, dt, lib=lib)
            assert np.array_equal(y, O.dequantize(codes, scales, n, fmt, G, dt, lib=lib))


def pin_schedule_closed_forms(lib):
    """bpw(0) = 8 - 6/a and bpw(T) = 8 - 6/(a + c); the mean over t = 0..T-1
    of an increasing function lies below its integral mean by at most
    (f(T) - f(0))/T, and that integral mean is 8 - (6/c) ln((a + c)/a)."""
    g = golden("aquavit_schedule.json")
    for a, c, T in ((g["a"], g["c"], g["steps"]), (0.5, 2.0, 300), (1.5, 8.0, 64)):
        f0, fT = O.aquavit_bpw(0, T, a, c, lib=lib), O.aquavit_bpw(T, T, a, c, lib=lib)
        assert abs(f0 - (8 - 6 / a)) < 1e-12 and abs(fT - (8 - 6 / (a + c))) < 1e-12, (a, c)
        mean = math.fsum(O.aquavit_bpw(t, T, a, c, lib=lib) for t in range(T)) / T
        integral = 8 - (6 / c) * math.log((a + c) / a)
        assert 0 <= integral - mean <= (fT - f0) / T + 1e-12, (a, c, T, mean, integral)
        assert all(O.aquavit_bpw(t + 1, T, a, c, lib=lib) > O.aquavit_bpw(t, T, a, c, lib=lib)
                   for t in range(T))


def pin_schedule_pick(lib):
    """The pairs: every available width maps to its own (b, G); the default
    schedule starts at 2-bit/G=1024 and ends at 6-bit/G=32 as printed; no
    pair wider than 7.00 is used; the pick is the nearest width (brute force
    over the 18 pairs) and never decreases along the schedule."""
    g = golden("aquavit_schedule.json")
    pairs = [(b, G, b + Fraction(32, G)) for b in (2, 4, 6) for G in BLOCKS]
    for b, G, w in pairs:
        assert O.aquavit_pick(float(w), lib=lib)[:2] == (b, G), (b, G)
    T, a, c = g["steps"], g["a"], g["c"]
    first = O.aquavit_pick(O.aquavit_bpw(0, T, a, c, lib=lib), lib=lib)
    last = O.aquavit_pick(O.aquavit_bpw(T, T, a, c, lib=lib), lib=lib)
    assert (first[0], first[1], f"{first[2]:.2f}") == (g["first_pair"]["bits"], g["first_pair"]["G"],
                                                       g["first_pair"]["bpw_printed"])
    assert (last[0], last[1], f"{last[2]:.2f}") == (g["last_pair"]["bits"], g["last_pair"]["G"],
                                                    g["last_pair"]["bpw_printed"])
    assert O.aquavit_pick(8.5, lib=lib)[:2] == (6, 32) and O.aquavit_pick(0.0, lib=lib)[:2] == (2, 1024)
    for target in np.linspace(1.0, 8.0, 701):
        b, G, w = O.aquavit_pick(float(target), lib=lib)
        best = min(abs(float(p[2]) - target) for p in pairs)
        assert abs(w - target) == best and w == float(b + Fraction(32, G)), target
    prev = 0.0
    for t in range(T + 1):
        w = O.aquavit_pick(O.aquavit_bpw(t, T, a, c, lib=lib), lib=lib)[2]
        assert w >= prev
        prev = w


# ---------------------------------------------------------------------------
# The ring reduce-scatter that qgZ replaces ([ZeRO++] "QGZ keeps reductions in
# full precision while sending quantized gradients"; reading R15).
# ---------------------------------------------------------------------------

def pin_ring_small_n(lib):
    """One or two shards: the ring has no intermediate requantization, so it is
    the one-hop reduce exactly."""
    r = rng(41)
    n = 3000
    for N in (1, 2):
        xs = [(r.laplace(0, 1e-3, n)).astype(np.float32) for _ in range(N)]
        q = [O.quantize(x, O.INT4, 128, lib=lib) for x in xs]
        a = O.reduce_ring([c for c, _ in q], [sc for _, sc in q], n, O.INT4, 128, O.INT8, 64,
                          want_sum=True, lib=lib)
        b = O.reduce([c for c, _ in q], [sc for _, sc in q], n, O.INT4, 128, O.INT8, 64,
                     want_sum=True, lib=lib)
        assert np.array_equal(a[0], b[0]) and np.array_equal(as_u32(a[1]), as_u32(b[1]))
        assert np.array_equal(as_u32(a[2]), as_u32(b[2])), N


def as_u32(a):
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def pin_ring_exact_sums(lib):
    """int8, G = 32, values q * 2^-9: in every block shard s holds +-127 at
    element s, where the other shards hold 0, and small integers elsewhere,
    so that no prefix sum leaves [-127, 127]. Every shard and every partial
    sum then has block absmax 127 * 2^-9, i.e. scale exactly 2^-9, every
    (re)quantization is exact, and the ring's fp32 result equals the integer
    sum."""
    k, N, nb = -9, 6, 64
    for G in (32, 128):
        r = np.random.default_rng([9, G])
        ints = []
        for s in range(N):
            q = r.integers(-127 // N, 127 // N + 1, nb * G)
            for s2 in range(N):
                q[s2::G] = 0
            q[s::G] = 127 * np.where(r.random(nb) < 0.5, 1, -1)
            ints.append(q.astype(np.int64))
        xs = [(q * 2.0 ** k).astype(np.float32) for q in ints]
        qs = [O.quantize(x, O.INT8, G, lib=lib) for x in xs]
        _, _, sm = O.reduce_ring([c for c, _ in qs], [sc for _, sc in qs], nb * G, O.INT8, G, O.INT8,
                                 G, want_sum=True, lib=lib)
        assert np.array_equal(sm, (np.sum(ints, axis=0) * 2.0 ** k).astype(np.float32)), G


def pin_ring_requantizes_partials(lib):
    """Three int8 shards of one block: 127 at element 0 of shard 0, 2^-7 at
    element 1 of shard 1, zeros in shard 2. The ring requantizes 127 + 2^-7
    with scale 1, which rounds the small term away (result 127 and 0); the
    one-hop reduce keeps it; a ring run in the reverse order keeps it too."""
    G, n = 32, 32
    x0 = np.zeros(n, np.float32); x0[0] = 127.0
    x1 = np.zeros(n, np.float32); x1[1] = 2.0 ** -7
    x2 = np.zeros(n, np.float32)
    q = [O.quantize(x, O.INT8, G, lib=lib) for x in (x0, x1, x2)]
    _, _, ring = O.reduce_ring([c for c, _ in q], [sc for _, sc in q], n, O.INT8, G, O.INT8, G,
                               want_sum=True, lib=lib)
    _, _, one = O.reduce([c for c, _ in q], [sc for _, sc in q], n, O.INT8, G, O.INT8, G,
                         want_sum=True, lib=lib)
    assert ring[0] == 127.0 and ring[1] == 0.0 and np.all(ring[2:] == 0.0)
    assert one[0] == 127.0 and abs(float(one[1]) - 2.0 ** -7) < 2.0 ** -20
    q.reverse()
    _, _, rev = O.reduce_ring([c for c, _ in q], [sc for _, sc in q], n, O.INT8, G, O.INT8, G,
                              want_sum=True, lib=lib)
    assert rev[1] != 0.0


# ---------------------------------------------------------------------------
# The dequantization fused into the consumer GEMM (the oracle's reading R16)
# ---------------------------------------------------------------------------

def _int_weights(r, N, K, G, qmax_):
    """An N x K integer matrix whose every G-block holds +-qmax: its block
    scales are exactly 1, so the dequantized (and bf16) weights are the
    integers themselves."""
    W = r.integers(-qmax_, qmax_ + 1, size=(N, K)).astype(np.int64)
    W[:, ::G] = qmax_ * np.where(r.random((N, K // G)) < 0.5, -1, 1)
    return W


def pin_gemm_small_integers(lib):
    """Small-integer operands: every product and partial sum is an integer, so
    y and the sums of magnitudes equal int64 matrix products of the integer
    matrices built here (non-square, so a transposed operand fails)."""
    r = rng(301)
    for fmt, G in ((O.INT8, 32), (O.INT4, 64), (O.INT2, 128)):
        M, N, K = 3, 5, 256
        W = _int_weights(r, N, K, G, qmax(fmt))
        X = r.integers(-16, 17, size=(M, K)).astype(np.int64)
        codes, scales = O.quantize(W.astype(np.float32).ravel(), fmt, G, lib=lib)
        assert np.all(scales == 1.0)
        xb = torch_bf16_bits(X.astype(np.float32).ravel())
        y, absy = O.gemm_dequant(xb, M, K, codes, scales, fmt, G, N, lib=lib)
        assert np.array_equal(y.reshape(M, N), (X @ W.T).astype(np.float64))
        assert np.array_equal(absy.reshape(M, N), (np.abs(X) @ np.abs(W).T).astype(np.float64))


def pin_gemm_bf16_weights_exact_sum(lib):
    """Random weights and activations: the weight operand is the bf16 rounding
    (torch) of the fp32 product code * scale (numpy float32), the codes read
    back from the bit stream by the pinned unpacking helper, and y is the
    exact rational sum of the products."""
    r = rng(302)
    for fmt, G in ((O.INT4, 32), (O.INT8, 64), (O.E4M3, 32), (O.INT6, 64)):
        M, N, K = 2, 3, 128
        w32 = (r.standard_normal(N * K) * 0.02).astype(np.float32)
        codes, scales = O.quantize(w32, fmt, G, lib=lib)
        if fmt == O.E4M3:
            import torch

            q = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).float().numpy()
        else:
            q = unpack_codes(codes, N * K, O.BITS[fmt]).astype(np.float32)
        wq = (q * np.repeat(scales, G)).astype(np.float32)
        wb = bf16_to_f32(torch_bf16_bits(wq)).reshape(N, K)
        xb = torch_bf16_bits(r.standard_normal(M * K).astype(np.float32))
        X = bf16_to_f32(xb).reshape(M, K)
        y, absy = O.gemm_dequant(xb, M, K, codes, scales, fmt, G, N, lib=lib)
        for m in range(M):
            for n in range(N):
                exact = sum(Fraction(float(X[m, k])) * Fraction(float(wb[n, k])) for k in range(K))
                assert abs(Fraction(float(y[m * N + n])) - exact) <= Fraction(2) ** -50 * abs(exact) + Fraction(2) ** -1000
                mag = sum(abs(Fraction(float(X[m, k])) * Fraction(float(wb[n, k]))) for k in range(K))
                assert abs(Fraction(float(absy[m * N + n])) - mag) <= Fraction(2) ** -50 * mag


def pin_gemm_identity_gives_dequantized_weights(lib):
    """x = I (M = K): y[m][n] is the bf16-dequantized weight element (n, m),
    the pinned dequantize's output transposed; sampled positions only."""
    r = rng(303)
    K = N = 64
    w32 = (r.standard_normal(N * K) * 0.02).astype(np.float32)
    codes, scales = O.quantize(w32, O.INT4, 32, lib=lib)
    wd = bf16_to_f32(O.dequantize(codes, scales, N * K, O.INT4, 32, O.BF16, lib=lib)).reshape(N, K)
    xb = torch_bf16_bits(np.eye(K, dtype=np.float32).ravel())
    rows, cols = r.integers(0, K, 200), r.integers(0, N, 200)
    y, _ = O.gemm_dequant(xb, K, K, codes, scales, O.INT4, 32, N, rows=rows, cols=cols, lib=lib)
    assert np.array_equal(y, wd[cols, rows].astype(np.float64))


FAST_PINS = [
    pin_bpw_endpoints, pin_bpw_formula, pin_zeropp_payload, pin_bit_layout,
    pin_e4m3_points, pin_e4m3_vs_library, pin_f16_vs_library, pin_bf16_vs_library,
    pin_rounding_exhaustive_16bit, pin_rounding_fractions, pin_exact_multiples_and_ties,
    pin_zero_and_tiny_blocks, pin_e4m3_quantize, pin_block_independence, pin_odd_symmetry,
    pin_power_of_two_scaling, pin_roundtrip_bound,
    pin_idempotence, pin_dequant_values, pin_reduce_zero_shard_neutral, pin_reduce_single_shard, pin_reduce_pow2_exact,
    pin_reduce_order, pin_reduce_plain_sum_and_bound, pin_reduce_two_roundings,
    pin_fp8_reduce_no_overflow, pin_fp8_accumulate, pin_fp8_accumulate_cancellation, pin_fp8_accumulate_two_roundings,
    pin_reordered_quantize_identity, pin_two_hop_ownership, pin_two_hop_exact_sums,
    pin_two_hop_order, pin_il_size, pin_il_hand_records, pin_il_is_a_regrouping,
    pin_schedule_closed_forms, pin_schedule_pick, pin_ring_small_n, pin_ring_exact_sums,
    pin_ring_requantizes_partials, pin_gemm_small_integers, pin_gemm_bf16_weights_exact_sum,
    pin_gemm_identity_gives_dequantized_weights,
]
