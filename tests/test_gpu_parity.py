"""GPU kernels against the oracle, element by element, through the C ABI.

Sizes span several 1024-element tiles plus a ragged tail with a partial last
block; every code format, block size and element type is covered. Codes,
scales, dequantized values and sums must match bit for bit: the kernels keep
the definition's order of operations (shard order included), so no tolerance
applies.
"""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, bytes_dev, mixed_input, oracle_quantize, to_dev, to_host

pytestmark = pytest.mark.gpu

FORMATS = (O.INT2, O.INT4, O.INT6, O.INT8, O.E4M3)
BLOCKS = (32, 64, 128, 256, 512, 1024)
DTYPES = (O.BF16, O.F16, O.F32)
N_MAIN = 5 * 1024 + 333  # five full tiles and a ragged tail (partial block for every G)


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    return zq


def fid(v):
    return {O.INT2: "int2", O.INT4: "int4", O.INT6: "int6", O.INT8: "int8", O.E4M3: "e4m3",
            }.get(v, str(v))


def dname(v):
    return {O.F32: "f32", O.F16: "f16", O.BF16: "bf16"}[v]


def gpu_quantize(zq, x, dtype, fmt, G):
    codes, scales = zq.quantize(to_dev(x, dtype), fmt, G)
    return to_host(codes), to_host(scales)


def assert_same_codes(got, want, label=""):
    if not np.array_equal(got, want):
        bad = np.flatnonzero(got != want)
        raise AssertionError(f"{label}: {bad.size} code bytes differ, first at {bad[:8]}: "
                             f"got {got[bad[:8]]} want {want[bad[:8]]}")


def assert_same_bits(got, want, label=""):
    g, w = as_bits(got), as_bits(want)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{label}: {bad.size} values differ, first at {bad[:8]}: "
                             f"got {got[bad[:8]]} want {want[bad[:8]]}")


# ---------------------------------------------------------------------------
# quantize
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
@pytest.mark.parametrize("fmt", FORMATS, ids=fid)
@pytest.mark.parametrize("G", BLOCKS)
def test_quantize_matches_oracle(zq, dtype, fmt, G):
    x = mixed_input(N_MAIN, dtype, seed=1000 + G, G=G)
    codes, scales = gpu_quantize(zq, x, dtype, fmt, G)
    want_c, want_s = oracle_quantize(x, dtype, fmt, G)
    assert_same_bits(scales, want_s, "scales")
    assert_same_codes(codes, want_c, "codes")


@pytest.mark.parametrize("n", [1, 2, 31, 32, 33, 511, 512, 1023, 1024, 1025, 2048, 3 * 1024 + 1])
@pytest.mark.parametrize("fmt", FORMATS, ids=fid)
def test_quantize_edge_sizes(zq, n, fmt):
    for G in (32, 1024):
        x = mixed_input(n, O.BF16, seed=n, G=G)
        codes, scales = gpu_quantize(zq, x, O.BF16, fmt, G)
        want_c, want_s = oracle_quantize(x, O.BF16, fmt, G)
        assert_same_bits(scales, want_s, f"scales n={n} G={G}")
        assert_same_codes(codes, want_c, f"codes n={n} G={G}")


@pytest.mark.parametrize("fmt", FORMATS, ids=fid)
def test_quantize_near_rounding_boundaries(zq, fmt):
    """Values placed on, and one or two binary32 ulps either side of, every
    rounding boundary of every code: the fast path's guard must send all the
    close calls to the exact division."""
    G = 128
    rng = np.random.default_rng(7)
    blocks = []
    for k in range(64):
        m = np.float32(rng.uniform(0.5, 2.0) * 2.0 ** rng.integers(-20, 20))
        qmax = 448.0 if fmt == O.E4M3 else float((1 << (O.BITS[fmt] - 1)) - 1)
        s = np.float32(np.float64(m) / qmax)
        if fmt == O.E4M3:
            grid = O.decode_array("e4m3", np.arange(0x7F, dtype=np.uint32)).astype(np.float64)
            mids = (grid[1:] + grid[:-1]) / 2
            t = rng.choice(mids, G - 1)
        else:
            t = rng.integers(-int(qmax), int(qmax), G - 1) + 0.5
        vals = (t * np.float64(s)).astype(np.float32)
        vals = np.nextafter(vals, vals * 2, dtype=np.float32) if k % 3 == 1 else vals
        vals = np.nextafter(vals, np.float32(0), dtype=np.float32) if k % 3 == 2 else vals
        vals = np.where(np.abs(vals) > m, np.sign(vals) * m, vals).astype(np.float32)
        blocks.append(np.concatenate([[m], vals * np.where(rng.random(G - 1) < 0.5, -1, 1)]))
    x = np.concatenate(blocks).astype(np.float32)
    codes, scales = gpu_quantize(zq, x, O.F32, fmt, G)
    want_c, want_s = O.quantize(x, fmt, G)
    assert_same_bits(scales, want_s, "scales")
    assert_same_codes(codes, want_c, "codes")


def test_e4m3_conversion_exhaustive_near_midpoints(zq):
    """Blocks led by 448 have scale exactly 1, so codes are the E4M3 conversion
    of the inputs themselves: every E4M3 value and midpoint, +-3 ulps."""
    grid = O.decode_array("e4m3", np.arange(0x7F, dtype=np.uint32)).astype(np.float32)
    mids = ((grid[1:].astype(np.float64) + grid[:-1]) / 2).astype(np.float32)
    pts = np.concatenate([grid, mids])
    around = [pts]
    for k in (1, 2, 3):
        up, dn = pts.copy(), pts.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(1e9))
            dn = np.nextafter(dn, np.float32(-1e9))
        around += [up, dn]
    vals = np.concatenate(around)
    vals = vals[np.abs(vals) <= 448]
    vals = np.concatenate([vals, -vals])
    G = 128
    nb = -(-vals.size // (G - 1))
    vals = np.concatenate([vals, np.zeros(nb * (G - 1) - vals.size, np.float32)])
    x = np.concatenate([np.full((nb, 1), 448.0, np.float32), vals.reshape(nb, G - 1)], axis=1).ravel()
    codes, scales = gpu_quantize(zq, x, O.F32, O.E4M3, G)
    assert np.all(scales == 1.0)
    want_c, _ = O.quantize(x, O.E4M3, G)
    assert_same_codes(codes, want_c, "e4m3")


def test_e4m3_conversion_every_binary32_to_448(zq):
    """The same scale-1 blocks over every binary32 value whose magnitude lies
    in [2^-11, 448], both signs (331,350,018 values; every smaller magnitude
    is below half the smallest E4M3 subnormal, 2^-10), every binary32
    subnormal and zero, and 2^24 seeded samples of the normal range below
    2^-11: all against the oracle's conversion, on every host core."""
    import time

    import fullsize as F

    t0 = time.time()
    G = 128
    mag = np.concatenate([
        np.arange(0x3A000000, 0x43E00000 + 1, dtype=np.uint32),  # 2^-11 .. 448
        np.arange(0, 0x00800000, dtype=np.uint32),  # zero and the subnormals
        np.random.default_rng(11).integers(0x00800000, 0x3A000000, 1 << 24, dtype=np.uint32)])
    vals = np.concatenate([mag, mag | np.uint32(0x80000000)]).view(np.float32)
    del mag
    nb = -(-vals.size // (G - 1))
    x = np.zeros((nb, G), np.float32)
    x[:, 0] = 448.0
    x[:, 1:] = np.concatenate([vals, np.zeros(nb * (G - 1) - vals.size, np.float32)]).reshape(nb, G - 1)
    x = x.reshape(-1)
    del vals
    codes, scales = gpu_quantize(zq, x, O.F32, O.E4M3, G)
    assert np.all(scales == 1.0)
    n = F.check_roundtrip("e4m3 conversion", x, O.F32, O.E4M3, G, codes, scales)
    assert n == x.size
    print(f"\n[e4m3] {n:,} elements (every binary32 in [2^-11, 448] of both signs among them) "
          f"compared on {F.cores()} host cores in {time.time() - t0:.1f} s")


def test_quantize_subnormal_scales(zq):
    """bf16 subnormal inputs give subnormal scales; the exact path (with its
    clamp) must agree with the definition."""
    rng = np.random.default_rng(3)
    bits = rng.integers(0, 0x0080, 4096).astype(np.uint16)  # bf16 subnormals and zero
    bits[rng.random(4096) < 0.5] |= 0x8000
    for fmt in FORMATS:
        codes, scales = gpu_quantize(zq, bits, O.BF16, fmt, 32)
        want_c, want_s = O.quantize(bits, fmt, 32, dtype=O.BF16)
        assert_same_bits(scales, want_s, f"scales {fid(fmt)}")
        assert_same_codes(codes, want_c, f"codes {fid(fmt)}")
    # fp32 subnormals where the clamp to qmax decides the code
    x = (np.array([300, -300, 299, 255, 254, -256, 3, 0] * 512, np.float64) * 2.0 ** -149).astype(np.float32)
    codes, scales = gpu_quantize(zq, x, O.F32, O.INT8, 32)
    want_c, want_s = O.quantize(x, O.INT8, 32)
    assert_same_bits(scales, want_s, "scales clamp")
    assert_same_codes(codes, want_c, "codes clamp")


def test_quantize_extreme_scales(zq):
    """fp32 blocks whose scale sits at the edges of the fast paths: near the
    largest binary32, around 2^126 (above it the reciprocal is subnormal and
    the run must take the exact path), around 2^-100 (below it the block
    scale and the fix-up use the IEEE division) and near 2^-126. Each block
    holds random values and exact half-integer multiples of a power of two."""
    rng = np.random.default_rng(11)
    G = 32
    s_targets = [3.0e38, 2.0 ** 127, 1.5 * 2.0 ** 126, 2.0 ** 126, 0.999 * 2.0 ** 126,
                 2.0 ** 100, 1.0, 2.0 ** -99, 2.0 ** -100, 0.999 * 2.0 ** -100, 2.0 ** -120,
                 2.0 ** -125, 1.001 * 2.0 ** -126, 2.0 ** -126]
    for fmt in FORMATS:
        d = 448.0 if fmt == O.E4M3 else float((1 << (O.BITS[fmt] - 1)) - 1)
        blocks = []
        for st in s_targets:
            m = min(st * d, 3.4e38)
            v = rng.standard_normal(G)
            blocks.append((v / np.abs(v).max() * m).astype(np.float32))
            p2 = 2.0 ** np.floor(np.log2(m / d))  # a power of two near the scale
            k = rng.integers(-int(d), int(d), G) + 0.5
            t = np.clip(k * p2, -3.4e38, 3.4e38).astype(np.float32)
            t[0] = np.float32(min(d * p2, 3.4e38))
            blocks.append(t)
        x = np.concatenate(blocks)
        assert np.all(np.isfinite(x))
        codes, scales = gpu_quantize(zq, x, O.F32, fmt, G)
        want_c, want_s = O.quantize(x, fmt, G)
        assert_same_bits(scales, want_s, f"scales {fid(fmt)}")
        assert_same_codes(codes, want_c, f"codes {fid(fmt)}")


def test_quantize_unaligned_32B_source(zq):
    """A source that is 16- but not 32-byte aligned takes the 128-bit load path."""
    import torch

    x = mixed_input(8 * 1024 + 8, O.BF16, seed=5)
    t = to_dev(x, O.BF16)
    sub = t[8:]  # 16 bytes past a 256-byte aligned allocation
    assert sub.data_ptr() % 32 == 16
    codes, scales = zq.quantize(sub, O.INT4, 128)
    want_c, want_s = O.quantize(x[8:], O.INT4, 128, dtype=O.BF16)
    assert_same_codes(to_host(codes), want_c, "codes")
    assert_same_bits(to_host(scales), want_s, "scales")
    del torch


# ---------------------------------------------------------------------------
# dequantize (codes from the oracle, never from the GPU)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("out", DTYPES, ids=dname)
@pytest.mark.parametrize("fmt", FORMATS, ids=fid)
@pytest.mark.parametrize("G", BLOCKS)
def test_dequantize_matches_oracle(zq, out, fmt, G):
    import torch

    x = mixed_input(N_MAIN, O.F32, seed=2000 + G, G=G)
    c, s = O.quantize(x, fmt, G)
    y = zq.dequantize(bytes_dev(c), bytes_dev(s), x.size, fmt, G,
                      out_dtype={O.F32: torch.float32, O.F16: torch.float16, O.BF16: torch.bfloat16}[out])
    want = O.dequantize(c, s, x.size, fmt, G, out)
    assert_same_bits(to_host(y), want, "dequantized")


@pytest.mark.parametrize("n", [1, 17, 32, 1000, 1024, 1025, 4097])
def test_dequantize_edge_sizes(zq, n):
    import torch

    for fmt in FORMATS:
        x = mixed_input(n, O.F32, seed=n + 1)
        c, s = O.quantize(x, fmt, 64)
        y = zq.dequantize(bytes_dev(c), bytes_dev(s), n, fmt, 64, out_dtype=torch.bfloat16)
        assert_same_bits(to_host(y), O.dequantize(c, s, n, fmt, 64, O.BF16), f"n={n}")


# ---------------------------------------------------------------------------
# quantized reduce
# ---------------------------------------------------------------------------

def _oracle_shards(N, n, fmt, G, seed, scale=1e-4):
    from blockwise_quantized_zero_gb300 import inputs

    out = []
    for r in range(N):
        x = inputs.laplace_f32(n, scale * (1 + r), seed, stream=r)
        if n >= 4 * 1024:
            x[1024:1024 + 128] = 0.0
        out.append(O.quantize(x, fmt, G))
    return out


def _gpu_reduce(zq, shards, n, fin, Gin, fout, Gout, want_sum=True):
    codes = [bytes_dev(c) for c, _ in shards]
    scales = [bytes_dev(s) for _, s in shards]
    oc, os_, sm = zq.reduce_quantized(codes, scales, n, fin, Gin, fout, Gout,
                                      sum_out=True if want_sum else None)
    zq.device_status()  # no bounded device-side wait ran out
    return to_host(oc), to_host(os_), (to_host(sm) if want_sum else None)


REDUCE_CASES = [
    (O.INT4, 128, O.INT4, 128), (O.INT4, 128, O.INT8, 256), (O.INT8, 256, O.INT4, 128),
    (O.E4M3, 128, O.E4M3, 128), (O.INT2, 32, O.INT6, 1024), (O.INT6, 64, O.INT2, 512),
    (O.INT8, 1024, O.E4M3, 32), (O.E4M3, 64, O.INT8, 64),
]


@pytest.mark.parametrize("fin,Gin,fout,Gout", REDUCE_CASES,
                         ids=[f"{fid(a)}g{b}-{fid(c)}g{d}" for a, b, c, d in REDUCE_CASES])
@pytest.mark.parametrize("N", [1, 3, 8])
def test_reduce_matches_oracle(zq, fin, Gin, fout, Gout, N):
    n = N_MAIN
    shards = _oracle_shards(N, n, fin, Gin, seed=31 + N)
    oc, os_, sm = _gpu_reduce(zq, shards, n, fin, Gin, fout, Gout)
    wc, ws, wsum = O.reduce([c for c, _ in shards], [s for _, s in shards], n, fin, Gin, fout, Gout,
                            want_sum=True)
    assert_same_bits(sm, wsum, "sum")
    assert_same_bits(os_, ws, "scales")
    assert_same_codes(oc, wc, "codes")


def test_reduce_all_format_pairs(zq):
    n = 2 * 1024 + 77
    for fin in FORMATS:
        shards = _oracle_shards(4, n, fin, 128, seed=fin)
        for fout in FORMATS:
            oc, os_, sm = _gpu_reduce(zq, shards, n, fin, 128, fout, 256)
            wc, ws, wsum = O.reduce([c for c, _ in shards], [s for _, s in shards], n, fin, 128,
                                    fout, 256, want_sum=True)
            assert_same_bits(sm, wsum, f"sum {fid(fin)}->{fid(fout)}")
            assert_same_bits(os_, ws, f"scales {fid(fin)}->{fid(fout)}")
            assert_same_codes(oc, wc, f"codes {fid(fin)}->{fid(fout)}")


def test_reduce_many_shards_and_no_sum(zq):
    n = 3 * 1024 + 5
    shards = _oracle_shards(64, n, O.INT4, 128, seed=64)
    oc, os_, _ = _gpu_reduce(zq, shards, n, O.INT4, 128, O.INT4, 128, want_sum=False)
    wc, ws, _ = O.reduce([c for c, _ in shards], [s for _, s in shards], n, O.INT4, 128, O.INT4, 128)
    assert_same_bits(os_, ws, "scales")
    assert_same_codes(oc, wc, "codes")


def test_reduce_order_is_shard_order(zq):
    """1 + 2^-24 + 2^-24 sums to 1 left to right but to 1 + 2^-23 right to left."""
    n, G = 1024, 32
    shards = [O.quantize(np.full(n, np.float32(v)), O.INT2, G) for v in (1.0, 2.0 ** -24, 2.0 ** -24)]
    _, _, sm = _gpu_reduce(zq, shards, n, O.INT2, G, O.INT8, G)
    assert np.all(sm == np.float32(1.0))
    _, _, sm = _gpu_reduce(zq, shards[::-1], n, O.INT2, G, O.INT8, G)
    assert np.all(sm == np.float32(1.0 + 2.0 ** -23))


# ---------------------------------------------------------------------------
# FP8 accumulate
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", DTYPES, ids=dname)
@pytest.mark.parametrize("G", BLOCKS)
def test_fp8_accumulate_matches_oracle(zq, dtype, G):
    n = N_MAIN
    codes = np.zeros(O.codes_bytes(O.E4M3, n), np.uint8)
    scales = np.zeros(O.num_blocks(n, G), np.float32)
    dc, ds = bytes_dev(codes), bytes_dev(scales)
    for step in range(4):
        from blockwise_quantized_zero_gb300 import inputs

        g32 = inputs.normal_f32(n, 1e-3, 4, stream=step)
        g32[::501] *= 30
        if step == 2:
            g32[:G] = 0.0
        g = {O.BF16: inputs.to_bf16_bits(g32), O.F16: g32.astype(np.float16), O.F32: g32}[dtype]
        zq.fp8_accumulate(dc, ds, to_dev(g, dtype), G)
        codes, scales = O.fp8_accumulate(codes, scales, g, G, grad_dtype=dtype)
        assert_same_bits(to_host(ds), scales, f"scales step {step}")
        assert_same_codes(to_host(dc), codes, f"codes step {step}")


@pytest.mark.parametrize("n", [1, 100, 1024, 1025, 2 * 1024 + 130])
def test_fp8_accumulate_edge_sizes(zq, n):
    from blockwise_quantized_zero_gb300 import inputs

    G = 128
    codes = np.zeros(O.codes_bytes(O.E4M3, n), np.uint8)
    scales = np.zeros(O.num_blocks(n, G), np.float32)
    dc, ds = bytes_dev(codes), bytes_dev(scales)
    for step in range(3):
        g = inputs.to_bf16_bits(inputs.normal_f32(n, 1e-3, 9, stream=step))
        zq.fp8_accumulate(dc, ds, to_dev(g, O.BF16), G)
        codes, scales = O.fp8_accumulate(codes, scales, g, G, grad_dtype=O.BF16)
    assert_same_bits(to_host(ds), scales, "scales")
    assert_same_codes(to_host(dc), codes, "codes")


def test_round_trip_through_the_gpu_only(zq):
    """GPU quantize then GPU dequantize equals the oracle's round trip."""
    import torch

    x = mixed_input(64 * 1024 + 7, O.BF16, seed=77)
    for fmt in FORMATS:
        c, s = zq.quantize(to_dev(x, O.BF16), fmt, 256)
        y = zq.dequantize(c, s, x.size, fmt, 256, out_dtype=torch.bfloat16)
        wc, ws = O.quantize(x, fmt, 256, dtype=O.BF16)
        assert_same_bits(to_host(y), O.dequantize(wc, ws, x.size, fmt, 256, O.BF16), fid(fmt))


@pytest.mark.parametrize("fmt", [O.INT8, O.INT4, O.E4M3])
def test_quantize_every_finite_fp16_value(zq, fmt):
    """Every finite binary16 bit pattern (subnormals, zeros of both signs,
    the largest values) as quantize input: blocks of 32 consecutive patterns,
    so each block's scale and every code depend on the exact widening."""
    import torch

    bits = np.arange(1 << 16, dtype=np.uint32)
    finite = bits[(bits & 0x7C00) != 0x7C00].astype(np.uint16)
    n = finite.size - finite.size % 32
    x = finite[:n].view(np.float16)
    c, s = zq.quantize(torch.from_numpy(x.copy()).cuda(), fmt, 32)
    wc, ws = O.quantize(x, fmt, 32)
    assert np.array_equal(to_host(c), wc)
    assert np.array_equal(as_bits(to_host(s)), as_bits(ws))
