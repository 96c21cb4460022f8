"""Aquavit's metadata-interleaved record layout on the GPU (through the C ABI)
against the oracle, bit for bit: the record stream of the quantize kernel and
the values of the dequantize kernel, for every integer width, block size and
element type, ragged sizes, and the full 8192x8192 bf16 shard on every
element."""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, mixed_input, to_dev, to_host

pytestmark = pytest.mark.gpu

INT_FORMATS = [O.INT2, O.INT4, O.INT6, O.INT8]
BLOCKS = [32, 64, 128, 256, 512, 1024]
DTYPES = [O.F32, O.F16, O.BF16]
N_MAIN = 5 * 1024 + 333  # five full tiles and a ragged tail (partial block for every G)
WIN = 2048


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    yield zq
    torch.cuda.empty_cache()


def _oracle_records(x, dtype, fmt, G):
    return O.quantize_interleaved(x, fmt, G, dtype=dtype if dtype == O.BF16 else None)


def _torch_dtype(dt):
    import torch

    return {O.F32: torch.float32, O.F16: torch.float16, O.BF16: torch.bfloat16}[dt]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("fmt", INT_FORMATS)
@pytest.mark.parametrize("G", BLOCKS)
def test_quantize_interleaved_matches_oracle(zq, dtype, fmt, G):
    x = mixed_input(N_MAIN, dtype, seed=fmt * 100 + G + dtype, G=G)
    rec = zq.quantize_interleaved(to_dev(x, dtype), fmt, G)
    want = _oracle_records(x, dtype, fmt, G)
    got = to_host(rec)
    assert got.size == want.size == zq.interleaved_bytes(fmt, N_MAIN, G)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:6]}"


@pytest.mark.parametrize("n", [1, 31, 32, 33, 511, 1023, 1024, 1025, 3 * 1024 + 1])
@pytest.mark.parametrize("fmt,G", [(O.INT4, 32), (O.INT6, 1024), (O.INT2, 64), (O.INT8, 256)])
def test_quantize_interleaved_edge_sizes(zq, n, fmt, G):
    x = mixed_input(n, O.BF16, seed=n, G=G)
    got = to_host(zq.quantize_interleaved(to_dev(x, O.BF16), fmt, G))
    assert np.array_equal(got, _oracle_records(x, O.BF16, fmt, G))


@pytest.mark.parametrize("out", DTYPES)
@pytest.mark.parametrize("fmt", INT_FORMATS)
@pytest.mark.parametrize("G", BLOCKS)
def test_dequantize_interleaved_matches_oracle(zq, out, fmt, G):
    from helpers import bytes_dev

    x = mixed_input(N_MAIN, O.F32, seed=7 * fmt + G, G=G)
    rec = _oracle_records(x, O.F32, fmt, G)
    y = zq.dequantize_interleaved(bytes_dev(rec), N_MAIN, fmt, G, out_dtype=_torch_dtype(out))
    want = O.dequantize_interleaved(rec, N_MAIN, fmt, G, out)
    assert np.array_equal(as_bits(to_host(y)), as_bits(want))


def test_interleaved_regroups_the_planar_gpu_result(zq):
    """The same tensor through both layouts on the GPU: record k is planar
    scale k followed by planar block k's codes, and both dequantize alike."""
    import torch

    n, G, fmt = 64 * 1024 + 96, 128, O.INT4
    x = mixed_input(n, O.BF16, seed=5, G=G)
    xd = to_dev(x, O.BF16)
    c, s = zq.quantize(xd, fmt, G)
    rec = to_host(zq.quantize_interleaved(xd, fmt, G)).tobytes()
    hc, hs = to_host(c).tobytes(), to_host(s)
    cb = G * 4 // 8
    for k in range(n // G):
        r = rec[k * (4 + cb):(k + 1) * (4 + cb)]
        assert r[:4] == hs[k:k + 1].tobytes() and r[4:] == hc[k * cb:(k + 1) * cb], k
    y1 = zq.dequantize(c, s, n, fmt, G, out_dtype=torch.bfloat16)
    y2 = zq.dequantize_interleaved(zq.quantize_interleaved(xd, fmt, G), n, fmt, G,
                                   out_dtype=torch.bfloat16)
    assert torch.equal(y1, y2)


def test_aquavit_schedule_run(zq):
    """A 24-step ascending schedule: every step quantizes into records at the
    step's (b, G) and dequantizes; the result equals the planar path's."""
    import torch

    x = to_dev(mixed_input(256 * 1024, O.BF16, seed=9), O.BF16)
    n, seen = x.numel(), set()
    for t in range(25):
        fmt, G, _, width = zq.aquavit_schedule(t, 24)
        seen.add((fmt, G))
        rec = zq.quantize_interleaved(x, fmt, G)
        assert rec.numel() * 8 == n * width
        y = zq.dequantize_interleaved(rec, n, fmt, G)
        c, s = zq.quantize(x, fmt, G)
        assert torch.equal(y, zq.dequantize(c, s, n, fmt, G)), (t, fmt, G)
    assert (O.INT2, 1024) in seen and (O.INT6, 32) in seen


def test_full_shard_every_element(zq):
    """8192x8192 bf16 (the weight shard of the benchmark), every pair of the
    schedule plus int8: every record and every dequantized value checked
    against the oracle, chunk by chunk of whole blocks."""
    import time

    import torch

    import fullsize as F
    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    x = inputs.weight_shard_bf16()
    xd = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()
    n = x.size
    total = 0
    for b in (2, 4, 6, 8):
        for G in BLOCKS:
            rec = zq.quantize_interleaved(xd, b, G)
            y = to_host(zq.dequantize_interleaved(rec, n, b, G, out_dtype=torch.bfloat16))
            hr = to_host(rec)
            R = 4 + G * b // 8

            def chunk(span, b=b, G=G, R=R, hr=hr, y=y):
                lo, hi = span
                want = O.quantize_interleaved(np.ascontiguousarray(x[lo:hi]), b, G, dtype=O.BF16)
                F.same(f"b={b} G={G}", "records", lo, hr[(lo // G) * R:(hi // G) * R], want)
                wy = O.dequantize_interleaved(want, hi - lo, b, G, O.BF16)
                F.same(f"b={b} G={G}", "dequantized values", lo, y[lo:hi], wy)
                return hi - lo

            total += sum(F.pmap(chunk, F.chunks(n)))
            del rec
    assert total == 24 * n
    print(f"\n[full-size parity] interleaved records: {total:,} elements compared bit for bit on "
          f"{F.cores()} host cores in {time.time() - t0:.1f} s")
