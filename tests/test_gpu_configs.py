"""The five benchmark workloads at full size, through the same C-ABI calls the
benchmark times, checked against the oracle on sampled windows.

Blocks are independent and start on 32-bit word boundaries, so the oracle can
quantize (or reduce, or accumulate) any window of whole blocks on its own and
must reproduce the GPU's bytes for that window exactly. Windows: the first and
the last 2048 elements and a seeded random set of 2048-element windows aligned
to 1024, which covers every block size and both runs of every warp tile.
"""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, to_host

pytestmark = pytest.mark.gpu

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


def windows(n: int, count: int, seed: int):
    rng = np.random.default_rng(seed)
    starts = {0, ((n - WIN) // 1024) * 1024}
    starts |= set((rng.integers(0, (n - WIN) // 1024, count) * 1024).tolist())
    return sorted(starts)


def code_window(codes: np.ndarray, fmt: int, lo: int, hi: int) -> np.ndarray:
    b = O.BITS[fmt]
    return codes[lo * b // 8: (hi * b + 7) // 8]


def check_quantize(host_in, dtype, dev_codes, dev_scales, fmt, G, wins, label):
    codes, scales = to_host(dev_codes), to_host(dev_scales)
    for lo in wins:
        hi = lo + WIN
        wc, ws = O.quantize(host_in[lo:hi], fmt, G, dtype=dtype if dtype == O.BF16 else None)
        nbytes = WIN * O.BITS[fmt] // 8
        assert np.array_equal(code_window(codes, fmt, lo, hi), wc[:nbytes]), (label, lo)
        assert np.array_equal(as_bits(scales[lo // G: hi // G]), as_bits(ws)), (label, lo)
    return codes, scales


def bf16_dev(bits):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def test_qwz_fp16_full(zq):
    """1 Mi fp16 weights with outliers, int8 G=256: every element checked."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    x = inputs.weights_fp16_outliers()
    c, s = zq.quantize(torch.from_numpy(x).cuda(), zq.INT8, 256)
    wc, ws = O.quantize(x, O.INT8, 256)
    assert np.array_equal(to_host(c), wc) and np.array_equal(as_bits(to_host(s)), as_bits(ws))
    for out, od in ((torch.float32, O.F32), (torch.float16, O.F16)):
        y = zq.dequantize(c, s, x.size, zq.INT8, 256, out_dtype=out)
        assert np.array_equal(as_bits(to_host(y)), as_bits(O.dequantize(wc, ws, x.size, O.INT8, 256, od)))


def test_gm_sweep_full(zq):
    """8192x8192 bf16, all 24 (b, G) pairs, quantize + dequantize -> bf16."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    x = inputs.weight_shard_bf16()
    xd = bf16_dev(x)
    n = x.size
    wins = windows(n, 12, seed=2)
    for b in (2, 4, 6, 8):
        for G in (1024, 512, 256, 128, 64, 32):
            c, s = zq.quantize(xd, b, G)
            y = zq.dequantize(c, s, n, b, G, out_dtype=torch.bfloat16)
            hc, hs = check_quantize(x, O.BF16, c, s, b, G, wins, f"b={b} G={G}")
            hy = to_host(y)
            for lo in wins[:4]:
                want = O.dequantize(code_window(hc, b, lo, lo + WIN), hs[lo // G:(lo + WIN) // G],
                                    WIN, b, G, O.BF16)
                assert np.array_equal(hy[lo:lo + WIN], want), (b, G, lo)
            assert zq.codes_bytes(b, n) + 4 * zq.num_blocks(n, G) == n * b // 8 + 4 * n // G


def test_qgz_reduce_full(zq):
    """8 shards x 134,217,728 fp32 Laplace gradients, int4 G=128 -> int4 G=128
    and -> int8 G=256 with the fp32 sums."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    N, n = 8, 134217728
    wins = windows(n, 6, seed=3)
    host_win = [[] for _ in wins]
    codes, scales = [], []
    for r in range(N):
        x = inputs.gradient_shard_f32(n, shard=r)
        for k, lo in enumerate(wins):
            host_win[k].append(x[lo:lo + WIN].copy())
        c, s = zq.quantize(torch.from_numpy(x).cuda(), zq.INT4, 128)
        if r == 0:
            check_quantize(x, O.F32, c, s, O.INT4, 128, wins, "shard 0")
        codes.append(c)
        scales.append(s)
        del x
    for fout, Gout in ((zq.INT4, 128), (zq.INT8, 256)):
        oc, os_, sm = zq.reduce_quantized(codes, scales, n, zq.INT4, 128, fout, Gout, sum_out=True)
        zq.device_status()
        hoc, hos, hsm = to_host(oc), to_host(os_), to_host(sm)
        for k, lo in enumerate(wins):
            sh = [O.quantize(xw, O.INT4, 128) for xw in host_win[k]]
            wc, ws, wsum = O.reduce([c for c, _ in sh], [s for _, s in sh], WIN, O.INT4, 128, fout,
                                    Gout, want_sum=True)
            assert np.array_equal(as_bits(hsm[lo:lo + WIN]), as_bits(wsum)), (fout, lo)
            assert np.array_equal(as_bits(hos[lo // Gout:(lo + WIN) // Gout]), as_bits(ws)), (fout, lo)
            assert np.array_equal(code_window(hoc, fout, lo, lo + WIN), wc[:WIN * O.BITS[fout] // 8])
        del oc, os_, sm
    del codes, scales
    torch.cuda.empty_cache()


def test_agoq_fp8_full(zq):
    """E4M3 main gradient of 268,435,456 elements: 4 accumulate steps, then the
    8-shard FP8 reduce of its slices."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    n, G, steps, N = 268435456, 128, 4, 8
    wins = windows(n, 6, seed=4)
    mc = torch.zeros(zq.codes_bytes(zq.E4M3, n), dtype=torch.uint8, device="cuda")
    ms = torch.zeros(zq.num_blocks(n, G), dtype=torch.float32, device="cuda")
    hc = {lo: np.zeros(WIN, np.uint8) for lo in wins}
    hs = {lo: np.zeros(WIN // G, np.float32) for lo in wins}
    for k in range(steps):
        g = inputs.gradient_bf16(n, step=k)
        zq.fp8_accumulate(mc, ms, bf16_dev(g), G)
        for lo in wins:
            hc[lo], hs[lo] = O.fp8_accumulate(hc[lo], hs[lo], g[lo:lo + WIN], G, grad_dtype=O.BF16)
        del g
    dmc, dms = to_host(mc), to_host(ms)
    for lo in wins:
        assert np.array_equal(dmc[lo:lo + WIN], hc[lo]), lo
        assert np.array_equal(as_bits(dms[lo // G:(lo + WIN) // G]), as_bits(hs[lo])), lo
    m = n // N
    sc = [mc[r * m:(r + 1) * m] for r in range(N)]
    ss = [ms[r * m // G:(r + 1) * m // G] for r in range(N)]
    oc, os_, sm = zq.reduce_quantized(sc, ss, m, zq.E4M3, G, zq.E4M3, G, sum_out=True)
    hoc, hos, hsm = to_host(oc), to_host(os_), to_host(sm)
    for lo in windows(m, 6, seed=5):
        ic = [dmc[r * m + lo:r * m + lo + WIN] for r in range(N)]
        isc = [dms[(r * m + lo) // G:(r * m + lo + WIN) // G] for r in range(N)]
        wc, ws, wsum = O.reduce(ic, isc, WIN, O.E4M3, G, O.E4M3, G, want_sum=True)
        assert np.array_equal(as_bits(hsm[lo:lo + WIN]), as_bits(wsum)), lo
        assert np.array_equal(as_bits(hos[lo // G:(lo + WIN) // G]), as_bits(ws)), lo
        assert np.array_equal(hoc[lo:lo + WIN], wc[:WIN]), lo
    del mc, ms, oc, os_, sm, sc, ss
    torch.cuda.empty_cache()


def test_llama70b_layer_full(zq):
    """The seven Llama-3-70B layer matrices, int8 G=256 and 6-bit G=32, quantize
    + dequantize -> bf16."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    total = 0
    for name, r, c, bits in inputs.llama70b_layer_bf16():
        n = r * c
        total += n
        xd = bf16_dev(bits)
        wins = windows(n, 4, seed=r + c)
        for b, G in ((8, 256), (6, 32)):
            dc, ds = zq.quantize(xd, b, G)
            hc, hs = check_quantize(bits, O.BF16, dc, ds, b, G, wins, f"{name} b={b}")
            y = to_host(zq.dequantize(dc, ds, n, b, G, out_dtype=torch.bfloat16))
            for lo in wins[:2]:
                want = O.dequantize(code_window(hc, b, lo, lo + WIN), hs[lo // G:(lo + WIN) // G],
                                    WIN, b, G, O.BF16)
                assert np.array_equal(y[lo:lo + WIN], want), (name, b, lo)
            del dc, ds
        del xd
    assert total == 855638016
    torch.cuda.empty_cache()
