"""The five benchmark workloads at full size, through the same C-ABI calls the
benchmark times, compared with the oracle on EVERY element.

Each GPU output (codes, scales, dequantized values, fp32 sums) is copied to
the host and compared bit for bit with the oracle, run on whole-block chunks
of the same seeded inputs over all host cores (tests/fullsize.py). Nothing
the GPU computed is an oracle input: the reduce and the FP8 reduce take the
shards the oracle itself quantized or accumulated.
"""
import time

import numpy as np
import pytest

import oracle as O
import fullsize as F
from helpers import as_bits, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    yield zq
    torch.cuda.empty_cache()


def bf16_dev(bits):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


def _report(label, elements, t0):
    print(f"\n[full-size parity] {label}: {elements:,} elements compared bit for bit on "
          f"{F.cores()} host cores in {time.time() - t0:.1f} s")


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
    """8192x8192 bf16, all 24 (b, G) pairs, quantize + dequantize -> bf16:
    every code, scale and dequantized value of every pair."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    x = inputs.weight_shard_bf16()
    xd = bf16_dev(x)
    n = x.size
    total = 0
    for b in (2, 4, 6, 8):
        for G in (1024, 512, 256, 128, 64, 32):
            c, s = zq.quantize(xd, b, G)
            y = zq.dequantize(c, s, n, b, G, out_dtype=torch.bfloat16)
            total += F.check_roundtrip(f"b={b} G={G}", x, O.BF16, b, G, to_host(c), to_host(s),
                                       to_host(y), O.BF16)
            assert zq.codes_bytes(b, n) + 4 * zq.num_blocks(n, G) == n * b // 8 + 4 * n // G
            del c, s, y
    assert total == 24 * n
    _report("gm_sweep (24 pairs, quantize + dequantize)", total, t0)


def _gradient_shards(zq, N, n, fmt, G):
    """The qgZ gradient shards: seeded fp32 gradients quantized on the GPU
    (checked on every element against the oracle's quantization, which the
    oracle side keeps as its reduce input)."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    dev, ref = [], []
    for r in range(N):
        x = inputs.gradient_shard_f32(n, shard=r)
        c, s = zq.quantize(torch.from_numpy(x).cuda(), fmt, G)
        wc, ws = F.oracle_quantize_full(x, fmt, G)
        F.same(f"shard {r}", "codes", 0, to_host(c), wc)
        F.same(f"shard {r}", "scales", 0, to_host(s), ws)
        dev.append((c, s))
        ref.append((wc, ws))
        del x
    return dev, ref


def test_qgz_reduce_full(zq):
    """8 shards x 134,217,728 fp32 Laplace gradients, int4 G=128 -> int4 G=128
    and -> int8 G=256 with the fp32 sums: every element."""
    import torch

    t0 = time.time()
    N, n = 8, 134217728
    dev, ref = _gradient_shards(zq, N, n, zq.INT4, 128)
    total = 0
    for fout, Gout in ((zq.INT4, 128), (zq.INT8, 256)):
        oc, os_, sm = zq.reduce_quantized([c for c, _ in dev], [s for _, s in dev], n, zq.INT4, 128,
                                          fout, Gout, sum_out=True)
        zq.device_status()
        total += F.check_reduce(f"reduce -> {O.BITS[fout]}-bit G={Gout}", ref, n, O.INT4, 128, fout,
                                Gout, to_host(oc), to_host(os_), to_host(sm))
        del oc, os_, sm
    del dev
    torch.cuda.empty_cache()
    assert total == 2 * n
    _report("qgz_reduce (8 shard quantizations, 2 reductions)", total + N * n, t0)


def test_agoq_fp8_full(zq):
    """E4M3 main gradient of 268,435,456 elements: 4 accumulate steps (every
    element after every step), then the 8-shard FP8 reduce of its slices."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    n, G, steps, N = 268435456, 128, 4, 8
    mc = torch.zeros(zq.codes_bytes(zq.E4M3, n), dtype=torch.uint8, device="cuda")
    ms = torch.zeros(zq.num_blocks(n, G), dtype=torch.float32, device="cuda")
    hc = np.zeros(n, np.uint8)
    hs = np.zeros(n // G, np.float32)
    for k in range(steps):
        g = inputs.gradient_bf16(n, step=k)
        zq.fp8_accumulate(mc, ms, bf16_dev(g), G)
        F.fp8_accumulate_full(hc, hs, g, G, grad_dtype=O.BF16)
        F.same(f"accumulate step {k}", "codes", 0, to_host(mc), hc)
        F.same(f"accumulate step {k}", "scales", 0, to_host(ms), hs)
        del g
    m = n // N
    sc = [mc[r * m:(r + 1) * m] for r in range(N)]
    ss = [ms[r * m // G:(r + 1) * m // G] for r in range(N)]
    oc, os_, sm = zq.reduce_quantized(sc, ss, m, zq.E4M3, G, zq.E4M3, G, sum_out=True)
    zq.device_status()
    ref = [(hc[r * m:(r + 1) * m], hs[r * m // G:(r + 1) * m // G]) for r in range(N)]
    total = F.check_reduce("FP8 reduce 8 x n/8", ref, m, O.E4M3, G, O.E4M3, G, to_host(oc),
                           to_host(os_), to_host(sm))
    assert total == m
    del mc, ms, oc, os_, sm, sc, ss
    torch.cuda.empty_cache()
    _report("agoq_fp8 (4 accumulate steps + FP8 reduce)", steps * n + m, t0)


def test_llama70b_layer_full(zq):
    """The seven Llama-3-70B layer matrices, int8 G=256 and 6-bit G=32, quantize
    + dequantize -> bf16, in the benchmark's form (one multi-tensor quantize
    and one multi-tensor dequantize call per scheme): every element of every
    matrix against the oracle; the per-matrix calls give the same bytes."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    layer = list(inputs.llama70b_layer_bf16())
    xds = [bf16_dev(bits) for _, _, _, bits in layer]
    ns = [r * c for _, r, c, _ in layer]
    assert sum(ns) == 855638016
    checked = 0
    for b, G in ((8, 256), (6, 32)):
        cs, ss = zq.quantize_multi(xds, b, G)
        ys = zq.dequantize_multi(cs, ss, ns, b, G, out_dtype=torch.bfloat16)
        for (name, r, c, bits), dc, ds, y, xd in zip(layer, cs, ss, ys, xds):
            checked += F.check_roundtrip(f"{name} b={b} G={G}", bits, O.BF16, b, G, to_host(dc),
                                         to_host(ds), to_host(y), O.BF16)
            c1, s1 = zq.quantize(xd, b, G)
            assert torch.equal(c1, dc) and torch.equal(s1.view(torch.int32), ds.view(torch.int32)), name
            y1 = zq.dequantize(c1, s1, r * c, b, G, out_dtype=torch.bfloat16)
            assert torch.equal(y1.view(torch.int16), y.view(torch.int16)), name
            del c1, s1, y1
        del cs, ss, ys
    assert checked == 2 * sum(ns)
    del xds
    torch.cuda.empty_cache()
    _report("llama70b (2 schemes, batched quantize + dequantize; per-matrix calls equal)", checked, t0)
