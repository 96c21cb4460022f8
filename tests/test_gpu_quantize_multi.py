"""zq_quantize_multi (one launch over a list of tensors) against the oracle,
bit for bit, through the C ABI: ragged sizes (empty, shorter than a tile,
partial last tiles), every element type and format, more tensors than one
launch holds, and the 512-copy form of the 1 Mi-element fp16 workload."""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, mixed_input, oracle_quantize, to_dev, to_host

pytestmark = pytest.mark.gpu

SIZES = [0, 1, 31, 1023, 1024, 5000, 64 * 1024 + 3, 1 << 18, 3 * 1024 + 77, 2048]


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    return zq


def _check(zq, xs, dtype, fmt, G):
    srcs = [to_dev(x, dtype) for x in xs]
    codes, scales = zq.quantize_multi(srcs, fmt, G)
    for k, x in enumerate(xs):
        wc, ws = oracle_quantize(x, dtype, fmt, G)
        assert np.array_equal(to_host(codes[k]), wc), (k, x.size, "codes")
        assert np.array_equal(as_bits(to_host(scales[k])), as_bits(ws)), (k, x.size, "scales")


@pytest.mark.parametrize("dtype", [O.BF16, O.F16, O.F32])
@pytest.mark.parametrize("fmt,G", [(O.INT8, 256), (O.INT4, 128), (O.INT2, 32), (O.INT6, 1024),
                                   (O.E4M3, 64)])
def test_quantize_multi_ragged_list(zq, dtype, fmt, G):
    xs = [mixed_input(n, dtype, seed=40 + i, G=G) for i, n in enumerate(SIZES)]
    _check(zq, xs, dtype, fmt, G)


def test_quantize_multi_more_tensors_than_one_launch(zq):
    """300 tensors (two launches), sizes cycling through the ragged list."""
    xs = [mixed_input(SIZES[i % len(SIZES)] + (i % 3), O.BF16, seed=500 + i, G=128) for i in range(300)]
    _check(zq, xs, O.BF16, O.INT4, 128)


def test_quantize_multi_equals_single_calls_on_the_fp16_workload(zq):
    """512 copies of the 1 Mi-element fp16 weights with outliers (int8 G=256):
    the batched call writes exactly what one zq_quantize call per copy writes."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    x = torch.from_numpy(inputs.weights_fp16_outliers()).cuda()
    srcs = [x] + [x.clone() for _ in range(511)]
    codes, scales = zq.quantize_multi(srcs, zq.INT8, 256)
    c1, s1 = zq.quantize(x, zq.INT8, 256)
    wc, ws = O.quantize(inputs.weights_fp16_outliers(), O.INT8, 256)
    assert np.array_equal(to_host(c1), wc) and np.array_equal(as_bits(to_host(s1)), as_bits(ws))
    for k in range(512):
        assert torch.equal(codes[k], c1) and torch.equal(scales[k].view(torch.int32), s1.view(torch.int32)), k


@pytest.mark.parametrize("fmt,G", [(O.INT8, 256), (O.INT4, 128), (O.INT2, 32), (O.INT6, 1024),
                                   (O.E4M3, 64)])
@pytest.mark.parametrize("out", [O.BF16, O.F16, O.F32])
def test_dequantize_multi_ragged_list(zq, fmt, G, out):
    """zq_dequantize_multi of oracle-made codes (never GPU-made) on the ragged
    list, against the oracle's dequantize of each tensor."""
    import torch

    from helpers import bytes_dev

    qs = [oracle_quantize(mixed_input(n, O.F32, seed=60 + i, G=G), O.F32, fmt, G)
          for i, n in enumerate(SIZES)]
    td = {O.BF16: torch.bfloat16, O.F16: torch.float16, O.F32: torch.float32}[out]
    ys = zq.dequantize_multi([bytes_dev(c) for c, _ in qs], [bytes_dev(s) for _, s in qs], SIZES,
                             fmt, G, out_dtype=td)
    for k, ((c, s), n) in enumerate(zip(qs, SIZES)):
        want = O.dequantize(c, s, n, fmt, G, out)
        assert np.array_equal(as_bits(to_host(ys[k])), as_bits(want)), (k, n)


def test_dequantize_multi_llama_layer_equals_single_calls(zq):
    """The seven Llama-3-70B layer matrices (1/8 of the rows), int6 G=32: one
    batched dequantize writes exactly what one call per matrix writes."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    xs = [torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
          for _, _, _, bits in inputs.llama70b_layer_bf16(scale_rows=8)]
    codes, scales = zq.quantize_multi(xs, zq.INT6, 32)
    ys = zq.dequantize_multi(codes, scales, [x.numel() for x in xs], zq.INT6, 32,
                             out_dtype=torch.bfloat16)
    for x, c, s, y in zip(xs, codes, scales, ys):
        c1, s1 = zq.quantize(x, zq.INT6, 32)
        assert torch.equal(c, c1) and torch.equal(s.view(torch.int32), s1.view(torch.int32))
        assert torch.equal(y.view(torch.int16), zq.dequantize(c1, s1, x.numel(), zq.INT6, 32,
                                                              out_dtype=torch.bfloat16).view(torch.int16))
