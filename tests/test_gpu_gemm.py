"""The dequant-fused GEMM (zq_gemm_dequant, tcgen05 tensor cores) against the
oracle, through the C ABI.

Weights are quantized by the oracle (never by the GPU). Two kinds of check:

* exact: small-integer activations and weights whose block scales are 1, so
  every product and partial sum is an integer below 2^24 and the fp32 result
  cannot depend on the order of the additions: the GPU must equal the integer
  product exactly (fp32 output), or its single bf16 rounding (bf16 output);
* bounded: random operands against the oracle's exact sum, within the error
  bound of an fp32 accumulation of K/16 tensor-core steps in any order,
  |y - exact| <= (K/16) 2^-22 sum_k |x w|, plus half a bf16 ulp of y
  (2^-9 |y|, taken as 2^-8) for bf16 output.

Shapes cover each output tile the launcher picks (256 x 256 with one
accumulator, 256 x 128, 128 x 128 and 128 x 64 with two; checked through
zq_gemm_plan), several tiles per
CTA (the stage ring and the accumulators wrap), a ragged last row tile, every
code format and several block sizes, and the split-K form for few rows
(128 x 256 and 128 x 128 tiles over clusters of 2, 4 and 8 CTAs; each case
checks through zq_gemm_plan that the split path is the one taken).
"""
import numpy as np
import pytest

import oracle as O
from helpers import bytes_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    return zq


def _bf16_bits(x32):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def _bf16_dev(bits, M, K):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda().reshape(M, K)


def _int_weights(r, N, K, G, fmt):
    top = 448 if fmt == O.E4M3 else (1 << (O.BITS[fmt] - 1)) - 1
    lim = 16 if fmt == O.E4M3 else top
    W = r.integers(-lim, lim + 1, size=(N, K)).astype(np.int64)
    W[:, ::G] = top * np.where(r.random((N, K // G)) < 0.5, -1, 1)  # block scale exactly 1
    return W


EXACT_CASES = [  # (M, N, K, fmt, G): tiles 256x256 / 128x128 / 128x64, ragged M, all formats
    (4096 - 57, 2560, 1024, O.INT8, 128),
    (1024, 2560, 512, O.INT4, 64),
    (200, 1024, 768, O.INT2, 256),
    (1024, 2560, 512, O.INT6, 32),
    (1500, 1536, 1024, O.E4M3, 512),
]


@pytest.mark.parametrize("M,N,K,fmt,G", EXACT_CASES)
def test_gemm_exact_small_integers(zq, M, N, K, fmt, G):
    import torch

    r = np.random.default_rng(M + N + K + fmt)
    W = _int_weights(r, N, K, G, fmt)
    X = r.integers(-16, 17, size=(M, K)).astype(np.int64)
    codes, scales = O.quantize(W.astype(np.float32).ravel(), fmt, G)
    assert np.all(scales == 1.0)
    xd = _bf16_dev(_bf16_bits(X.astype(np.float32).ravel()), M, K)
    want = X.astype(np.float64) @ W.astype(np.float64).T  # exact: integers below 2^53
    assert np.abs(want).max() < 2 ** 24
    y = zq.gemm_dequant(xd, bytes_dev(codes), bytes_dev(scales), fmt, G, N)
    yb = zq.gemm_dequant(xd, bytes_dev(codes), bytes_dev(scales), fmt, G, N, out_dtype=torch.bfloat16)
    zq.device_status()
    got = to_host(y)
    bad = np.argwhere(got != want.astype(np.float32))
    assert bad.size == 0, f"{len(bad)} outputs differ, first at {bad[:4].tolist()}"
    assert np.array_equal(to_host(yb), _bf16_bits(want.astype(np.float32).ravel()).reshape(M, N))


BOUND_CASES = [  # tiles 256x128 / 128x64
    (2048, 2560, 1024, O.INT8, 256),
    (4096, 2560, 512, O.INT4, 32),
    (768, 2560, 512, O.INT4, 128),
    (128, 1024, 2048, O.INT4, 32),
    (1000, 1536, 512, O.E4M3, 128),
]


EDGE_CASES = [(1, 64, 64, O.INT8, 64), (1, 128, 64, O.INT4, 32), (129, 192, 128, O.INT6, 128),
              (300, 64, 1024, O.INT2, 1024)]


@pytest.mark.parametrize("M,N,K,fmt,G", BOUND_CASES)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_random_within_fp32_accumulation_bound(zq, M, N, K, fmt, G, out):
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    w32 = inputs.normal_f32(N * K, 0.02, 200 + fmt, stream=K)
    codes, scales = O.quantize(w32, fmt, G)
    xb = _bf16_bits(inputs.normal_f32(M * K, 1.0, 201, stream=M))
    od = torch.float32 if out == "f32" else torch.bfloat16
    y = to_host(zq.gemm_dequant(_bf16_dev(xb, M, K), bytes_dev(codes), bytes_dev(scales), fmt, G, N,
                                out_dtype=od))
    zq.device_status()
    r = np.random.default_rng(7)
    cnt = 4096
    rows = np.concatenate([r.integers(0, M, cnt), np.full(N, M - 1), np.zeros(N, np.int64)])
    cols = np.concatenate([r.integers(0, N, cnt), np.arange(N), np.arange(N)])
    ref, mag = O.gemm_dequant(xb, M, K, codes, scales, fmt, G, N, rows=rows, cols=cols)
    got = y[rows, cols].astype(np.float64) if out == "f32" else \
        (y[rows, cols].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tol = (K / 16) * 2.0 ** -22 * mag + (2.0 ** -8 * np.abs(ref) if out == "bf16" else 0.0)
    err = np.abs(got - ref)
    worst = float(np.max(err / np.maximum(tol, 1e-300)))
    assert np.all(err <= tol), f"worst error {worst:.3f} of the bound"


SPLIT_CASES = [  # few rows: K split over clusters (the plan on GB300 in the comment)
    (1, 512, 2048, O.INT8, 256),     # 128 x 128 tiles, 8 CTAs a tile
    (77, 1024, 4096, O.INT4, 128),   # 128 x 128, 8
    (255, 1024, 8192, O.INT6, 64),   # 128 x 128, 8, two row tiles
    (1, 6144, 2048, O.INT8, 128),    # 128 x 256, 4
    (77, 6144, 2048, O.INT2, 32),    # 128 x 256, 4
    (1, 12288, 4096, O.INT4, 64),    # 128 x 256, 2
    (200, 6144, 4096, O.E4M3, 512),  # 128 x 256, 2, two row tiles
    (150, 2048, 4096, O.INT8, 256),  # 128 x 256, 8, two row tiles
    (1, 3072, 2048, O.INT6, 32),     # 128 x 256, 8
]


@pytest.mark.parametrize("M,N,K,fmt,G", SPLIT_CASES)
def test_gemm_split_k_exact_small_integers(zq, M, N, K, fmt, G):
    """Problems with too few output tiles for the GPU, where K is split over
    the CTAs of a cluster and the partial tiles are summed in rank order:
    exact on integer operands, like the unsplit tiles."""
    import torch

    assert zq.gemm_plan(M, N, K)[2] > 1, zq.gemm_plan(M, N, K)  # the split path is the one tested
    r = np.random.default_rng(M * 3 + N + K + fmt)
    W = _int_weights(r, N, K, G, fmt)
    X = r.integers(-16, 17, size=(M, K)).astype(np.int64)
    codes, scales = O.quantize(W.astype(np.float32).ravel(), fmt, G)
    assert np.all(scales == 1.0)
    xd = _bf16_dev(_bf16_bits(X.astype(np.float32).ravel()), M, K)
    want = X.astype(np.float64) @ W.astype(np.float64).T
    assert np.abs(want).max() < 2 ** 24
    y = zq.gemm_dequant(xd, bytes_dev(codes), bytes_dev(scales), fmt, G, N)
    yb = zq.gemm_dequant(xd, bytes_dev(codes), bytes_dev(scales), fmt, G, N, out_dtype=torch.bfloat16)
    zq.device_status()
    bad = np.argwhere(to_host(y) != want.astype(np.float32))
    assert bad.size == 0, f"{len(bad)} outputs differ, first at {bad[:4].tolist()}"
    assert np.array_equal(to_host(yb), _bf16_bits(want.astype(np.float32).ravel()).reshape(M, N))


@pytest.mark.parametrize("M,N,K,fmt,G", [(128, 8192, 8192, O.INT8, 256), (1, 1024, 8192, O.INT4, 128),
                                         (96, 8192, 28672, O.INT8, 256)])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_gemm_split_k_random_within_bound(zq, M, N, K, fmt, G, out):
    """Few-token shapes of the Llama-3-70B projections (q / down at 128 and
    96 tokens, k at one token): random operands, every output of a sampled
    set against the oracle within the fp32 accumulation bound, which covers
    the split sum ((p0 + p1) + ...) as well."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    assert zq.gemm_plan(M, N, K)[2] > 1, zq.gemm_plan(M, N, K)
    w32 = inputs.normal_f32(N * K, 0.02, 210 + fmt, stream=K)
    codes, scales = O.quantize(w32, fmt, G)
    xb = _bf16_bits(inputs.normal_f32(M * K, 1.0, 211, stream=M))
    od = torch.float32 if out == "f32" else torch.bfloat16
    y = to_host(zq.gemm_dequant(_bf16_dev(xb, M, K), bytes_dev(codes), bytes_dev(scales), fmt, G, N,
                                out_dtype=od))
    zq.device_status()
    r = np.random.default_rng(9)
    rows = np.concatenate([r.integers(0, M, 2048), np.full(N, M - 1)])
    cols = np.concatenate([r.integers(0, N, 2048), np.arange(N)])
    ref, mag = O.gemm_dequant(xb, M, K, codes, scales, fmt, G, N, rows=rows, cols=cols)
    got = y[rows, cols].astype(np.float64) if out == "f32" else \
        (y[rows, cols].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tol = (K / 16) * 2.0 ** -22 * mag + (2.0 ** -8 * np.abs(ref) if out == "bf16" else 0.0)
    err = np.abs(got - ref)
    assert np.all(err <= tol), f"worst error {float(np.max(err / np.maximum(tol, 1e-300))):.3f} of the bound"


@pytest.mark.parametrize("M,N,K,fmt,G", EDGE_CASES)
def test_gemm_edge_shapes_exact(zq, M, N, K, fmt, G):
    """One row, the smallest N and K (one k-block), a row tile of one row."""
    r = np.random.default_rng(M * 7 + N + K)
    W = _int_weights(r, N, K, G, fmt)
    X = r.integers(-16, 17, size=(M, K)).astype(np.int64)
    codes, scales = O.quantize(W.astype(np.float32).ravel(), fmt, G)
    y = zq.gemm_dequant(_bf16_dev(_bf16_bits(X.astype(np.float32).ravel()), M, K), bytes_dev(codes),
                        bytes_dev(scales), fmt, G, N)
    zq.device_status()
    assert np.array_equal(to_host(y), (X.astype(np.float64) @ W.astype(np.float64).T).astype(np.float32))


def test_gemm_cases_cover_every_plan(zq):
    """The cases of this file reach every tile the launcher can pick (by its
    cost model, zq_gemm_plan): 256 x 256, 256 x 128, 128 x 128 and 128 x 64
    unsplit, and 128 x 256 and 128 x 128 split over clusters of 2, 4 and 8."""
    cases = EXACT_CASES + BOUND_CASES + EDGE_CASES + SPLIT_CASES
    plans = {zq.gemm_plan(M, N, K) for M, N, K, _, _ in cases}
    unsplit = {(bm, bn) for bm, bn, sp in plans if sp == 1}
    assert {(256, 256), (256, 128), (128, 128), (128, 64)} <= unsplit, plans
    assert {sp for _, _, sp in plans} >= {2, 4, 8}, plans
    assert {bn for _, bn, sp in plans if sp > 1} == {128, 256}, plans


def test_gemm_empty_problem_enqueues_nothing(zq):
    import torch

    codes = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(64 * 64 // 32, dtype=torch.float32, device="cuda")
    x = torch.zeros(0, 64, dtype=torch.bfloat16, device="cuda")
    assert zq.gemm_dequant(x, codes, scales, O.INT8, 32, 64).shape == (0, 64)
    zq.device_status()


def test_gemm_llama70b_layer_sampled(zq):
    """The benchmark configuration: the seven Llama-3-70B layer projections
    applied to 4096 tokens of bf16 activations. Each seeded bf16 matrix of the
    layer (listed input x output features) is read as the N x K weight of the
    projection (N = its output features, K = its input features; the same
    N(0, 0.02) bytes), quantized int8 G=256 by the oracle. 4096 sampled
    outputs of each projection, plus a whole output row and column, against
    the oracle within the fp32 accumulation bound (bf16 output)."""
    import torch

    import fullsize as F
    from blockwise_quantized_zero_gb300 import inputs

    M, fmt, G = 4096, O.INT8, 256
    xs = {}
    r = np.random.default_rng(11)
    for name, rows, cols, bits in inputs.llama70b_layer_bf16():
        N, K = cols, rows  # output features x input features
        codes, scales = F.oracle_quantize_full(bits, fmt, G, dtype=O.BF16)
        if K not in xs:
            xs[K] = _bf16_bits(inputs.normal_f32(M * K, 1.0, 300, stream=K))
        xb = xs[K]
        y = to_host(zq.gemm_dequant(_bf16_dev(xb, M, K), bytes_dev(codes), bytes_dev(scales), fmt, G,
                                    N, out_dtype=torch.bfloat16))
        zq.device_status()
        mrow, ncol = int(r.integers(0, M)), int(r.integers(0, N))
        rows_ = np.concatenate([r.integers(0, M, 4096), np.full(N, mrow), np.arange(M)])
        cols_ = np.concatenate([r.integers(0, N, 4096), np.arange(N), np.full(M, ncol)])
        ref, mag = O.gemm_dequant(xb, M, K, codes, scales, fmt, G, N, rows=rows_, cols=cols_)
        got = (y[rows_, cols_].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        tol = (K / 16) * 2.0 ** -22 * mag + 2.0 ** -8 * np.abs(ref)
        err = np.abs(got - ref)
        assert np.all(err <= tol), (name, float(np.max(err / tol)))
        del codes, scales, y
    torch.cuda.empty_cache()
