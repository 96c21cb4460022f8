"""qgZ's tensor-slice reordering and two-hop reduce on the GPU (through the C
ABI) against the oracle, bit for bit: codes, scales, the hop-1 results and the
final fp32 sums, for several node x GPU shapes, formats and element types."""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, bytes_dev, mixed_input, to_dev, to_host

pytestmark = pytest.mark.gpu

SHAPES = [(2, 2), (2, 4), (4, 2), (3, 2), (1, 3), (3, 1)]


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    return zq


def _same(got, want, label):
    g, w = as_bits(got), as_bits(want)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{label}: {bad.size} differ, first at {bad[:6]}")


@pytest.mark.parametrize("A,L", SHAPES)
@pytest.mark.parametrize("dtype,fmt,G", [(O.BF16, O.INT4, 128), (O.F32, O.INT8, 256),
                                         (O.F16, O.E4M3, 64), (O.F32, O.INT2, 32),
                                         (O.BF16, O.INT6, 1024)])
def test_quantize_reordered_matches_oracle(zq, A, L, dtype, fmt, G):
    n = A * L * 2048
    x = mixed_input(n, dtype, seed=A * 100 + L + fmt, G=G)
    c, s = zq.quantize_reordered(to_dev(x, dtype), fmt, G, A, L)
    wc, ws = O.quantize_reordered(x, fmt, G, A, L, dtype=dtype if dtype == O.BF16 else None)
    _same(to_host(s), ws, "scales")
    _same(to_host(c), wc, "codes")


def _gradients(P, n, seed):
    from blockwise_quantized_zero_gb300 import inputs

    return [inputs.laplace_f32(n, 1e-4 * (1 + g % 5), seed, stream=g) for g in range(P)]


@pytest.mark.parametrize("A,L", SHAPES)
@pytest.mark.parametrize("fin,Gin,fmid,Gmid,fout,Gout", [
    (O.INT4, 128, O.INT4, 128, O.INT4, 128),
    (O.INT8, 256, O.E4M3, 64, O.INT8, 32),
    (O.E4M3, 128, O.INT4, 1024, O.E4M3, 128),
])
def test_two_hop_matches_oracle(zq, A, L, fin, Gin, fmid, Gmid, fout, Gout):
    P = A * L
    n = P * 4096 * 2
    xs = _gradients(P, n, seed=70 + A * 10 + L)
    qs = [O.quantize_reordered(x, fin, Gin, A, L) for x in xs]
    mid, out, sums = zq.reduce_two_hop([bytes_dev(c) for c, _ in qs], [bytes_dev(s) for _, s in qs],
                                       A, L, n, fin, Gin, fmid, Gmid, fout, Gout, sums=True)
    zq.device_status()
    wmid, wout, wsums = O.reduce_two_hop([c for c, _ in qs], [s for _, s in qs], A, L, n, fin, Gin,
                                         fmid, Gmid, fout, Gout, want_sum=True)
    for g in range(P):
        _same(to_host(mid[g][1]), wmid[g][1], f"GPU {g} hop-1 scales")
        _same(to_host(mid[g][0]), wmid[g][0], f"GPU {g} hop-1 codes")
        _same(to_host(sums[g]), wsums[g], f"GPU {g} sums")
        _same(to_host(out[g][1]), wout[g][1], f"GPU {g} scales")
        _same(to_host(out[g][0]), wout[g][0], f"GPU {g} codes")


def test_reordered_quantize_then_two_hop_end_to_end(zq):
    """GPU-only chain (reordered quantize of every GPU's fp32 gradient, then
    both hops) against the oracle's chain on the same inputs."""
    A, L = 2, 4
    P, n = A * L, A * L * 4096 * 4
    xs = _gradients(P, n, seed=91)
    qd = [zq.quantize_reordered(to_dev(x, O.F32), O.INT4, 128, A, L) for x in xs]
    _, out, sums = zq.reduce_two_hop([c for c, _ in qd], [s for _, s in qd], A, L, n, O.INT4, 128,
                                     O.INT4, 128, O.INT4, 128, sums=True)
    zq.device_status()
    qs = [O.quantize_reordered(x, O.INT4, 128, A, L) for x in xs]
    _, wout, wsums = O.reduce_two_hop([c for c, _ in qs], [s for _, s in qs], A, L, n, O.INT4, 128,
                                      O.INT4, 128, O.INT4, 128, want_sum=True)
    for g in range(P):
        _same(to_host(sums[g]), wsums[g], f"GPU {g} sums")
        _same(to_host(out[g][0]), wout[g][0], f"GPU {g} codes")


def test_two_hop_argument_errors(zq):
    """Chunks must be a multiple of 4096 elements; too many GPUs and aliasing
    outputs are refused before any work."""
    import torch

    A, L = 2, 2
    P = 4
    n = P * 4096
    c = [torch.zeros(zq.codes_bytes(O.INT4, n), dtype=torch.uint8, device="cuda") for _ in range(P)]
    s = [torch.zeros(zq.num_blocks(n, 128), dtype=torch.float32, device="cuda") for _ in range(P)]
    with pytest.raises(zq.ZQError, match="INVALID_ARG"):
        zq.reduce_two_hop(c, s, A, L, n - P * 1024, O.INT4, 128, O.INT4, 128, O.INT4, 128)
    mid = [(zq.empty_codes(O.INT4, A * n // P, "cuda"), zq.empty_scales(A * n // P, 128, "cuda"))
           for _ in range(P)]
    out = [(mid[g][0], mid[g][1]) for g in range(P)]  # outputs on top of the hop-1 buffers
    with pytest.raises(zq.ZQError, match="ALIAS"):
        zq.reduce_two_hop(c, s, A, L, n, O.INT4, 128, O.INT4, 128, O.INT4, 128, mid=mid, out=out)


def test_two_hop_full_size_sampled(zq):
    """The benchmark configuration (2 nodes x 4 GPUs, 134,217,728 fp32 per GPU,
    int4 G=128 throughout), through the same calls the benchmark times. GPU
    g's final chunk is the sum of chunk g of every gradient, so a window of
    whole blocks of it follows from the same window of chunk g on every GPU:
    the oracle quantizes those windows, sums them node by node (hop 1) and
    over the nodes (hop 2), and must reproduce the GPU's codes, scales and
    fp32 sums there."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    A, L, n, G = 2, 4, 134217728, 128
    P, m = A * L, n // (A * L)
    hx, qd = [], []
    for g in range(P):
        x = inputs.gradient_shard_f32(n, shard=g)
        xd = torch.from_numpy(x).cuda()
        qd.append(zq.quantize_reordered(xd, O.INT4, G, A, L))
        del xd
        hx.append(x)
    _, out, sums = zq.reduce_two_hop([c for c, _ in qd], [s for _, s in qd], A, L, n, O.INT4, G,
                                     O.INT4, G, O.INT4, G, sums=True)
    zq.device_status()
    W = 4096
    rng = np.random.default_rng(17)
    for g, lo in [(0, 0), (P - 1, m - W)] + [(int(rng.integers(0, P)), int(rng.integers(0, (m - W) // G)) * G)
                                             for _ in range(4)]:
        win = [O.quantize(np.ascontiguousarray(hx[g2][g * m + lo:g * m + lo + W]), O.INT4, G)
               for g2 in range(P)]
        mid = []
        for a2 in range(A):  # hop 1: node a2's GPUs in order
            part = [win[a2 * L + l2] for l2 in range(L)]
            mc, ms, _ = O.reduce([c for c, _ in part], [s for _, s in part], W, O.INT4, G, O.INT4, G)
            mid.append((mc, ms))
        wc, ws, wsum = O.reduce([c for c, _ in mid], [s for _, s in mid], W, O.INT4, G, O.INT4, G,
                                want_sum=True)
        _same(to_host(sums[g][lo:lo + W]), wsum, f"GPU {g} sums at {lo}")
        _same(to_host(out[g][1][lo // G:(lo + W) // G]), ws, f"GPU {g} scales at {lo}")
        _same(to_host(out[g][0][lo // 2:(lo + W) // 2]), wc, f"GPU {g} codes at {lo}")
