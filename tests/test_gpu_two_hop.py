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


def test_two_hop_full_size_every_element(zq):
    """The benchmark configuration (2 nodes x 4 GPUs, 134,217,728 fp32 per GPU,
    int4 G=128 throughout), through the same calls the benchmark times, on
    every element: each GPU's reordered quantization, every hop-1 result and
    every final chunk with its fp32 sums. The oracle quantizes each gradient
    chunk by chunk (chunk c at its slice position), then, for each window of
    whole blocks of final chunk g = a*L + l, sums that window of chunk g over
    each node's GPUs in order (hop 1: the window of GPU (a2, l)'s hop-1 result
    at chunk a) and over the nodes in order (hop 2)."""
    import time

    import torch

    import fullsize as F
    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    A, L, n, G = 2, 4, 134217728, 128
    P, m = A * L, n // (A * L)
    qd, ref = [], []
    for g in range(P):
        x = inputs.gradient_shard_f32(n, shard=g)
        qd.append(zq.quantize_reordered(torch.from_numpy(x).cuda(), O.INT4, G, A, L))
        codes = np.empty(O.codes_bytes(O.INT4, n), np.uint8)
        scales = np.empty(n // G, np.float32)

        def chunk(c):
            pos = O.slice_position(c, A, L)
            wc, ws = O.quantize(np.ascontiguousarray(x[c * m:(c + 1) * m]), O.INT4, G)
            codes[pos * m // 2:(pos + 1) * m // 2] = wc
            scales[pos * m // G:(pos + 1) * m // G] = ws

        F.pmap(chunk, range(P))
        F.same(f"GPU {g} reordered quantize", "codes", 0, to_host(qd[g][0]), codes)
        F.same(f"GPU {g} reordered quantize", "scales", 0, to_host(qd[g][1]), scales)
        ref.append((codes, scales))
        del x
    mid, out, sums = zq.reduce_two_hop([c for c, _ in qd], [s for _, s in qd], A, L, n, O.INT4, G,
                                       O.INT4, G, O.INT4, G, sums=True)
    zq.device_status()
    hmid = [(to_host(c), to_host(s)) for c, s in mid]
    hout = [(to_host(c), to_host(s)) for c, s in out]
    hsum = [to_host(s) for s in sums]

    def window(job):
        g, lo, hi = job
        a, l = divmod(g, L)
        w = hi - lo
        mids = []
        for a2 in range(A):  # hop 1 on node a2: its GPUs in order, slice position l*A + a
            off = (l * A + a) * m + lo
            part = [ref[a2 * L + l2] for l2 in range(L)]
            mc, ms, _ = O.reduce([F.code_slice(c, O.INT4, off, off + w) for c, _ in part],
                                 [s[off // G:(off + w) // G] for _, s in part], w, O.INT4, G,
                                 O.INT4, G)
            moff = a * m + lo  # in GPU (a2, l)'s hop-1 result
            gm = hmid[a2 * L + l]
            F.same(f"GPU {a2 * L + l} hop 1", "codes", moff, F.code_slice(gm[0], O.INT4, moff, moff + w), mc)
            F.same(f"GPU {a2 * L + l} hop 1", "scales", moff, gm[1][moff // G:(moff + w) // G], ms)
            mids.append((mc, ms))
        wc, ws, wsum = O.reduce([c for c, _ in mids], [s for _, s in mids], w, O.INT4, G, O.INT4, G,
                                want_sum=True)
        F.same(f"GPU {g} hop 2", "fp32 sums", lo, hsum[g][lo:hi], wsum)
        F.same(f"GPU {g} hop 2", "scales", lo, hout[g][1][lo // G:hi // G], ws)
        F.same(f"GPU {g} hop 2", "codes", lo, F.code_slice(hout[g][0], O.INT4, lo, hi), wc)
        return w

    total = sum(F.pmap(window, [(g, lo, hi) for g in range(P) for lo, hi in F.chunks(m)]))
    assert total == n
    print(f"\n[full-size parity] qgz_two_hop: {P} reordered quantizations ({P * n:,} elements), "
          f"{P} hop-1 results ({A * n:,}) and {P} final chunks ({n:,}) compared bit for bit on "
          f"{F.cores()} host cores in {time.time() - t0:.1f} s")
