"""The ring reduce-scatter's hops on the GPU (zq_reduce_ring through the C
ABI) against the oracle's ring, bit for bit (codes, scales and fp32 sums),
and the accuracy comparison with the one-hop reduce at full size."""
import numpy as np
import pytest

import oracle as O
from helpers import as_bits, bytes_dev, to_host

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


def _shards(N, n, fmt, G, seed):
    from blockwise_quantized_zero_gb300 import inputs

    xs = [inputs.laplace_f32(n, 1e-4 * (1 + r % 3), seed, stream=r) for r in range(N)]
    return xs, [O.quantize(x, fmt, G) for x in xs]


def _same(got, want, label):
    g, w = as_bits(got), as_bits(want)
    if not np.array_equal(g, w):
        bad = np.flatnonzero(g != w)
        raise AssertionError(f"{label}: {bad.size} differ, first at {bad[:6]}")


@pytest.mark.parametrize("N", [1, 2, 3, 8])
@pytest.mark.parametrize("fmt,G,fout,Gout", [(O.INT4, 128, O.INT4, 128), (O.INT8, 256, O.INT8, 32),
                                             (O.E4M3, 128, O.E4M3, 128), (O.INT2, 32, O.INT6, 64)])
def test_ring_matches_oracle(zq, N, fmt, G, fout, Gout):
    n = 9 * 1024 + 300  # several CTA tiles and a ragged tail
    _, q = _shards(N, n, fmt, G, seed=N * 10 + fmt)
    c, s, sm = zq.reduce_ring([bytes_dev(c) for c, _ in q], [bytes_dev(s) for _, s in q], n, fmt, G,
                              fout, Gout, sum_out=True)
    zq.device_status()
    wc, ws, wsm = O.reduce_ring([c for c, _ in q], [s for _, s in q], n, fmt, G, fout, Gout,
                                want_sum=True)
    _same(to_host(sm), wsm, "sums")
    _same(to_host(s), ws, "scales")
    _same(to_host(c), wc, "codes")


def test_ring_full_size_sampled_and_less_accurate(zq):
    """8 shards x 134,217,728 int4 G=128 (the qgZ reduce workload): the ring's
    sums and codes on sampled windows of whole blocks equal the oracle's ring
    on those windows, and its error against the exact sum of the gradients
    exceeds the one-hop reduce's."""
    import torch

    from blockwise_quantized_zero_gb300 import inputs

    N, n, G = 8, 134217728, 128
    dc, ds, hx = [], [], []
    for r in range(N):
        x = inputs.gradient_shard_f32(n, shard=r)
        xd = torch.from_numpy(x).cuda()
        c, s = zq.quantize(xd, O.INT4, G)
        dc.append(c)
        ds.append(s)
        del xd
        hx.append(x)
    c, s, sm = zq.reduce_ring(dc, ds, n, O.INT4, G, O.INT4, G, sum_out=True)
    _, _, one = zq.reduce_quantized(dc, ds, n, O.INT4, G, O.INT4, G, sum_out=True)
    zq.device_status()
    rng = np.random.default_rng(3)
    W = 4096
    starts = sorted({0, n - W} | set((rng.integers(0, (n - W) // 1024, 6) * 1024).tolist()))
    hsm, hone, hc, hs = to_host(sm), to_host(one), to_host(c), to_host(s)
    err_ring = err_one = ref = 0.0
    for lo in starts:
        q = [O.quantize(x[lo:lo + W], O.INT4, G) for x in hx]
        wc, ws, wsm = O.reduce_ring([a for a, _ in q], [b for _, b in q], W, O.INT4, G, O.INT4, G,
                                    want_sum=True)
        _same(hsm[lo:lo + W], wsm, f"sums at {lo}")
        _same(hs[lo // G:(lo + W) // G], ws, f"scales at {lo}")
        _same(hc[lo // 2:(lo + W) // 2], wc, f"codes at {lo}")
        exact = np.sum([x[lo:lo + W].astype(np.float64) for x in hx], axis=0)
        err_ring += float(np.sum((hsm[lo:lo + W] - exact) ** 2))
        err_one += float(np.sum((hone[lo:lo + W] - exact) ** 2))
        ref += float(np.sum(exact ** 2))
    assert np.sqrt(err_ring / ref) > 1.3 * np.sqrt(err_one / ref)
