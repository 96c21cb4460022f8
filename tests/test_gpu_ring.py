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


def test_ring_full_size_every_element_and_less_accurate(zq):
    """8 shards x 134,217,728 int4 G=128 (the qgZ reduce workload): the ring's
    fp32 sums, codes and scales equal the oracle's ring on every element (the
    oracle runs the ring on each chunk of whole blocks of the oracle-made
    shards: every hop works block by block), and on the first 16,777,216
    elements its error against the exact sum of the gradients exceeds the
    one-hop reduce's."""
    import time

    import torch

    import fullsize as F
    from blockwise_quantized_zero_gb300 import inputs

    t0 = time.time()
    N, n, G, M = 8, 134217728, 128, 1 << 24
    dc, ds, ref = [], [], []
    exact = np.zeros(M, np.float64)
    for r in range(N):
        x = inputs.gradient_shard_f32(n, shard=r)
        c, s = zq.quantize(torch.from_numpy(x).cuda(), O.INT4, G)
        ref.append(F.oracle_quantize_full(x, O.INT4, G))
        dc.append(c)
        ds.append(s)
        exact += x[:M]
        del x
    c, s, sm = zq.reduce_ring(dc, ds, n, O.INT4, G, O.INT4, G, sum_out=True)
    _, _, one = zq.reduce_quantized(dc, ds, n, O.INT4, G, O.INT4, G, sum_out=True)
    zq.device_status()
    hsm, hc, hs = to_host(sm), to_host(c), to_host(s)

    def chunk(span):
        lo, hi = span
        wc, ws, wsm = O.reduce_ring([F.code_slice(a, O.INT4, lo, hi) for a, _ in ref],
                                    [b[lo // G:hi // G] for _, b in ref], hi - lo, O.INT4, G,
                                    O.INT4, G, want_sum=True)
        F.same("ring", "fp32 sums", lo, hsm[lo:hi], wsm)
        F.same("ring", "scales", lo, hs[lo // G:hi // G], ws)
        F.same("ring", "codes", lo, F.code_slice(hc, O.INT4, lo, hi), wc)
        return hi - lo

    assert sum(F.pmap(chunk, F.chunks(n))) == n
    hone = to_host(one[:M])
    err_ring = float(np.sum((hsm[:M] - exact) ** 2))
    err_one = float(np.sum((hone - exact) ** 2))
    assert np.sqrt(err_ring) > 1.3 * np.sqrt(err_one)
    print(f"\n[full-size parity] ring_study: {n:,} ring outputs compared bit for bit on "
          f"{F.cores()} host cores in {time.time() - t0:.1f} s")
