"""zq_reduce_quantized_static, the reduce entry point that allocates nothing,
called through the C ABI.

It exists for callers that cannot allocate device memory (for instance code
whose device memory is owned by another allocator that has reserved most of
HBM) and still need a reduce over more shards than fit in kernel parameters:
its shard pointer table is a static device array shared by all calls. Its
results must be bit-identical to zq_reduce_quantized's, on consecutive calls
(the table keeps the previous call's entries), and to the definition beyond
64 shards, where zq_reduce_quantized refuses. This file is named to be
collected last.
"""
import ctypes

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
    return zq


def _shards(N, n, fmt, G, seed):
    from blockwise_quantized_zero_gb300 import inputs

    out = []
    for r in range(N):
        x = inputs.laplace_f32(n, 1e-4 * (1 + r % 7), seed, stream=r)
        out.append(O.quantize(x, fmt, G))
    return out


def _call(zq, entry, shards, n, fin, Gin, fout, Gout):
    """One reduce through the C ABI into freshly zeroed outputs (fp32 sums too)."""
    import torch

    codes = [bytes_dev(c) for c, _ in shards]
    scales = [bytes_dev(s) for _, s in shards]
    oc = torch.zeros(zq.codes_bytes(fout, n), dtype=torch.uint8, device="cuda")
    os_ = torch.zeros(zq.num_blocks(n, Gout), dtype=torch.float32, device="cuda")
    sm = torch.zeros(n, dtype=torch.float32, device="cuda")
    N = len(shards)
    cp = (ctypes.c_void_p * N)(*[c.data_ptr() for c in codes])
    sp = (ctypes.c_void_p * N)(*[s.data_ptr() for s in scales])
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = getattr(zq.lib(), entry)(cp, sp, N, n, fin, Gin, oc.data_ptr(), os_.data_ptr(), fout,
                                      Gout, sm.data_ptr(), st)
    assert status == 0, (entry, status)
    assert zq.lib().zq_device_status(st) == 0
    return to_host(oc), to_host(os_), to_host(sm)


def _same(a, b, label):
    for x, y, part in zip(a, b, ("codes", "scales", "sums")):
        assert np.array_equal(as_bits(x), as_bits(y)), f"{label}: {part} differ"


def test_static_reduce_equals_reduce_on_two_calls_in_a_row(zq):
    n = 5 * 1024 + 333  # ragged tail with a partial block
    first = (_shards(8, n, O.INT4, 128, seed=71), O.INT4, 128, O.INT8, 256)
    second = (_shards(3, n, O.E4M3, 64, seed=72), O.E4M3, 64, O.INT4, 128)
    for k, (sh, fin, Gin, fout, Gout) in enumerate((first, second)):
        want = _call(zq, "zq_reduce_quantized", sh, n, fin, Gin, fout, Gout)
        got = _call(zq, "zq_reduce_quantized_static", sh, n, fin, Gin, fout, Gout)
        _same(got, want, f"call {k}")


def test_static_reduce_beyond_64_shards_matches_the_definition(zq):
    n = 3 * 8192 + 1024 + 77  # several CTA tiles, a partial one and a ragged tail
    for k, N in enumerate((100, 65)):
        sh = _shards(N, n, O.INT4, 128, seed=80 + k)
        got = _call(zq, "zq_reduce_quantized_static", sh, n, O.INT4, 128, O.INT4, 128)
        wc, ws, wsum = O.reduce([c for c, _ in sh], [s for _, s in sh], n, O.INT4, 128, O.INT4,
                                128, want_sum=True)
        _same(got, (wc, ws, wsum), f"N={N}")


def test_static_reduce_at_the_shard_limit(zq):
    """ZQ_STATIC_MAX_SHARDS shards (every table slot, the last shard batch and
    the table's end) on a small ragged tensor, against the definition."""
    N, n = zq.STATIC_MAX_SHARDS, 1024 + 77
    sh = _shards(N, n, O.INT2, 32, seed=90)
    got = _call(zq, "zq_reduce_quantized_static", sh, n, O.INT2, 32, O.INT4, 64)
    wc, ws, wsum = O.reduce([c for c, _ in sh], [s for _, s in sh], n, O.INT2, 32, O.INT4, 64,
                            want_sum=True)
    _same(got, (wc, ws, wsum), f"N={N}")


def test_static_reduce_refuses_while_capturing(zq):
    """A call on a stream that is being captured returns ZQ_ERR_INVALID_ARG with
    nothing enqueued (its table copies would read the caller's host arrays again
    at every replay); the capture itself stays valid, and the next ordinary
    call works."""
    import torch

    n = 4096
    sh = _shards(3, n, O.INT4, 128, seed=95)
    codes = [bytes_dev(c) for c, _ in sh]
    scales = [bytes_dev(s) for _, s in sh]
    oc = torch.zeros(zq.codes_bytes(O.INT4, n), dtype=torch.uint8, device="cuda")
    os_ = torch.zeros(zq.num_blocks(n, 128), dtype=torch.float32, device="cuda")
    marker = torch.zeros(1, dtype=torch.float32, device="cuda")
    cp = (ctypes.c_void_p * 3)(*[c.data_ptr() for c in codes])
    sp = (ctypes.c_void_p * 3)(*[s.data_ptr() for s in scales])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
            status = zq.lib().zq_reduce_quantized_static(cp, sp, 3, n, O.INT4, 128, oc.data_ptr(),
                                                         os_.data_ptr(), O.INT4, 128, None, st)
            marker.add_(1.0)
    assert status == 1, status  # ZQ_ERR_INVALID_ARG
    g.replay()
    torch.cuda.synchronize()
    assert marker.item() == 1.0  # the rest of the capture replays
    assert int(oc.count_nonzero()) == 0 and int(os_.count_nonzero()) == 0  # nothing was enqueued
    got = zq.reduce_quantized_static(codes, scales, n, O.INT4, 128, O.INT4, 128)
    zq.device_status()
    wc, ws, _ = O.reduce([c for c, _ in sh], [s for _, s in sh], n, O.INT4, 128, O.INT4, 128)
    assert np.array_equal(to_host(got[0]), wc) and np.array_equal(as_bits(to_host(got[1])), as_bits(ws))
