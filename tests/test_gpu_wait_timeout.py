"""The bounded device-side waits run out cleanly (no GPU fault, no hang).

The reduce kernels wait on shared-memory barriers for their bulk copies, each
wait bounded in time; a wait that runs out sets a device error word that
zq_device_status reports as ZQ_ERR_TIMEOUT. zq_wait_selftest runs those same
wait routines on a barrier that nothing completes, with a short limit, so the
timeout path is exercised without breaking any copy. Afterwards the error
word is clear and the next reduce is exact.
"""
import time

import numpy as np
import pytest

import oracle as O
from helpers import as_bits, bytes_dev, to_host

pytestmark = pytest.mark.gpu

TIMEOUT = 6  # ZQ_ERR_TIMEOUT


@pytest.fixture(scope="module")
def zq():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import blockwise_quantized_zero_gb300 as zq

    zq.lib()
    return zq


def test_wait_runs_out_and_is_reported(zq):
    import torch

    zq.device_status()  # start from a clear error word
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    zq.wait_selftest(5000)
    with pytest.raises(zq.ZQError) as e:
        zq.device_status()
    dt = time.perf_counter() - t0
    assert e.value.status == TIMEOUT
    assert 0.004 < dt < 1.0, dt  # the 5 ms limit, not the reduce's 2 s
    zq.device_status()  # reading the word cleared it


def test_reduce_after_a_timeout_is_clean_and_exact(zq):
    from blockwise_quantized_zero_gb300 import inputs

    zq.wait_selftest(1000)
    with pytest.raises(zq.ZQError):
        zq.device_status()
    n = 3 * 8192 + 1024 + 77
    sh = [O.quantize(inputs.laplace_f32(n, 1e-4, 60, stream=r), O.INT4, 128) for r in range(8)]
    oc, os_, sm = zq.reduce_quantized([bytes_dev(c) for c, _ in sh], [bytes_dev(s) for _, s in sh],
                                      n, O.INT4, 128, O.INT8, 256, sum_out=True)
    zq.device_status()
    wc, ws, wsum = O.reduce([c for c, _ in sh], [s for _, s in sh], n, O.INT4, 128, O.INT8, 256,
                            want_sum=True)
    assert np.array_equal(as_bits(to_host(sm)), as_bits(wsum))
    assert np.array_equal(as_bits(to_host(os_)), as_bits(ws))
    assert np.array_equal(to_host(oc), wc)
