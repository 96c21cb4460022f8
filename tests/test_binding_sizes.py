"""The binding refuses buffers too small for the call before reaching the C
ABI (which takes raw pointers and cannot know buffer sizes). Checked on CPU
with stand-in tensor objects that only report their size."""
import pytest

import blockwise_quantized_zero_gb300 as zq


class FakeCuda:
    is_cuda = True

    def __init__(self, nbytes, elem=1):
        self._n, self._e = nbytes // elem, elem

    def is_contiguous(self):
        return True

    def numel(self):
        return self._n

    def element_size(self):
        return self._e


def test_need_accepts_enough_and_refuses_less():
    zq._need(FakeCuda(4096), 4096, "codes")
    zq._need(FakeCuda(8192, 4), 4096, "scales")
    with pytest.raises(ValueError, match="holds 4092 bytes"):
        zq._need(FakeCuda(4092), 4096, "codes")


def test_need_pair_uses_the_format_sizes():
    n, G = 1000, 128
    zq._need_pair(FakeCuda(zq.codes_bytes(zq.INT4, n)), FakeCuda(4 * zq.num_blocks(n, G), 4),
                  zq.INT4, n, G, "x")
    with pytest.raises(ValueError, match="x codes"):
        zq._need_pair(FakeCuda(zq.codes_bytes(zq.INT4, n) - 4), FakeCuda(4 * 8, 4),
                      zq.INT4, n, G, "x")
    with pytest.raises(ValueError, match="x scales"):
        zq._need_pair(FakeCuda(zq.codes_bytes(zq.INT4, n)), FakeCuda(4 * 7, 4), zq.INT4, n, G, "x")
    # an unknown format or block size needs nothing here: the C ABI reports it
    zq._need_pair(FakeCuda(0), FakeCuda(0, 4), 5, n, 48, "x")


def test_cpu_tensors_are_refused():
    class Cpu(FakeCuda):
        is_cuda = False

    with pytest.raises(ValueError, match="must be a CUDA tensor"):
        zq._need(Cpu(16), 16, "codes")
