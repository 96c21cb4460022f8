"""The chunked, multi-threaded oracle comparison used by the full-size GPU
parity tests (tests/fullsize.py), checked on the CPU: splitting a tensor into
chunks of whole blocks and running the oracle on them in parallel gives
exactly the whole-tensor oracle call's bytes, and a single flipped bit in the
compared output is caught."""
import numpy as np
import pytest

import oracle as O
import fullsize as F
from blockwise_quantized_zero_gb300 import inputs

N = 2 * F.CHUNK + 3 * 1024 + 77  # three chunks, the last one ragged with a partial block


def _x():
    return inputs.to_bf16_bits(inputs.normal_f32(N, 0.02, 123))


@pytest.mark.parametrize("fmt,G", [(O.INT6, 32), (O.INT2, 1024), (O.E4M3, 128)])
def test_chunked_quantize_equals_whole_call(fmt, G):
    x = _x()
    wc, ws = O.quantize(x, fmt, G, dtype=O.BF16)
    cc, cs = F.oracle_quantize_full(x, fmt, G, dtype=O.BF16)
    assert np.array_equal(cc, wc) and np.array_equal(F.bits(cs), F.bits(ws))
    y = O.dequantize(wc, ws, N, fmt, G, O.BF16)
    assert F.check_roundtrip("whole", x, O.BF16, fmt, G, wc, ws, y, O.BF16) == N


def test_flipped_bit_is_caught():
    x = _x()
    wc, ws = O.quantize(x, O.INT4, 128, dtype=O.BF16)
    y = O.dequantize(wc, ws, N, O.INT4, 128, O.BF16)
    rng = np.random.default_rng(5)
    for part in ("codes", "scales", "dequantized values"):
        c, s, yy = wc.copy(), ws.copy(), y.copy()
        target = {"codes": c, "scales": s.view(np.uint32), "dequantized values": yy}[part]
        i = int(rng.integers(target.size // 2, target.size))  # past the first chunk
        target[i] ^= 1
        with pytest.raises(AssertionError, match=part):
            F.check_roundtrip("planted", x, O.BF16, O.INT4, 128, c, s, yy, O.BF16)


def test_chunked_reduce_and_accumulate_equal_whole_calls():
    n = N - 77  # the reduce shards: several chunks, whole blocks
    shards = [O.quantize(inputs.laplace_f32(n, 1e-4, 9, stream=r), O.INT4, 128) for r in range(3)]
    wc, ws, wsum = O.reduce([c for c, _ in shards], [s for _, s in shards], n, O.INT4, 128, O.INT8,
                            256, want_sum=True)
    assert F.check_reduce("whole", shards, n, O.INT4, 128, O.INT8, 256, wc, ws, wsum) == n
    bad = wsum.copy()
    bad[n - 5] = np.nextafter(bad[n - 5], np.float32(1))
    with pytest.raises(AssertionError, match="fp32 sums"):
        F.check_reduce("planted", shards, n, O.INT4, 128, O.INT8, 256, wc, ws, bad)

    g = inputs.to_bf16_bits(inputs.normal_f32(n, 1e-3, 10))
    c0, s0 = np.zeros(n, np.uint8), np.zeros(n // 128, np.float32)
    c1, s1 = O.fp8_accumulate(c0, s0, g, 128, grad_dtype=O.BF16)
    F.fp8_accumulate_full(c0, s0, g, 128, grad_dtype=O.BF16)
    assert np.array_equal(c0, c1) and np.array_equal(F.bits(s0), F.bits(s1))
