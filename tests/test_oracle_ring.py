"""The ring reduce-scatter that qgZ replaces ([ZeRO++] "QGZ keeps reductions in
full precision while sending quantized gradients"; reading R15 of the oracle):
pins of the oracle's ring, and the accuracy comparison the pages claim.

The pages say the ring's N sequential dequantize-add-requantize steps lose
precision and that qgZ's single requantization avoids it. Measured here with
the oracle on Laplace gradients (the qgZ workload's distribution): the fp32
result of each scheme against the exact (float64) sum of the unquantized
gradients."""
import numpy as np
import pytest

import oracle as O
import pins


def test_pins_hold_for_the_oracle():
    lib = O.load()
    for pin in (pins.pin_ring_small_n, pins.pin_ring_exact_sums, pins.pin_ring_requantizes_partials):
        pin(lib)


def _errors(N, fmt, G, n=16384, seed=0):
    r = np.random.default_rng([seed, N, fmt, G])
    xs = [r.laplace(0, 1e-4, n).astype(np.float32) for _ in range(N)]
    q = [O.quantize(x, fmt, G) for x in xs]
    exact = np.sum([x.astype(np.float64) for x in xs], axis=0)
    _, _, one = O.reduce([c for c, _ in q], [s for _, s in q], n, fmt, G, fmt, G, want_sum=True)
    _, _, ring = O.reduce_ring([c for c, _ in q], [s for _, s in q], n, fmt, G, fmt, G,
                               want_sum=True)
    rel = lambda y: float(np.sqrt(np.mean((y - exact) ** 2)) / np.sqrt(np.mean(exact ** 2)))  # noqa: E731
    return rel(one), rel(ring)


@pytest.mark.parametrize("fmt,G", [(O.INT4, 128), (O.INT8, 256)])
def test_ring_loses_precision_one_hop_does_not_grow(fmt, G):
    """The ring's relative RMS error exceeds the one-hop reduce's and grows
    with the number of hops; the one-hop error stays at the level of a single
    quantization of each input (it does not grow with N)."""
    res = {N: _errors(N, fmt, G) for N in (2, 4, 8, 16)}
    one2, ring2 = res[2]
    assert ring2 == one2  # two shards: no intermediate requantization
    for N in (4, 8, 16):
        one, ring = res[N]
        assert ring > 1.3 * one, (N, one, ring)
        assert one < 1.5 * one2, (N, one, one2)
    assert res[16][1] > res[8][1] > res[4][1]
