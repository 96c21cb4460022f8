"""Pins of the oracle's qgZ hierarchy: tensor-slice reordering and the two-hop
reduce ([ZeRO++] sections "Two-hop communication prevents QGZ traffic from
multiplying across GPUs" and "Tensor-slice reordering fixes incorrect gradient
placement"; readings R10-R12 of the oracle).

The pages state the goal, not a formula: after the intra-node and the
inter-node reduction every GPU must hold the chunk assigned to it. The pins
check exactly that, and the arithmetic, against facts that do not come from
the oracle:
  * ownership: a gradient that is zero except for one chunk on one GPU ends
    up, after both hops, on the owner of that chunk and nowhere else;
  * exact sums: inputs built so that every quantization and requantization is
    exact give, after both hops, fp32 sums equal to the integer sum over all
    GPUs (computed with int64 here);
  * the reordering is a transposition: identity for one node or one GPU per
    node, and its own inverse with the roles of A and L exchanged.
"""
import numpy as np

import oracle as O
import pins

M = 1024  # chunk elements (one tile)


def test_reordering_is_the_chunk_grid_transpose():
    for A, L in ((1, 4), (4, 1), (1, 1)):
        assert [O.slice_position(c, A, L) for c in range(A * L)] == list(range(A * L))
    for A, L in ((2, 2), (2, 4), (4, 2), (3, 5)):
        P = A * L
        pos = [O.slice_position(c, A, L) for c in range(P)]
        assert sorted(pos) == list(range(P))  # a permutation
        back = [O.slice_position(p, L, A) for p in pos]  # transpose of the transpose
        assert back == list(range(P))
    # two nodes of two GPUs: the middle chunks trade places, the outer ones stay
    assert [O.slice_position(c, 2, 2) for c in range(4)] == [0, 2, 1, 3]


def test_pins_hold_for_the_oracle():
    lib = O.load()
    for pin in (pins.pin_reordered_quantize_identity, pins.pin_two_hop_ownership,
                pins.pin_two_hop_exact_sums, pins.pin_two_hop_order):
        pin(lib)


def test_pins_catch_a_wrong_hierarchy():
    """The ownership pin is sharp: with the reordering left out (chunks kept in
    place), chunks land on the wrong GPU for A, L > 1."""
    A, L = 2, 4
    P, n = A * L, A * L * M
    g_star, c_star = 0, 1
    xs = [np.zeros(n, np.float32) for _ in range(P)]
    xs[g_star][c_star * M:(c_star + 1) * M] = 1.0
    q = [O.quantize(x, O.INT4, 128) for x in xs]  # no reordering
    _, out, _ = O.reduce_two_hop([c for c, _ in q], [s for _, s in q], A, L, n, O.INT4, 128,
                                 O.INT4, 128, O.INT4, 128)
    owners = [g for g in range(P) if np.any(out[g][1] != 0)]
    assert owners != [c_star]
