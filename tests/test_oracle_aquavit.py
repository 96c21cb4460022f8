"""Pins of the oracle's Aquavit additions ([Aquavit] summary of the
implementation, Section 5.1-5.3, Eq. 6; readings R13 and R14 of the oracle):
the metadata-interleaved record layout and the ascending width schedule.

The layout is checked against hand-built byte streams and against the planar
codec it regroups; the schedule against its closed forms, the printed first
and last (b, G) pairs and a brute-force nearest-width search."""
import math

import numpy as np
import pytest

import oracle as O
import pins


def test_pins_hold_for_the_oracle():
    lib = O.load()
    for pin in (pins.pin_il_size, pins.pin_il_hand_records, pins.pin_il_is_a_regrouping,
                pins.pin_schedule_closed_forms, pins.pin_schedule_pick):
        pin(lib)


@pytest.mark.parametrize("fmt", [O.INT2, O.INT4, O.INT6, O.INT8])
@pytest.mark.parametrize("G", [32, 1024])
def test_interleaved_roundtrip_bound(fmt, G):
    """|x - D(Q(x))| <= s/2 (1 + 2^-22) per block, as for the planar codec."""
    n = 5 * G + 17
    x = (np.random.default_rng(fmt * 7 + G).standard_normal(n) * 0.02).astype(np.float32)
    rec = O.quantize_interleaved(x, fmt, G)
    y = O.dequantize_interleaved(rec, n, fmt, G, O.F32)
    _, scales = O.quantize(x, fmt, G)
    s = np.repeat(scales, G)[:n].astype(np.float64)
    assert np.all(np.abs(x.astype(np.float64) - y) <= s / 2 * (1 + 2.0 ** -22))


def test_e4m3_has_no_interleaved_form():
    with pytest.raises(ValueError):
        O.quantize_interleaved(np.zeros(256, np.float32), O.E4M3, 128)


def test_printed_mean_is_not_reproduced():
    """The page prints a mean of 5.79 bits over 1000 steps. The continuous
    schedule gives 5.74 and the nearest available widths 5.76: recorded here
    so that a change in either shows up."""
    g = pins.golden("aquavit_schedule.json")
    T, a, c = g["steps"], g["a"], g["c"]
    cont = math.fsum(O.aquavit_bpw(t, T, a, c) for t in range(T)) / T
    picked = math.fsum(O.aquavit_pick(O.aquavit_bpw(t, T, a, c))[2] for t in range(T)) / T
    assert f"{cont:.2f}" == "5.74" and f"{picked:.2f}" == "5.76"
    assert not g["mean_reproduced"] and g["mean_bpw_printed"] == "5.79"
