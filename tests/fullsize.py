"""Every-element comparison of full-size GPU results with the oracle.

Blocks are independent, and with chunks of whole 1024-element tiles every
chunk's codes start on a 32-bit word boundary, so a tensor splits into
chunks that the oracle quantizes (dequantizes, reduces, accumulates) on its
own and that must reproduce the GPU's bytes for that chunk exactly. The
oracle's entry points keep no state between calls, and its foreign calls
release the interpreter lock, so the chunks run on every host core at once,
one thread each: the oracle itself stays the plain single-threaded C code.

The oracle's inputs are always the seeded host inputs (and, for a reduce or
a dequantize, codes the oracle made from them): nothing the GPU computed is
ever fed to the oracle. The GPU's outputs are copied to the host and compared
chunk by chunk, bit for bit.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as O

CHUNK = 1 << 20  # elements: a multiple of every block size and of the 1024-element tile


def cores() -> int:
    return len(os.sched_getaffinity(0))


def pmap(fn, items):
    """fn over items on every host core (threads), results in order."""
    items = list(items)
    with ThreadPoolExecutor(max(1, min(cores(), len(items)))) as ex:
        return list(ex.map(fn, items))


def chunks(n: int, chunk: int = CHUNK):
    return [(lo, min(n, lo + chunk)) for lo in range(0, n, chunk)]


def code_slice(codes: np.ndarray, fmt: int, lo: int, hi: int) -> np.ndarray:
    """The packed codes of elements [lo, hi) (lo a multiple of 32)."""
    start = lo * O.BITS[fmt] // 8
    return codes[start:start + O.codes_bytes(fmt, hi - lo)]


def bits(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _first_diff(a: np.ndarray, b: np.ndarray) -> int:
    d = np.flatnonzero(bits(a) != bits(b))
    return int(d[0]) if d.size else -1


def _fail(label: str, part: str, lo: int, a, b):
    i = _first_diff(a, b)
    raise AssertionError(f"{label}: {part} differ in the chunk at element {lo} (first at offset "
                         f"{i} of the {part}: GPU {bits(a)[i]!r}, oracle {bits(b)[i]!r})")


def same(label: str, part: str, lo: int, got: np.ndarray, want: np.ndarray):
    if got.shape != want.shape or not np.array_equal(bits(got), bits(want)):
        if got.shape != want.shape:
            raise AssertionError(f"{label}: {part} shapes {got.shape} vs {want.shape} at {lo}")
        _fail(label, part, lo, got, want)


def check_roundtrip(label: str, x: np.ndarray, dtype: int | None, fmt: int, G: int,
                    codes: np.ndarray, scales: np.ndarray, y: np.ndarray | None = None,
                    out_dtype: int | None = None) -> int:
    """Quantize every chunk of the host input with the oracle and compare with
    the GPU's codes and scales; then, if y is given, dequantize the oracle's
    codes to out_dtype and compare with the GPU's y. Returns the element count."""
    n = x.size
    assert codes.size == O.codes_bytes(fmt, n) and scales.size == O.num_blocks(n, G)

    def work(span):
        lo, hi = span
        wc, ws = O.quantize(np.ascontiguousarray(x[lo:hi]), fmt, G,
                            dtype=dtype if dtype == O.BF16 else None)
        same(label, "codes", lo, code_slice(codes, fmt, lo, hi), wc)
        same(label, "scales", lo, scales[lo // G:(hi + G - 1) // G], ws)
        if y is not None:
            wy = O.dequantize(wc, ws, hi - lo, fmt, G, out_dtype)
            same(label, "dequantized values", lo, y[lo:hi], wy)
        return hi - lo

    return sum(pmap(work, chunks(n)))


def oracle_quantize_full(x: np.ndarray, fmt: int, G: int, dtype: int | None = None):
    """(codes, scales) of a whole tensor, computed chunk by chunk in parallel
    (identical to one oracle call on the whole tensor: blocks are independent)."""
    n = x.size
    codes = np.empty(O.codes_bytes(fmt, n), np.uint8)
    scales = np.empty(O.num_blocks(n, G), np.float32)

    def work(span):
        lo, hi = span
        wc, ws = O.quantize(np.ascontiguousarray(x[lo:hi]), fmt, G, dtype=dtype)
        start = lo * O.BITS[fmt] // 8
        codes[start:start + wc.size] = wc
        scales[lo // G:lo // G + ws.size] = ws

    pmap(work, chunks(n))
    return codes, scales


def check_reduce(label: str, shards, n: int, fin: int, Gin: int, fout: int, Gout: int,
                 codes: np.ndarray, scales: np.ndarray, sums: np.ndarray | None = None) -> int:
    """The oracle's shard-ordered reduce of every chunk of the oracle-made
    shards [(codes, scales), ...] against the GPU's codes, scales and sums."""

    def work(span):
        lo, hi = span
        sc = [code_slice(c, fin, lo, hi) for c, _ in shards]
        ss = [s[lo // Gin:(hi + Gin - 1) // Gin] for _, s in shards]
        wc, ws, wsum = O.reduce(sc, ss, hi - lo, fin, Gin, fout, Gout, want_sum=sums is not None)
        if sums is not None:
            same(label, "fp32 sums", lo, sums[lo:hi], wsum)
        same(label, "scales", lo, scales[lo // Gout:(hi + Gout - 1) // Gout], ws)
        same(label, "codes", lo, code_slice(codes, fout, lo, hi), wc)
        return hi - lo

    return sum(pmap(work, chunks(n)))


def fp8_accumulate_full(codes: np.ndarray, scales: np.ndarray, grad: np.ndarray, G: int,
                        grad_dtype: int | None = None):
    """One oracle FP8 accumulate step over a whole main gradient, in place,
    chunk by chunk in parallel."""

    def work(span):
        lo, hi = span
        c, s = O.fp8_accumulate(codes[lo:hi], scales[lo // G:hi // G], grad[lo:hi], G,
                                grad_dtype=grad_dtype)
        codes[lo:hi] = c
        scales[lo // G:hi // G] = s

    pmap(work, chunks(codes.size))
