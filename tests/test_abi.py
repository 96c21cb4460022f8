"""The C ABI without a GPU: libzq.so loads, exports every symbol declared in
include/zq.h, and rejects every bad argument before touching the device."""
import ctypes
import os
import re

import pytest

import blockwise_quantized_zero_gb300 as zq
import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zq.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, ALIAS = 0, 1, 2, 3, 4
BASE = 0x7F0000000000  # fake device addresses: never dereferenced by these calls


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zq_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def L():
    return zq.lib()


def test_header_declares_the_entry_points():
    names = declared_functions()
    for f in ("zq_quantize", "zq_dequantize", "zq_reduce_quantized", "zq_fp8_accumulate",
              "zq_codes_bytes", "zq_num_blocks", "zq_status_string", "zq_last_cuda_error",
              "zq_device_status"):
        assert f in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_size_helpers_match_the_oracle(L):
    for fmt in zq.FORMATS:
        for n in (0, 1, 31, 32, 33, 1000, 1 << 20, 67108864 + 5):
            assert zq.codes_bytes(fmt, n) == O.codes_bytes(fmt, n)
    for G in zq.BLOCK_SIZES:
        for n in (0, 1, G - 1, G, G + 1, 855638016):
            assert zq.num_blocks(n, G) == O.num_blocks(n, G)
    assert zq.codes_bytes(3, 10) == 0 and zq.codes_bytes(zq.INT4, -1) == 0
    assert zq.num_blocks(10, 48) == 0 and zq.num_blocks(-1, 32) == 0


def test_status_strings(L):
    for s in range(7):
        assert L.zq_status_string(s)
    assert L.zq_last_cuda_error() == 0


def q(L, src=BASE, dt=zq.BF16, n=4096, fmt=zq.INT8, G=256, codes=BASE + (1 << 24),
      scales=BASE + (1 << 26)):
    return L.zq_quantize(src, dt, n, fmt, G, codes, scales, None)


def test_quantize_argument_errors(L):
    assert q(L, fmt=3) == UNSUPPORTED
    assert q(L, dt=7) == UNSUPPORTED
    assert q(L, n=-1) == INVALID
    assert q(L, G=48) == INVALID and q(L, G=16) == INVALID and q(L, G=2048) == INVALID
    assert q(L, n=0, src=None, codes=None, scales=None) == OK  # empty: nothing to do
    assert q(L, src=None) == INVALID and q(L, codes=None) == INVALID and q(L, scales=None) == INVALID
    assert q(L, src=BASE + 8) == MISALIGNED and q(L, codes=BASE + (1 << 24) + 4) == MISALIGNED
    assert q(L, scales=BASE + (1 << 26) + 2) == MISALIGNED
    assert q(L, codes=BASE + 4096) == ALIAS  # codes inside the 8 KiB source
    assert q(L, scales=BASE + (1 << 24) + 1024) == ALIAS  # scales inside the codes


def test_dequantize_argument_errors(L):
    c, s, d = BASE, BASE + (1 << 24), BASE + (1 << 26)
    assert L.zq_dequantize(c, s, 4096, 5, 256, d, zq.BF16, None) == UNSUPPORTED
    assert L.zq_dequantize(c, s, 4096, zq.INT4, 256, d, 9, None) == UNSUPPORTED
    assert L.zq_dequantize(c, s, -5, zq.INT4, 256, d, zq.BF16, None) == INVALID
    assert L.zq_dequantize(c, s, 4096, zq.INT4, 100, d, zq.BF16, None) == INVALID
    assert L.zq_dequantize(None, s, 4096, zq.INT4, 256, d, zq.BF16, None) == INVALID
    assert L.zq_dequantize(c, s, 4096, zq.INT4, 256, d + 16 + 8, zq.BF16, None) == MISALIGNED
    assert L.zq_dequantize(c, s, 4096, zq.INT4, 256, c + 512, zq.BF16, None) == ALIAS
    assert L.zq_dequantize(c, s, 0, zq.INT4, 256, d, zq.BF16, None) == OK


def test_reduce_argument_errors(L):
    N, n = 4, 4096
    cp = (ctypes.c_void_p * N)(*[BASE + i * (1 << 20) for i in range(N)])
    sp = (ctypes.c_void_p * N)(*[BASE + (1 << 28) + i * (1 << 20) for i in range(N)])
    oc, os_, sm = BASE + (1 << 30), BASE + (1 << 31), BASE + (1 << 32)

    def r(**kw):
        a = dict(codes=cp, scales=sp, N=N, n=n, fin=zq.INT4, Gin=128, oc=oc, os=os_, fout=zq.INT4,
                 Gout=128, sm=sm)
        a.update(kw)
        return L.zq_reduce_quantized(a["codes"], a["scales"], a["N"], a["n"], a["fin"], a["Gin"],
                                     a["oc"], a["os"], a["fout"], a["Gout"], a["sm"], None)

    assert r(fin=1) == UNSUPPORTED and r(fout=0x49) == UNSUPPORTED
    assert r(N=0) == INVALID and r(N=65) == INVALID
    assert r(Gin=2048) == INVALID and r(Gout=8) == INVALID and r(n=-1) == INVALID
    assert r(n=0) == OK
    assert r(codes=None) == INVALID and r(oc=None) == INVALID
    bad = (ctypes.c_void_p * N)(*([BASE] + [None] * (N - 1)))
    assert r(codes=bad) == INVALID
    mis = (ctypes.c_void_p * N)(*[BASE + i * (1 << 20) + (8 if i == 2 else 0) for i in range(N)])
    assert r(codes=mis) == MISALIGNED
    assert r(sm=sm + 4) == MISALIGNED
    assert r(oc=BASE + 64) == ALIAS  # output codes on top of shard 0
    assert r(sm=BASE + (1 << 28) + 16) == ALIAS  # sum on top of shard 0's scales
    assert r(os=oc + 16) == ALIAS


def test_static_reduce_shard_limit(L):
    """zq_reduce_quantized_static takes up to ZQ_STATIC_MAX_SHARDS shards and
    refuses more before any work (n = 0 stops after the argument checks)."""
    N = zq.STATIC_MAX_SHARDS + 1
    cp = (ctypes.c_void_p * N)(*[BASE + i * (1 << 20) for i in range(N)])
    sp = (ctypes.c_void_p * N)(*[BASE + (1 << 31) + i * (1 << 20) for i in range(N)])
    oc, os_, sm = BASE + (1 << 33), BASE + (1 << 34), BASE + (1 << 35)

    def r(entry, nshards, n):
        return getattr(L, entry)(cp, sp, nshards, n, zq.INT4, 128, oc, os_, zq.INT4, 128, sm, None)

    assert r("zq_reduce_quantized_static", N, 4096) == INVALID
    assert r("zq_reduce_quantized_static", 0, 4096) == INVALID
    assert r("zq_reduce_quantized_static", N - 1, 0) == OK
    assert r("zq_reduce_quantized_static", 65, 0) == OK
    assert r("zq_reduce_quantized", 65, 0) == INVALID


def test_fp8_accumulate_argument_errors(L):
    c, s, g = BASE, BASE + (1 << 24), BASE + (1 << 26)
    assert L.zq_fp8_accumulate(c, s, g, 5, 4096, 128, None) == UNSUPPORTED
    assert L.zq_fp8_accumulate(c, s, g, zq.BF16, 4096, 100, None) == INVALID
    assert L.zq_fp8_accumulate(c, s, g, zq.BF16, -1, 128, None) == INVALID
    assert L.zq_fp8_accumulate(None, s, g, zq.BF16, 4096, 128, None) == INVALID
    assert L.zq_fp8_accumulate(c, s, g + 4, zq.BF16, 4096, 128, None) == MISALIGNED
    assert L.zq_fp8_accumulate(c, s, c + 1024, zq.BF16, 4096, 128, None) == ALIAS
    assert L.zq_fp8_accumulate(c, c + 2048, g, zq.BF16, 4096, 128, None) == ALIAS
    assert L.zq_fp8_accumulate(c, s, g, zq.BF16, 0, 128, None) == OK


def test_interleaved_size_matches_the_oracle(L):
    for fmt in (zq.INT2, zq.INT4, zq.INT6, zq.INT8):
        for G in zq.BLOCK_SIZES:
            for n in (0, 1, G - 1, G, G + 1, 3 * G, 67108864 + 5):
                assert zq.interleaved_bytes(fmt, n, G) == O.il_bytes(fmt, n, G), (fmt, G, n)
    assert zq.interleaved_bytes(zq.E4M3, 4096, 128) == 0 and O.il_bytes(O.E4M3, 4096, 128) == -1
    assert zq.interleaved_bytes(zq.INT4, 4096, 48) == 0 and zq.interleaved_bytes(zq.INT4, -1, 32) == 0


def test_interleaved_argument_errors(L):
    src, rec, dst = BASE, BASE + (1 << 24), BASE + (1 << 26)
    qi = lambda **k: L.zq_quantize_interleaved(k.get("src", src), k.get("dt", zq.BF16),  # noqa: E731
                                               k.get("n", 4096), k.get("fmt", zq.INT4),
                                               k.get("G", 128), k.get("rec", rec), None)
    assert qi(fmt=zq.E4M3) == UNSUPPORTED and qi(fmt=3) == UNSUPPORTED and qi(dt=7) == UNSUPPORTED
    assert qi(n=-1) == INVALID and qi(G=48) == INVALID
    assert qi(n=0, src=None, rec=None) == OK
    assert qi(src=None) == INVALID and qi(rec=None) == INVALID
    assert qi(src=src + 8) == MISALIGNED and qi(rec=rec + 4) == MISALIGNED
    assert qi(rec=src + 4096) == ALIAS  # records inside the 8 KiB source
    di = lambda **k: L.zq_dequantize_interleaved(k.get("rec", rec), k.get("n", 4096),  # noqa: E731
                                                 k.get("fmt", zq.INT4), k.get("G", 128),
                                                 k.get("dst", dst), k.get("dt", zq.BF16), None)
    assert di(fmt=zq.E4M3) == UNSUPPORTED and di(dt=9) == UNSUPPORTED
    assert di(n=-5) == INVALID and di(G=100) == INVALID and di(rec=None) == INVALID
    assert di(dst=dst + 8) == MISALIGNED and di(dst=rec + 1024) == ALIAS
    assert di(n=0) == OK


def test_aquavit_schedule_matches_the_oracle(L):
    """Host-only arithmetic: the library's schedule and pair choice against the
    oracle's for the pages' default and two other settings, every step."""
    for a, c, T in ((0.9, 5.0, 1000), (0.5, 2.0, 300), (2.0, 9.0, 77)):
        for t in range(T + 1):
            fmt, G, want, width = zq.aquavit_schedule(t, T, a, c)
            b, oG, ow = O.aquavit_pick(O.aquavit_bpw(t, T, a, c))
            assert (fmt, G, width) == (b, oG, ow), (a, c, T, t)
            assert want == O.aquavit_bpw(t, T, a, c)


def test_aquavit_schedule_argument_errors(L):
    f, G = ctypes.c_int(0), ctypes.c_int64(0)
    s = lambda t, T, a=0.9, c=5.0, fp=ctypes.byref(f), gp=ctypes.byref(G): \
        L.zq_aquavit_schedule(t, T, a, c, fp, gp, None, None)  # noqa: E731
    assert s(0, 1000) == OK and (f.value, G.value) == (zq.INT2, 1024)
    assert s(1000, 1000) == OK and (f.value, G.value) == (zq.INT6, 32)
    assert s(-1, 10) == INVALID and s(11, 10) == INVALID and s(0, 0) == INVALID
    assert s(0, 10, a=0.0) == INVALID and s(0, 10, c=-1.0) == INVALID
    assert s(0, 10, a=float("nan")) == INVALID and s(0, 10, c=float("inf")) == INVALID
    assert s(0, 10, fp=None) == INVALID and s(0, 10, gp=None) == INVALID


def test_reduce_ring_argument_errors(L):
    N, n = 4, 4096
    cp = (ctypes.c_void_p * N)(*[BASE + i * (1 << 20) for i in range(N)])
    sp = (ctypes.c_void_p * N)(*[BASE + (1 << 28) + i * (1 << 20) for i in range(N)])
    oc, os_, sm = BASE + (1 << 30), BASE + (1 << 31), BASE + (1 << 32)
    pc = (ctypes.c_void_p * 2)(BASE + (1 << 33), BASE + (1 << 33) + (1 << 20))
    ps = (ctypes.c_void_p * 2)(BASE + (1 << 34), BASE + (1 << 34) + (1 << 20))

    def r(**kw):
        a = dict(N=N, n=n, fmt=zq.INT4, G=128, pc=pc, ps=ps, fout=zq.INT4, Gout=128, sm=sm)
        a.update(kw)
        return L.zq_reduce_ring(cp, sp, a["N"], a["n"], a["fmt"], a["G"], a["pc"], a["ps"], oc, os_,
                                a["fout"], a["Gout"], a["sm"], None)

    assert r(fmt=5) == UNSUPPORTED and r(N=0) == INVALID and r(N=65) == INVALID
    assert r(G=48) == INVALID and r(n=-1) == INVALID and r(n=0) == OK
    assert r(pc=None) == INVALID and r(ps=None) == INVALID  # three or more shards need partials
    bad = (ctypes.c_void_p * 2)(BASE + (1 << 33) + 4, BASE + (1 << 33) + (1 << 20))
    assert r(pc=bad) == MISALIGNED
    onto_input = (ctypes.c_void_p * 2)(BASE + (1 << 20), BASE + (1 << 33) + (1 << 20))
    assert r(pc=onto_input) == ALIAS
    same = (ctypes.c_void_p * 2)(BASE + (1 << 33), BASE + (1 << 33))
    assert r(pc=same) == ALIAS
    onto_out = (ctypes.c_void_p * 2)(oc, BASE + (1 << 33) + (1 << 20))
    assert r(pc=onto_out) == ALIAS


def test_wait_selftest_limit_checked_before_the_device(L):
    """The wait self-test accepts 1 .. 100000 microseconds; other limits are
    refused before anything is enqueued (no device needed to see that)."""
    for bad in (0, -1, 100001, 1 << 40):
        assert L.zq_wait_selftest(bad, None) == INVALID


def test_gemm_dequant_argument_errors(L):
    """zq_gemm_dequant refuses bad formats, output types, shapes, alignment and
    overlap before touching the device; empty problems enqueue nothing."""
    x, c, s, y = BASE, BASE + (1 << 30), BASE + (2 << 30), BASE + (3 << 30)
    g = L.zq_gemm_dequant
    g.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                  ctypes.c_void_p]
    assert g(x, 128, 512, c, s, 3, 128, 256, y, O.F32, None) == UNSUPPORTED
    assert g(x, 128, 512, c, s, O.INT8, 128, 256, y, O.F16, None) == UNSUPPORTED
    assert g(x, 0, 512, c, s, O.INT8, 128, 256, y, O.F32, None) == OK
    assert g(x, 128, 512, c, s, O.INT8, 128, 0, y, O.F32, None) == OK
    assert g(x, 128, 500, c, s, O.INT8, 128, 256, y, O.F32, None) == INVALID   # K % 64
    assert g(x, 128, 512, c, s, O.INT8, 128, 250, y, O.F32, None) == INVALID   # N % 64
    assert g(x, 128, 64, c, s, O.INT8, 128, 256, y, O.F32, None) == INVALID    # G does not divide K
    assert g(x, 128, 512, c, s, O.INT8, 48, 256, y, O.F32, None) == INVALID    # block size
    assert g(x, -1, 512, c, s, O.INT8, 128, 256, y, O.F32, None) == INVALID
    assert g(None, 128, 512, c, s, O.INT8, 128, 256, y, O.F32, None) == INVALID
    assert g(x + 8, 128, 512, c, s, O.INT8, 128, 256, y, O.F32, None) == MISALIGNED
    assert g(x, 128, 512, c, s, O.INT8, 128, 256, x + 4096, O.F32, None) == ALIAS
    assert g(x, 128, 512, c, s, O.INT8, 128, 256, c + 64, O.BF16, None) == ALIAS


def test_gemm_plan(L):
    """zq_gemm_plan refuses bad sizes and null outputs; a problem with
    thousands of rows gets an unsplit 256-row tile, one with a hundred rows
    and a long K a 128-row tile with K split over a cluster. (Without a
    device the plan uses a default SM count; the choice is the same.)"""
    p = L.zq_gemm_plan
    I = ctypes.c_int
    p.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(I), ctypes.POINTER(I),
                  ctypes.POINTER(I)]
    bm, bn, sp = I(), I(), I()
    out = (ctypes.byref(bm), ctypes.byref(bn), ctypes.byref(sp))
    assert p(128, 250, 512, *out) == INVALID
    assert p(128, 256, 500, *out) == INVALID
    assert p(-1, 256, 512, *out) == INVALID
    assert p(128, 256, 512, None, out[1], out[2]) == INVALID
    assert p(4096, 8192, 8192, *out) == OK and (bm.value, bn.value, sp.value) == (256, 256, 1)
    assert p(128, 8192, 8192, *out) == OK and bm.value == 128 and sp.value in (2, 4, 8)
    assert p(1, 64, 64, *out) == OK and (bm.value, bn.value, sp.value) == (128, 64, 1)


def _plan_model(M, N, K, sms, wave):
    """The tile cost model of zq_gemm_dequant as its source comment states it:
    waves x (k-blocks a CTA x time a k-block) + fixed time, over the unsplit
    persistent shapes and, up to 512 rows, split-K over clusters of 2, 4, 8."""
    kb = K // 64
    best, plan = float("inf"), (128, 64, 1)
    for bm, bn, t in ((256, 256, 0.885), (256, 128, 0.60), (128, 128, 0.49), (128, 64, 0.42)):
        if N % bn:
            continue
        tiles = -(-M // bm) * (N // bn)
        cost = -(-tiles // sms) * (kb * t) + 3.0
        if cost < best:
            best, plan = cost, (bm, bn, 1)
    if M <= 512:
        for bn, t in ((256, 0.664), (128, 0.49)):
            if N % bn:
                continue
            tiles = -(-M // 128) * (N // bn)
            for cs in (2, 4, 8):
                if kb < 4 * cs:
                    continue
                cost = -(-(tiles * cs) // wave(cs)) * (kb / cs * t + 11.0)
                if cost < best:
                    best, plan = cost, (128, bn, cs)
    return plan


def test_gemm_plan_follows_the_cost_model(L):
    """Without a device the launcher plans with its fallback SM count (148)
    and cluster waves (148 // cs * cs); its choice must be the documented cost
    model's on a spread of shapes (few tokens to large problems, every tile
    and split)."""
    I = ctypes.c_int
    p = L.zq_gemm_plan
    p.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(I), ctypes.POINTER(I),
                  ctypes.POINTER(I)]
    bm, bn, sp = I(), I(), I()
    checked = set()
    for M in (1, 16, 77, 128, 200, 256, 300, 512, 513, 1024, 2148, 4096, 8192):
        for N in (64, 192, 512, 1024, 1536, 2560, 4096, 8192, 28672):
            for K in (64, 512, 2048, 8192, 28672):
                assert p(M, N, K, ctypes.byref(bm), ctypes.byref(bn), ctypes.byref(sp)) == OK
                want = _plan_model(M, N, K, 148, lambda cs: 148 // cs * cs)
                assert (bm.value, bn.value, sp.value) == want, (M, N, K, want)
                checked.add(want)
    assert {(256, 256, 1), (256, 128, 1), (128, 128, 1), (128, 64, 1)} <= checked
    assert {s for _, _, s in checked} >= {1, 2, 4, 8}


def test_quantize_multi_argument_errors(L):
    """zq_quantize_multi: bad format / type, negative counts and sizes, null,
    misaligned and overlapping buffers are refused before any work."""
    def call(srcs, ns, codes, scales, fmt=O.INT8, dt=O.F16, G=256, count=None):
        k = len(srcs) if count is None else count
        arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)  # noqa: E731
        return L.zq_quantize_multi(arr(srcs), (ctypes.c_int64 * max(1, len(ns)))(*ns), k, dt, fmt, G,
                                   arr(codes), arr(scales), None)

    s0, s1 = BASE, BASE + (1 << 24)
    c0, c1 = BASE + (2 << 24), BASE + (3 << 24)
    k0, k1 = BASE + (4 << 24), BASE + (5 << 24)
    assert call([s0], [1024], [c0], [k0], fmt=3) == UNSUPPORTED
    assert call([s0], [1024], [c0], [k0], dt=7) == UNSUPPORTED
    assert call([s0], [1024], [c0], [k0], count=-1) == INVALID
    assert call([s0], [1024], [c0], [k0], count=0) == OK
    assert call([s0], [1024], [c0], [k0], G=100) == INVALID
    assert call([s0, s1], [1024, -5], [c0, c1], [k0, k1]) == INVALID
    assert call([s0, None], [1024, 8], [c0, c1], [k0, k1]) == INVALID
    assert call([s0, 0], [1024, 0], [c0, 0], [k0, 0]) != MISALIGNED  # empty tensors: pointers ignored
    assert call([s0, s1 + 8], [1024, 1024], [c0, c1], [k0, k1]) == MISALIGNED
    assert call([s0, s1], [1024, 1024], [c0, c0 + 512], [k0, k1]) == ALIAS   # outputs overlap
    assert call([s0, s1], [1024, 1024], [c0, s0], [k0, k1]) == ALIAS         # output on an input
    assert call([s0, s1], [1024, 1024], [c0, c1], [k0, c1 + 128]) == ALIAS   # scales on codes
    assert call([s0, s0], [1024, 1024], [c0, c1], [k0, k1]) != ALIAS         # shared input is fine


def test_dequantize_multi_argument_errors(L):
    def call(codes, scales, ns, dsts, fmt=O.INT8, dt=O.BF16, G=256, count=None):
        k = len(ns) if count is None else count
        arr = lambda xs: (ctypes.c_void_p * max(1, len(xs)))(*xs)  # noqa: E731
        return L.zq_dequantize_multi(arr(codes), arr(scales), (ctypes.c_int64 * max(1, len(ns)))(*ns), k,
                                     fmt, G, arr(dsts), dt, None)

    c0, c1 = BASE, BASE + (1 << 24)
    s0, s1 = BASE + (2 << 24), BASE + (3 << 24)
    d0, d1 = BASE + (4 << 24), BASE + (5 << 24)
    assert call([c0], [s0], [1024], [d0], fmt=3) == UNSUPPORTED
    assert call([c0], [s0], [1024], [d0], dt=9) == UNSUPPORTED
    assert call([c0], [s0], [1024], [d0], count=-2) == INVALID
    assert call([c0], [s0], [1024], [d0], count=0) == OK
    assert call([c0, c1], [s0, s1], [1024, -1], [d0, d1]) == INVALID
    assert call([c0, c1], [s0, s1], [1024, 1024], [d0, d1 + 4]) == MISALIGNED
    assert call([c0, c1], [s0, s1], [1024, 1024], [d0, d0 + 1024]) == ALIAS   # outputs overlap
    assert call([c0, c1], [s0, s1], [1024, 1024], [d0, c1]) == ALIAS          # output on codes
