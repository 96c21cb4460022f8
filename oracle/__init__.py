"""Oracle for the blockwise quantize / pack / dequantize / reduce path.

TEST INFRASTRUCTURE, NOT PRODUCT CODE. Only the test suite, the package smoke
check and the benchmark's CPU-baseline leg may import this package. The
product library never loads it, and this package never loads the product.

The arithmetic lives in ``zq_oracle.c`` (plain single-threaded C, compiled
with ``-O2 -ffp-contract=off`` so that every binary32 operation is rounded
once, as written). This module only compiles it, loads it with ctypes and
marshals numpy arrays. Parity status of every function is stated in
``zq_oracle.c``'s header and in the tests that pin it.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "zq_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD_DIR, "libzq_oracle.so")

# gcc flags: IEEE binary32 arithmetic with no contraction into FMA and no
# value-changing optimisations; the same flags on x86-64 and aarch64.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]

F32, F16, BF16 = 0, 1, 2
INT2, INT4, INT6, INT8, E4M3 = 2, 4, 6, 8, 0x48
BITS = {INT2: 2, INT4: 4, INT6: 6, INT8: 8, E4M3: 8}

# Outputs are pre-filled with this byte (and scales with NaN) so that a byte
# the oracle forgets to write shows up in the checks.
GARBAGE = 0xA5

_lock = threading.Lock()
_lib = None


def build(src: str = _SRC, out: str = _LIB, extra_flags=()) -> str:
    """Compile ``src`` into the shared library ``out`` with gcc; return ``out``."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _stale() -> bool:
    return not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)


def _declare(lib):
    i64, i32, u32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_uint32, ctypes.c_void_p
    lib.orc_codes_bytes.argtypes = [i32, i64]
    lib.orc_codes_bytes.restype = i64
    lib.orc_num_blocks.argtypes = [i64, i64]
    lib.orc_num_blocks.restype = i64
    for name in ("orc_f16_decode", "orc_bf16_decode", "orc_e4m3_decode"):
        getattr(lib, name).argtypes = [u32]
        getattr(lib, name).restype = ctypes.c_float
    for name in ("orc_f16_encode", "orc_bf16_encode", "orc_e4m3_encode"):
        getattr(lib, name).argtypes = [ctypes.c_float]
        getattr(lib, name).restype = u32
    lib.orc_quantize.argtypes = [vp, i32, i64, i32, i64, vp, vp]
    lib.orc_dequantize.argtypes = [vp, vp, i64, i32, i64, vp, i32]
    lib.orc_reduce.argtypes = [vp, vp, i32, i64, i32, i64, vp, vp, i32, i64, vp]
    lib.orc_fp8_accumulate.argtypes = [vp, vp, vp, i32, i64, i64]
    lib.orc_quantize_reordered.argtypes = [vp, i32, i64, i32, i64, i32, i32, vp, vp]
    lib.orc_reduce_two_hop.argtypes = [vp, vp, i32, i32, i64, i32, i64, vp, vp, i32, i64, vp, vp,
                                       i32, i64, vp]
    lib.orc_il_bytes.argtypes = [i32, i64, i64]
    lib.orc_il_bytes.restype = i64
    lib.orc_quantize_interleaved.argtypes = [vp, i32, i64, i32, i64, vp]
    lib.orc_dequantize_interleaved.argtypes = [vp, i64, i32, i64, vp, i32]
    lib.orc_aquavit_bpw.argtypes = [i64, i64, ctypes.c_double, ctypes.c_double]
    lib.orc_aquavit_bpw.restype = ctypes.c_double
    lib.orc_aquavit_pick.argtypes = [ctypes.c_double, ctypes.POINTER(i32), ctypes.POINTER(i64)]
    lib.orc_aquavit_pick.restype = ctypes.c_double
    lib.orc_reduce_ring.argtypes = [vp, vp, i32, i64, i32, i64, vp, vp, vp, vp, i32, i64, vp]
    lib.orc_reduce_ring.restype = i32
    lib.orc_encode_n.argtypes = [i32, vp, i64, vp]
    lib.orc_decode_n.argtypes = [i32, vp, i64, vp]
    lib.orc_encode_n.restype = i32
    lib.orc_decode_n.restype = i32
    lib.orc_gemm_dequant.argtypes = [vp, i64, i64, vp, vp, i32, i64, i64, vp, vp, i64, vp, vp]
    lib.orc_gemm_dequant.restype = i32
    for name in ("orc_quantize", "orc_dequantize", "orc_reduce", "orc_fp8_accumulate",
                 "orc_quantize_interleaved", "orc_dequantize_interleaved"):
        getattr(lib, name).restype = i32
    return lib


def load(path: str | None = None):
    """Load the compiled oracle (building it first if it is missing or stale)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            if _stale():
                build()
            _lib = _declare(ctypes.CDLL(_LIB))
    return _lib


# ---------------------------------------------------------------------------
# numpy conveniences. 16-bit floats travel as uint16 bit patterns (bf16 has no
# numpy dtype); fp16 arrays may also be passed as np.float16.
# ---------------------------------------------------------------------------

def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _dtype_code(a: np.ndarray, dtype: int | None) -> int:
    if dtype is not None:
        return dtype
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float16:
        return F16
    raise ValueError("pass dtype= for uint16 (bf16/f16) bit patterns")


def codes_bytes(fmt: int, n: int, lib=None) -> int:
    return int((lib or load()).orc_codes_bytes(fmt, n))


def num_blocks(n: int, G: int, lib=None) -> int:
    return int((lib or load()).orc_num_blocks(n, G))


def quantize(x: np.ndarray, fmt: int, G: int, dtype: int | None = None, lib=None):
    """Return (codes uint8[codes_bytes], scales float32[num_blocks])."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    n = x.size
    codes = np.full(codes_bytes(fmt, n, lib), GARBAGE, dtype=np.uint8)
    scales = np.full(max(num_blocks(n, G, lib), 0), np.nan, dtype=np.float32)
    rc = lib.orc_quantize(_ptr(x), _dtype_code(x, dtype), n, fmt, G, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return codes, scales


_OUT_NP = {F32: np.float32, F16: np.uint16, BF16: np.uint16}


def dequantize(codes: np.ndarray, scales: np.ndarray, n: int, fmt: int, G: int, out_dtype: int,
               lib=None) -> np.ndarray:
    """Return the dequantized values (float32, or uint16 bit patterns for f16/bf16)."""
    lib = lib or load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    out = np.full(n * np.dtype(_OUT_NP[out_dtype]).itemsize, GARBAGE, np.uint8).view(_OUT_NP[out_dtype])
    rc = lib.orc_dequantize(_ptr(codes), _ptr(scales), n, fmt, G, _ptr(out), out_dtype)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def reduce(codes_list, scales_list, n: int, fmt_in: int, G_in: int, fmt_out: int, G_out: int,
           want_sum: bool = False, lib=None):
    """Return (codes, scales, sum_or_None) of the shard-ordered quantized reduce."""
    lib = lib or load()
    codes_list = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    scales_list = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    N = len(codes_list)
    cp = (ctypes.c_void_p * N)(*[_ptr(c) for c in codes_list])
    sp = (ctypes.c_void_p * N)(*[_ptr(s) for s in scales_list])
    out_codes = np.full(codes_bytes(fmt_out, n, lib), GARBAGE, dtype=np.uint8)
    out_scales = np.full(max(num_blocks(n, G_out, lib), 0), np.nan, dtype=np.float32)
    sum_out = np.full(n, np.nan, dtype=np.float32) if want_sum else None
    rc = lib.orc_reduce(ctypes.addressof(cp), ctypes.addressof(sp), N, n, fmt_in, G_in,
                        _ptr(out_codes), _ptr(out_scales), fmt_out, G_out,
                        _ptr(sum_out) if want_sum else None)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out_codes, out_scales, sum_out


def il_bytes(fmt: int, n: int, G: int, lib=None) -> int:
    """Bytes of the interleaved record stream (-1: no interleaved form)."""
    return int((lib or load()).orc_il_bytes(fmt, n, G))


def quantize_interleaved(x: np.ndarray, fmt: int, G: int, dtype: int | None = None,
                         lib=None) -> np.ndarray:
    """Return the record stream (uint8[il_bytes]): per block its fp32 scale, then its codes."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    n = x.size
    nbytes = il_bytes(fmt, n, G, lib)
    if nbytes < 0:
        raise ValueError("oracle rejected the arguments")
    rec = np.full(nbytes, GARBAGE, dtype=np.uint8)
    if lib.orc_quantize_interleaved(_ptr(x), _dtype_code(x, dtype), n, fmt, G, _ptr(rec)) != 0:
        raise ValueError("oracle rejected the arguments")
    return rec


def dequantize_interleaved(rec: np.ndarray, n: int, fmt: int, G: int, out_dtype: int,
                           lib=None) -> np.ndarray:
    """Dequantize a record stream (float32, or uint16 bit patterns for f16/bf16)."""
    lib = lib or load()
    rec = np.ascontiguousarray(rec, dtype=np.uint8)
    out = np.full(n * np.dtype(_OUT_NP[out_dtype]).itemsize, GARBAGE, np.uint8).view(_OUT_NP[out_dtype])
    if lib.orc_dequantize_interleaved(_ptr(rec), n, fmt, G, _ptr(out), out_dtype) != 0:
        raise ValueError("oracle rejected the arguments")
    return out


def aquavit_bpw(t: int, T: int, a: float = 0.9, c: float = 5.0, lib=None) -> float:
    """Target width of the ascending schedule at step t of T."""
    return float((lib or load()).orc_aquavit_bpw(t, T, a, c))


def aquavit_pick(bpw: float, lib=None):
    """(b, G, width) of the available pair nearest to a target width."""
    lib = lib or load()
    b, G = ctypes.c_int(0), ctypes.c_int64(0)
    w = lib.orc_aquavit_pick(bpw, ctypes.byref(b), ctypes.byref(G))
    return b.value, G.value, float(w)


def reduce_ring(codes_list, scales_list, n: int, fmt: int, G: int, fmt_out: int, G_out: int,
                want_sum: bool = False, lib=None):
    """The ring reduce-scatter's hops for one chunk: (codes, scales, sum_or_None)."""
    lib = lib or load()
    codes_list = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    scales_list = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    N = len(codes_list)
    cp = (ctypes.c_void_p * N)(*[_ptr(c) for c in codes_list])
    sp = (ctypes.c_void_p * N)(*[_ptr(s) for s in scales_list])
    part_c = [np.zeros(codes_bytes(fmt, n, lib), np.uint8) for _ in range(2)]
    part_s = [np.zeros(max(num_blocks(n, G, lib), 1), np.float32) for _ in range(2)]
    pcp = (ctypes.c_void_p * 2)(*[_ptr(c) for c in part_c])
    psp = (ctypes.c_void_p * 2)(*[_ptr(s) for s in part_s])
    out_codes = np.full(codes_bytes(fmt_out, n, lib), GARBAGE, dtype=np.uint8)
    out_scales = np.full(max(num_blocks(n, G_out, lib), 0), np.nan, dtype=np.float32)
    sum_out = np.full(n, np.nan, dtype=np.float32) if want_sum else None
    rc = lib.orc_reduce_ring(ctypes.addressof(cp), ctypes.addressof(sp), N, n, fmt, G,
                             ctypes.addressof(pcp), ctypes.addressof(psp), _ptr(out_codes),
                             _ptr(out_scales), fmt_out, G_out, _ptr(sum_out) if want_sum else None)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return out_codes, out_scales, sum_out


def slice_position(c: int, A: int, L: int) -> int:
    """Where chunk c sits in the reordered layout (the transpose of the A x L grid)."""
    return (c % L) * A + c // L


def quantize_reordered(x: np.ndarray, fmt: int, G: int, A: int, L: int, dtype: int | None = None,
                       lib=None):
    """Quantize with tensor-slice reordering: (codes, scales) of the whole tensor,
    chunk c of n/(A*L) elements stored at slice position slice_position(c)."""
    lib = lib or load()
    x = np.ascontiguousarray(x)
    n = x.size
    codes = np.full(codes_bytes(fmt, n, lib), GARBAGE, dtype=np.uint8)
    scales = np.full(max(num_blocks(n, G, lib), 0), np.nan, dtype=np.float32)
    rc = lib.orc_quantize_reordered(_ptr(x), _dtype_code(x, dtype), n, fmt, G, A, L, _ptr(codes),
                                    _ptr(scales))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return codes, scales


def reduce_two_hop(codes_list, scales_list, A: int, L: int, n: int, fmt_in: int, G_in: int,
                   fmt_mid: int, G_mid: int, fmt_out: int, G_out: int, want_sum: bool = False,
                   lib=None):
    """Two-hop reduce over P = A*L simulated GPUs. Returns (mid, out, sums): mid and
    out are lists of (codes, scales) per GPU (A*n/P and n/P elements), sums a list
    of fp32 arrays (or None)."""
    lib = lib or load()
    P = A * L
    if len(codes_list) != P or len(scales_list) != P:
        raise ValueError("need one codes and one scales array per GPU")
    m = n // P
    codes_list = [np.ascontiguousarray(c, dtype=np.uint8) for c in codes_list]
    scales_list = [np.ascontiguousarray(s, dtype=np.float32) for s in scales_list]
    mid = [(np.full(codes_bytes(fmt_mid, A * m, lib), GARBAGE, np.uint8),
            np.full(num_blocks(A * m, G_mid, lib), np.nan, np.float32)) for _ in range(P)]
    out = [(np.full(codes_bytes(fmt_out, m, lib), GARBAGE, np.uint8),
            np.full(num_blocks(m, G_out, lib), np.nan, np.float32)) for _ in range(P)]
    sums = [np.full(m, np.nan, np.float32) for _ in range(P)] if want_sum else None

    def arr(items):
        return (ctypes.c_void_p * P)(*[_ptr(a) for a in items])

    # every pointer array is bound to a name so that it outlives the call
    ic, is_ = arr(codes_list), arr(scales_list)
    mc, ms = arr([c for c, _ in mid]), arr([s for _, s in mid])
    oc, os_ = arr([c for c, _ in out]), arr([s for _, s in out])
    sp = arr(sums) if want_sum else None
    rc = lib.orc_reduce_two_hop(
        ctypes.addressof(ic), ctypes.addressof(is_), A, L, n, fmt_in, G_in, ctypes.addressof(mc),
        ctypes.addressof(ms), fmt_mid, G_mid, ctypes.addressof(oc), ctypes.addressof(os_), fmt_out,
        G_out, ctypes.addressof(sp) if want_sum else None)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return mid, out, sums


def fp8_accumulate(codes: np.ndarray, scales: np.ndarray, grad: np.ndarray, G: int,
                   grad_dtype: int | None = None, lib=None):
    """Return new (codes, scales) after one in-place FP8 accumulate step (inputs untouched)."""
    lib = lib or load()
    codes = np.array(codes, dtype=np.uint8, copy=True)
    scales = np.array(scales, dtype=np.float32, copy=True)
    grad = np.ascontiguousarray(grad)
    rc = lib.orc_fp8_accumulate(_ptr(codes), _ptr(scales), _ptr(grad),
                                _dtype_code(grad, grad_dtype), grad.size, G)
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return codes, scales


_KIND = {"f16": F16, "bf16": BF16, "e4m3": E4M3}


def encode_array(kind: str, x: np.ndarray, lib=None) -> np.ndarray:
    """Round float32 values to f16 / bf16 / e4m3 bit patterns (uint32 array)."""
    lib = lib or load()
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.zeros(x.size, dtype=np.uint32)
    if lib.orc_encode_n(_KIND[kind], _ptr(x), x.size, _ptr(out)) != 0:
        raise ValueError(kind)
    return out


def decode_array(kind: str, c: np.ndarray, lib=None) -> np.ndarray:
    """Decode f16 / bf16 / e4m3 bit patterns to float32."""
    lib = lib or load()
    c = np.ascontiguousarray(c, dtype=np.uint32)
    out = np.zeros(c.size, dtype=np.float32)
    if lib.orc_decode_n(_KIND[kind], _ptr(c), c.size, _ptr(out)) != 0:
        raise ValueError(kind)
    return out


def e4m3_decode(c: int, lib=None) -> float:
    return float((lib or load()).orc_e4m3_decode(c))


def e4m3_encode(x: float, lib=None) -> int:
    return int((lib or load()).orc_e4m3_encode(x))


def f16_decode(h: int, lib=None) -> float:
    return float((lib or load()).orc_f16_decode(h))


def f16_encode(x: float, lib=None) -> int:
    return int((lib or load()).orc_f16_encode(x))


def bf16_decode(h: int, lib=None) -> float:
    return float((lib or load()).orc_bf16_decode(h))


def bf16_encode(x: float, lib=None) -> int:
    return int((lib or load()).orc_bf16_encode(x))


def gemm_dequant(x_bf16: np.ndarray, M: int, K: int, codes: np.ndarray, scales: np.ndarray,
                 fmt: int, G: int, N: int, rows=None, cols=None, lib=None):
    """Dequant-fused GEMM reference (reading R16 of zq_oracle.c): returns (y, absy),
    float64, for the listed output positions (all M x N, row-major, when rows and
    cols are None): y = x W_hat^T exactly, absy = the sums of |products|."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    if rows is None:
        rr, cc = np.meshgrid(np.arange(M, dtype=np.int64), np.arange(N, dtype=np.int64), indexing="ij")
        rows, cols = rr.ravel(), cc.ravel()
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    y = np.zeros(rows.size, np.float64)
    absy = np.zeros(rows.size, np.float64)
    rc = lib.orc_gemm_dequant(_ptr(x), M, K, _ptr(codes), _ptr(scales), fmt, G, N, _ptr(rows),
                              _ptr(cols), rows.size, _ptr(y), _ptr(absy))
    if rc != 0:
        raise ValueError("oracle rejected the arguments")
    return y, absy
