"""zq -- blockwise quantize / pack / dequantize / quantized reduce / FP8 accumulate
on one GB300 GPU.

This module is a thin binding over the C ABI of ``libzq.so`` (``include/zq.h``):
it only marshals arguments. torch supplies device memory and the current CUDA
stream; every step of the computation runs in the library's CUDA kernels. If
the library is missing the calls raise; there is no fallback.

The operations (see ``include/zq.h`` for the exact definitions):
  * ``quantize``          blockwise symmetric quantization to packed 2/4/6/8-bit
                          codes or E4M3 bytes, one fp32 scale per G elements
                          (ZeRO++ qwZ; Aquavit granularity modulation; AGoQ);
  * ``dequantize``        codes * scale, rounded to the output type;
  * ``reduce_quantized``  N quantized shards -> fp32 sum in shard order ->
                          requantized (ZeRO++ qgZ; AGoQ local reduce);
  * ``fp8_accumulate``    in-place E4M3 main-gradient update (AGoQ QuanGrad);
  * ``quantize_reordered`` / ``reduce_two_hop``  qgZ's tensor-slice reordering
                          fused into quantize, and its intra-node + inter-node
                          reduce (ZeRO++ two-hop communication);
  * ``reduce_ring``       the ring reduce-scatter's dequantize-add-requantize
                          hops, for comparison with the one-hop reduce;
  * ``quantize_interleaved`` / ``dequantize_interleaved``  Aquavit's metadata-
                          interleaved block records (scale, then codes);
  * ``aquavit_schedule``  Aquavit's ascending width schedule -> (b, G);
  * ``gemm_dequant``      y = x @ bf16(dequantize(W)).T on the tensor cores,
                          the dequantization fused into the GEMM (AGoQ kernel
                          fusion; the consumer of qwZ's gathered weights).
"""
from __future__ import annotations

import ctypes
import os
import threading

F32, F16, BF16 = 0, 1, 2
INT2, INT4, INT6, INT8, E4M3 = 2, 4, 6, 8, 0x48
FORMATS = (INT2, INT4, INT6, INT8, E4M3)
BLOCK_SIZES = (32, 64, 128, 256, 512, 1024)
BITS = {INT2: 2, INT4: 4, INT6: 6, INT8: 8, E4M3: 8}
MAX_SHARDS = 64
STATIC_MAX_SHARDS = 1024

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libzq.so")

STATUS = {0: "ZQ_OK", 1: "ZQ_ERR_INVALID_ARG", 2: "ZQ_ERR_UNSUPPORTED", 3: "ZQ_ERR_MISALIGNED",
          4: "ZQ_ERR_ALIAS", 5: "ZQ_ERR_CUDA", 6: "ZQ_ERR_TIMEOUT"}

_lock = threading.Lock()
_lib = None


class ZQError(RuntimeError):
    def __init__(self, status: int, call: str):
        self.status = status
        msg = f"{call} failed: {STATUS.get(status, status)}"
        if status == 5:
            msg += f" (cudaError {lib().zq_last_cuda_error()})"
        super().__init__(msg)


def _declare(L):
    i32, i64, vp, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t
    L.zq_codes_bytes.argtypes = [i32, i64]
    L.zq_codes_bytes.restype = sz
    L.zq_num_blocks.argtypes = [i64, i64]
    L.zq_num_blocks.restype = i64
    L.zq_quantize.argtypes = [vp, i32, i64, i32, i64, vp, vp, vp]
    L.zq_dequantize.argtypes = [vp, vp, i64, i32, i64, vp, i32, vp]
    L.zq_reduce_quantized.argtypes = [vp, vp, i32, i64, i32, i64, vp, vp, i32, i64, vp, vp]
    L.zq_reduce_quantized_static.argtypes = [vp, vp, i32, i64, i32, i64, vp, vp, i32, i64, vp, vp]
    L.zq_reduce_quantized_static.restype = i32
    L.zq_fp8_accumulate.argtypes = [vp, vp, vp, i32, i64, i64, vp]
    L.zq_gemm_dequant.argtypes = [vp, i64, i64, vp, vp, i32, i64, i64, vp, i32, vp]
    L.zq_gemm_dequant.restype = i32
    L.zq_gemm_plan.argtypes = [i64, i64, i64, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int),
                               ctypes.POINTER(ctypes.c_int)]
    L.zq_gemm_plan.restype = i32
    L.zq_quantize_multi.argtypes = [vp, vp, i32, i32, i32, i64, vp, vp, vp]
    L.zq_quantize_multi.restype = i32
    L.zq_dequantize_multi.argtypes = [vp, vp, vp, i32, i32, i64, vp, i32, vp]
    L.zq_dequantize_multi.restype = i32
    L.zq_wait_selftest.argtypes = [i64, vp]
    L.zq_wait_selftest.restype = i32
    for f in ("zq_quantize", "zq_dequantize", "zq_reduce_quantized", "zq_fp8_accumulate"):
        getattr(L, f).restype = i32
    L.zq_interleaved_bytes.argtypes = [i32, i64, i64]
    L.zq_interleaved_bytes.restype = sz
    L.zq_quantize_interleaved.argtypes = [vp, i32, i64, i32, i64, vp, vp]
    L.zq_quantize_interleaved.restype = i32
    L.zq_dequantize_interleaved.argtypes = [vp, i64, i32, i64, vp, i32, vp]
    L.zq_dequantize_interleaved.restype = i32
    L.zq_aquavit_schedule.argtypes = [i64, i64, ctypes.c_double, ctypes.c_double,
                                      ctypes.POINTER(i32), ctypes.POINTER(i64),
                                      ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_double)]
    L.zq_aquavit_schedule.restype = i32
    L.zq_reduce_ring.argtypes = [vp, vp, i32, i64, i32, i64, vp, vp, vp, vp, i32, i64, vp, vp]
    L.zq_reduce_ring.restype = i32
    L.zq_status_string.argtypes = [i32]
    L.zq_status_string.restype = ctypes.c_char_p
    L.zq_last_cuda_error.argtypes = []
    L.zq_last_cuda_error.restype = i32
    L.zq_device_status.argtypes = [vp]
    L.zq_device_status.restype = i32
    L.zq_quantize_reordered.argtypes = [vp, i32, i64, i32, i64, i32, i32, vp, vp, vp]
    L.zq_quantize_reordered.restype = i32
    L.zq_reduce_two_hop.argtypes = [vp, vp, i32, i32, i64, i32, i64, vp, vp, i32, i64, vp, vp, i32,
                                    i64, vp, vp]
    L.zq_reduce_two_hop.restype = i32
    return L


def lib():
    """The loaded libzq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        with _lock:
            if _lib is None:
                if not os.path.exists(LIB_PATH):
                    raise RuntimeError(
                        f"{LIB_PATH} is missing: build it with "
                        "`python -m blockwise_quantized_zero_gb300.build` (no CPU fallback exists)")
                _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def codes_bytes(fmt: int, n: int) -> int:
    return int(lib().zq_codes_bytes(fmt, n))


def num_blocks(n: int, G: int) -> int:
    return int(lib().zq_num_blocks(n, G))


# ---------------------------------------------------------------------------
# torch-facing wrappers (argument marshalling only)
# ---------------------------------------------------------------------------

def _torch():
    import torch

    return torch


def dtype_code(dt) -> int:
    torch = _torch()
    return {torch.float32: F32, torch.float16: F16, torch.bfloat16: BF16}[dt]


def torch_dtype(code: int):
    torch = _torch()
    return {F32: torch.float32, F16: torch.float16, BF16: torch.bfloat16}[code]


def _stream(t, stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(status: int, call: str):
    if status != 0:
        raise ZQError(status, call)


def _cuda_contig(t, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need(t, nbytes: int, name: str):
    """t must be a contiguous CUDA tensor of at least nbytes bytes (the C ABI
    takes raw pointers, so the binding refuses buffers the kernels would
    overrun)."""
    _cuda_contig(t, name)
    have = t.numel() * t.element_size()
    if have < nbytes:
        raise ValueError(f"{name} holds {have} bytes; the call needs {nbytes}")


def _need_pair(codes, scales, fmt: int, n: int, G: int, name: str):
    _need(codes, codes_bytes(fmt, n), f"{name} codes")
    _need(scales, 4 * num_blocks(n, G), f"{name} scales")


def empty_codes(fmt: int, n: int, device):
    torch = _torch()
    return torch.empty(codes_bytes(fmt, n), dtype=torch.uint8, device=device)


def empty_scales(n: int, G: int, device):
    torch = _torch()
    return torch.empty(num_blocks(n, G), dtype=torch.float32, device=device)


def quantize(src, fmt: int, G: int, codes=None, scales=None, stream=None):
    """Quantize a CUDA tensor (fp32/fp16/bf16, flattened) -> (codes uint8, scales fp32)."""
    _cuda_contig(src, "src")
    n = src.numel()
    codes = empty_codes(fmt, n, src.device) if codes is None else codes
    scales = empty_scales(n, G, src.device) if scales is None else scales
    _need_pair(codes, scales, fmt, n, G, "output")
    _check(lib().zq_quantize(src.data_ptr(), dtype_code(src.dtype), n, fmt, G, codes.data_ptr(),
                             scales.data_ptr(), _stream(src, stream)), "zq_quantize")
    return codes, scales


def dequantize(codes, scales, n: int, fmt: int, G: int, out_dtype=None, out=None, stream=None):
    """Dequantize packed codes -> a CUDA tensor of n elements (default bf16)."""
    torch = _torch()
    _need_pair(codes, scales, fmt, n, G, "input")
    if out is None:
        out = torch.empty(n, dtype=out_dtype or torch.bfloat16, device=codes.device)
    _need(out, max(n, 0) * out.element_size(), "out")
    _check(lib().zq_dequantize(codes.data_ptr(), scales.data_ptr(), n, fmt, G, out.data_ptr(),
                               dtype_code(out.dtype), _stream(codes, stream)), "zq_dequantize")
    return out


def reduce_ring(codes_list, scales_list, n: int, fmt: int, G: int, fmt_out: int, G_out: int,
                out_codes=None, out_scales=None, sum_out=None, partials=None, stream=None):
    """The ring reduce-scatter's hops (dequantize, add, requantize per hop) for
    one chunk -> (codes, scales, sum or None). partials: two (codes, scales)
    buffer pairs in (fmt, G), allocated here when not given."""
    torch = _torch()
    N = len(codes_list)
    if N != len(scales_list):
        raise ValueError("codes_list and scales_list differ in length")
    dev = codes_list[0].device
    out_codes = empty_codes(fmt_out, n, dev) if out_codes is None else out_codes
    out_scales = empty_scales(n, G_out, dev) if out_scales is None else out_scales
    if sum_out is True:
        sum_out = torch.empty(n, dtype=torch.float32, device=dev)
    if partials is None and N >= 3:
        partials = [(empty_codes(fmt, n, dev), empty_scales(n, G, dev)) for _ in range(2)]
    for r in range(N):
        _need_pair(codes_list[r], scales_list[r], fmt, n, G, f"shard {r}")
    _need_pair(out_codes, out_scales, fmt_out, n, G_out, "output")
    if sum_out is not None:
        _need(sum_out, 4 * max(n, 0), "sum_out")
    if partials and N >= 3:
        for k, (pc_, ps_) in enumerate(partials[:2]):
            _need_pair(pc_, ps_, fmt, n, G, f"partial {k}")
    cp = (ctypes.c_void_p * N)(*[c.data_ptr() for c in codes_list])
    sp = (ctypes.c_void_p * N)(*[s.data_ptr() for s in scales_list])
    pc = (ctypes.c_void_p * 2)(*[c.data_ptr() for c, _ in partials]) if partials else None
    ps = (ctypes.c_void_p * 2)(*[s.data_ptr() for _, s in partials]) if partials else None
    _check(lib().zq_reduce_ring(cp, sp, N, n, fmt, G, pc, ps, out_codes.data_ptr(),
                                out_scales.data_ptr(), fmt_out, G_out,
                                sum_out.data_ptr() if sum_out is not None else None,
                                _stream(out_codes, stream)), "zq_reduce_ring")
    return out_codes, out_scales, sum_out


def interleaved_bytes(fmt: int, n: int, G: int) -> int:
    """Bytes of the metadata-interleaved record stream (0: integer formats only)."""
    return int(lib().zq_interleaved_bytes(fmt, n, G))


def quantize_interleaved(src, fmt: int, G: int, records=None, stream=None):
    """Quantize a CUDA tensor into one uint8 stream of block records (fp32 scale, then codes)."""
    torch = _torch()
    _cuda_contig(src, "src")
    n = src.numel()
    if records is None:
        records = torch.empty(max(interleaved_bytes(fmt, n, G), 1), dtype=torch.uint8,
                              device=src.device)
    _need(records, interleaved_bytes(fmt, n, G), "records")
    _check(lib().zq_quantize_interleaved(src.data_ptr(), dtype_code(src.dtype), n, fmt, G,
                                         records.data_ptr(), _stream(src, stream)),
           "zq_quantize_interleaved")
    return records


def dequantize_interleaved(records, n: int, fmt: int, G: int, out_dtype=None, out=None,
                           stream=None):
    """Dequantize a record stream -> a CUDA tensor of n elements (default bf16)."""
    torch = _torch()
    _need(records, interleaved_bytes(fmt, n, G), "records")
    if out is None:
        out = torch.empty(n, dtype=out_dtype or torch.bfloat16, device=records.device)
    _need(out, max(n, 0) * out.element_size(), "out")
    _check(lib().zq_dequantize_interleaved(records.data_ptr(), n, fmt, G, out.data_ptr(),
                                           dtype_code(out.dtype), _stream(records, stream)),
           "zq_dequantize_interleaved")
    return out


def aquavit_schedule(t: int, T: int, a: float = 0.9, c: float = 5.0):
    """(format, G, target width, pair width) of the ascending schedule at step t of T."""
    fmt, G = ctypes.c_int(0), ctypes.c_int64(0)
    want, width = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check(lib().zq_aquavit_schedule(t, T, a, c, ctypes.byref(fmt), ctypes.byref(G),
                                     ctypes.byref(want), ctypes.byref(width)),
           "zq_aquavit_schedule")
    return fmt.value, G.value, want.value, width.value


def _reduce(entry: str, codes_list, scales_list, n, fmt_in, G_in, fmt_out, G_out, out_codes,
            out_scales, sum_out, stream):
    torch = _torch()
    N = len(codes_list)
    if N != len(scales_list):
        raise ValueError("codes_list and scales_list differ in length")
    dev = codes_list[0].device
    out_codes = empty_codes(fmt_out, n, dev) if out_codes is None else out_codes
    out_scales = empty_scales(n, G_out, dev) if out_scales is None else out_scales
    if sum_out is True:
        sum_out = torch.empty(n, dtype=torch.float32, device=dev)
    for r in range(N):
        _need_pair(codes_list[r], scales_list[r], fmt_in, n, G_in, f"shard {r}")
    _need_pair(out_codes, out_scales, fmt_out, n, G_out, "output")
    if sum_out is not None:
        _need(sum_out, 4 * max(n, 0), "sum_out")
    cp = (ctypes.c_void_p * N)(*[c.data_ptr() for c in codes_list])
    sp = (ctypes.c_void_p * N)(*[s.data_ptr() for s in scales_list])
    _check(getattr(lib(), entry)(cp, sp, N, n, fmt_in, G_in, out_codes.data_ptr(),
                                 out_scales.data_ptr(), fmt_out, G_out,
                                 sum_out.data_ptr() if sum_out is not None else None,
                                 _stream(out_codes, stream)), entry)
    return out_codes, out_scales, sum_out


def quantize_reordered(src, fmt: int, G: int, nodes: int, gpus_per_node: int, codes=None,
                       scales=None, stream=None):
    """Quantize with qgZ's tensor-slice reordering (see zq_quantize_reordered)."""
    _cuda_contig(src, "src")
    n = src.numel()
    codes = empty_codes(fmt, n, src.device) if codes is None else codes
    scales = empty_scales(n, G, src.device) if scales is None else scales
    _need_pair(codes, scales, fmt, n, G, "output")
    _check(lib().zq_quantize_reordered(src.data_ptr(), dtype_code(src.dtype), n, fmt, G, nodes,
                                       gpus_per_node, codes.data_ptr(), scales.data_ptr(),
                                       _stream(src, stream)), "zq_quantize_reordered")
    return codes, scales


def reduce_two_hop(codes_list, scales_list, nodes: int, gpus_per_node: int, n: int, fmt_in: int,
                   G_in: int, fmt_mid: int, G_mid: int, fmt_out: int, G_out: int, mid=None,
                   out=None, sums=None, stream=None):
    """qgZ's two-hop reduce over P = nodes * gpus_per_node simulated GPUs (see
    zq_reduce_two_hop). mid / out: lists of (codes, scales) per GPU, allocated
    when None; sums: None, True (allocate) or a list of fp32 tensors.
    Returns (mid, out, sums)."""
    torch = _torch()
    P = nodes * gpus_per_node
    if len(codes_list) != P or len(scales_list) != P:
        raise ValueError("need one codes and one scales tensor per GPU")
    dev = codes_list[0].device
    m = n // P
    if mid is None:
        mid = [(empty_codes(fmt_mid, nodes * m, dev), empty_scales(nodes * m, G_mid, dev))
               for _ in range(P)]
    if out is None:
        out = [(empty_codes(fmt_out, m, dev), empty_scales(m, G_out, dev)) for _ in range(P)]
    if sums is True:
        sums = [torch.empty(m, dtype=torch.float32, device=dev) for _ in range(P)]
    if len(mid) != P or len(out) != P or (sums is not None and len(sums) != P):
        raise ValueError("need one mid, out (and sums) buffer per GPU")
    for g in range(P):
        _need_pair(codes_list[g], scales_list[g], fmt_in, n, G_in, f"GPU {g} input")
        _need_pair(mid[g][0], mid[g][1], fmt_mid, nodes * m, G_mid, f"GPU {g} mid")
        _need_pair(out[g][0], out[g][1], fmt_out, m, G_out, f"GPU {g} output")
        if sums is not None:
            _need(sums[g], 4 * max(m, 0), f"GPU {g} sums")

    def arr(ts):
        return (ctypes.c_void_p * P)(*[t.data_ptr() for t in ts])

    ic, is_ = arr(codes_list), arr(scales_list)
    mc, ms = arr([c for c, _ in mid]), arr([s for _, s in mid])
    oc, os_ = arr([c for c, _ in out]), arr([s for _, s in out])
    sp = arr(sums) if sums is not None else None
    _check(lib().zq_reduce_two_hop(ic, is_, nodes, gpus_per_node, n, fmt_in, G_in, mc, ms, fmt_mid,
                                   G_mid, oc, os_, fmt_out, G_out, sp,
                                   _stream(codes_list[0], stream)), "zq_reduce_two_hop")
    return mid, out, sums


def reduce_quantized(codes_list, scales_list, n: int, fmt_in: int, G_in: int, fmt_out: int,
                     G_out: int, out_codes=None, out_scales=None, sum_out=None, stream=None):
    """Shard-ordered fp32 sum of N quantized shards, requantized.

    ``sum_out``: None (not written), True (allocate), or an fp32 tensor of n.
    Returns (out_codes, out_scales, sum_out_or_None)."""
    return _reduce("zq_reduce_quantized", codes_list, scales_list, n, fmt_in, G_in, fmt_out,
                   G_out, out_codes, out_scales, sum_out, stream)


def reduce_quantized_static(codes_list, scales_list, n: int, fmt_in: int, G_in: int,
                            fmt_out: int, G_out: int, out_codes=None, out_scales=None,
                            sum_out=None, stream=None):
    """reduce_quantized for up to 1024 shards through zq_reduce_quantized_static,
    which allocates nothing (its shard table is a static device array shared by
    all calls: calls that overlap on the GPU race). Outputs are allocated here
    only when not given; a caller that cannot allocate passes them in."""
    return _reduce("zq_reduce_quantized_static", codes_list, scales_list, n, fmt_in, G_in,
                   fmt_out, G_out, out_codes, out_scales, sum_out, stream)


def fp8_accumulate(main_codes, main_scales, grad, G: int, stream=None):
    """In place: main (E4M3 codes + scales) <- Q8(D8(main) + grad)."""
    _cuda_contig(grad, "grad")
    _need_pair(main_codes, main_scales, E4M3, grad.numel(), G, "main")
    _check(lib().zq_fp8_accumulate(main_codes.data_ptr(), main_scales.data_ptr(), grad.data_ptr(),
                                   dtype_code(grad.dtype), grad.numel(), G,
                                   _stream(grad, stream)), "zq_fp8_accumulate")
    return main_codes, main_scales


def device_status(stream=None):
    """Wait for the stream, then raise ZQError if a kernel's bounded device-side
    wait ran out since the last check (the library's device error words)."""
    torch = _torch()
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib().zq_device_status(ctypes.c_void_p(st.cuda_stream)), "zq_device_status")


def wait_selftest(limit_us: int = 5000, stream=None):
    """Enqueue the bounded-wait self-test (zq_wait_selftest): a kernel whose
    waits on a barrier that nothing completes run out after limit_us, so the
    next device_status() raises ZQError(ZQ_ERR_TIMEOUT)."""
    torch = _torch()
    st = stream if stream is not None else torch.cuda.current_stream()
    _check(lib().zq_wait_selftest(int(limit_us), ctypes.c_void_p(st.cuda_stream)),
           "zq_wait_selftest")


def gemm_dequant(x, w_codes, w_scales, fmt: int, G: int, N: int, out_dtype=None, out=None,
                 stream=None):
    """y = x @ W_hat.T with W_hat the bf16 dequantization of the N x K weight held
    as (w_codes, w_scales) in (fmt, G) layout (zq_gemm_dequant). x: CUDA bf16
    tensor M x K. Returns y (M x N, fp32 unless out_dtype / out say bf16)."""
    torch = _torch()
    _cuda_contig(x, "x")
    if x.dtype != torch.bfloat16 or x.dim() != 2:
        raise ValueError("x must be a 2-D bf16 tensor")
    M, K = x.shape
    _need_pair(w_codes, w_scales, fmt, N * K, G, "weight")
    if out is None:
        out = torch.empty(M, N, dtype=out_dtype or torch.float32, device=x.device)
    _cuda_contig(out, "out")
    if out.numel() != M * N:
        raise ValueError("out must hold M x N elements")
    _check(lib().zq_gemm_dequant(x.data_ptr(), M, K, w_codes.data_ptr(), w_scales.data_ptr(), fmt,
                                 G, N, out.data_ptr(), dtype_code(out.dtype), _stream(x, stream)),
           "zq_gemm_dequant")
    return out


def gemm_plan(M: int, N: int, K: int):
    """The output tile gemm_dequant uses for an M x N x K problem on the
    current device: (rows, columns, CTAs sharing a tile's K range)
    (zq_gemm_plan)."""
    bm, bn, sp = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(lib().zq_gemm_plan(int(M), int(N), int(K), ctypes.byref(bm), ctypes.byref(bn),
                              ctypes.byref(sp)), "zq_gemm_plan")
    return bm.value, bn.value, sp.value


def quantize_multi(srcs, fmt: int, G: int, codes=None, scales=None, stream=None):
    """zq_quantize of every tensor in `srcs` (same dtype) in one batched call
    (zq_quantize_multi). Returns the lists (codes, scales); outputs are
    allocated when not given."""
    torch = _torch()
    srcs = list(srcs)
    if not srcs:
        return [], []
    dt = srcs[0].dtype
    for t in srcs:
        _cuda_contig(t, "src")
        if t.dtype != dt:
            raise ValueError("all tensors must have one dtype")
    if codes is None:
        codes = [empty_codes(fmt, t.numel(), t.device) for t in srcs]
    if scales is None:
        scales = [empty_scales(t.numel(), G, t.device) for t in srcs]
    for t, c, s in zip(srcs, codes, scales):
        _need_pair(c, s, fmt, t.numel(), G, "output")
    k = len(srcs)

    def arr(ts):
        return (ctypes.c_void_p * k)(*[t.data_ptr() for t in ts])

    sp, cp, kp = arr(srcs), arr(codes), arr(scales)
    ns = (ctypes.c_int64 * k)(*[t.numel() for t in srcs])
    _check(lib().zq_quantize_multi(sp, ns, k, dtype_code(dt), fmt, G, cp, kp,
                                   _stream(srcs[0], stream)), "zq_quantize_multi")
    return codes, scales


def dequantize_multi(codes_list, scales_list, ns, fmt: int, G: int, out_dtype=None, outs=None,
                     stream=None):
    """zq_dequantize of every (codes, scales, n) in one batched call
    (zq_dequantize_multi). Returns the list of outputs (allocated when not
    given; float32 unless out_dtype says otherwise)."""
    torch = _torch()
    codes_list, scales_list, ns = list(codes_list), list(scales_list), [int(v) for v in ns]
    k = len(ns)
    if k == 0:
        return []
    if len(codes_list) != k or len(scales_list) != k:
        raise ValueError("need one codes and one scales tensor per size")
    dev = codes_list[0].device
    if outs is None:
        outs = [torch.empty(n, dtype=out_dtype or torch.float32, device=dev) for n in ns]
    dt = outs[0].dtype
    for c, s, n, o in zip(codes_list, scales_list, ns, outs):
        _need_pair(c, s, fmt, n, G, "input")
        _cuda_contig(o, "out")
        if o.dtype != dt or o.numel() < n:
            raise ValueError("outputs must share one dtype and hold n elements")

    def arr(ts):
        return (ctypes.c_void_p * k)(*[t.data_ptr() for t in ts])

    cp, sp, op = arr(codes_list), arr(scales_list), arr(outs)
    nv = (ctypes.c_int64 * k)(*ns)
    _check(lib().zq_dequantize_multi(cp, sp, nv, k, fmt, G, op, dtype_code(dt),
                                     _stream(codes_list[0], stream)), "zq_dequantize_multi")
    return outs
