"""Benchmark of the blockwise quantize / pack / dequantize / reduce path on GB300.

One JSON line (rank 0) per run. Default workload (``--workload llama70b``,
the largest single-GPU configuration): one Llama-3-70B decoder layer's bf16
weights (q, o 8192x8192; k, v 8192x1024; gate, up 8192x28672; down
28672x8192; 855,638,016 elements ~ N(0, 0.02)) quantized to int8 G=256 and to
6-bit G=32, then dequantized to bf16 (28 launches per step). Metric: GB/s of
algorithmic input+output bytes. The same run then times the kernel families
of the other configurations (``--configs``, reported under ``configs``):
qwz_fp16 (1 Mi fp16 weights with outliers, int8 G=256, batched over 512
tensors), gm_sweep (8192x8192 bf16, b in {2,4,6,8} x G in {1024..32}),
qgz_reduce (8 int4 shards of 134,217,728 gradients -> int4 G=128 and int8
G=256), agoq_fp8 (E4M3 main gradient of 268,435,456 elements, 4 accumulate
steps + 8-shard FP8 reduce), llama70b_batched (the headline layer through one
multi-tensor quantize and one multi-tensor dequantize call per scheme) and
llama70b_gemm (the layer's projections on 4096 tokens with the dequantization
fused into the tensor-core GEMM). Further workloads (``--workload``): qgz_two_hop
(qgZ's reordered quantize and two-hop reduce, 2 nodes x 4 GPUs simulated),
aquavit_schedule (the 1000-step ascending width schedule, in the metadata-
interleaved and the planar layout) and ring_study (the ring reduce-scatter's
hops against the one-hop reduce, with their errors).

After every timed region the library's device error words are read
(zq_device_status); if a bounded device-side wait ran out, no number is
printed and the run exits non-zero.

Timing: CUDA events on the launching stream, W untimed warm-up steps, then K
timed steps bracketed by a barrier and a synchronize; the max over ranks is
reported. Every kernel of a step reads and writes its own buffers, so each
step touches several GB (far more than the 126 MB L2) and no flush is needed.
Inputs are seeded and synthetic (blockwise_quantized_zero_gb300.inputs).

``--impl reference`` times the oracle (plain single-threaded C) on a bounded
sample of the same workload instead. The GPU run also times the oracle on one
core (``cpu_baseline``) and on every host core (``cpu_baseline_all_cores``,
one process per core).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GB/s moved (in+out) per kernel and % of GB300 HBM peak, vs CPU oracle"
UNIT = "GB/s"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def packed_bytes(fmt: int, n: int, G: int) -> int:
    bits = 8 if fmt == 0x48 else fmt
    return ((n * bits + 31) // 32) * 4 + 4 * ((n + G - 1) // G)


def fmt_name(fmt: int) -> str:
    return "e4m3" if fmt == 0x48 else f"int{fmt}"


# ---------------------------------------------------------------------------
# environment: peaks, clocks
# ---------------------------------------------------------------------------

def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 tensor-core TFLOP/s: (burst, sustained, source)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]), "measured"
    except Exception:  # noqa: BLE001
        return 1900.0, 1700.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            import tempfile

            fd, self.path = tempfile.mkstemp(prefix="zq_clocks_", suffix=".csv")
            os.close(fd)
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not self.path:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        sm = sorted(r[0] for r in rows)
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class Launch:
    """One timed unit: `fn` enqueues `kernels` launches of one kernel family
    that move `nbytes` algorithmic bytes in total."""

    __slots__ = ("label", "family", "nbytes", "fn", "kernels", "flops")

    def __init__(self, label, family, nbytes, fn, kernels=1, flops=0):
        self.label, self.family, self.nbytes, self.fn = label, family, nbytes, fn
        self.kernels, self.flops = kernels, flops


class ForkedStreams:
    """Side streams forked from the current stream and joined back to it, for
    end-to-end steps whose items are independent: item k runs on side stream
    k % N with buffer set k % N, so one item's device-to-host copies overlap
    another item's host-to-device copies (the host link is full duplex).
    Each stream reuses its buffer set only after its own previous item, in
    stream order. Four streams (measured on gm_sweep: 2 -> 279, 3 -> 303,
    4 -> 308 GB/s end to end) keep both link directions busier than two."""

    N = 4

    def __init__(self, make_set):
        import torch

        self.streams = [torch.cuda.Stream() for _ in range(self.N)]
        self.sets = [make_set() for _ in range(self.N)]

    def run(self, items, fn):
        import torch

        cur = torch.cuda.current_stream()
        for st in self.streams:
            st.wait_stream(cur)
        for k, item in enumerate(items):
            with torch.cuda.stream(self.streams[k % self.N]):
                fn(item, self.sets[k % self.N])
        for st in self.streams:
            cur.wait_stream(st)


def _dev_bf16(bits: np.ndarray):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


class GMSweep:
    """8192x8192 bf16 ~ N(0, 0.02); b in {2,4,6,8} x G in {1024..32}; Q then D -> bf16."""

    name = "gm_sweep"
    dtype = "bf16 in, int2/4/6/8 codes + fp32 scales, bf16 out (fp32 arithmetic)"
    rows, cols = 8192, 8192
    bits = (2, 4, 6, 8)
    blocks = (1024, 512, 256, 128, 64, 32)

    def __init__(self, pair=None):
        from blockwise_quantized_zero_gb300 import inputs

        self.n = self.rows * self.cols
        self.pairs = [(b, G) for b in self.bits for G in self.blocks]
        if pair is not None:  # one (b, G) pair only, e.g. for a profiler capture
            self.pairs = [pair]
        self.host = inputs.weight_shard_bf16(self.rows, self.cols)

    def config(self):
        return {"workload": "gm_sweep: one 8192x8192 bf16 weight shard (67,108,864 elements, "
                            "N(0,0.02)); quantize + dequantize->bf16 for b in {2,4,6,8} x "
                            "G in {1024,512,256,128,64,32}",
                "elements": self.n, "pairs": len(self.pairs),
                "pair_subset": None if len(self.pairs) == 24 else [list(p) for p in self.pairs],
                "l2": "no flush: each of the 48 launches per step reads and writes its own "
                      "buffers (7.7 GB touched per step >> 126 MB L2)"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq

        src0 = _dev_bf16(self.host)
        self.src = [src0] + [src0.clone() for _ in self.pairs[1:]]
        self.codes = [zq.empty_codes(b, self.n, "cuda") for b, _ in self.pairs]
        self.scales = [zq.empty_scales(self.n, G, "cuda") for _, G in self.pairs]
        self.out = [torch.empty(self.n, dtype=torch.bfloat16, device="cuda") for _ in self.pairs]
        self.zq = zq

    def launches(self):
        zq, n = self.zq, self.n
        out = []
        for i, (b, G) in enumerate(self.pairs):
            nb = 2 * n + packed_bytes(b, n, G)
            out.append(Launch(f"quantize bf16 {fmt_name(b)} G={G}", "quantize", nb,
                              lambda i=i, b=b, G=G: zq.quantize(self.src[i], b, G, self.codes[i],
                                                                self.scales[i])))
        for i, (b, G) in enumerate(self.pairs):
            nb = 2 * n + packed_bytes(b, n, G)
            out.append(Launch(f"dequantize {fmt_name(b)} G={G} bf16", "dequantize", nb,
                              lambda i=i, b=b, G=G: zq.dequantize(self.codes[i], self.scales[i], n,
                                                                  b, G, out=self.out[i])))
        return out

    # end to end: every C-ABI call gets host buffers
    def setup_e2e(self):
        import torch

        zq, n = self.zq, self.n
        self.h_src = torch.from_numpy(self.host.view(np.int16)).view(torch.bfloat16).pin_memory()
        cmax = max(zq.codes_bytes(b, n) for b in self.bits)
        smax = zq.num_blocks(n, 32)

        def make_set():
            dev = dict(device="cuda")
            return dict(h_codes=torch.empty(cmax, dtype=torch.uint8).pin_memory(),
                        h_scales=torch.empty(smax, dtype=torch.float32).pin_memory(),
                        h_out=torch.empty(n, dtype=torch.bfloat16).pin_memory(),
                        d_src=torch.empty(n, dtype=torch.bfloat16, **dev),
                        d_codes=torch.empty(cmax, dtype=torch.uint8, **dev),
                        d_scales=torch.empty(smax, dtype=torch.float32, **dev),
                        d_codes2=torch.empty(cmax, dtype=torch.uint8, **dev),
                        d_scales2=torch.empty(smax, dtype=torch.float32, **dev),
                        d_out=torch.empty(n, dtype=torch.bfloat16, **dev))

        self.fork = ForkedStreams(make_set)
        h2d = d2h = 0
        for b, G in self.pairs:
            cb, sb = self.zq.codes_bytes(b, n), 4 * self.zq.num_blocks(n, G)
            h2d += 2 * n + cb + sb
            d2h += cb + sb + 2 * n
        return h2d, d2h

    def e2e_step(self):
        """Per pair: host src -> quantize -> host codes; host codes -> dequantize
        -> host out. Pairs alternate between two streams (ForkedStreams)."""
        zq, n = self.zq, self.n

        def one(pair, B):
            b, G = pair
            cb, nb = zq.codes_bytes(b, n), zq.num_blocks(n, G)
            B["d_src"].copy_(self.h_src, non_blocking=True)
            zq.quantize(B["d_src"], b, G, B["d_codes"][:cb], B["d_scales"][:nb])
            B["h_codes"][:cb].copy_(B["d_codes"][:cb], non_blocking=True)
            B["h_scales"][:nb].copy_(B["d_scales"][:nb], non_blocking=True)
            B["d_codes2"][:cb].copy_(B["h_codes"][:cb], non_blocking=True)
            B["d_scales2"][:nb].copy_(B["h_scales"][:nb], non_blocking=True)
            zq.dequantize(B["d_codes2"][:cb], B["d_scales2"][:nb], n, b, G, out=B["d_out"])
            B["h_out"].copy_(B["d_out"], non_blocking=True)

        self.fork.run(self.pairs, one)

    def step_bytes(self):
        return sum(2 * (2 * self.n + packed_bytes(b, self.n, G)) for b, G in self.pairs)

    # CPU oracle on a bounded sample (the first `sample` elements)
    def oracle_sample(self, sample=1 << 24):
        import oracle as O

        x = np.ascontiguousarray(self.host[:sample])

        def run():
            for b, G in self.pairs:
                c, s = O.quantize(x, b, G, dtype=O.BF16)
                O.dequantize(c, s, sample, b, G, O.BF16)

        nbytes = sum(2 * (2 * sample + packed_bytes(b, sample, G)) for b, G in self.pairs)
        desc = (f"first {sample:,} elements ({sample // self.cols} rows) of the shard, all 24 "
                "(b, G) pairs, quantize + dequantize->bf16, single thread")
        return run, nbytes, desc


class QwzFP16:
    """1,048,576 fp16 weights ~ N(0, 0.02) with 0.1% x50 outliers (seed 0);
    int8 G=256 quantize and dequantize -> fp32. One call moves 3.2 MB and
    takes microseconds, so a step replays CUDA graphs of 512 calls on 512
    distinct tensors (1.6-2.7 GB per graph, far beyond L2); the single-call
    latency is reported beside it."""

    name = "qwz_fp16"
    dtype = "fp16 in, int8 codes + fp32 scales, fp32 out (fp32 arithmetic)"
    copies = 512
    n = 1 << 20
    G = 256
    streams = 8  # the graph's independent calls run as this many concurrent chains

    def __init__(self):
        from blockwise_quantized_zero_gb300 import inputs

        self.host = inputs.weights_fp16_outliers(self.n)

    def config(self):
        return {"workload": "qwz_fp16: one fp16 tensor of 1,048,576 elements N(0,0.02) with 0.1% "
                            "outliers x50 (seed 0), int8 G=256 quantize + dequantize->fp32; "
                            "timed as CUDA graphs of 512 independent calls on 512 distinct copies, "
                            "and as one multi-tensor quantize call over the 512 copies",
                "elements": self.n, "batched_copies": self.copies,
                "graph_chains": self.streams,
                "l2": "no flush: 512 distinct buffers per graph (1.6-2.7 GB per replay)",
                "single_call_us": getattr(self, "single_call_us", None)}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq

        self.zq = zq
        src0 = torch.from_numpy(self.host).cuda()
        self.src = [src0] + [src0.clone() for _ in range(self.copies - 1)]
        self.codes = [zq.empty_codes(zq.INT8, self.n, "cuda") for _ in range(self.copies)]
        self.scales = [zq.empty_scales(self.n, self.G, "cuda") for _ in range(self.copies)]
        self.out = [torch.empty(self.n, dtype=torch.float32, device="cuda") for _ in range(self.copies)]
        # single-call latency through the C ABI, host launch included
        for _ in range(20):
            zq.quantize(self.src[0], zq.INT8, self.G, self.codes[0], self.scales[0])
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(200):
            zq.quantize(self.src[i % 8], zq.INT8, self.G, self.codes[i % 8], self.scales[i % 8])
        torch.cuda.synchronize()
        self.single_call_us = round((time.perf_counter() - t0) / 200 * 1e6, 2)
        s = torch.cuda.Stream()
        self.gq, self.gd = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            for i in range(self.copies):  # warm the launch paths before capture
                zq.quantize(self.src[i], zq.INT8, self.G, self.codes[i], self.scales[i])
                zq.dequantize(self.codes[i], self.scales[i], self.n, zq.INT8, self.G, out=self.out[i])
        torch.cuda.synchronize()
        # The calls are independent, so each graph forks into `streams` chains
        # (call i on chain i % streams) that join at its end; the GPU runs the
        # chains concurrently, each chain's calls in order.
        side = [torch.cuda.Stream() for _ in range(self.streams)]

        def capture(graph, call):
            with torch.cuda.graph(graph, stream=s):
                for st in side:
                    st.wait_stream(s)
                for i in range(self.copies):
                    with torch.cuda.stream(side[i % self.streams]):
                        call(i)
                for st in side:
                    s.wait_stream(st)

        capture(self.gq, lambda i: zq.quantize(self.src[i], zq.INT8, self.G, self.codes[i],
                                               self.scales[i]))
        # the multi-tensor call (two launches of 256 tensors), captured so that
        # its host-side argument checks are not timed as device time
        zq.quantize_multi(self.src, zq.INT8, self.G, self.codes, self.scales)
        torch.cuda.synchronize()
        self.gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.gm, stream=s):
            zq.quantize_multi(self.src, zq.INT8, self.G, self.codes, self.scales)
        capture(self.gd, lambda i: zq.dequantize(self.codes[i], self.scales[i], self.n, zq.INT8,
                                                 self.G, out=self.out[i]))
        torch.cuda.synchronize()

    def launches(self):
        n, k = self.n, self.copies
        pb = packed_bytes(8, n, self.G)
        zq = self.zq
        return [Launch(f"quantize fp16 int8 G=256 x{k} (graph)", "quantize", k * (2 * n + pb),
                       self.gq.replay, kernels=k),
                Launch(f"dequantize int8 G=256 f32 x{k} (graph)", "dequantize", k * (pb + 4 * n),
                       self.gd.replay, kernels=k),
                Launch(f"quantize fp16 int8 G=256 x{k} (one multi-tensor call, graph)",
                       "quantize_multi", k * (2 * n + pb), self.gm.replay, kernels=(k + 255) // 256)]

    def setup_e2e(self):
        import torch

        zq, n = self.zq, self.n
        self.e_copies = 64
        self.h_src = torch.from_numpy(self.host).pin_memory()
        self.fork = ForkedStreams(lambda: dict(
            h_codes=torch.empty(zq.codes_bytes(zq.INT8, n), dtype=torch.uint8).pin_memory(),
            h_scales=torch.empty(zq.num_blocks(n, self.G), dtype=torch.float32).pin_memory(),
            h_out=torch.empty(n, dtype=torch.float32).pin_memory()))
        pb = packed_bytes(8, n, self.G)
        return self.e_copies * (2 * n + pb), self.e_copies * (pb + 4 * n)

    def e2e_step(self):
        """64 calls, each from host memory to host memory; the calls alternate
        between two streams (ForkedStreams)."""
        zq, n = self.zq, self.n

        def one(i, B):
            self.src[i].copy_(self.h_src, non_blocking=True)
            zq.quantize(self.src[i], zq.INT8, self.G, self.codes[i], self.scales[i])
            B["h_codes"].copy_(self.codes[i], non_blocking=True)
            B["h_scales"].copy_(self.scales[i], non_blocking=True)
            self.codes[i].copy_(B["h_codes"], non_blocking=True)
            self.scales[i].copy_(B["h_scales"], non_blocking=True)
            zq.dequantize(self.codes[i], self.scales[i], n, zq.INT8, self.G, out=self.out[i])
            B["h_out"].copy_(self.out[i], non_blocking=True)

        self.fork.run(range(self.e_copies), one)

    def e2e_bytes(self):
        pb = packed_bytes(8, self.n, self.G)
        return self.e_copies * (2 * self.n + pb + pb + 4 * self.n)

    def oracle_sample(self, sample=None):
        import oracle as O

        # whole-tensor round trips; `sample` elements are rounded to whole tensors
        reps = 256 if sample is None else max(1, sample // self.n)
        x = self.host if sample is None or sample >= self.n else self.host[:max(1024, sample)]
        m = x.size

        def run():
            for _ in range(reps):
                c, s = O.quantize(x, O.INT8, self.G)
                O.dequantize(c, s, m, O.INT8, self.G, O.F32)

        pb = packed_bytes(8, m, self.G)
        return run, reps * (2 * m + pb + pb + 4 * m), \
            f"{reps} quantize + dequantize->fp32 round trips of {m:,} elements of the fp16 tensor, single thread"


class QgzReduce:
    """8 gradient shards of 134,217,728 fp32 ~ Laplace(0, 1e-4) (seed 3,
    stream = shard), pre-quantized to int4 G=128 (setup, not timed); a step
    reduces them to int4 G=128 and, separately, to int8 G=256."""

    name = "qgz_reduce"
    dtype = "int4 codes + fp32 scales in, fp32 sums, int4/int8 codes out"
    N = 8
    n = 134217728

    def config(self):
        return {"workload": "qgz_reduce: 8 simulated peer shards of 134,217,728 fp32 gradients "
                            "~Laplace(0,1e-4), pre-quantized to int4 G=128; fused dequant -> fp32 "
                            "sum in shard order -> requant to int4 G=128 and to int8 G=256",
                "elements": self.n, "shards": self.N,
                "l2": "no flush: 570 MB of shard input per launch >> 126 MB L2"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq
        from blockwise_quantized_zero_gb300 import inputs

        self.zq = zq
        self.codes, self.scales, self.host_sample = [], [], []
        for r in range(self.N):
            x = inputs.gradient_shard_f32(self.n, shard=r)
            self.host_sample.append(x[: 1 << 26].copy())
            c, s = zq.quantize(torch.from_numpy(x).cuda(), zq.INT4, 128)
            self.codes.append(c)
            self.scales.append(s)
            del x
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self.oc4, self.os4 = zq.empty_codes(zq.INT4, self.n, "cuda"), zq.empty_scales(self.n, 128, "cuda")
        self.oc8, self.os8 = zq.empty_codes(zq.INT8, self.n, "cuda"), zq.empty_scales(self.n, 256, "cuda")

    def launches(self):
        zq, n, N = self.zq, self.n, self.N
        inb = N * packed_bytes(4, n, 128)
        return [
            Launch("reduce 8x int4 G=128 -> int4 G=128", "reduce", inb + packed_bytes(4, n, 128),
                   lambda: zq.reduce_quantized(self.codes, self.scales, n, zq.INT4, 128, zq.INT4, 128,
                                               self.oc4, self.os4)),
            Launch("reduce 8x int4 G=128 -> int8 G=256", "reduce", inb + packed_bytes(8, n, 256),
                   lambda: zq.reduce_quantized(self.codes, self.scales, n, zq.INT4, 128, zq.INT8, 256,
                                               self.oc8, self.os8)),
        ]

    def setup_e2e(self):
        import torch

        zq, n = self.zq, self.n
        self.h_codes = [c.cpu().pin_memory() for c in self.codes]
        self.h_scales = [s.cpu().pin_memory() for s in self.scales]
        self.h_oc = torch.empty(zq.codes_bytes(zq.INT8, n), dtype=torch.uint8).pin_memory()
        self.h_os = torch.empty(zq.num_blocks(n, 128), dtype=torch.float32).pin_memory()
        inb = self.N * packed_bytes(4, n, 128)
        return 2 * inb, packed_bytes(4, n, 128) + packed_bytes(8, n, 256)

    def e2e_step(self):
        """Shards from host memory, results to host memory, for both reductions."""
        zq, n = self.zq, self.n
        for fout, G, oc, os_ in ((zq.INT4, 128, self.oc4, self.os4), (zq.INT8, 256, self.oc8, self.os8)):
            for r in range(self.N):
                self.codes[r].copy_(self.h_codes[r], non_blocking=True)
                self.scales[r].copy_(self.h_scales[r], non_blocking=True)
            zq.reduce_quantized(self.codes, self.scales, n, zq.INT4, 128, fout, G, oc, os_)
            self.h_oc[: oc.numel()].copy_(oc, non_blocking=True)
            self.h_os[: os_.numel()].copy_(os_, non_blocking=True)

    def oracle_sample(self, sample=1 << 26):
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        host = getattr(self, "host_sample", None)
        if host is None or host[0].size < sample:
            host = [inputs.gradient_shard_f32(sample, shard=r) for r in range(self.N)]
        sh = [O.quantize(np.ascontiguousarray(x[:sample]), O.INT4, 128) for x in host]

        def run():
            O.reduce([c for c, _ in sh], [s for _, s in sh], sample, O.INT4, 128, O.INT4, 128)
            O.reduce([c for c, _ in sh], [s for _, s in sh], sample, O.INT4, 128, O.INT8, 256)

        inb = self.N * packed_bytes(4, sample, 128)
        nbytes = 2 * inb + packed_bytes(4, sample, 128) + packed_bytes(8, sample, 256)
        return run, nbytes, (f"first {sample:,} elements of each of the 8 shards, both reductions, "
                             "single thread")


class RingStudy(QgzReduce):
    """The ring reduce-scatter that qgZ replaces, against qgZ's one-hop
    reduce, on the qgz_reduce shards (8 x 134,217,728 int4 G=128 from
    Laplace(0, 1e-4) gradients): one-hop = one launch that dequantizes all 8
    shards, sums in fp32 and requantizes once; ring = 7 sequential hops, each
    a dequantize-add-requantize of [partial, next shard] with the partial in
    int4 G=128. Both keep the fp32 sums. After the timed steps the fp32
    results are compared with the exact (float64) sum of the unquantized
    gradients on the first 16,777,216 elements."""

    name = "ring_study"
    dtype = "int4 codes + fp32 scales in, fp32 sums, int4 codes out (fp32 arithmetic)"

    def config(self):
        c = {"workload": "ring_study: 8 simulated peer shards of 134,217,728 fp32 gradients "
                         "~Laplace(0,1e-4), pre-quantized to int4 G=128; qgZ one-hop reduce "
                         "(dequant all, fp32 sum, requant once) vs ring reduce-scatter (7 "
                         "sequential dequant-add-requant hops, partials in int4 G=128); fp32 sums "
                         "kept by both",
             "elements": self.n, "shards": self.N,
             "l2": "no flush: 570 MB of shard input per one-hop launch; each ring hop reads "
                   "142 MB and writes 71 MB (>> 126 MB L2 across hops)"}
        if hasattr(self, "sum_one"):
            c["accuracy"] = self.accuracy()
        return c

    def setup(self):
        super().setup()
        zq, n = self.zq, self.n
        import torch

        self.sum_one = torch.empty(n, dtype=torch.float32, device="cuda")
        self.sum_ring = torch.empty(n, dtype=torch.float32, device="cuda")
        self.ocr, self.osr = zq.empty_codes(zq.INT4, n, "cuda"), zq.empty_scales(n, 128, "cuda")
        self.partials = [(zq.empty_codes(zq.INT4, n, "cuda"), zq.empty_scales(n, 128, "cuda"))
                         for _ in range(2)]

    def _one(self):
        zq = self.zq
        zq.reduce_quantized(self.codes, self.scales, self.n, zq.INT4, 128, zq.INT4, 128, self.oc4,
                            self.os4, sum_out=self.sum_one)

    def _ring(self):
        zq = self.zq
        zq.reduce_ring(self.codes, self.scales, self.n, zq.INT4, 128, zq.INT4, 128, self.ocr,
                       self.osr, sum_out=self.sum_ring, partials=self.partials)

    def launches(self):
        n, N = self.n, self.N
        p4 = packed_bytes(4, n, 128)
        return [Launch("one-hop reduce 8x int4 G=128 -> int4 G=128 + fp32 sums", "reduce one-hop",
                       N * p4 + p4 + 4 * n, self._one),
                Launch("ring 7 hops of 2x int4 G=128 -> int4 G=128 (+ fp32 sums at the end)",
                       "reduce ring hop", (N - 1) * 3 * p4 + 4 * n, self._ring, kernels=N - 1)]

    def accuracy(self, m=1 << 24):
        import torch

        torch.cuda.synchronize()
        exact = np.zeros(m, np.float64)
        for x in self.host_sample:
            exact += x[:m].astype(np.float64)
        ref = float(np.sqrt(np.mean(exact ** 2)))
        out = {"elements": m, "reference": "float64 sum of the unquantized fp32 gradients"}
        for key, t in (("one_hop", self.sum_one), ("ring", self.sum_ring)):
            e = t[:m].cpu().numpy().astype(np.float64) - exact
            out[key] = {"rel_rms_error": round(float(np.sqrt(np.mean(e ** 2))) / ref, 5),
                        "max_abs_error": float(np.max(np.abs(e)))}
        return out

    def setup_e2e(self):
        import torch

        zq, n = self.zq, self.n
        self.h_codes = [c.cpu().pin_memory() for c in self.codes]
        self.h_scales = [s.cpu().pin_memory() for s in self.scales]
        self.h_oc = torch.empty(zq.codes_bytes(zq.INT4, n), dtype=torch.uint8).pin_memory()
        self.h_os = torch.empty(zq.num_blocks(n, 128), dtype=torch.float32).pin_memory()
        inb = self.N * packed_bytes(4, n, 128)
        return inb, 2 * packed_bytes(4, n, 128)

    def e2e_step(self):
        """Shards from host memory once; both schemes; both results to host memory."""
        for r in range(self.N):
            self.codes[r].copy_(self.h_codes[r], non_blocking=True)
            self.scales[r].copy_(self.h_scales[r], non_blocking=True)
        for run, oc, os_ in ((self._one, self.oc4, self.os4), (self._ring, self.ocr, self.osr)):
            run()
            self.h_oc.copy_(oc, non_blocking=True)
            self.h_os.copy_(os_, non_blocking=True)

    def e2e_bytes(self):
        return sum(l.nbytes for l in self.launches())

    def oracle_sample(self, sample=1 << 24):
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        host = getattr(self, "host_sample", None)
        if host is None or host[0].size < sample:
            host = [inputs.gradient_shard_f32(sample, shard=r) for r in range(self.N)]
        sh = [O.quantize(np.ascontiguousarray(x[:sample]), O.INT4, 128) for x in host]

        def run():
            O.reduce([c for c, _ in sh], [s for _, s in sh], sample, O.INT4, 128, O.INT4, 128,
                     want_sum=True)
            O.reduce_ring([c for c, _ in sh], [s for _, s in sh], sample, O.INT4, 128, O.INT4, 128,
                          want_sum=True)

        p4 = packed_bytes(4, sample, 128)
        nbytes = self.N * p4 + p4 + 4 * sample + (self.N - 1) * 3 * p4 + 4 * sample
        return run, nbytes, (f"first {sample:,} elements of each of the 8 shards, one-hop and ring, "
                             "single thread")


class QgzTwoHop:
    """qgZ's hierarchy simulated on one GPU: 2 nodes x 4 GPUs, each holding a
    134,217,728-element fp32 gradient ~ Laplace(0, 1e-4) (seed 3, stream = GPU,
    like qgz_reduce's shards). A step quantizes every gradient to int4 G=128
    with tensor-slice reordering, then runs the two-hop reduce: intra-node
    reduce + requantize to int4 G=128, inter-node reduce + requantize to int4
    G=128 (two reduce launches, one per hop, each over all 8 GPUs' problems)."""

    name = "qgz_two_hop"
    dtype = "fp32 gradients in, int4 codes + fp32 scales between the hops and out"
    A, L = 2, 4
    n = 134217728

    def config(self):
        return {"workload": "qgz_two_hop: 2 nodes x 4 GPUs simulated as buffers, 134,217,728 fp32 "
                            "gradients ~Laplace(0,1e-4) per GPU; quantize with tensor-slice "
                            "reordering (int4 G=128), intra-node reduce -> int4 G=128, inter-node "
                            "reduce -> int4 G=128",
                "elements_per_gpu": self.n, "nodes": self.A, "gpus_per_node": self.L,
                "l2": "no flush: 512 MB of fp32 gradient per quantize launch, 35-71 MB of codes "
                      "per reduce launch, 0.9 GB of codes per step >> 126 MB L2"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq
        from blockwise_quantized_zero_gb300 import inputs

        self.zq = zq
        P, n = self.A * self.L, self.n
        self.P, self.m = P, n // P
        self.x, self.host_sample = [], []
        for g in range(P):
            h = inputs.gradient_shard_f32(n, shard=g)
            self.host_sample.append(h[: 1 << 24].copy())
            self.x.append(torch.from_numpy(h).cuda())
            del h
        self.q = [(zq.empty_codes(zq.INT4, n, "cuda"), zq.empty_scales(n, 128, "cuda"))
                  for _ in range(P)]
        am = self.A * self.m
        self.mid = [(zq.empty_codes(zq.INT4, am, "cuda"), zq.empty_scales(am, 128, "cuda"))
                    for _ in range(P)]
        self.out = [(zq.empty_codes(zq.INT4, self.m, "cuda"), zq.empty_scales(self.m, 128, "cuda"))
                    for _ in range(P)]

    def _reduce_bytes(self, k=1):
        P, A, L, m = self.P, self.A, self.L, self.m
        hop1 = P * (L + 1) * packed_bytes(4, A * m, 128)
        hop2 = P * (A + 1) * packed_bytes(4, m, 128)
        return hop1 + hop2

    def two_hop(self):
        zq = self.zq
        zq.reduce_two_hop([c for c, _ in self.q], [s for _, s in self.q], self.A, self.L, self.n,
                          zq.INT4, 128, zq.INT4, 128, zq.INT4, 128, mid=self.mid, out=self.out)

    def launches(self):
        zq, n = self.zq, self.n
        out = []
        for g in range(self.P):
            out.append(Launch(f"quantize reordered fp32 int4 G=128 GPU {g}", "quantize",
                              4 * n + packed_bytes(4, n, 128),
                              lambda g=g: zq.quantize_reordered(self.x[g], zq.INT4, 128, self.A,
                                                                self.L, *self.q[g])))
        out.append(Launch("two-hop reduce (one launch per hop, int4 G=128)", "reduce",
                          self._reduce_bytes(), self.two_hop, kernels=2))
        return out

    def setup_e2e(self):
        import torch

        self.h_x = [x.cpu().pin_memory() for x in self.x]
        self.h_out = [(torch.empty(c.numel(), dtype=torch.uint8).pin_memory(),
                       torch.empty(s.numel(), dtype=torch.float32).pin_memory())
                      for c, s in self.out]
        d2h = sum(c.numel() + 4 * s.numel() for c, s in self.out)
        return sum(4 * x.numel() for x in self.x), d2h

    def e2e_bytes(self):
        return self.step_bytes()

    def step_bytes(self):
        return self.P * (4 * self.n + packed_bytes(4, self.n, 128)) + self._reduce_bytes()

    def e2e_step(self):
        """Every GPU's fp32 gradient from host memory, the reduced chunks to host memory."""
        zq = self.zq
        for g in range(self.P):
            self.x[g].copy_(self.h_x[g], non_blocking=True)
            zq.quantize_reordered(self.x[g], zq.INT4, 128, self.A, self.L, *self.q[g])
        self.two_hop()
        for (c, s), (hc, hs) in zip(self.out, self.h_out):
            hc.copy_(c, non_blocking=True)
            hs.copy_(s, non_blocking=True)

    def oracle_sample(self, sample=1 << 24):
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        P = self.A * self.L
        sample = max(P * 4096, sample - sample % (P * 4096))
        host = getattr(self, "host_sample", None)
        if host is None or host[0].size < sample:
            host = [inputs.gradient_shard_f32(sample, shard=g) for g in range(P)]
        xs = [np.ascontiguousarray(x[:sample]) for x in host]

        def run():
            qs = [O.quantize_reordered(x, O.INT4, 128, self.A, self.L) for x in xs]
            O.reduce_two_hop([c for c, _ in qs], [s for _, s in qs], self.A, self.L, sample,
                             O.INT4, 128, O.INT4, 128, O.INT4, 128)

        m = sample // P
        nbytes = (P * (4 * sample + packed_bytes(4, sample, 128))
                  + P * (self.L + 1) * packed_bytes(4, self.A * m, 128)
                  + P * (self.A + 1) * packed_bytes(4, m, 128))
        return run, nbytes, (f"first {sample:,} elements of each of the 8 GPUs' gradients, "
                             "reordered quantize and both hops, single thread")


class AgoqFP8:
    """E4M3 main gradient of 268,435,456 elements, G=128; a step adds 4
    micro-batch bf16 gradients ~ N(0, 1e-3) (seed 4, stream = micro-batch) in
    place, then reduces 8 shards of n/8 elements to one E4M3 output with its
    own scales (the slices of the main gradient stand in for the slice every
    peer sends after the all-to-all)."""

    name = "agoq_fp8"
    dtype = "e4m3 codes + fp32 scales, bf16 gradients in, fp32 sums"
    n = 268435456
    G = 128
    steps = 4
    N = 8

    def config(self):
        return {"workload": "agoq_fp8: E4M3 main gradient of 268,435,456 elements, fp32 scale per "
                            "128-block; 4 accumulate steps of bf16 N(0,1e-3) gradients "
                            "(dequant -> add in fp32 -> requant, in place), then an 8-shard FP8 "
                            "local reduce of 8 x 33,554,432 elements in fp32 and requant",
                "elements": self.n, "micro_batches": self.steps, "reduce_shards": self.N,
                "l2": "no flush: 1.1 GB moved per accumulate launch >> 126 MB L2"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq
        from blockwise_quantized_zero_gb300 import inputs

        self.zq = zq
        self.mc = torch.zeros(zq.codes_bytes(zq.E4M3, self.n), dtype=torch.uint8, device="cuda")
        self.ms = torch.zeros(zq.num_blocks(self.n, self.G), dtype=torch.float32, device="cuda")
        self.grads = []
        for k in range(self.steps):
            g = inputs.gradient_bf16(self.n, step=k)
            if k == 0:
                self.host_grad0 = g[: 1 << 26].copy()
            self.grads.append(_dev_bf16(g))
            del g
        m = self.n // self.N
        self.sc = [self.mc[r * m:(r + 1) * m] for r in range(self.N)]
        self.ss = [self.ms[r * m // self.G:(r + 1) * m // self.G] for r in range(self.N)]
        self.oc = zq.empty_codes(zq.E4M3, m, "cuda")
        self.os = zq.empty_scales(m, self.G, "cuda")
        for g in self.grads:  # the reduce's inputs hold an accumulated gradient from the start
            zq.fp8_accumulate(self.mc, self.ms, g, self.G)
        torch.cuda.synchronize()

    def launches(self):
        zq, n, G = self.zq, self.n, self.G
        acc_bytes = 2 * packed_bytes(0x48, n, G) + 2 * n
        m = n // self.N
        out = [Launch(f"fp8_accumulate e4m3 G=128 step {k}", "fp8_accumulate", acc_bytes,
                      lambda k=k: zq.fp8_accumulate(self.mc, self.ms, self.grads[k], G))
               for k in range(self.steps)]
        out.append(Launch("reduce 8x e4m3 G=128 -> e4m3 G=128", "reduce",
                          (self.N + 1) * packed_bytes(0x48, m, G),
                          lambda: zq.reduce_quantized(self.sc, self.ss, m, zq.E4M3, G, zq.E4M3, G,
                                                      self.oc, self.os)))
        return out

    def setup_e2e(self):
        import torch

        self.h_grad = self.grads[0].cpu().pin_memory()
        self.h_mc = torch.empty(self.mc.numel(), dtype=torch.uint8).pin_memory()
        self.h_ms = torch.empty(self.ms.numel(), dtype=torch.float32).pin_memory()
        self.h_oc = torch.empty(self.oc.numel(), dtype=torch.uint8).pin_memory()
        self.h_os = torch.empty(self.os.numel(), dtype=torch.float32).pin_memory()
        return (self.steps * 2 * self.n + self.mc.numel() + 4 * self.ms.numel(),
                self.mc.numel() + 4 * self.ms.numel() + self.oc.numel() + 4 * self.os.numel())

    def e2e_step(self):
        """Host main gradient in, 4 host micro-batch gradients, host results out."""
        zq, G = self.zq, self.G
        self.mc.copy_(self.h_mc, non_blocking=True)
        self.ms.copy_(self.h_ms, non_blocking=True)
        for k in range(self.steps):
            self.grads[k].copy_(self.h_grad, non_blocking=True)
            zq.fp8_accumulate(self.mc, self.ms, self.grads[k], G)
        m = self.n // self.N
        zq.reduce_quantized(self.sc, self.ss, m, zq.E4M3, G, zq.E4M3, G, self.oc, self.os)
        self.h_mc.copy_(self.mc, non_blocking=True)
        self.h_ms.copy_(self.ms, non_blocking=True)
        self.h_oc.copy_(self.oc, non_blocking=True)
        self.h_os.copy_(self.os, non_blocking=True)

    def oracle_sample(self, sample=1 << 26):
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        g = getattr(self, "host_grad0", None)
        if g is None or g.size < sample:
            g = inputs.gradient_bf16(sample, step=0)
        g = np.ascontiguousarray(g[:sample])
        G = self.G

        def run():
            c = np.zeros(sample, np.uint8)
            s = np.zeros(sample // G, np.float32)
            for _ in range(self.steps):
                c, s = O.fp8_accumulate(c, s, g, G, grad_dtype=O.BF16)
            m = sample // self.N
            O.reduce([c[r * m:(r + 1) * m] for r in range(self.N)],
                     [s[r * m // G:(r + 1) * m // G] for r in range(self.N)], m, O.E4M3, G, O.E4M3, G)

        acc = self.steps * (2 * packed_bytes(0x48, sample, G) + 2 * sample)
        red = (self.N + 1) * packed_bytes(0x48, sample // self.N, G)
        return run, acc + red, (f"{sample:,}-element main gradient: 4 accumulate steps + 8-shard "
                                "reduce of its slices, single thread")


class Llama70B:
    """One Llama-3-70B decoder layer's bf16 weights (7 matrices, 855,638,016
    elements, N(0, 0.02), seed 5): int8 G=256 and 6-bit G=32 quantize +
    dequantize -> bf16, one call per matrix (`llama70b_batched`: per scheme one
    zq_quantize_multi and one zq_dequantize_multi call over the seven matrices,
    with the same results)."""

    name = "llama70b"
    dtype = "bf16 in, int8 / int6 codes + fp32 scales, bf16 out (fp32 arithmetic)"
    schemes = ((8, 256), (6, 32))
    batched = False

    def config(self):
        how = ("per scheme one multi-tensor quantize and one multi-tensor dequantize call over the "
               "seven matrices" if self.batched else "one call per matrix")
        return {"workload": "llama70b: one Llama-3-70B decoder layer in bf16 (q,o 8192x8192; k,v "
                            "8192x1024; gate,up 8192x28672; down 28672x8192; 855,638,016 elements, "
                            "N(0,0.02)), quantize + dequantize->bf16 at int8 G=256 and 6-bit G=32",
                "elements": 855638016, "calls": how,
                "l2": "no flush: each launch streams whole matrices (1.7 GB in, 0.7-0.9 GB out)"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq
        from blockwise_quantized_zero_gb300 import inputs

        self.zq = zq
        self.mats = []
        for name, r, c, bits in inputs.llama70b_layer_bf16():
            if name == "q":
                self.host_q = bits.copy()
            self.mats.append((name, r * c, _dev_bf16(bits)))
            del bits
        self.buf = {}
        for b, G in self.schemes:
            for name, n, _ in self.mats:
                self.buf[(b, G, name)] = (zq.empty_codes(b, n, "cuda"), zq.empty_scales(n, G, "cuda"),
                                          torch.empty(n, dtype=torch.bfloat16, device="cuda"))

    def launches(self):
        zq = self.zq
        out = []
        for b, G in self.schemes:
            if self.batched:
                xs = [x for _, _, x in self.mats]
                cs = [self.buf[(b, G, name)][0] for name, _, _ in self.mats]
                ss = [self.buf[(b, G, name)][1] for name, _, _ in self.mats]
                ys = [self.buf[(b, G, name)][2] for name, _, _ in self.mats]
                ns = [n for _, n, _ in self.mats]
                nb = sum(2 * n + packed_bytes(b, n, G) for n in ns)
                out.append(Launch(f"quantize bf16 int{b} G={G} layer (one multi-tensor call)",
                                  "quantize", nb,
                                  lambda xs=xs, b=b, G=G, cs=cs, ss=ss: zq.quantize_multi(xs, b, G, cs, ss)))
                out.append(Launch(f"dequantize int{b} G={G} bf16 layer (one multi-tensor call)",
                                  "dequantize", nb,
                                  lambda cs=cs, ss=ss, ns=ns, b=b, G=G, ys=ys: zq.dequantize_multi(
                                      cs, ss, ns, b, G, outs=ys)))
                continue
            for name, n, x in self.mats:
                c, s, y = self.buf[(b, G, name)]
                nb = 2 * n + packed_bytes(b, n, G)
                out.append(Launch(f"quantize bf16 int{b} G={G} {name}", "quantize", nb,
                                  lambda x=x, b=b, G=G, c=c, s=s: zq.quantize(x, b, G, c, s)))
            for name, n, x in self.mats:
                c, s, y = self.buf[(b, G, name)]
                nb = 2 * n + packed_bytes(b, n, G)
                out.append(Launch(f"dequantize int{b} G={G} bf16 {name}", "dequantize", nb,
                                  lambda n=n, b=b, G=G, c=c, s=s, y=y: zq.dequantize(c, s, n, b, G, out=y)))
        return out

    def setup_e2e(self):
        import torch

        name, n, x = self.mats[4]  # gate, 8192 x 28672
        assert n % (4 * 1024) == 0
        self.e_name, self.e_n = name, n
        self.fork = ForkedStreams(dict)
        self.h_x = x.cpu().pin_memory()
        self.h_c = torch.empty(n, dtype=torch.uint8).pin_memory()
        self.h_s = torch.empty(n // 32, dtype=torch.float32).pin_memory()
        self.h_y = torch.empty(n, dtype=torch.bfloat16).pin_memory()
        h2d = d2h = 0
        for b, G in self.schemes:
            pb = packed_bytes(b, n, G)
            h2d += 2 * n + pb
            d2h += pb + 2 * n
        return h2d, d2h

    def e2e_step(self):
        """The gate matrix from host memory through both schemes, results to
        host, in four row chunks per scheme (chunk boundaries are block
        boundaries, so the results are those of whole-matrix calls). Items
        alternate between two streams (ForkedStreams); with four chunks per
        scheme a chunk's two items share a stream, so no slice is touched by
        both streams."""
        zq, n = self.zq, self.e_n
        x = self.mats[4][2]
        q = n // 4
        items = [(b, G, j) for b, G in self.schemes for j in range(4)]

        def one(item, _):
            b, G, j = item
            c, s, y = self.buf[(b, G, self.e_name)]
            lo, hi = j * q, (j + 1) * q
            clo, chi = lo * b // 8, hi * b // 8
            x[lo:hi].copy_(self.h_x[lo:hi], non_blocking=True)
            zq.quantize(x[lo:hi], b, G, c[clo:chi], s[lo // G:hi // G])
            self.h_c[clo:chi].copy_(c[clo:chi], non_blocking=True)
            self.h_s[lo // G:hi // G].copy_(s[lo // G:hi // G], non_blocking=True)
            c[clo:chi].copy_(self.h_c[clo:chi], non_blocking=True)
            s[lo // G:hi // G].copy_(self.h_s[lo // G:hi // G], non_blocking=True)
            zq.dequantize(c[clo:chi], s[lo // G:hi // G], hi - lo, b, G, out=y[lo:hi])
            self.h_y[lo:hi].copy_(y[lo:hi], non_blocking=True)

        self.fork.run(items, one)

    def e2e_bytes(self):
        n = self.e_n
        return sum(2 * (2 * n + packed_bytes(b, n, G)) for b, G in self.schemes)

    def oracle_sample(self, sample=1 << 26):
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        x = getattr(self, "host_q", None)
        if x is None or x.size < sample:
            x = next(inputs.llama70b_layer_bf16(scale_rows=4))[3]
        sample = min(sample, x.size)
        x = np.ascontiguousarray(x[:sample])

        def run():
            for b, G in self.schemes:
                c, s = O.quantize(x, b, G, dtype=O.BF16)
                O.dequantize(c, s, sample, b, G, O.BF16)

        nbytes = sum(2 * (2 * sample + packed_bytes(b, sample, G)) for b, G in self.schemes)
        return run, nbytes, (f"first {sample:,} elements of the q projection, int8 G=256 and 6-bit "
                             "G=32 round trips, single thread")


class Llama70BBatched(Llama70B):
    """The Llama-3-70B layer round trip through the multi-tensor calls (4 launches a step)."""

    name = "llama70b_batched"
    batched = True


class Llama70BGemm:
    """The dequantization fused into the consumer GEMM: one Llama-3-70B
    decoder layer's seven projections (N x K weights: q, o 8192 x 8192; k, v
    1024 x 8192; gate, up 28672 x 8192; down 8192 x 28672, the layer's seeded
    N(0, 0.02) bf16 matrices), held as int8 G=256 codes (qwZ's weight format),
    applied to 4096 tokens of bf16 activations with zq_gemm_dequant, bf16
    output. The bf16 weights are never materialized. For context the same
    layer is also timed unfused (zq_dequantize to bf16, then cuBLAS bf16
    matmul) during setup; that path is not part of the step."""

    name = "llama70b_gemm"
    dtype = "bf16 activations x int8 G=256 weights (dequantized to bf16 on chip), fp32 accumulate, bf16 out"
    M = 4096
    fmt, G = 8, 256

    def config(self):
        return {"workload": "llama70b_gemm: the seven projections of one Llama-3-70B decoder layer "
                            "(855,638,016 weights, int8 G=256) on 4096 bf16 tokens, dequantization "
                            "fused into the tcgen05 GEMM",
                "tokens": self.M, "weights": 855638016,
                "context_unfused_ms_per_step": getattr(self, "unfused_ms", None),
                "context_cublas_bf16_ms_per_step": getattr(self, "cublas_ms", None),
                "l2": "no flush: 0.9 GB of weights and 1.2 GB of activations/outputs per step"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq
        from blockwise_quantized_zero_gb300 import inputs

        self.zq = zq
        self.mats = []
        for name, r, c, bits in inputs.llama70b_layer_bf16():
            N, K = c, r  # output features x input features
            w = _dev_bf16(bits)
            codes, scales = zq.quantize(w, self.fmt, self.G)
            self.mats.append((name, N, K, codes, scales))
            del w, bits
        self.x = {}
        for K in sorted({K for _, _, K, _, _ in self.mats}):
            self.x[K] = _dev_bf16(inputs.to_bf16_bits(inputs.normal_f32(self.M * K, 1.0, 7, stream=K))
                                  ).reshape(self.M, K)
        self.y = {name: torch.empty(self.M, N, dtype=torch.bfloat16, device="cuda")
                  for name, N, _, _, _ in self.mats}
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        self._context()

    def _context(self):
        """The unfused alternative on the same layer: dequantize to bf16, then
        cuBLAS bf16 matmul (torch.matmul); and the matmul alone."""
        import torch

        zq = self.zq
        wb = {name: torch.empty(N, K, dtype=torch.bfloat16, device="cuda")
              for name, N, K, _, _ in self.mats}

        def unfused():
            for name, N, K, c, s in self.mats:
                zq.dequantize(c, s, N * K, self.fmt, self.G, out=wb[name].view(-1))
                torch.matmul(self.x[K], wb[name].t(), out=self.y[name])

        def matmul_only():
            for name, N, K, _, _ in self.mats:
                torch.matmul(self.x[K], wb[name].t(), out=self.y[name])

        out = []
        for fn in (unfused, matmul_only):
            for _ in range(2):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(5):
                fn()
            e1.record()
            torch.cuda.synchronize()
            out.append(round(e0.elapsed_time(e1) / 5, 3))
        self.unfused_ms, self.cublas_ms = out
        del wb
        torch.cuda.empty_cache()

    def launches(self):
        zq, M = self.zq, self.M
        out = []
        for name, N, K, c, s in self.mats:
            nb = 2 * M * K + packed_bytes(self.fmt, N * K, self.G) + 2 * M * N
            out.append(Launch(f"gemm_dequant int8 G=256 {name} {M}x{N}x{K}", "gemm_dequant", nb,
                              lambda name=name, N=N, K=K, c=c, s=s: zq.gemm_dequant(
                                  self.x[K], c, s, self.fmt, self.G, N, out=self.y[name]),
                              flops=2 * M * N * K))
        return out

    def setup_e2e(self):
        """End to end: the q projection's activations from host memory, its
        output back to host memory (weights stay resident, as gathered)."""
        import torch

        _, N, K, _, _ = self.mats[0]
        self.h_x = self.x[K].cpu().pin_memory()
        self.h_y = torch.empty(self.M, N, dtype=torch.bfloat16).pin_memory()
        return 2 * self.M * K, 2 * self.M * N

    def e2e_step(self):
        name, N, K, c, s = self.mats[0]
        self.x[K].copy_(self.h_x, non_blocking=True)
        self.zq.gemm_dequant(self.x[K], c, s, self.fmt, self.G, N, out=self.y[name])
        self.h_y.copy_(self.y[name], non_blocking=True)

    def e2e_bytes(self):
        _, N, K, _, _ = self.mats[0]
        return 2 * self.M * K + packed_bytes(self.fmt, N * K, self.G) + 2 * self.M * N

    def oracle_sample(self, sample=1 << 12):
        """The oracle's exact dequant-fused products for `sample` output
        elements of the q projection (K = 8192 products each)."""
        import oracle as O
        from blockwise_quantized_zero_gb300 import inputs

        K = N = 8192
        rows = 64
        w = next(inputs.llama70b_layer_bf16(scale_rows=128))[3]  # 64 x 8192 of the q matrix
        codes, scales = O.quantize(w, self.fmt, self.G, dtype=O.BF16)
        x = inputs.to_bf16_bits(inputs.normal_f32(rows * K, 1.0, 7, stream=K))
        r = np.random.default_rng(0)
        rr, cc = r.integers(0, rows, sample), r.integers(0, rows, sample)

        def run():
            O.gemm_dequant(x, rows, K, codes, scales, self.fmt, self.G, rows, rows=rr, cols=cc)

        nbytes = sample * (2 * K + K + 4 * K // self.G + 2)
        return run, nbytes, (f"{sample:,} outputs of a {rows} x {rows} x {K} slice of the q "
                             "projection, single thread")


class AquavitSchedule:
    """Aquavit's weight codec over its ascending schedule: bpw(t) = 8 -
    6/(a + c t/T) with (a, c) = (0.9, 5) and T = 1000 steps, each step's width
    mapped to the nearest available b + 32/G (b in {2,4,6}). A benchmark step
    is one whole schedule on the 8192x8192 bf16 weight shard (N(0, 0.02),
    seed 2): every schedule step quantizes the shard at its (b, G) and
    dequantizes it to bf16, once in the metadata-interleaved record layout and
    once in the planar layout, so the two layouts compare on the same calls.
    Calls rotate over 8 buffer sets (no call finds its inputs in L2)."""

    name = "aquavit_schedule"
    dtype = "bf16 in, int2/4/6 codes + fp32 scales (interleaved records or planar), bf16 out"
    rows, cols = 8192, 8192
    a, c = 0.9, 5.0
    slots = 8

    def __init__(self, T=1000):
        from blockwise_quantized_zero_gb300 import inputs

        if T < 1:
            raise SystemExit("the schedule needs at least one step")
        self.T = T
        self.n = self.rows * self.cols
        self.host = inputs.weight_shard_bf16(self.rows, self.cols)

    def config(self):
        return {"workload": f"aquavit_schedule: one 8192x8192 bf16 weight shard (N(0,0.02)); the "
                            f"{self.T}-step ascending schedule bpw = 8 - 6/(0.9 + 5 t/{self.T}), each step "
                            "quantize + dequantize->bf16 at its nearest (b, G); interleaved "
                            "records and planar layout, each for the whole schedule",
                "elements": self.n, "schedule_steps": self.T, "a": self.a, "c": self.c,
                "pairs": {f"{b}:{G}": k for (b, G), k in sorted(self.counts.items())}
                if hasattr(self, "counts") else None,
                "mean_bpw": getattr(self, "mean_bpw", None),
                "l2": "no flush: calls rotate over 8 buffer sets of 134 MB source + output each"}

    def setup(self):
        import torch

        import blockwise_quantized_zero_gb300 as zq

        self.zq = zq
        counts = {}
        width = 0.0
        for t in range(self.T):
            fmt, G, _, w = zq.aquavit_schedule(t, self.T, self.a, self.c)
            counts[(fmt, G)] = counts.get((fmt, G), 0) + 1
            width += w
        self.counts, self.mean_bpw = counts, round(width / self.T, 5)
        n, S = self.n, self.slots
        src0 = _dev_bf16(self.host)
        self.src = [src0] + [src0.clone() for _ in range(S - 1)]
        rmax = max(zq.interleaved_bytes(b, n, G) for b, G in counts)
        self.rec = [torch.empty(rmax, dtype=torch.uint8, device="cuda") for _ in range(S)]
        self.codes = [torch.empty(zq.codes_bytes(6, n), dtype=torch.uint8, device="cuda")
                      for _ in range(S)]
        self.scales = [torch.empty(zq.num_blocks(n, 32), dtype=torch.float32, device="cuda")
                       for _ in range(S)]
        self.out = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(S)]

    def _calls(self, k, body):
        def run():
            for j in range(k):
                body(j % self.slots)
        return run

    def launches(self):
        zq, n = self.zq, self.n
        out = []
        for (b, G), k in sorted(self.counts.items()):
            nb = 2 * n + packed_bytes(b, n, G)
            rb, cb, sb = zq.interleaved_bytes(b, n, G), zq.codes_bytes(b, n), zq.num_blocks(n, G)
            out.append(Launch(f"quantize_il bf16 {fmt_name(b)} G={G} x{k}", "quantize_il", k * nb,
                              self._calls(k, lambda i, b=b, G=G, rb=rb: zq.quantize_interleaved(
                                  self.src[i], b, G, self.rec[i][:rb])), kernels=k))
            out.append(Launch(f"dequantize_il {fmt_name(b)} G={G} bf16 x{k}", "dequantize_il",
                              k * nb, self._calls(k, lambda i, b=b, G=G, rb=rb:
                                                  zq.dequantize_interleaved(
                                                      self.rec[i][:rb], n, b, G, out=self.out[i])),
                              kernels=k))
            out.append(Launch(f"quantize bf16 {fmt_name(b)} G={G} x{k}", "quantize", k * nb,
                              self._calls(k, lambda i, b=b, G=G, cb=cb, sb=sb: zq.quantize(
                                  self.src[i], b, G, self.codes[i][:cb], self.scales[i][:sb])),
                              kernels=k))
            out.append(Launch(f"dequantize {fmt_name(b)} G={G} bf16 x{k}", "dequantize", k * nb,
                              self._calls(k, lambda i, b=b, G=G, cb=cb, sb=sb: zq.dequantize(
                                  self.codes[i][:cb], self.scales[i][:sb], n, b, G,
                                  out=self.out[i])), kernels=k))
        return out

    def step_bytes(self):
        return sum(2 * 2 * k * (2 * self.n + packed_bytes(b, self.n, G))
                   for (b, G), k in self.counts.items())

    # end to end: each of the 18 pairs once, interleaved records through host memory
    def setup_e2e(self):
        import torch

        zq, n = self.zq, self.n
        self.h_src = torch.from_numpy(self.host.view(np.int16)).view(torch.bfloat16).pin_memory()
        rmax = self.rec[0].numel()

        def make_set():
            dev = dict(device="cuda")
            return dict(h_rec=torch.empty(rmax, dtype=torch.uint8).pin_memory(),
                        h_out=torch.empty(n, dtype=torch.bfloat16).pin_memory(),
                        d_src=torch.empty(n, dtype=torch.bfloat16, **dev),
                        d_rec=torch.empty(rmax, dtype=torch.uint8, **dev),
                        d_rec2=torch.empty(rmax, dtype=torch.uint8, **dev),
                        d_out=torch.empty(n, dtype=torch.bfloat16, **dev))

        self.fork = ForkedStreams(make_set)
        h2d = sum(2 * n + zq.interleaved_bytes(b, n, G) for b, G in self.counts)
        d2h = sum(zq.interleaved_bytes(b, n, G) + 2 * n for b, G in self.counts)
        return h2d, d2h

    def e2e_step(self):
        """Per pair: host src -> quantize_interleaved -> host records; host
        records -> dequantize_interleaved -> host out (pairs alternate between
        two streams)."""
        zq, n = self.zq, self.n

        def one(pair, B):
            b, G = pair
            rb = zq.interleaved_bytes(b, n, G)
            B["d_src"].copy_(self.h_src, non_blocking=True)
            zq.quantize_interleaved(B["d_src"], b, G, B["d_rec"][:rb])
            B["h_rec"][:rb].copy_(B["d_rec"][:rb], non_blocking=True)
            B["d_rec2"][:rb].copy_(B["h_rec"][:rb], non_blocking=True)
            zq.dequantize_interleaved(B["d_rec2"][:rb], n, b, G, out=B["d_out"])
            B["h_out"].copy_(B["d_out"], non_blocking=True)

        self.fork.run(sorted(self.counts), one)

    def e2e_bytes(self):
        return sum(2 * (2 * self.n + packed_bytes(b, self.n, G)) for b, G in self.counts)

    def oracle_sample(self, sample=1 << 22):
        import oracle as O

        x = np.ascontiguousarray(self.host[:sample])
        pairs = sorted({O.aquavit_pick(O.aquavit_bpw(t, self.T, self.a, self.c))[:2]
                        for t in range(self.T)})

        def run():
            for b, G in pairs:
                rec = O.quantize_interleaved(x, b, G, dtype=O.BF16)
                O.dequantize_interleaved(rec, sample, b, G, O.BF16)

        nbytes = sum(2 * (2 * sample + packed_bytes(b, sample, G)) for b, G in pairs)
        desc = (f"first {sample:,} elements of the shard, each of the schedule's {len(pairs)} "
                "(b, G) pairs once, interleaved quantize + dequantize->bf16, single thread")
        return run, nbytes, desc


class Llama70BGemmFew(Llama70BGemm):
    """The same fused GEMM on 128 tokens (a few-token forward: decode or a
    small micro-batch). Every projection has fewer 128-row output tiles than
    the GPU has SMs, so the launcher splits K over clusters of CTAs (128 x 256
    tiles, 4 CTAs a tile, for q, o and down; 128 x 128 tiles, 8 CTAs, for k
    and v; 256 x 128 unsplit tiles for gate and up). At 128 tokens an int8
    weight byte carries 256 flops, so the weights' HBM time and the tensor
    time are about equal; both rooflines are reported."""

    name = "llama70b_gemm_t128"
    M = 128

    def config(self):
        c = super().config()
        c["workload"] = ("llama70b_gemm_t128: the seven projections of one Llama-3-70B decoder layer "
                         "(855,638,016 weights, int8 G=256) on 128 bf16 tokens, dequantization fused "
                         "into the tcgen05 GEMM, K split over clusters where the tiles are too few")
        c["l2"] = "no flush: 0.9 GB of int8 weights per step >> 126 MB L2"
        return c


WORKLOADS = {"gm_sweep": GMSweep, "qwz_fp16": QwzFP16, "qgz_reduce": QgzReduce,
             "agoq_fp8": AgoqFP8, "llama70b": Llama70B, "qgz_two_hop": QgzTwoHop,
             "llama70b_gemm": Llama70BGemm, "llama70b_gemm_t128": Llama70BGemmFew,
             "llama70b_batched": Llama70BBatched,
             "aquavit_schedule": AquavitSchedule, "ring_study": RingStudy}


# ---------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if _cuda_ok() else "gloo"
        if backend == "nccl":
            import torch

            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def _cuda_ok():
    try:
        import torch

        return torch.cuda.is_available()
    except Exception:  # noqa: BLE001
        return False


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(per_rank_bytes: float, elapsed_s: list[float], world: int) -> tuple[float, float]:
    """Whole-job throughput: bytes of all ranks over the slowest rank's time."""
    t = max(elapsed_s)
    return world * per_rank_bytes / t / 1e9, t


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

REFERENCE_BUDGET_S = 120.0  # whole reference run (warm-up + timed steps)


def reference_sample(wl, steps: int, warmup: int) -> int:
    """Sample size per step so that (steps + warmup) steps of the oracle take
    about REFERENCE_BUDGET_S, from a calibration run on a small sample."""
    probe = 1 << 16
    run, _, _ = wl.oracle_sample(probe)
    t0 = time.perf_counter()
    run()
    per_elem = (time.perf_counter() - t0) / probe
    target = REFERENCE_BUDGET_S / max(1, steps + warmup)
    n = int(target / max(per_elem, 1e-12))
    return max(1 << 14, min(1 << 26, (n // 1024) * 1024))


def make_workload(args):
    if args.pair:
        if args.workload != "gm_sweep":
            raise SystemExit("--pair applies to --workload gm_sweep only")
        b, G = (int(v) for v in args.pair.split(":"))
        return GMSweep(pair=(b, G))
    if args.schedule_steps is not None:
        if args.workload != "aquavit_schedule":
            raise SystemExit("--schedule-steps applies to --workload aquavit_schedule only")
        return AquavitSchedule(T=args.schedule_steps)
    return WORKLOADS[args.workload]()


def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl = make_workload(args)
    sample = args.oracle_sample if args.oracle_sample else reference_sample(wl, args.steps, args.warmup)
    run, nbytes, desc = wl.oracle_sample(sample)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = (time.perf_counter() - t0) / args.steps
    value = nbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic", "config": wl.config(),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def _oracle_sample(wl, sample):
    return wl.oracle_sample() if sample is None else wl.oracle_sample(sample)


def time_cpu_baseline(wl, sample):
    run, nbytes, desc = _oracle_sample(wl, sample)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": desc, "seconds": round(dt, 2)}


def _oracle_core_worker(name, sample, barrier, queue):
    """One process of the all-cores oracle timing: the unchanged single-threaded
    oracle on `sample` elements of the workload, started together with the
    other processes (host data only; no GPU)."""
    try:
        wl = WORKLOADS[name]()
        run, nbytes, desc = _oracle_sample(wl, sample)
        barrier.wait(timeout=900)
        t0 = time.monotonic()
        run()
        queue.put((t0, time.monotonic(), nbytes, desc))
    except Exception as e:  # reported by the parent
        queue.put(("error", repr(e)))


def time_cpu_all_cores(wl, sample):
    """The oracle on every host core this process may use: one spawned process
    per core, each on an equal share of the single-core sample (a whole copy of
    it when the workload's sample is not an element count), started at a
    barrier; the wall time runs from the first start to the last end."""
    import inspect
    import multiprocessing as mp

    cores = len(os.sched_getaffinity(0))
    if sample is None:
        sample = inspect.signature(wl.oracle_sample).parameters["sample"].default
    per = max(8192, (sample // cores) // 8192 * 8192) if isinstance(sample, int) else sample
    ctx = mp.get_context("spawn")
    barrier, queue = ctx.Barrier(cores), ctx.Queue()
    procs = [ctx.Process(target=_oracle_core_worker, args=(wl.name, per, barrier, queue))
             for _ in range(cores)]
    for p in procs:
        p.start()
    res = [queue.get(timeout=1800) for _ in procs]
    for p in procs:
        p.join()
    bad = [r for r in res if r[0] == "error"]
    if bad:
        return {"error": bad[0][1], "cores": cores}
    t0, t1 = min(r[0] for r in res), max(r[1] for r in res)
    nbytes = sum(r[2] for r in res)
    return {"value": round(nbytes / (t1 - t0) / 1e9, 4), "unit": UNIT, "cores": cores,
            "kind": "oracle", "sample": f"{cores} processes, each: {res[0][3]}",
            "seconds": round(t1 - t0, 2)}


# The configurations timed after the headline workload in the same run (the
# other single-GPU workloads of the method: the batched 1 Mi fp16 round trip,
# the granularity sweep, the qgZ reduce and the AGoQ FP8 accumulate + reduce;
# the headline layer again through the multi-tensor calls; then the
# dequantization fused into the consumer GEMM, on 4096 and on 128 tokens).
EXTRA_CONFIGS = ("qwz_fp16", "gm_sweep", "qgz_reduce", "agoq_fp8", "llama70b_batched",
                 "llama70b_gemm", "llama70b_gemm_t128")
EXTRA_STEPS = 20  # timed steps per extra configuration (at most --steps)
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, the ~8 TB/s nominal figure


def check_device(zq, what: str):
    """Refuse to report a number measured while a bounded device-side wait ran
    out (the kernels' outputs would then be incomplete)."""
    try:
        zq.device_status()
    except zq.ZQError as e:
        raise SystemExit(f"bench.py: {what}: {e}; a bounded device-side wait ran out, so no "
                         "number is reported") from None


def _groups(launches):
    """Maximal runs of consecutive launches of one kernel family."""
    groups = []
    for i, l in enumerate(launches):
        if groups and groups[-1][0] == l.family:
            groups[-1][1].append(i)
        else:
            groups.append((l.family, [i]))
    return groups


def family_table(fam, peak):
    out = {}
    burst, sustained, _ = measured_tensor_peak()
    for k, v in fam.items():
        row = {"gbs": round(v[1] / (v[0] / 1e3) / 1e9, 1),
               "frac": round(v[1] / (v[0] / 1e3) / 1e9 / peak, 4),
               "frac_of_nominal_hbm": round(v[1] / (v[0] / 1e3) / 1e9 / NOMINAL_HBM_GBS, 4),
               "bytes_per_launch": int(v[1] / v[2]),
               "us_per_launch": round(v[0] / v[2] * 1e3, 2), "launches": v[2]}
        if v[3]:  # a contraction: its roofline is the tensor-core rate
            tf = v[3] / (v[0] / 1e3) / 1e12
            row.update({"tflops": round(tf, 1), "frac_of_bf16_burst": round(tf / burst, 4),
                        "frac_of_bf16_sustained": round(tf / sustained, 4),
                        "flops_per_launch": int(v[3] / v[2])})
            row["bound"] = "tensor"
        out[k] = row
    return out


def time_steps(launches, steps, world, stream, per_launch=True):
    """Time `steps` steps of `launches` in up to three regions (see run_gpu).
    Returns (elapsed seconds of the back-to-back region, max over ranks;
    per-family [ms, bytes, launches]; per-label [ms, bytes, count] or None)."""
    import torch

    groups = _groups(launches)

    def step(evs=None):
        for i, l in enumerate(launches):
            if evs is not None:
                evs[i][0].record(stream)
            l.fn()
            if evs is not None:
                evs[i][1].record(stream)

    def ev():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    gevs = [[ev() for _ in groups] for _ in range(steps)]
    evs = [[ev() for _ in launches] for _ in range(steps)] if per_launch else None
    t_start, t_end = ev()
    barrier(world)
    torch.cuda.synchronize()
    t_start.record(stream)
    for _ in range(steps):
        step()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    for k in range(steps):
        for gi, (_, idx) in enumerate(groups):
            gevs[k][gi][0].record(stream)
            for i in idx:
                launches[i].fn()
            gevs[k][gi][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    if per_launch:
        for k in range(steps):
            step(evs[k])
        torch.cuda.synchronize()
        barrier(world)
    elapsed = max_over_ranks(t_start.elapsed_time(t_end) / 1e3, world)
    fam = {}
    for k in range(steps):
        for gi, (family, idx) in enumerate(groups):
            f = fam.setdefault(family, [0.0, 0, 0, 0])
            f[0] += gevs[k][gi][0].elapsed_time(gevs[k][gi][1])
            f[1] += sum(launches[i].nbytes for i in idx)
            f[2] += sum(launches[i].kernels for i in idx)
            f[3] += sum(launches[i].flops for i in idx)
    per_label = None
    if per_launch:
        per_label = {}
        for k in range(steps):
            for i, l in enumerate(launches):
                pl = per_label.setdefault(l.label, [0.0, 0, 0])
                pl[0] += evs[k][i][0].elapsed_time(evs[k][i][1])
                pl[1] += l.nbytes
                pl[2] += 1
    return elapsed, fam, per_label


def run_extra_config(name, args, world):
    """Set up one more workload, time its kernel families (same protocol as the
    headline, fewer steps), check the device error words, free it."""
    import torch

    import blockwise_quantized_zero_gb300 as zq

    t0 = time.perf_counter()
    wl = WORKLOADS[name]()
    wl.setup()
    launches = wl.launches()
    stream = torch.cuda.current_stream()
    steps = max(1, min(args.steps, EXTRA_STEPS))
    for _ in range(args.warmup):
        for l in launches:
            l.fn()
    torch.cuda.synchronize()
    elapsed, fam, _ = time_steps(launches, steps, world, stream, per_launch=False)
    check_device(zq, name)
    peak, _ = measured_peak()
    step_bytes = sum(l.nbytes for l in launches)
    value, _ = aggregate(step_bytes * steps, [elapsed], world)
    out = {"config": wl.config(), "value": round(value, 2), "unit": UNIT,
           "frac": round(value / peak, 4), "steps": steps, "warmup": args.warmup,
           "ms_per_step": round(elapsed / steps * 1e3, 3),
           "families": family_table(fam, peak),
           "gpu_launches": sum(l.kernels for l in launches) * steps,
           "device_status": "ok", "wall_s": None}
    del launches, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    out["wall_s"] = round(time.perf_counter() - t0, 1)
    return out


def run_gpu(args, rank, world, local):
    import torch

    import blockwise_quantized_zero_gb300 as zq

    torch.cuda.set_device(local)
    wl = make_workload(args)
    wl.setup()
    launches = wl.launches()
    stream = torch.cuda.current_stream()
    step_bytes = sum(l.nbytes for l in launches)
    for _ in range(args.warmup):
        for l in launches:
            l.fn()
    torch.cuda.synchronize()
    check_device(zq, f"{wl.name} warm-up")

    # Three timed regions of K steps each (time_steps). The first runs the
    # launches back to back, as a user's stream does (the kernels use
    # programmatic dependent launch, which an event recorded between two
    # launches would defeat): it gives `value`. The second records events only
    # where the kernel family changes, so each family's launches still run back
    # to back: its group times give each family's average launch duration for
    # the roofline. The third brackets every launch with an event pair, for the
    # per-launch table (isolated launches, so it includes each launch's start-up).
    with ClockSampler(local) as clocks:
        elapsed_max, fam, per_label = time_steps(launches, args.steps, world, stream)
    check_device(zq, f"{wl.name} timed steps")
    value, _ = aggregate(step_bytes * args.steps, [elapsed_max], world)

    dominant = max(fam, key=lambda k: fam[k][0])
    peak, peak_src = measured_peak()
    ms_sum, nbytes, count, flops = fam[dominant]
    achieved = nbytes / (ms_sum / 1e3) / 1e9
    traffic = lookup_traffic(wl.name, dominant)
    if flops:  # a contraction: the tensor-core roofline (burst: the family runs alone)
        burst, _, tsrc = measured_tensor_peak()
        tf = flops / (ms_sum / 1e3) / 1e12
        roofline = {"bound": "tensor", "kernel": dominant, "achieved": round(tf, 1),
                    "peak": burst, "peak_source": f"{tsrc} bf16_tflops (cuBLAS bf16 GEMM, burst)",
                    "unit": "TFLOP/s", "frac": round(tf / burst, 4), "traffic": traffic,
                    "algorithmic_flops_per_launch": int(flops / count),
                    "us_per_launch": round(ms_sum / count * 1e3, 2)}
    else:
        roofline = {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                    "peak": peak, "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)",
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                    "frac_of_nominal_hbm": round(achieved / NOMINAL_HBM_GBS, 4),
                    "nominal_hbm_gbs": NOMINAL_HBM_GBS,
                    "target_uses": "frac (of the measured copy peak)",
                    "algorithmic_bytes_per_launch": int(nbytes / count),
                    "us_per_launch": round(ms_sum / count * 1e3, 2)}
    kpl = {l.label: l.kernels for l in launches}
    kernels = {k: {"gbs": round(v[1] / (v[0] / 1e3) / 1e9, 1),
                   "frac": round(v[1] / (v[0] / 1e3) / 1e9 / peak, 3),
                   "us_per_launch": round(v[0] / (v[2] * kpl[k]) * 1e3, 2),
                   "launches": v[2] * kpl[k]}
               for k, v in per_label.items()}

    # end to end through the C ABI with host buffers
    h2d, d2h = wl.setup_e2e()
    wl.e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_steps = max(1, min(args.steps, 3))
    barrier(world)
    e0.record(stream)
    for _ in range(e2e_steps):
        wl.e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    check_device(zq, f"{wl.name} end-to-end steps")
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_bytes = wl.e2e_bytes() if hasattr(wl, "e2e_bytes") else step_bytes
    e2e_value = world * e2e_bytes * e2e_steps / e2e_t / 1e9
    main_config = wl.config()
    gpu_launches = sum(l.kernels for l in launches) * args.steps
    del launches

    # the other configurations of the method, timed in the same run
    extra = {}
    names = [] if args.configs in ("", "none") else [c for c in args.configs.split(",") if c]
    for name in names:
        if name not in WORKLOADS or name == args.workload:
            continue
        extra[name] = run_extra_config(name, args, world)

    cpu = time_cpu_baseline(wl, args.oracle_sample) if (rank == 0 and world == 1 and not args.no_cpu) else None
    cpu_all = (time_cpu_all_cores(wl, args.oracle_sample)
               if (rank == 0 and world == 1 and not args.no_cpu) else None)
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_max / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic (seeded, blockwise_quantized_zero_gb300.inputs)",
            "config": dict(main_config, parallelism=f"replicas x{world} (no collective)"),
            "frac_of_peak": round(value / peak, 4),
            "frac_of_nominal_hbm": round(value / NOMINAL_HBM_GBS, 4),
            "roofline": roofline,
            "kernels": kernels,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": gpu_launches,
            "gpu_launches_note": "per timed region (the value's); two more regions of as many "
                                 "launches time the kernel families (events only between "
                                 "families) and each launch alone (the kernels table); the "
                                 "configs entries count their own launches",
            "families": family_table(fam, peak),
            "configs": extra,
            "device_status": "ok (checked after every timed region)",
            "clocks": clocks.summary()}
    return line


# The DRAM bytes per launch in profiles/ncu_traffic.json were captured on
# particular kernel sources: the fused GEMM's family on all of csrc/, the
# codec families (quantize, dequantize, reduce, FP8 accumulate and their
# variants) on csrc/ without the GEMM's own files. A capture whose source set
# has changed since is not reported.
GEMM_ONLY_SOURCES = ("zq_gemm.cu", "zq_gemm.cuh", "zq_tc.cuh")


def source_set(family: str) -> str:
    return "gemm" if family.startswith("gemm") else "codec"


def lookup_traffic(workload: str, family: str):
    """DRAM bytes per launch of a workload's kernel family from the committed
    ncu summaries, if they were taken on the current kernel sources; None
    otherwise."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:  # noqa: BLE001
        return None
    sset = source_set(family)
    if d.get("source_sets", {}).get(sset) != csrc_sha(sset):
        return None
    return d.get("workloads", {}).get(workload, {}).get(family)


def csrc_sha(sset: str = "gemm") -> str:
    """Hash of the kernel sources of a source set ("gemm": all of csrc/;
    "codec": csrc/ without the GEMM's own files)."""
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blockwise_quantized_zero_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if sset == "codec" and name in GEMM_ONLY_SOURCES:
            continue
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def parse_args(argv=None):
    """The command line, checked: at least 3 warm-up steps for the GPU arm,
    and the options that serve one workload (--pair, --schedule-steps) only
    with that workload."""
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["zq", "reference"], default="zq")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="llama70b")
    ap.add_argument("--configs", default=",".join(EXTRA_CONFIGS),
                    help="comma-separated workloads whose kernel families are also timed in the "
                         "same run (default: the other single-GPU configurations; 'none' to skip)")
    ap.add_argument("--oracle-sample", type=int, default=None,
                    help="elements in the CPU-oracle sample (default: the workload's own)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    ap.add_argument("--schedule-steps", type=int, default=None,
                    help="aquavit_schedule: schedule length T (default 1000, the pages' run); "
                         "shorter schedules serve profiler captures")
    ap.add_argument("--pair", default=None,
                    help="gm_sweep only: run just one (b, G) pair, given as b:G (for profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "zq":
        ap.error("at least 3 warm-up steps")
    if args.pair is not None:
        if args.workload != "gm_sweep":
            ap.error("--pair applies to --workload gm_sweep only")
        try:
            b, G = (int(v) for v in args.pair.split(":"))
        except ValueError:
            ap.error("--pair takes b:G, for example 4:128")
        if b not in (2, 4, 6, 8) or G not in (32, 64, 128, 256, 512, 1024):
            ap.error("--pair: b in {2, 4, 6, 8} and G a power of two in [32, 1024]")
    if args.schedule_steps is not None and args.workload != "aquavit_schedule":
        ap.error("--schedule-steps applies to --workload aquavit_schedule only")
    return args


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_init()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_gpu(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
