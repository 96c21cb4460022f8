"""Benchmark of the blockwise quantize / pack / dequantize / reduce path on GB300.

One JSON line (rank 0) per run. Default workload (``--workload gm_sweep``):
granularity-modulation sweep on one 8192x8192 bf16 weight shard ~ N(0, 0.02):
for every b in {2,4,6,8} and G in {1024,...,32}, quantize then dequantize to
bf16 (48 kernel launches per step). Metric: GB/s of algorithmic input+output
bytes. Other workloads (``--workload``): qwz_fp16 (1 Mi fp16 weights with
outliers, int8 G=256, batched over 512 tensors), qgz_reduce (8 int4 shards of
134,217,728 gradients -> int4 G=128 and int8 G=256), agoq_fp8 (E4M3 main
gradient of 268,435,456 elements, 4 accumulate steps + 8-shard FP8 reduce),
llama70b (one Llama-3-70B layer, int8 G=256 and 6-bit G=32 round trips).

Timing: CUDA events on the launching stream, W untimed warm-up steps, then K
timed steps bracketed by a barrier and a synchronize; the max over ranks is
reported. Every kernel of a step reads and writes its own buffers, so each
step touches several GB (far more than the 126 MB L2) and no flush is needed.
Inputs are seeded and synthetic (blockwise_quantized_zero_gb300.inputs).

``--impl reference`` times the oracle (plain single-threaded C) on a bounded
sample of the same workload instead.
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
    __slots__ = ("label", "family", "nbytes", "fn")

    def __init__(self, label, family, nbytes, fn):
        self.label, self.family, self.nbytes, self.fn = label, family, nbytes, fn


def _dev_bf16(bits: np.ndarray):
    import torch

    return torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()


class GMSweep:
    """8192x8192 bf16 ~ N(0, 0.02); b in {2,4,6,8} x G in {1024..32}; Q then D -> bf16."""

    name = "gm_sweep"
    rows, cols = 8192, 8192
    bits = (2, 4, 6, 8)
    blocks = (1024, 512, 256, 128, 64, 32)

    def __init__(self):
        from blockwise_quantized_zero_gb300 import inputs

        self.n = self.rows * self.cols
        self.pairs = [(b, G) for b in self.bits for G in self.blocks]
        self.host = inputs.weight_shard_bf16(self.rows, self.cols)

    def config(self):
        return {"workload": "gm_sweep: one 8192x8192 bf16 weight shard (67,108,864 elements, "
                            "N(0,0.02)); quantize + dequantize->bf16 for b in {2,4,6,8} x "
                            "G in {1024,512,256,128,64,32}",
                "elements": self.n, "pairs": len(self.pairs),
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

        zq = self.zq
        self.h_src = torch.from_numpy(self.host.view(np.int16)).view(torch.bfloat16).pin_memory()
        cmax = max(zq.codes_bytes(b, self.n) for b in self.bits)
        smax = zq.num_blocks(self.n, 32)
        self.h_codes = torch.empty(cmax, dtype=torch.uint8).pin_memory()
        self.h_scales = torch.empty(smax, dtype=torch.float32).pin_memory()
        self.h_out = torch.empty(self.n, dtype=torch.bfloat16).pin_memory()
        self.d_src = torch.empty(self.n, dtype=torch.bfloat16, device="cuda")
        self.d_codes = torch.empty(cmax, dtype=torch.uint8, device="cuda")
        self.d_scales = torch.empty(smax, dtype=torch.float32, device="cuda")
        self.d_codes2 = torch.empty(cmax, dtype=torch.uint8, device="cuda")
        self.d_scales2 = torch.empty(smax, dtype=torch.float32, device="cuda")
        self.d_out = torch.empty(self.n, dtype=torch.bfloat16, device="cuda")
        h2d = d2h = 0
        for b, G in self.pairs:
            cb, sb = self.zq.codes_bytes(b, self.n), 4 * self.zq.num_blocks(self.n, G)
            h2d += 2 * self.n + cb + sb
            d2h += cb + sb + 2 * self.n
        return h2d, d2h

    def e2e_step(self):
        """Per pair: host src -> quantize -> host codes; host codes -> dequantize -> host out."""
        zq, n = self.zq, self.n
        for b, G in self.pairs:
            cb, nb = zq.codes_bytes(b, n), zq.num_blocks(n, G)
            self.d_src.copy_(self.h_src, non_blocking=True)
            zq.quantize(self.d_src, b, G, self.d_codes[:cb], self.d_scales[:nb])
            self.h_codes[:cb].copy_(self.d_codes[:cb], non_blocking=True)
            self.h_scales[:nb].copy_(self.d_scales[:nb], non_blocking=True)
            self.d_codes2[:cb].copy_(self.h_codes[:cb], non_blocking=True)
            self.d_scales2[:nb].copy_(self.h_scales[:nb], non_blocking=True)
            zq.dequantize(self.d_codes2[:cb], self.d_scales2[:nb], n, b, G, out=self.d_out)
            self.h_out.copy_(self.d_out, non_blocking=True)

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


WORKLOADS = {"gm_sweep": GMSweep}


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

def run_reference(args, rank, world):
    if rank != 0:
        return None
    wl = WORKLOADS[args.workload]()
    run, nbytes, desc = wl.oracle_sample(args.oracle_sample)
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
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": wl.config(),
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    return line


def time_cpu_baseline(wl, sample):
    run, nbytes, desc = wl.oracle_sample(sample)
    t0 = time.perf_counter()
    run()
    dt = time.perf_counter() - t0
    return {"value": round(nbytes / dt / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": desc, "seconds": round(dt, 2)}


def run_gpu(args, rank, world, local):
    import torch

    torch.cuda.set_device(local)
    wl = WORKLOADS[args.workload]()
    wl.setup()
    launches = wl.launches()
    stream = torch.cuda.current_stream()
    step_bytes = sum(l.nbytes for l in launches)

    def step(evs=None):
        for i, l in enumerate(launches):
            if evs is not None:
                evs[i][0].record(stream)
            l.fn()
            if evs is not None:
                evs[i][1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in launches] for _ in range(args.steps)]
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier(world)
        torch.cuda.synchronize()
        t_start.record(stream)
        for k in range(args.steps):
            step(evs[k])
        t_end.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    elapsed = t_start.elapsed_time(t_end) / 1e3
    elapsed_max = max_over_ranks(elapsed, world)
    value, _ = aggregate(step_bytes * args.steps, [elapsed_max], world)

    # per-kernel-family launch durations
    fam = {}
    per_label = {}
    for k in range(args.steps):
        for i, l in enumerate(launches):
            ms = evs[k][i][0].elapsed_time(evs[k][i][1])
            f = fam.setdefault(l.family, [0.0, 0, 0])
            f[0] += ms
            f[1] += l.nbytes
            f[2] += 1
            pl = per_label.setdefault(l.label, [0.0, 0, 0])
            pl[0] += ms
            pl[1] += l.nbytes
            pl[2] += 1
    dominant = max(fam, key=lambda k: fam[k][0])
    peak, peak_src = measured_peak()
    ms_sum, nbytes, count = fam[dominant]
    achieved = nbytes / (ms_sum / 1e3) / 1e9
    traffic = lookup_traffic(dominant)
    kernels = {k: {"gbs": round(v[1] / (v[0] / 1e3) / 1e9, 1),
                   "frac": round(v[1] / (v[0] / 1e3) / 1e9 / peak, 3),
                   "us_per_launch": round(v[0] / v[2] * 1e3, 2), "launches": v[2]}
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
    e2e_t = max_over_ranks(e0.elapsed_time(e1) / 1e3, world)
    e2e_value = world * step_bytes * e2e_steps / e2e_t / 1e9

    cpu = time_cpu_baseline(wl, args.oracle_sample) if (rank == 0 and world == 1 and not args.no_cpu) else None
    if rank != 0:
        return None
    line = {"metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(elapsed_max / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16->int2/4/6/8 (fp32 scale math)",
            "data": "synthetic (seeded, blockwise_quantized_zero_gb300.inputs)",
            "config": dict(wl.config(), parallelism=f"replicas x{world} (no collective)"),
            "frac_of_peak": round(value / peak, 4),
            "roofline": {"bound": "hbm", "kernel": dominant, "achieved": round(achieved, 1),
                         "peak": peak, "peak_source": f"{peak_src} hbm_gbs (STREAM-style copy)",
                         "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": traffic,
                         "algorithmic_bytes_per_launch": int(nbytes / count),
                         "us_per_launch": round(ms_sum / count * 1e3, 2)},
            "kernels": kernels,
            "cpu_baseline": cpu,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps},
            "gpu_launches": len(launches) * args.steps,
            "clocks": clocks.summary()}
    return line


def lookup_traffic(family: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; None otherwise."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:  # noqa: BLE001
        return None
    if d.get("csrc_sha") != csrc_sha():
        return None
    return d.get("families", {}).get(family)


def csrc_sha() -> str:
    import hashlib

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "blockwise_quantized_zero_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["zq", "reference"], default="zq")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="gm_sweep")
    ap.add_argument("--oracle-sample", type=int, default=1 << 24)
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-oracle baseline leg")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "zq":
        ap.error("at least 3 warm-up steps")
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
