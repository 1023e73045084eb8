#!/usr/bin/env python3
"""Benchmark of the TACO ASH+DS FP8 codec hot path on GB300.

One step = one pass of the two-shot AllReduce's on-GPU path over the
GPT-6.7B-shaped workload (P = 4 shards of bf16 [8192, 4096], block 128):
fused compress of all four shards (one launch), shard reduce (FP8 -> FP32
sum -> requantise, one launch), decompress of the result to fp32 (one
launch).  Inputs are resident in HBM before the timed region and larger than
L2 (268 MB of bf16 per step), so no L2 flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  ``value`` is algorithmic HBM bytes moved per
step (reads + writes of the three kernels) x steps x ranks / max-over-ranks
time, in GB/s.  On one GPU the step is the two-shot reduce with its P
shards resident in that GPU's memory.  Under torchrun (N > 1), or with
``--exchange`` on one GPU (an NCCL group of one), each rank holds one
activation of the same shape and a step is the two-shot AllReduce across
the ranks: compress, All-to-All of codes and scalars (NCCL), shard reduce of
the received chunks, AllGather, decompress.  ``--replicas`` runs
independent replicas of the one-GPU path under torchrun instead (no
data-path collective).

After the timed region, a sampling phase of a fixed number of steps (60 by
default, whatever K is) records a CUDA event after every launch; the first
sampled step is dropped.  The per-kernel figures and the roofline come from
these samples, so they do not depend on K.  Side legs (GPT-2.7B and GPT-13B
shapes, INT8 codec, AGoQ, LAAQ) time single kernels from CUDA-graph replays.

``--impl reference`` times the CPU oracle (the plain reference
implementation of the method) on bounded samples of the same workload, on
all host cores.
"""

from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "ASH+DS FP8 compress/decompress/reduce GB/s and % of GB300 HBM roofline"
HEADLINE = "gpt6.7b_p4x8192x4096_n128"
GPT27B = "gpt2.7b_4096x2560_n128"
GPT13B = "gpt13b_p8x8192x5120_n256"
FALLBACK_HBM_GBS = 6800.0
# GB300 HBM3e, nominal: 8 stacks, 7.9 TB/s (NVIDIA's published figure).  Used
# only when the device attributes cannot be read.
SPEC_NOMINAL_GBS = 7900.0
L2_BYTES = 129 * 2**20
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "fp8_communication_compression_gb300", "csrc", f)
                  for f in ("codec_kernels.cu", "codec_math.cuh", "device_utils.cuh")]


def algorithmic_bytes(P: int, n: int, block: int, out_bytes: int = 4, fused: bool = False) -> dict:
    """Bytes each launch must move at minimum (reads + writes), per step of
    the two-shot local path over P shards of n elements each: the bf16
    input, one code byte per element and two fp32 scalars (alpha, s) per
    block, and the decompressed output of ``out_bytes`` per element.  The
    one-call reduce + decompress (``fused``) does not re-read the compressed
    sum."""
    nb = n // block
    comp = P * (2 * n + n + 8 * nb)             # bf16 in; codes + alpha + s out
    red_in = P * (n + 8 * nb)                   # P compressed shards in
    red_out = n + 8 * nb                        # the compressed sum out
    dec_out = out_bytes * n                     # its reconstruction out
    if fused:
        return {"compress": comp, "reduce_decompress": red_in + red_out + dec_out}
    return {"compress": comp, "reduce": red_in + red_out, "decompress": red_out + dec_out}


def codec_bytes(n: int, block: int, out_bytes: int = 4) -> dict:
    """Algorithmic bytes of one compress and one decompress of n elements."""
    nb = n // block
    return {"compress": 2 * n + n + 8 * nb, "decompress": n + 8 * nb + out_bytes * n}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def spec_hbm_gbs(device_index: int = 0):
    """Spec DRAM bandwidth: peak memory clock x 2 (double data rate) x bus
    width, read from the device attributes through the CUDA driver API
    (torch does not expose the memory clock).  Falls back to the nominal
    figure when the attributes cannot be read.  Returns (GB/s, source)."""
    try:
        cu = ctypes.CDLL("libcuda.so.1")
        if cu.cuInit(0) != 0:
            raise OSError("cuInit failed")
        dev = ctypes.c_int()
        if cu.cuDeviceGet(ctypes.byref(dev), int(device_index)) != 0:
            raise OSError("cuDeviceGet failed")
        clk, bus = ctypes.c_int(), ctypes.c_int()
        # CU_DEVICE_ATTRIBUTE_MEMORY_CLOCK_RATE (kHz), ..._GLOBAL_MEMORY_BUS_WIDTH (bits)
        if cu.cuDeviceGetAttribute(ctypes.byref(clk), 36, dev) != 0 or \
                cu.cuDeviceGetAttribute(ctypes.byref(bus), 37, dev) != 0:
            raise OSError("cuDeviceGetAttribute failed")
        if clk.value > 0 and bus.value > 0:
            gbs = clk.value * 1e3 * 2 * bus.value / 8 / 1e9
            return gbs, (f"device attributes: memory clock {clk.value / 1e3:.0f} MHz x 2 (DDR) x "
                         f"{bus.value}-bit bus")
    except (OSError, AttributeError):
        pass
    return SPEC_NOMINAL_GBS, "nominal 7.9 TB/s (device attributes unavailable)"


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per compress launch from the committed ncu summary, or None
    once the kernel source has changed since those counters were taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        if t.get("source_digest") == kernel_source_digest():
            return t.get("dram_bytes_per_launch")
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, interval_ms: int = 50):
        self.proc = None
        self.interval_ms = interval_ms

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 f"-lms", str(self.interval_ms)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                text=True)
        except Exception:
            self.proc = None
        return self

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": n}


def replica_seed(base_seed: int, rank: int) -> int:
    """Seed of a shard on ``rank``: each replica draws its own data."""
    return base_seed + 1000 * rank


def max_over_ranks(value_ms: float, dist, device=None) -> float:
    """Largest per-rank time (the job takes as long as its slowest rank)."""
    if dist is None:
        return value_ms
    import torch

    t = torch.tensor([value_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_step: int, steps: int, world: int, max_ms: float) -> float:
    """Aggregate throughput: every rank moves bytes_per_step per step."""
    return bytes_per_step * steps * world / (max_ms / 1e3) / 1e9


def summarize(ms: list) -> dict:
    """Mean, median, spread and count of per-launch times (ms -> us)."""
    us = [m * 1e3 for m in ms]
    return {"us_mean": statistics.mean(us), "us_median": statistics.median(us), "us_min": min(us),
            "us_max": max(us), "samples": len(us)}


# ------------------------------------------------------------ host workers --
# Input generation and the oracle baseline run in worker processes started
# with "spawn" (safe whatever the parent's CUDA state).

def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def worker_pool(n: int):
    import concurrent.futures as cf
    import multiprocessing as mp

    return cf.ProcessPoolExecutor(max_workers=max(1, n), mp_context=mp.get_context("spawn"))


def _tp_shard(args):
    from fp8_communication_compression_gb300 import workloads as W

    seed, rows, d, channel_scale, spikes, block = args
    return W.tp_activation(seed, rows, d, channel_scale=channel_scale, spikes=spikes, block=block)


def _named_shard(args):
    from fp8_communication_compression_gb300 import workloads as W

    name, p = args
    return W.shard_input(name, p)


def make_inputs(rank: int, rows: int | None = None, pool=None):
    from fp8_communication_compression_gb300 import workloads as W

    w = dict(W.WORKLOADS[HEADLINE])
    if rows is not None:
        w["rows"] = rows
    jobs = [(replica_seed(w["seeds"][p], rank), w["rows"], w["d"], w["channel_scale"], w["spikes"],
             w["block"]) for p in range(w["shards"])]
    shards = list(pool.map(_tp_shard, jobs)) if pool else [_tp_shard(j) for j in jobs]
    return w, np.stack(shards)


def _oracle_path_rows(task):
    """Worker: the oracle's two-shot local path (compress every shard,
    reduce, decompress) on rows r0..r1 of the shards held in shared memory.
    Returns the decompressed rows' sum, so that the work is not dead."""
    from multiprocessing import shared_memory

    import oracle

    shm_name, shape, r0, r1, block = task
    shm = shared_memory.SharedMemory(name=shm_name)
    view = np.ndarray(shape, dtype=np.uint16, buffer=shm.buf)
    sub = [view[p, r0:r1].copy() for p in range(shape[0])]  # copies: the segment is closed next
    del view
    shm.close()
    comp = [oracle.compress(s, block) for s in sub]
    rc, ra, rs = oracle.reduce_shards(*zip(*comp), block)
    return float(oracle.decompress(rc, ra, rs, block).sum())


class SharedShards:
    """bf16 shard bits [P, rows, d] in a shared-memory segment for the pool."""

    def __init__(self, bits: np.ndarray):
        from multiprocessing import shared_memory

        self.shm = shared_memory.SharedMemory(create=True, size=bits.nbytes)
        np.ndarray(bits.shape, dtype=np.uint16, buffer=self.shm.buf)[...] = bits
        self.shape = tuple(bits.shape)

    def tasks(self, rows: int, pieces: int, block: int):
        step = max(1, -(-rows // pieces))
        return [(self.shm.name, self.shape, r, min(rows, r + step), block) for r in range(0, rows, step)]

    def close(self):
        self.shm.close()
        self.shm.unlink()


def oracle_wall_seconds(pool, shards: SharedShards, rows: int, cores: int, block: int) -> float:
    """Wall time of the oracle path over the first ``rows`` rows of every
    shard, split over ``cores`` workers (a few row ranges each)."""
    tasks = shards.tasks(rows, 4 * cores, block)
    t0 = time.perf_counter()
    list(pool.map(_oracle_path_rows, tasks))
    return time.perf_counter() - t0


def cpu_baseline(bits: np.ndarray, w: dict, sample_rows: int, pool, cores: int) -> dict:
    """The oracle, as it stands, timed twice: single-threaded on the first
    ``sample_rows`` rows of every shard, and on all host cores (one worker
    process per core, row ranges handed out in turn) over the whole
    workload.  Both run compress of each shard, reduce and decompress."""
    import oracle

    P, block, rows = bits.shape[0], w["block"], bits.shape[1]
    sub = [np.ascontiguousarray(bits[p, :sample_rows]) for p in range(P)]
    n1 = sample_rows * w["d"]
    t0 = time.perf_counter()
    comp = [oracle.compress(s, block) for s in sub]
    rc, ra, rs = oracle.reduce_shards(*zip(*comp), block)
    oracle.decompress(rc, ra, rs, block)
    dt1 = time.perf_counter() - t0
    single = sum(algorithmic_bytes(P, n1, block).values()) / dt1 / 1e9
    shards = SharedShards(bits)
    try:
        oracle_wall_seconds(pool, shards, min(rows, 4 * cores), cores, block)  # workers load the oracle
        dtn = oracle_wall_seconds(pool, shards, rows, cores, block)
    finally:
        shards.close()
    n = rows * w["d"]
    allc = sum(algorithmic_bytes(P, n, block).values()) / dtn / 1e9
    return {"value": allc, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"all {rows} rows of each of the {P} shards ({P * n} elements compressed, {n} reduced "
                      f"and decompressed) on {cores} worker processes, {dtn:.1f} s wall",
            "single_thread": {"value": single, "unit": "GB/s", "cores": 1,
                              "sample": f"first {sample_rows} of {rows} rows of each of the {P} shards "
                                        f"({P * n1} elements compressed, {n1} reduced and decompressed), "
                                        f"{dt1:.1f} s"}}


def run_reference(args, rank: int, world: int) -> None:
    """The reference arm: the CPU oracle timed on bounded samples, on all
    host cores."""
    if rank != 0:
        return
    from fp8_communication_compression_gb300 import workloads as W
    import oracle

    oracle.build()
    w = W.WORKLOADS[HEADLINE]
    P, block, rows_s = w["shards"], w["block"], args.ref_rows
    cores = host_cores()
    n = rows_s * w["d"]
    step_bytes = sum(algorithmic_bytes(P, n, block).values())
    with worker_pool(cores) as pool:
        jobs = [(w["seeds"][p], rows_s, w["d"], True, False, block) for p in range(P)]
        bits = np.stack(list(pool.map(_tp_shard, jobs)))
        shards = SharedShards(bits)
        try:
            for _ in range(args.warmup):
                oracle_wall_seconds(pool, shards, rows_s, cores, block)
            dt = sum(oracle_wall_seconds(pool, shards, rows_s, cores, block) for _ in range(args.steps))
        finally:
            shards.close()
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"each step: {rows_s} of {w['rows']} rows of each of the {P} shards "
              f"(compress {P * n}, reduce and decompress {n} elements), split over {cores} worker processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "P": P, "rows": w["rows"], "d": w["d"], "block": block,
                   "sample_rows": rows_s},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------- GPU timing --

def time_launches(torch, fn, reps: int, stream, replays: int = 3) -> float:
    """Mean device time (ms) per launch of ``fn``: ``reps`` calls captured in
    one CUDA graph, and the graph replayed ``replays`` times between two CUDA
    events on ``stream``.  Replaying a graph keeps the host's per-call launch
    overhead out of the figure; it matters for launches of a few tens of
    microseconds, which the host cannot otherwise enqueue as fast as the GPU
    runs them."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        for _ in range(reps):
            fn()
    with torch.cuda.stream(stream):
        graph.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (reps * replays)
    del graph
    return ms


def sample_kernel_times(torch, launches, x, stream, samples: int) -> dict:
    """Per-launch device times of the step's launches: ``samples`` + 1 steps,
    each with a CUDA event before the first launch and after every launch;
    the first step is dropped (it follows the host's preceding work).  The
    events separate the launches, so each sample includes the launch's own
    start-up, which programmatic dependent launch hides in the unsampled
    step."""
    nl = len(launches)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nl + 1)] for _ in range(samples + 1)]
    for e in ev:
        e[0].record(stream)
        for i, (_, fn) in enumerate(launches):
            fn(x)
            e[i + 1].record(stream)
    torch.cuda.synchronize()
    return {name: [ev[k][i].elapsed_time(ev[k][i + 1]) for k in range(1, samples + 1)]
            for i, (name, _) in enumerate(launches)}


def kernel_entry(ms: float, nbytes: int, peak: float, **extra) -> dict:
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"us_per_launch": ms * 1e3, "algorithmic_bytes": nbytes, "gbs": gbs, "frac_of_peak": gbs / peak,
            **extra}


def agoq_leg(torch, api, peak: float) -> dict:
    """AGoQ accumulate over the 2^28-element buffer and the P=8 reduce of
    2^25-element shards; inputs larger than L2, timed per launch from graph
    replays."""
    from fp8_communication_compression_gb300 import workloads as W

    a = W.AGOQ
    n, block, P, ns = a["n_main"], a["block"], a["reduce_P"], a["n_shard"]
    g = torch.from_numpy(W.agoq_grad(a["grad_seeds"][0], n).view(np.int16)).cuda().view(torch.bfloat16)
    codes = torch.zeros(n, dtype=torch.uint8, device="cuda")
    scale = torch.ones(n // block, dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    api.agoq_fp8_accumulate(codes, scale, g, block)
    acc_ms = time_launches(torch, lambda: api.agoq_fp8_accumulate(codes, scale, g, block), 4, stream)
    acc_bytes = n * (1 + 2 + 1) + 2 * 4 * (n // block)
    del codes, scale
    sc = [torch.zeros(ns, dtype=torch.uint8, device="cuda") for _ in range(P)]
    ss = [torch.ones(ns // block, dtype=torch.float32, device="cuda") for _ in range(P)]
    for p in range(P):
        api.agoq_fp8_accumulate(sc[p], ss[p], g[p * ns:(p + 1) * ns], block)
    oc = torch.empty(ns, dtype=torch.uint8, device="cuda")
    os_ = torch.empty(ns // block, dtype=torch.float32, device="cuda")
    api.agoq_reduce_shards(sc, ss, block, oc, os_)
    red_ms = time_launches(torch, lambda: api.agoq_reduce_shards(sc, ss, block, oc, os_), 5, stream)
    red_bytes = (P + 1) * (ns + 4 * (ns // block))
    return {"accumulate": kernel_entry(acc_ms, acc_bytes, peak, workload=f"2^28 elements, n={block}"),
            "reduce": kernel_entry(red_ms, red_bytes, peak, workload=f"P={P} x 2^25 elements, n={block}")}


def int8_leg(torch, api, x, P: int, rows: int, d: int, block: int, peak: float) -> dict:
    """The INT8 variant of the codec (compress all shards, decompress one
    tensor of the same size) on the headline shards, timed per launch from
    graph replays."""
    n = rows * d
    nb = n // block
    codes = torch.empty((P, rows, d), dtype=torch.int8, device="cuda")
    alpha = torch.empty((P, nb), dtype=torch.float32, device="cuda")
    scale = torch.empty((P, nb), dtype=torch.float32, device="cuda")
    out = torch.empty((rows, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    comp = lambda: api.taco_compress_int8(x, block, codes=codes, alpha=alpha, scale=scale)
    it = [0]

    def dec():
        # one shard's codes (34 MB) fit in L2: consecutive launches rotate
        # over the P shards, so each reads codes that are not L2-resident
        p = it[0] % P
        it[0] += 1
        api.taco_decompress_int8(codes[p], alpha[p], scale[p], block, out=out)

    comp()
    dec()
    ms = {"compress_int8": time_launches(torch, comp, 10, stream),
          "decompress_int8": time_launches(torch, dec, 10, stream)}
    nbytes = {"compress_int8": P * (2 * n + n + 8 * nb), "decompress_int8": n + 8 * nb + 4 * n}
    return {k: kernel_entry(ms[k], nbytes[k], peak) for k in ms}


def laaq_leg(torch, api, peak: float) -> dict:
    """AGoQ LAAQ activation codec on a GPT-6.7B-shaped activation tensor
    (bf16 [8192, 4096]), block 128, 4/5/6/8 bits: quantize and dequantize to
    bf16, and at 4 bits SiLU and RMSNorm recomputed from the stored input,
    timed per launch from graph replays.  One tensor is 67 MB, below the
    129 MB L2, so launches rotate over a ring of three inputs and outputs
    (201 MB of inputs): each launch reads a tensor the previous two launches
    did not touch."""
    from fp8_communication_compression_gb300 import workloads as W

    rows, d, block = 8192, 4096, 128
    n = rows * d
    xs = [torch.from_numpy(W.tp_activation(600 + i, rows, d, channel_scale=True).view(np.int16))
          .cuda().view(torch.bfloat16).reshape(-1) for i in range(3)]
    stream = torch.cuda.current_stream()
    gamma = torch.linspace(0.5, 1.5, d, device="cuda")
    res = {}
    for bits in (4, 5, 6, 8):
        packed = [torch.empty(n * bits // 8, dtype=torch.uint8, device="cuda") for _ in range(3)]
        scale = [torch.empty(n // block, dtype=torch.float32, device="cuda") for _ in range(3)]
        out = [torch.empty(n, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
        it = {"q": 0, "d": 0}

        def quant():
            i = it["q"] % 3
            it["q"] += 1
            api.agoq_laaq_quantize(xs[i], block, bits, packed[i], scale[i])

        def dequant():
            i = it["d"] % 3
            it["d"] += 1
            api.agoq_laaq_dequantize(packed[i], scale[i], n, block, bits, out=out[i])

        def silu():
            i = it["d"] % 3
            it["d"] += 1
            api.agoq_laaq_dequantize_silu(packed[i], scale[i], n, block, bits, out=out[i])

        def rmsnorm():
            i = it["d"] % 3
            it["d"] += 1
            api.agoq_laaq_dequantize_rmsnorm(packed[i], scale[i], rows, d, gamma, 1e-6, block, bits,
                                             out=out[i].view(rows, d))

        for _ in range(3):
            quant()
            dequant()
        legs = [("quantize", quant, 2 * n + n * bits // 8 + 4 * (n // block)),
                ("dequantize", dequant, n * bits // 8 + 4 * (n // block) + 2 * n)]
        if bits == 4:  # the recomputations of AGoQ 2.A, from the 4-bit stored input
            legs += [("dequantize_silu", silu, n * bits // 8 + 4 * (n // block) + 2 * n),
                     ("dequantize_rmsnorm", rmsnorm, n * bits // 8 + 4 * (n // block) + 2 * n + 4 * d)]
        for name, fn, b in legs:
            res[f"{name}_{bits}bit"] = kernel_entry(time_launches(torch, fn, 12, stream), b, peak)
    return res


def gpt27b_leg(torch, api, peak: float) -> dict:
    """The GPT-2.7B-shaped round trip (one bf16 [4096, 2560] activation,
    n=128): compress, decompress to fp32, and the two back to back, timed per
    launch from graph replays, L2-flushed and warm.  The tensor and its
    outputs (74 MB) fit in the 129 MB L2, so the flushed figures rotate over
    12 copies in distinct buffers (888 MB): between two launches on the same
    copy, the launches on the other eleven move more than twice the L2.  The
    warm figures repeat the launch on one copy, whose data then stays in
    L2."""
    from fp8_communication_compression_gb300 import workloads as W

    w = W.WORKLOADS[GPT27B]
    rows, d, block = w["rows"], w["d"], w["block"]
    n, nb, R = rows * d, rows * d // block, 12
    bits = torch.from_numpy(W.shard_input(GPT27B, 0).view(np.int16)).cuda().view(torch.bfloat16)
    x = bits.unsqueeze(0).repeat(R, 1, 1).contiguous()
    codes = torch.empty((R, rows, d), dtype=torch.uint8, device="cuda")
    alpha = torch.empty((R, nb), dtype=torch.float32, device="cuda")
    scale = torch.empty((R, nb), dtype=torch.float32, device="cuda")
    out = torch.empty((R, rows, d), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream()
    it = [0]

    def comp(i):
        api.taco_compress(x[i], block, codes=codes[i], alpha=alpha[i], scale=scale[i])

    def dec(i):
        api.taco_decompress(codes[i], alpha[i], scale[i], block, out=out[i])

    def rotating(fn):
        def call():
            i = it[0] % R
            it[0] += 1
            fn(i)
        return call

    for i in range(R):
        comp(i)
        dec(i)
    b = codec_bytes(n, block)
    b["round_trip"] = b["compress"] + b["decompress"]
    fns = {"compress": comp, "decompress": dec, "round_trip": lambda i: (comp(i), dec(i))}
    res = {}
    for name, fn in fns.items():
        it[0] = 0
        flushed = time_launches(torch, rotating(fn), 2 * R, stream)
        warm = time_launches(torch, lambda: fn(0), 2 * R, stream)
        res[name] = kernel_entry(flushed, b[name], peak, l2="flushed (12-copy rotation)",
                                 warm=kernel_entry(warm, b[name], peak, l2="warm (one copy)"))
    res["round_trip"]["launches"] = "compress then decompress of the same copy (2 launches)"
    return res


def bf16_peak():
    """Measured dense bf16 tensor throughput (TFLOP/s, burst) from
    MEASURED_PEAKS.json, else the fallback figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured cuBLAS bf16 burst (MEASURED_PEAKS.json bf16_tflops)"
    except Exception:
        return 1900.0, "fallback 1.9 PFLOP/s bf16 burst (no MEASURED_PEAKS.json)"


def gemm_leg(torch, api, pool=None) -> dict:
    """The GEMM that produces a GPT-6.7B TP partial sum, with the compressor
    in its epilogue: the row-parallel MLP down-projection at TP = 4, A =
    [8192 tokens, 4096] activations, B = [4096, 4096] weights, Y = A B^T
    compressed per 128-element block (taco_gemm_compress).  Timed from graph
    replays beside the unfused path it replaces: cuBLAS (torch.matmul, bf16
    out) then taco_compress, and beside each of those two alone.  The
    operands (96 MB) stay in L2 across replays, as they would between the
    layer's tiles; the fused call's and cuBLAS's outputs are written every
    replay."""
    from fp8_communication_compression_gb300 import workloads as W

    M, N, K = 8192, 4096, 4096
    a_bits = pool.submit(_tp_shard, (900, M, K, True, False, 128)).result() if pool else \
        _tp_shard((900, M, K, True, False, 128))
    b_bits = W.f32_to_bf16_bits(np.random.default_rng(901).normal(0.0, 0.02, (N, K)).astype(np.float32))
    a = torch.from_numpy(a_bits.view(np.int16)).cuda().view(torch.bfloat16)
    b = torch.from_numpy(b_bits.view(np.int16)).cuda().view(torch.bfloat16)
    nb = M * N // 128
    codes = torch.empty((M, N), dtype=torch.uint8, device="cuda")
    alpha = torch.empty(nb, dtype=torch.float32, device="cuda")
    scale = torch.empty(nb, dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fused = lambda: api.taco_gemm_compress(a, b, codes=codes, alpha=alpha, scale=scale)
    fused_ns = lambda: api.taco_gemm_compress(a, b, codes=codes, alpha=alpha, scale=scale, split_tail=False)
    gemm = lambda: torch.matmul(a, b.t(), out=y)
    comp = lambda: api.taco_compress(y, 128, codes=codes, alpha=alpha, scale=scale)

    def unfused():
        gemm()
        comp()

    for fn in (fused, fused_ns, unfused):
        fn()
    ms = {"fused": time_launches(torch, fused, 10, stream),
          "fused_no_split_tail": time_launches(torch, fused_ns, 10, stream),
          "cublas_gemm": time_launches(torch, gemm, 10, stream),
          "compress": time_launches(torch, comp, 10, stream), "unfused": time_launches(torch, unfused, 10, stream)}
    flops = 2.0 * M * N * K
    peak, src = bf16_peak()
    out = {k: {"us_per_launch": v * 1e3, "tflops": flops / (v / 1e3) / 1e12 if k != "compress" else None}
           for k, v in ms.items()}
    for k in ("fused", "fused_no_split_tail", "cublas_gemm", "unfused"):
        out[k]["frac_of_bf16_peak"] = out[k]["tflops"] / peak
    out["shape"] = {"M": M, "N": N, "K": K, "block": 128}
    out["split_tail_workspace_bytes"] = api.gemm_workspace_bytes(M, N, K)
    out["bf16_peak_tflops"] = peak
    out["bf16_peak_source"] = src
    out["fused_vs_unfused_speedup"] = ms["unfused"] / ms["fused"]
    out["hbm_bytes_saved_per_call"] = 2 * 2 * M * N  # the bf16 Y written and read back
    return out


def agoq_gemm_leg(torch, api) -> dict:
    """The weight-gradient GEMM with the FP8 main-gradient accumulation in its
    epilogue (agoq_gemm_accumulate): a GPT-6.7B-shaped dW [4096, 4096] =
    dY^T X over 8192 tokens, added into an FP8 main gradient per 128-element
    block.  Timed from graph replays beside the path it replaces: cuBLAS
    (torch.matmul, bf16 out) then agoq_fp8_accumulate."""
    from fp8_communication_compression_gb300 import workloads as W

    M, N, K = 4096, 4096, 8192
    a_bits = W.agoq_grad(960, M * K).reshape(M, K)
    b_bits = W.f32_to_bf16_bits(np.random.default_rng(961).normal(0.0, 0.05, (N, K)).astype(np.float32))
    a = torch.from_numpy(a_bits.view(np.int16)).cuda().view(torch.bfloat16)
    b = torch.from_numpy(b_bits.view(np.int16)).cuda().view(torch.bfloat16)
    codes = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
    scale = torch.ones(M * N // 128, dtype=torch.float32, device="cuda")
    g = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fused = lambda: api.agoq_gemm_accumulate(a, b, codes, scale)
    fused_ns = lambda: api.agoq_gemm_accumulate(a, b, codes, scale, split_tail=False)
    gemm = lambda: torch.matmul(a, b.t(), out=g)
    acc = lambda: api.agoq_fp8_accumulate(codes.view(-1), scale, g.view(-1))

    def unfused():
        gemm()
        acc()

    for fn in (fused, fused_ns, unfused):
        fn()
    ms = {"fused": time_launches(torch, fused, 10, stream),
          "fused_no_split_tail": time_launches(torch, fused_ns, 10, stream),
          "cublas_gemm": time_launches(torch, gemm, 10, stream),
          "accumulate": time_launches(torch, acc, 10, stream), "unfused": time_launches(torch, unfused, 10, stream)}
    flops = 2.0 * M * N * K
    peak, src = bf16_peak()
    out = {k: {"us_per_launch": v * 1e3, "tflops": flops / (v / 1e3) / 1e12 if k != "accumulate" else None}
           for k, v in ms.items()}
    for k in ("fused", "fused_no_split_tail", "cublas_gemm", "unfused"):
        out[k]["frac_of_bf16_peak"] = out[k]["tflops"] / peak
    out["shape"] = {"M": M, "N": N, "K": K, "block": 128}
    out["split_tail_workspace_bytes"] = api.gemm_workspace_bytes(M, N, K)
    out["fused_vs_unfused_speedup"] = ms["unfused"] / ms["fused"]
    out["hbm_bytes_saved_per_call"] = 2 * 2 * M * N  # the bf16 gradient written and read back
    return out


def laaq_gemm_leg(torch, api, pool=None, bits: int = 4) -> dict:
    """The GEMM that produces an activation with AGoQ's 4-bit LAAQ
    quantisation in its epilogue (agoq_gemm_laaq_quantize): a GPT-6.7B-sized
    [8192 tokens, 4096] = X W^T with W [4096, 4096], stored as packed codes
    and a multiplier per 128-element block.  Timed from graph replays beside
    the path it replaces: cuBLAS (torch.matmul, bf16 out) then
    agoq_laaq_quantize."""
    from fp8_communication_compression_gb300 import workloads as W

    M, N, K = 8192, 4096, 4096
    a_bits = pool.submit(_tp_shard, (902, M, K, True, False, 128)).result() if pool else \
        _tp_shard((902, M, K, True, False, 128))
    b_bits = W.f32_to_bf16_bits(np.random.default_rng(903).normal(0.0, 0.02, (N, K)).astype(np.float32))
    a = torch.from_numpy(a_bits.view(np.int16)).cuda().view(torch.bfloat16)
    b = torch.from_numpy(b_bits.view(np.int16)).cuda().view(torch.bfloat16)
    packed = torch.empty(M * N * bits // 8, dtype=torch.uint8, device="cuda")
    scale = torch.empty(M * N // 128, dtype=torch.float32, device="cuda")
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    fused = lambda: api.agoq_gemm_laaq_quantize(a, b, bits, packed=packed, scale=scale)
    gemm = lambda: torch.matmul(a, b.t(), out=y)
    quant = lambda: api.agoq_laaq_quantize(y.view(-1), 128, bits, packed, scale)

    def unfused():
        gemm()
        quant()

    for fn in (fused, unfused):
        fn()
    ms = {"fused": time_launches(torch, fused, 10, stream), "cublas_gemm": time_launches(torch, gemm, 10, stream),
          "quantize": time_launches(torch, quant, 10, stream), "unfused": time_launches(torch, unfused, 10, stream)}
    flops = 2.0 * M * N * K
    peak, _ = bf16_peak()
    out = {k: {"us_per_launch": v * 1e3, "tflops": flops / (v / 1e3) / 1e12 if k != "quantize" else None}
           for k, v in ms.items()}
    for k in ("fused", "cublas_gemm", "unfused"):
        out[k]["frac_of_bf16_peak"] = out[k]["tflops"] / peak
    out["shape"] = {"M": M, "N": N, "K": K, "block": 128, "bits": bits}
    out["fused_vs_unfused_speedup"] = ms["unfused"] / ms["fused"]
    out["hbm_bytes_saved_per_call"] = 2 * 2 * M * N  # the bf16 activation written and read back
    return out


def gpt13b_leg(torch, api, peak: float, pool=None) -> dict:
    """The GPT-13B-shaped path (8 shards of [8192, 5120], n=256): per-launch
    device times (graph replays) of compress, reduce + decompress in one call,
    and the separate reduce and decompress."""
    from fp8_communication_compression_gb300 import workloads as W

    w = W.WORKLOADS[GPT13B]
    P, rows, d, block = w["shards"], w["rows"], w["d"], w["block"]
    jobs = [(GPT13B, p) for p in range(P)]
    shards = list(pool.map(_named_shard, jobs)) if pool else [_named_shard(j) for j in jobs]
    x = torch.empty((P, rows, d), dtype=torch.bfloat16, device="cuda")
    for p in range(P):
        x[p].view(torch.int16).copy_(torch.from_numpy(shards[p].view(np.int16)))
    del shards
    path = api.TwoShotLocal(P, rows, d, block, fused=True)
    for _ in range(3):
        path.run(x)
    stream = torch.cuda.current_stream()
    it = [0]

    def dec():
        # the reduced codes (42 MB) fit in L2: consecutive launches decompress
        # the P shards' codes in turn, same kernel and sizes, not L2-resident
        p = it[0] % P
        it[0] += 1
        api.taco_decompress(path.codes[p], path.alpha[p], path.scale[p], block, out=path.out)

    ms = {"compress": time_launches(torch, lambda: path.compress(x), 10, stream),
          "reduce_decompress": time_launches(torch, path.reduce_decompress, 10, stream),
          "reduce": time_launches(torch, path.reduce, 10, stream),
          "decompress": time_launches(torch, dec, 16, stream)}
    nb = dict(algorithmic_bytes(P, rows * d, block, fused=True))
    nb.update(algorithmic_bytes(P, rows * d, block, fused=False))
    return {k: kernel_entry(ms[k], nb[k], peak) for k in ms}


def exchange_bytes(world: int, rows: int, d: int, block: int, out_bytes: int = 4, stages: int = 1) -> dict:
    """Algorithmic bytes of one rank's kernels in one two-shot AllReduce over
    ``world`` ranks of a [rows, d] tensor: compress of the whole tensor, the
    reduce of ``world`` received chunks of R rows into one (R =
    ceil(rows / world), rounded up to a multiple of ``stages``), and the
    decompress of the ``world`` gathered chunks."""
    R = -(-(-(-rows // world)) // stages) * stages
    n, c = rows * d, R * d
    return {"compress": 3 * n + 8 * (n // block),
            "reduce": (world + 1) * (c + 8 * (c // block)),
            "decompress": world * (c + 8 * (c // block) + out_bytes * c)}


def run_exchange(args, rank: int, world: int, local: int, pool) -> None:
    """The two-shot AllReduce across the ranks (NCCL): each rank holds one
    bf16 [8192, 4096] activation of the GPT-6.7B shape (seeded by rank; with
    four ranks these are the headline's four shards) and every step runs
    compress, All-to-All, shard reduce, AllGather and decompress."""
    import torch
    import torch.distributed as dist

    from fp8_communication_compression_gb300 import api, exchange
    from fp8_communication_compression_gb300 import workloads as W

    w = W.WORKLOADS[HEADLINE]
    rows = args.rows or w["rows"]
    d, block = w["d"], w["block"]
    bits = pool.submit(_tp_shard, (rank, rows, d, w["channel_scale"], w["spikes"], block)).result()
    torch.cuda.set_device(local)
    if world == 1 and "MASTER_ADDR" not in os.environ:  # a group of one, without torchrun
        import socket

        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                                device_id=torch.device("cuda", local))
    else:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    ar = exchange.TwoShotAllReduce(rows, d, block, stages=args.exchange_stages)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler().start() if rank == 0 and not args.no_clocks else None
    time.sleep(0.2 if clocks else 0)
    for _ in range(args.warmup):
        ar.run(x)
    torch.cuda.synchronize()
    # one step as a CUDA graph (kernels and NCCL collectives), so that the
    # host's per-call cost (Python, the binding, torch.distributed) is not
    # timed; eager steps if the capture is refused
    graph, capture = None, "CUDA graph of one step (kernels and NCCL collectives), replayed"
    try:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            ar.run(x)
        stream.wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            ar.run(x)
    except Exception as exc:  # noqa: BLE001 - report and time eagerly
        graph = None
        capture = f"eager steps (graph capture failed: {type(exc).__name__})"
    torch.cuda.synchronize()
    step = graph.replay if graph is not None else (lambda: ar.run(x))
    for _ in range(3):
        step()
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dist.barrier()
    torch.cuda.synchronize()
    t_host = time.perf_counter()
    start.record(stream)
    for _ in range(K):
        step()
    end.record(stream)
    host_us = (time.perf_counter() - t_host) / K * 1e6
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(start.elapsed_time(end), dist, "cuda")
    # the captured graph holds the communicator's collectives: release it
    # (after the device has finished with it) before the process group goes
    step = None
    del graph
    torch.cuda.synchronize()
    # per-kernel figures: each local phase of a step (its launches for every
    # stage, no collective) captured in a CUDA graph and replayed, so that the
    # host's per-call cost is not timed
    names = ("compress", "reduce", "decompress")
    phases = {"compress": lambda: [ar.compress(x, k) for k in range(ar.S)],
              "reduce": lambda: [ar.reduce(k) for k in range(ar.S)],
              "decompress": lambda: [ar.decompress(k) for k in range(ar.S)]}
    ns = max(2, args.kernel_samples)
    per_phase_ms = {k: time_launches(torch, fn, 10, stream, replays=max(1, ns // 10)) for k, fn in phases.items()}
    # the AllReduce of a row-parallel layer fed by its GEMM (the GPT-6.7B
    # MLP down-projection at TP = 4: [rows, 4096] x [d, 4096]^T): the GEMM
    # with the compressor in its epilogue writing the send pieces
    # (run_gemm), against cuBLAS (bf16 out) then the exchange of that output
    layer = None
    if not args.no_gemm and all((r1 - r0) % 128 == 0 for j in range(ar.W) for k in range(ar.S)
                                for r0, r1 in [ar._piece(j, k)]):
        kg = 4096
        a_bits = pool.submit(_tp_shard, (100 + rank, rows, kg, True, False, block)).result()
        a = torch.from_numpy(a_bits.view(np.int16)).cuda().view(torch.bfloat16)
        w_bits = W.f32_to_bf16_bits(np.random.default_rng(110 + rank).normal(0.0, 0.02, (d, kg))
                                    .astype(np.float32))
        wt = torch.from_numpy(w_bits.view(np.int16)).cuda().view(torch.bfloat16)
        y = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
        fused = lambda: ar.run_gemm(a, wt)

        def unfused():
            torch.matmul(a, wt.t(), out=y)
            ar.run(y)

        fused()
        unfused()
        f_ms = time_launches(torch, fused, 5, stream, replays=2)
        u_ms = time_launches(torch, unfused, 5, stream, replays=2)
        layer = {"shape": {"M": rows, "N": d, "K": kg}, "fused_gemm_then_exchange_us": f_ms * 1e3,
                 "cublas_gemm_then_exchange_us": u_ms * 1e3, "speedup": u_ms / f_ms,
                 "timed_as": "graph replays of whole steps (GEMM, kernels and NCCL collectives)"}
    # end to end: pinned host input in, result out, every step
    h_in = torch.empty((rows, d), dtype=torch.bfloat16, pin_memory=True)
    h_in.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
    h_out = torch.empty((rows, d), dtype=torch.float32, pin_memory=True)
    E = max(1, args.e2e_steps)
    dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        x.copy_(h_in, non_blocking=True)
        h_out.copy_(ar.run(x), non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), dist, "cuda")
    flags = api.taco_device_error(clear=True)
    if rank == 0:
        peak, peak_src = hbm_peak()
        spec, spec_src = spec_hbm_gbs(local)
        nbytes = exchange_bytes(world, rows, d, block, stages=ar.S)
        step_bytes = sum(nbytes.values())
        kern = {k: kernel_entry(per_phase_ms[k], nbytes[k], peak, launches=(ar.S if k == "reduce" else ar.W * ar.S),
                                timed_as="graph replays of the phase's launches")
                for k in names}
        achieved = kern["compress"]["gbs"]
        line = {
            "metric": METRIC, "value": whole_job_gbs(step_bytes, K, world, elapsed_ms), "unit": "GB/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": elapsed_ms / K,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"two-shot AllReduce of one bf16 [{rows}, {d}] activation per rank "
                                   f"(GPT-6.7B shape, block {block}) across {world} ranks",
                       "rows": rows, "d": d, "block": block, "parallelism": f"tp{world} two-shot exchange (NCCL)",
                       "exchange_stages": ar.S, "timed_as": capture, "host_enqueue_us_per_step": host_us,
                       "bytes_per_step_per_rank": step_bytes,
                       "exchange_bytes_sent_per_rank": ar.bytes_exchanged(),
                       "l2": "inputs larger than L2, no flush"},
            "roofline": {"bound": "hbm", "kernel": f"taco_compress_kernel<{block}>", "achieved": achieved,
                         "peak": peak, "unit": "GB/s", "frac": achieved / peak, "traffic": None,
                         "peak_source": peak_src, "spec_peak": spec, "spec_peak_source": spec_src,
                         "frac_of_spec": achieved / spec},
            "kernels": kern,
            "row_parallel_layer": layer,
            "e2e": {"value": whole_job_gbs(step_bytes, E, world, e2e_ms), "unit": "GB/s",
                    "h2d_bytes_per_step": 2 * rows * d, "d2h_bytes_per_step": 4 * rows * d,
                    "api": "TwoShotAllReduce.run with pinned host copies in and out"},
            "gpu_launches": (2 * ar.W * ar.S + ar.S) * K,  # compress and decompress per piece, reduce per stage
            "clocks": clk,
            "watchdog_flags": flags,
        }
        print(json.dumps(line), flush=True)
    dist.barrier()
    torch.cuda.synchronize()
    dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--kernel-samples", type=int, default=60,
                    help="steps of the per-kernel sampling phase after the timed region")
    ap.add_argument("--e2e-chunks", type=int, default=4, help="row chunks of the host pipeline")
    ap.add_argument("--e2e-blocks", type=int, default=9, help="timed blocks of the end-to-end leg (median reported)")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="single-thread oracle sample rows per shard")
    ap.add_argument("--ref-rows", type=int, default=1024, help="reference arm rows per shard per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip nvidia-smi clock sampling")
    ap.add_argument("--no-agoq", action="store_true", help="skip the AGoQ accumulate/reduce leg")
    ap.add_argument("--no-int8", action="store_true", help="skip the INT8-codec leg")
    ap.add_argument("--no-laaq", action="store_true", help="skip the LAAQ activation-codec leg")
    ap.add_argument("--no-gpt27b", action="store_true", help="skip the GPT-2.7B-shaped round-trip leg")
    ap.add_argument("--no-gpt13b", action="store_true", help="skip the GPT-13B-shaped leg")
    ap.add_argument("--no-gemm", action="store_true",
                    help="skip the fused GEMM legs (compress, AGoQ accumulate, LAAQ quantise; with --exchange, "
                         "the GEMM-fed exchange)")
    ap.add_argument("--fused", action="store_true",
                    help="run reduce and decompress through the one-call entry point (taco_reduce_decompress)")
    ap.add_argument("--replicas", action="store_true",
                    help="under torchrun: independent replicas of the one-GPU path instead of the exchange")
    ap.add_argument("--exchange", action="store_true",
                    help="run the exchange path even on one rank (an NCCL group of one)")
    ap.add_argument("--exchange-stages", type=int, default=4,
                    help="pieces per chunk in the exchange (compress and decompress overlap the collectives)")
    ap.add_argument("--rows", type=int, default=None,
                    help="rows per shard (a smaller case of the same workload, e.g. for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    cores = max(1, host_cores() // max(1, int(os.environ.get("LOCAL_WORLD_SIZE", world))))
    pool = worker_pool(cores)

    import torch

    from fp8_communication_compression_gb300 import api

    if (world > 1 and not args.replicas) or args.exchange:
        run_exchange(args, rank, world, local, pool)
        pool.shutdown()
        return
    w, bits = make_inputs(rank, args.rows, pool)
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    P, rows, d, block = w["shards"], w["rows"], w["d"], w["block"]
    n = rows * d

    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    path = api.TwoShotLocal(P, rows, d, block, fused=args.fused)
    stream = torch.cuda.current_stream()

    # the clock sampler starts before the warm-up steps, so that no idle gap
    # separates the warm-up from the timed region
    clocks = ClockSampler().start() if rank == 0 and not args.no_clocks else None
    time.sleep(0.2 if clocks else 0)
    for _ in range(args.warmup):
        path.run(x)
    torch.cuda.synchronize()

    launches = path.launches()
    names = [nm for nm, _ in launches]
    nbytes = path.bytes_per_step()
    step_bytes = sum(nbytes.values())
    K = args.steps
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_host = time.perf_counter()
    start.record(stream)
    for _ in range(K):
        for _, fn in launches:
            fn(x)
    end.record(stream)
    host_us = (time.perf_counter() - t_host) / K * 1e6
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed_ms = start.elapsed_time(end)
    # keep the same work running until the clock sampler has a few samples
    soak = 0
    t_region = elapsed_ms / 1e3
    while clocks and t_region < 1.0:
        path.run(x)
        soak += 1
        if soak % 200 == 0:
            torch.cuda.synchronize()
            t_region += 200 * elapsed_ms / K / 1e3
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    elapsed_ms = max_over_ranks(elapsed_ms, dist, "cuda")

    # per-kernel figures: a sampling phase of a fixed number of steps
    samples = sample_kernel_times(torch, launches, x, stream, max(2, args.kernel_samples))

    # end to end through the public API with pinned host buffers
    e2e_ms = None
    if args.e2e_steps > 0:
        h_in = torch.empty((P, rows, d), dtype=torch.bfloat16, pin_memory=True)
        h_in.view(torch.int16).copy_(torch.from_numpy(bits.view(np.int16)))
        h_out = torch.empty((rows, d), dtype=torch.float32, pin_memory=True)
        pipe = api.HostPipeline(P, rows, d, block, chunks=args.e2e_chunks)
        for _ in range(3):
            pipe.run(h_in, h_out)
        torch.cuda.synchronize()
        # the host link is shared with other work on the same host: time
        # several blocks spread over a second or so and report their median
        e2e_blocks = []
        for b in range(args.e2e_blocks):
            if b:
                time.sleep(0.2)
            if dist:
                dist.barrier()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(args.e2e_steps):
                pipe.run(h_in, h_out)
            e1.record(stream)
            torch.cuda.synchronize()
            e2e_blocks.append(max_over_ranks(e0.elapsed_time(e1), dist, "cuda"))
        e2e_ms = statistics.median(e2e_blocks)
    peak, peak_src = hbm_peak()
    spec, spec_src = spec_hbm_gbs(local)
    extra = {}
    if rank == 0 and not args.no_int8:
        extra["int8_" + HEADLINE] = int8_leg(torch, api, x, P, rows, d, block, peak)
    if rank == 0:
        del path, x
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_gpt27b:
        extra[GPT27B] = gpt27b_leg(torch, api, peak)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_gpt13b:
        extra[GPT13B] = gpt13b_leg(torch, api, peak, pool)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_gemm:
        extra["gemm_compress_gpt6.7b_down_proj_8192x4096x4096"] = gemm_leg(torch, api, pool)
        extra["agoq_gemm_accumulate_gpt6.7b_dw_4096x4096x8192"] = agoq_gemm_leg(torch, api)
        extra["laaq_gemm_quantize_4bit_gpt6.7b_8192x4096x4096"] = laaq_gemm_leg(torch, api, pool)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_agoq:
        extra["agoq"] = agoq_leg(torch, api, peak)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_laaq:
        extra["laaq_8192x4096_n128"] = laaq_leg(torch, api, peak)
        torch.cuda.empty_cache()
    flags = api.taco_device_error(clear=True)

    if rank == 0:
        value = whole_job_gbs(step_bytes, K, world, elapsed_ms)
        kern = {}
        for name in names:
            st = summarize(samples[name])
            kern[name] = kernel_entry(st["us_mean"] / 1e3, nbytes[name], peak, **st)
        achieved = kern["compress"]["gbs"]
        ns = len(samples[names[0]])
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": HEADLINE if args.rows is None else f"{HEADLINE} (rows={rows})",
                       "P": P, "rows": rows, "d": d, "block": block,
                       "launches": names,
                       "kernel_events": (f"per-launch CUDA events in a sampling phase of {ns + 1} steps after "
                                         f"the timed region, first step dropped ({ns} samples per kernel)"),
                       "bytes_per_step": step_bytes,
                       "host_enqueue_us_per_step": host_us,
                       "input_bf16_bytes_per_step": 2 * P * n,
                       "l2": "inputs larger than L2 (268 MB bf16 read per step), no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": f"taco_compress_kernel<{block}>",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": committed_traffic(), "peak_source": peak_src,
                         "samples": ns,
                         "spec_peak": spec, "spec_peak_source": spec_src, "frac_of_spec": achieved / spec},
            "kernels": kern,
            "step_frac_of_peak": value / world / peak,
            "step_frac_of_spec": value / world / spec,
            "e2e": None if e2e_ms is None else {
                "value": whole_job_gbs(step_bytes, args.e2e_steps, world, e2e_ms), "unit": "GB/s",
                "h2d_bytes_per_step": 2 * P * n, "d2h_bytes_per_step": 4 * n,
                "blocks": f"median of {len(e2e_blocks)} blocks of {args.e2e_steps} steps, 0.2 s apart",
                "block_values": [round(whole_job_gbs(step_bytes, args.e2e_steps, world, t), 1) for t in e2e_blocks],
                "api": f"taco_host_pipeline_run via HostPipeline.run (pinned host in/out, {pipe.C} row chunks on 3 streams)"},
            "other_workloads": extra,
            # kernels per call: taco_reduce_decompress runs two
            "gpu_launches": sum(2 if nm == "reduce_decompress" else 1 for nm in names) * K,
            "clocks": clk,
            "watchdog_flags": flags,
        }
        if clk:
            line["clocks"]["window"] = (f"timed region plus {soak} further identical steps"
                                        if soak else "timed region")
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(bits, w, args.cpu_rows, pool, cores)
        print(json.dumps(line), flush=True)
    pool.shutdown()
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
