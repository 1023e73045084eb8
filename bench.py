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
time, in GB/s.  Under torchrun each rank runs its own replica on its own
shards (weak scaling, no data-path collective).

``--impl reference`` times the CPU oracle (the plain reference
implementation of the method) on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
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
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
KERNEL_SOURCES = [os.path.join(ROOT, "fp8_communication_compression_gb300", "csrc", f)
                  for f in ("codec_kernels.cu", "codec_math.cuh", "device_utils.cuh")]


def algorithmic_bytes(P: int, n: int, block: int, out_bytes: int = 4, fused: bool = False) -> dict:
    """Bytes each launch must move at minimum (reads + writes), per step of
    the two-shot local path over P shards of n elements."""
    nb = n // block
    comp = P * (2 * n + n + 8 * nb)             # bf16 in; codes + alpha + s out
    red_in = P * (n + 8 * nb)                   # P compressed shards in
    red_out = n + 8 * nb                        # the compressed sum out
    dec_out = out_bytes * n                     # its reconstruction out
    if fused:
        return {"compress": comp, "reduce_decompress": red_in + red_out + dec_out}
    return {"compress": comp, "reduce": red_in + red_out, "decompress": red_out + dec_out}


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def spec_hbm_gbs(torch):
    """Spec DRAM bandwidth from the device's attributes (memory clock x 2 for
    double data rate x bus width), or None where torch does not expose them.
    Context only: fractions are taken of the measured copy peak."""
    p = torch.cuda.get_device_properties(torch.cuda.current_device())
    clk_khz, bus_bits = getattr(p, "memory_clock_rate", None), getattr(p, "memory_bus_width", None)
    if not clk_khz or not bus_bits:
        return None
    return clk_khz * 1e3 * 2 * bus_bits / 8 / 1e9


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


def make_inputs(rank: int, rows: int | None = None):
    from fp8_communication_compression_gb300 import workloads as W

    w = dict(W.WORKLOADS[HEADLINE])
    if rows is not None:
        w["rows"] = rows
    shards = []
    for p in range(w["shards"]):
        seed = replica_seed(w["seeds"][p], rank)
        shards.append(W.tp_activation(seed, w["rows"], w["d"], channel_scale=w["channel_scale"],
                                      spikes=w["spikes"], block=w["block"]))
    return w, np.stack(shards)


def cpu_baseline(bits: np.ndarray, w: dict, sample_rows: int) -> dict:
    """The oracle, as it stands, on the first ``sample_rows`` rows of every
    shard: compress each shard, reduce, decompress.  Single-threaded."""
    import oracle

    P, block = bits.shape[0], w["block"]
    sub = [np.ascontiguousarray(bits[p, :sample_rows]) for p in range(P)]
    n = sample_rows * w["d"]
    t0 = time.perf_counter()
    comp = [oracle.compress(s, block) for s in sub]
    rc, ra, rs = oracle.reduce_shards(*zip(*comp), block)
    oracle.decompress(rc, ra, rs, block)
    dt = time.perf_counter() - t0
    total = sum(algorithmic_bytes(P, n, block).values())
    return {"value": total / dt / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {sample_rows} of {w['rows']} rows of each of the {P} shards "
                      f"({P * n} elements compressed, {n} reduced and decompressed), "
                      f"{dt:.1f} s single-threaded"}


def run_reference(args, rank: int, world: int) -> None:
    """The reference arm: the CPU oracle timed on bounded samples."""
    if rank != 0:
        return
    from fp8_communication_compression_gb300 import workloads as W
    import oracle

    oracle.build()
    w = W.WORKLOADS[HEADLINE]
    P, block, rows_s = w["shards"], w["block"], args.ref_rows
    bits = np.stack([W.tp_activation(w["seeds"][p], rows_s, w["d"], channel_scale=True, block=block)
                     for p in range(P)])
    n = rows_s * w["d"]
    step_bytes = sum(algorithmic_bytes(P, n, block).values())

    def step():
        comp = [oracle.compress(bits[p], block) for p in range(P)]
        rc, ra, rs = oracle.reduce_shards(*zip(*comp), block)
        oracle.decompress(rc, ra, rs, block)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = step_bytes * args.steps / dt / 1e9
    sample = (f"each step: {rows_s} of {w['rows']} rows of each of the {P} shards "
              f"(compress {P * n}, reduce and decompress {n} elements), single-threaded")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": HEADLINE, "P": P, "rows": w["rows"], "d": w["d"], "block": block,
                   "sample_rows": rows_s},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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
    out = {}
    for name, ms, b, units in (("accumulate", acc_ms, acc_bytes, f"2^28 elements, n={block}"),
                               ("reduce", red_ms, red_bytes, f"P={P} x 2^25 elements, n={block}")):
        gbs = b / (ms / 1e3) / 1e9
        out[name] = {"us_per_launch": ms * 1e3, "algorithmic_bytes": b, "gbs": gbs,
                     "frac_of_peak": gbs / peak, "workload": units}
    return out


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
    return {k: {"us_per_launch": ms[k] * 1e3, "algorithmic_bytes": nbytes[k],
                "gbs": nbytes[k] / (ms[k] / 1e3) / 1e9, "frac_of_peak": nbytes[k] / (ms[k] / 1e3) / 1e9 / peak}
            for k in ms}


def laaq_leg(torch, api, peak: float) -> dict:
    """AGoQ LAAQ activation codec on a GPT-6.7B-shaped activation tensor
    (bf16 [8192, 4096]), block 128, 4/5/6/8 bits: quantize and dequantize to
    bf16, timed per launch from graph replays.  One tensor is 67 MB, below the
    129 MB L2, so launches rotate over a ring of three inputs and outputs
    (201 MB of inputs): each launch reads a tensor the previous two launches
    did not touch."""
    from fp8_communication_compression_gb300 import workloads as W

    rows, d, block = 8192, 4096, 128
    n = rows * d
    xs = [torch.from_numpy(W.tp_activation(600 + i, rows, d, channel_scale=True).view(np.int16))
          .cuda().view(torch.bfloat16).reshape(-1) for i in range(3)]
    stream = torch.cuda.current_stream()
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

        for _ in range(3):
            quant()
            dequant()
        for name, fn, b in (("quantize", quant, 2 * n + n * bits // 8 + 4 * (n // block)),
                            ("dequantize", dequant, n * bits // 8 + 4 * (n // block) + 2 * n)):
            ms = time_launches(torch, fn, 12, stream)
            gbs = b / (ms / 1e3) / 1e9
            res[f"{name}_{bits}bit"] = {"us_per_launch": ms * 1e3, "algorithmic_bytes": b, "gbs": gbs,
                                        "frac_of_peak": gbs / peak}
    return res


def gpt13b_leg(torch, api, peak: float) -> dict:
    """The GPT-13B-shaped path (8 shards of [8192, 5120], n=256): per-launch
    device times (graph replays) of compress, reduce + decompress in one call,
    and the separate reduce and decompress."""
    from fp8_communication_compression_gb300 import workloads as W

    name = "gpt13b_p8x8192x5120_n256"
    w = W.WORKLOADS[name]
    P, rows, d, block = w["shards"], w["rows"], w["d"], w["block"]
    bits = np.stack([W.shard_input(name, p) for p in range(P)])
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    del bits
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
    return {k: {"us_per_launch": ms[k] * 1e3, "algorithmic_bytes": nb[k],
                "gbs": nb[k] / (ms[k] / 1e3) / 1e9, "frac_of_peak": nb[k] / (ms[k] / 1e3) / 1e9 / peak}
            for k in ms}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--kernel-events-every", type=int, default=10,
                    help="record per-kernel CUDA events on every N-th timed step")
    ap.add_argument("--e2e-chunks", type=int, default=4, help="row chunks of the host pipeline")
    ap.add_argument("--e2e-blocks", type=int, default=5, help="timed blocks of the end-to-end leg (median reported)")
    ap.add_argument("--cpu-rows", type=int, default=2048, help="oracle sample rows per shard")
    ap.add_argument("--ref-rows", type=int, default=128, help="reference arm rows per shard per step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true", help="skip nvidia-smi clock sampling")
    ap.add_argument("--no-agoq", action="store_true", help="skip the AGoQ accumulate/reduce leg")
    ap.add_argument("--no-int8", action="store_true", help="skip the INT8-codec leg")
    ap.add_argument("--no-laaq", action="store_true", help="skip the LAAQ activation-codec leg")
    ap.add_argument("--fused", action="store_true",
                    help="run reduce and decompress through the one-call entry point (taco_reduce_decompress)")
    ap.add_argument("--gpt13b", action="store_true",
                    help="also time the GPT-13B-shaped path (P=8, n=256; slow input generation)")
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

    import torch

    from fp8_communication_compression_gb300 import api

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    w, bits = make_inputs(rank, args.rows)
    P, rows, d, block = w["shards"], w["rows"], w["d"], w["block"]
    n = rows * d

    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    path = api.TwoShotLocal(P, rows, d, block, fused=args.fused)
    stream = torch.cuda.current_stream()

    for _ in range(args.warmup):
        path.run(x)
    torch.cuda.synchronize()

    launches = path.launches()
    names = [nm for nm, _ in launches]
    nbytes = path.bytes_per_step()
    step_bytes = sum(nbytes.values())
    K = args.steps
    # per-kernel events on every E-th step of the timed region; the other
    # steps run without events between their launches
    E = max(1, args.kernel_events_every)
    sampled = list(range(0, K, E))
    ev = {k: [torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)] for k in sampled}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler().start() if rank == 0 and not args.no_clocks else None
    time.sleep(0.2 if clocks else 0)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(K):
        e = ev.get(k)
        if e is None:
            for _, fn in launches:
                fn(x)
            continue
        e[0].record(stream)
        for i, (_, fn) in enumerate(launches):
            fn(x)
            e[i + 1].record(stream)
    end.record(stream)
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
    per = {name: statistics.mean(ev[k][i].elapsed_time(ev[k][i + 1]) for k in sampled)
           for i, name in enumerate(names)}

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
    spec = spec_hbm_gbs(torch)
    extra = {}
    if rank == 0 and not args.no_int8:
        extra["int8_" + HEADLINE] = int8_leg(torch, api, x, P, rows, d, block, peak)
    if rank == 0 and not args.no_agoq:
        del path, x
        torch.cuda.empty_cache()
        extra["agoq"] = agoq_leg(torch, api, peak)
        torch.cuda.empty_cache()
    if rank == 0 and not args.no_laaq:
        extra["laaq_8192x4096_n128"] = laaq_leg(torch, api, peak)
        torch.cuda.empty_cache()
    if rank == 0 and args.gpt13b:
        extra["gpt13b_p8x8192x5120_n256"] = gpt13b_leg(torch, api, peak)
        torch.cuda.empty_cache()
    flags = api.taco_device_error(clear=True)

    if rank == 0:
        value = whole_job_gbs(step_bytes, K, world, elapsed_ms)
        kern = {}
        for name in names:
            gbs = nbytes[name] / (per[name] / 1e3) / 1e9
            kern[name] = {"us_per_launch": per[name] * 1e3, "algorithmic_bytes": nbytes[name],
                          "gbs": gbs, "frac_of_peak": gbs / peak}
        achieved = kern["compress"]["gbs"]
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": args.warmup, "ms_per_step": elapsed_ms / K, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": HEADLINE if args.rows is None else f"{HEADLINE} (rows={rows})",
                       "P": P, "rows": rows, "d": d, "block": block,
                       "launches": names,
                       "kernel_events": f"per-launch CUDA events on every {E}th of the {K} timed steps",
                       "bytes_per_step": step_bytes,
                       "input_bf16_bytes_per_step": 2 * P * n,
                       "l2": "inputs larger than L2 (268 MB bf16 read per step), no flush",
                       "parallelism": f"replicas x{world}"},
            "roofline": {"bound": "hbm", "kernel": f"taco_compress_kernel<{block}>",
                         "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": committed_traffic(), "peak_source": peak_src,
                         "spec_peak": spec, "frac_of_spec": achieved / spec if spec else None},
            "kernels": kern,
            "step_frac_of_peak": value / world / peak,
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
            line["cpu_baseline"] = cpu_baseline(bits, w, args.cpu_rows)
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
