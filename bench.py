#!/usr/bin/env python3
"""Benchmark: batched decode over the 2-bit paged KV cache at the 27B geometry.

Workload (one step): 16 layers x 4 KV heads x head_dim 256, 24 query heads (GQA 6), 8 lanes
at a 40,960-token context after the step's append, pages scattered through one byte-sized
pool (8 x 40,960 x 9,216 B).  For every layer the step quantize-appends each lane's new
token (kv_quant_append) and runs paged_decode_attn for one query token per lane.  The step
is captured once in a CUDA graph and replayed.

Printed: one JSON line.  `value` = context tokens attended per second (lanes x 40,960 per
16-layer step, inputs resident in HBM); `e2e` = the same with the step's q/k/v copied from
pinned host memory and the outputs copied back inside the timed region; `roofline` = the
attention call's compressed-KV bytes over its CUDA-event duration against the measured HBM
copy bandwidth; `cpu_baseline` = the CPU oracle on a bounded sample of the same step.

`--impl reference` times the CPU oracle alone (the reference arm for this workload).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# page formats by name: the binding's (and the oracle's) format constant
FORMATS = {"hq2b": "FMT_HQ2B", "hq2b_had": "FMT_HQ2B_HAD", "hq2b_tok": "FMT_HQ2B_TOK", "fp8": "FMT_FP8",
           "bf16": "FMT_BF16"}
# bytes one head's one token costs for K plus V in each format
KV_BYTES = {"hq2b": 144, "hq2b_had": 144, "hq2b_tok": 144, "fp8": 512, "bf16": 1024}
WORKLOAD = dict(lanes=8, ctx=40960, layers=16, kv_heads=4, q_heads=24)
METRIC = "decode attn: compressed-KV tokens/s & achieved HBM GB/s (% of peak); prefill TFLOP/s"
UNIT = "tokens/s"


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


DECODE_SOURCES = ("decode_hq2b.cu", "kvq_internal.cuh", "attn_args.cuh", "append_ops.cuh", "mma_tma.cuh")
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_hq2b_main_27b_8x40960.md")


def _decode_source_hash():
    """sha256 of the decode kernel's sources with // comments and blank lines dropped, so that an
    edit of comments alone keeps a profile's counters valid."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in DECODE_SOURCES:
        with open(os.path.join(ROOT, "compressed_paged_kv_quant_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def _decode_traffic():
    """DRAM bytes per decode_hq2b_main launch from the committed ncu summary, if it was taken on
    the kernel source as it is now (its `traffic:` line records both); else None."""
    try:
        with open(DECODE_PROFILE) as f:
            for line in f:
                if line.startswith("traffic:"):
                    fields = dict(kv.split("=", 1) for kv in line[len("traffic:"):].split())
                    if fields.get("source_sha256") == _decode_source_hash():
                        return int(fields["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x: a job of N replicas takes as long as its slowest rank."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, tokens_per_step: int, ms: float) -> float:
    """Whole-job tokens per second: every rank processes tokens_per_step per step (weak scaling)."""
    return world * tokens_per_step / (ms / 1000.0)


def _config(extra=None, fmt="hq2b"):
    pages = {"fp8": "FP8 E4M3 pages (256 B/head/token each for K and V)",
             "bf16": "BF16 pages (512 B/head/token each for K and V)"}.get(fmt, "2-bit pages (72 B/head/token)")
    c = {"workload": "decode_27b_8x40960: 16 layers x 4 KV heads x 256, 24 q heads, 8 lanes x 40,960 tokens, "
                     f"{pages}, append + decode per layer",
         "lanes": WORKLOAD["lanes"], "context_tokens": WORKLOAD["ctx"], "layers": WORKLOAD["layers"],
         "kv_heads": WORKLOAD["kv_heads"], "q_heads": WORKLOAD["q_heads"], "head_dim": 256, "page_tokens": 64,
         "pool_bytes": WORKLOAD["lanes"] * WORKLOAD["ctx"] * WORKLOAD["layers"] * WORKLOAD["kv_heads"] * KV_BYTES[fmt],
         "l2_policy": "inputs larger than L2 (3.02 GB pool read per step)",
         "parallelism": "replicas only (one GPU per process)"}
    if extra:
        c.update(extra)
    return c


# ----------------------------------------------------------------------------- clocks
class Clocks:
    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="kvq_bench_clocks_", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                 "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "50", "-i", str(_device_index())],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 9:
                    continue
                try:
                    sm.append(float(f[1]))
                    mx = max(mx, float(f[2]))
                except ValueError:
                    continue
                for n, v in zip(names, f[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        except Exception:
            return None
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm),
                "window": "warm-up, timed decode steps, per-call timing and the end-to-end steps"}


def _device_index():
    v = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if v:
        ids = [x for x in v.split(",") if x.strip()]
        if local < len(ids) and ids[local].strip().isdigit():
            return int(ids[local])
    return local


# ----------------------------------------------------------------------------- CPU oracle arm
class OracleDecode:
    """The CPU oracle on lane 0 of the workload, layer 0's cache: set up once (host inputs,
    history appended, untimed), then timed per lane-layer decode (append of the step token +
    fp64 attention of all 24 query heads over the lane's 40,960 tokens).  The oracle's cost
    does not depend on the values, so one layer's cache stands in for every layer."""

    def __init__(self, seed=0, threads=None, fmt="FMT_HQ2B"):
        import numpy as np

        import oracle
        from compressed_paged_kv_quant_gb300 import synth
        self.oracle = oracle
        wl = synth.batched_decode_27b(seed=seed)
        self.wl, self.n = wl, wl.seq_len[0]
        n = self.n
        self.g = oracle.geom(getattr(oracle, fmt), 1, wl.num_kv_heads, wl.num_q_heads)
        npg = n // 64
        self.pool = np.zeros(npg * oracle.page_bytes(self.g), np.uint8)
        self.ring = np.zeros((1, 1, wl.num_kv_heads, 64, 256), np.uint16)
        self.pt = np.arange(npg, dtype=np.int32)[None, :]
        self.k = synth.kv_np_parallel(wl, 0, 0, 0, n, 0)
        self.v = synth.kv_np_parallel(wl, 0, 0, 0, n, 1)
        assert oracle.append(self.g, 0, self.pool, self.ring, self.pt, 1, [0], [n - 1], [0], self.k, self.v) == 0
        self.q = wl.q_np(0, 0, n - 1, 1)[0]
        self.threads = threads or max(1, min(os.cpu_count() or 1, wl.num_q_heads))

    def run(self, repeats):
        """Seconds for `repeats` lane-layer decode steps."""
        o, n = self.oracle, self.n
        heads = range(self.wl.num_q_heads)
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(self.threads) as ex:
            for _ in range(repeats):
                assert o.append(self.g, 0, self.pool, self.ring, self.pt, 1, [n - 1], [1], [n - 1], self.k, self.v) == 0
                list(ex.map(lambda j: o.attend(self.g, 0, self.pool, self.ring, 0, self.pt[0], 0, n, j, self.q[j], n,
                                               0.0625), heads))
        return time.perf_counter() - t0

    def value(self, repeats, seconds):
        """Context tokens per second in the benchmark's unit (16-layer steps)."""
        return repeats * self.n / self.wl.num_layers / seconds

    def describe(self, repeats):
        return (f"lane 0 of 8, {repeats} lane-layer decode steps on layer 0's cache (append of the step token + "
                f"fp64 attention of all {self.wl.num_q_heads} query heads over {self.n} tokens), {self.threads} "
                f"threads; scaled to 16-layer steps (context tokens per second)")


def run_reference(args):
    """The reference arm: the CPU oracle, as it stands, on the host cores; one step = one lane
    through all 16 layers (16 lane-layer decodes)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    od = OracleDecode(seed=args.seed)
    per_step = od.wl.num_layers
    for _ in range(args.warmup):
        od.run(1)
    secs = [od.run(per_step) for _ in range(args.steps)]
    value = od.value(per_step * args.steps, sum(secs))
    lane_layer_ms = 1000.0 * sum(secs) / (per_step * args.steps)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * WORKLOAD["lanes"] * WORKLOAD["ctx"] / value,
            "measured": {"lane_layer_ms": lane_layer_ms, "lane_layers_timed": per_step * args.steps,
                         "seconds": round(sum(secs), 2),
                         "ms_per_step_is": (f"derived: the measured lane-layer time x {WORKLOAD['lanes']} lanes x "
                                            f"{od.wl.num_layers} layers (one lane of the 8 was timed, through all "
                                            "16 layers' worth of decodes on one layer's cache)")},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": od.threads, "kind": "oracle",
                             "sample": od.describe(per_step) + f" per step, {args.steps} steps"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ----------------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch
    import torch.distributed as dist

    from compressed_paged_kv_quant_gb300 import build, kvq, synth
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    build.build()

    wl = synth.batched_decode_27b(seed=args.seed + rank, lanes=args.lanes, ctx=args.ctx, layers=args.layers)
    L, lanes, ctx = wl.num_layers, wl.lanes, wl.seq_len[0]
    H, Hq = wl.num_kv_heads, wl.num_q_heads
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl, getattr(kvq, FORMATS[args.format]), dev, fill=None, stream=stream.cuda_stream)
        dw.fill_history([n - 1 for n in wl.seq_len], chunk=16384)
        # one contiguous input buffer (q, k, v of every layer) and one output buffer per step
        n_q, n_kv = lanes * Hq * 256, lanes * H * 256
        step_in = torch.empty(L * (n_q + 2 * n_kv), dtype=torch.bfloat16, device=dev)
        q_v, k_v, v_v = [], [], []
        for l in range(L):
            base = l * (n_q + 2 * n_kv)
            q_v.append(step_in[base:base + n_q].view(lanes, Hq, 256))
            k_v.append(step_in[base + n_q:base + n_q + n_kv].view(lanes, H, 256))
            v_v.append(step_in[base + n_q + n_kv:base + n_q + 2 * n_kv].view(lanes, H, 256))
            q_v[l].copy_(dw.step_q(l))
            k, v = dw.step_kv(l)
            k_v[l].copy_(k)
            v_v[l].copy_(v)
        ws, _ = dw.decode_buffers()
        step_out = torch.empty((L, lanes, Hq, 256), dtype=torch.float32, device=dev)
    stream.synchronize()
    assert dw.cache.read_status() == 0

    def step():
        for l in range(L):
            if args.step_calls == "fused":
                dw.decode_step(l, q_v[l], k_v[l], v_v[l], ws, step_out[l])
            else:
                dw.append_step(l, k_v[l], v_v[l])
                dw.decode(l, q_v[l], ws, step_out[l])

    # capture one step in a CUDA graph
    with torch.cuda.stream(stream):
        step()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    stream.synchronize()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = Clocks()
    clocks.start()
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            g.replay()
    barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            g.replay()
        e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, world, dev)
    assert dw.cache.read_status() == 0, "device status flagged during the timed steps"
    tokens_per_step = lanes * ctx
    value = job_throughput(world, tokens_per_step, ms)

    # per-call duration of the attention: the L decode calls of one step captured alone in a
    # graph (no host launch gaps), CUDA events on the launching stream around its replays
    gd = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gd, stream=stream):
        for l in range(L):
            dw.decode(l, q_v[l], ws, step_out[l])
    stream.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(3):
            gd.replay()
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = max(3, args.steps)
        d0.record(stream)
        for _ in range(reps):
            gd.replay()
        d1.record(stream)
    stream.synchronize()
    call_ms = d0.elapsed_time(d1) / (reps * L)
    attn_bytes = lanes * ctx * H * KV_BYTES[args.format]   # K+V bytes one layer's attention reads
    peak, peak_src = _peaks()
    achieved = attn_bytes / (call_ms / 1000.0) / 1e9

    # end to end: the step's q/k/v from pinned host memory, outputs back to pinned host memory
    h_in = step_in.cpu().pin_memory()
    h_out = torch.empty(step_out.shape, dtype=step_out.dtype, pin_memory=True)
    h2d = h_in.numel() * h_in.element_size()
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        step_in.copy_(h_in, non_blocking=True)
        g.replay()
        h_out.copy_(step_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e_step()
    barrier()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            e2e_step()
        e1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    e2e_value = job_throughput(world, tokens_per_step, e2e_ms)
    clk = clocks.stop()

    moves = None if args.no_page_moves else run_page_moves(dw, stream)
    del dw, step_in, step_out, ws
    torch.cuda.empty_cache()
    prefill = None if (args.no_prefill or args.format != "hq2b") else run_prefill(args, dev, stream)
    prefill_fmts = None
    if not (args.no_prefill or args.no_legs or args.format != "hq2b"):
        prefill_fmts = {}
        for f in ("hq2b_tok", "hq2b_had", "fp8"):
            r = run_prefill(args, dev, stream, fmt=f, layers=1, steps=2)
            prefill_fmts[f] = {k: r[k] for k in ("ms_per_layer_attention", "tflops", "roofline")}
            torch.cuda.empty_cache()
    mixed = None if (args.no_legs or args.format != "hq2b") else run_mixed(args, dev, stream)
    needle = None if (args.no_legs or args.format != "hq2b") else run_needle(args, dev, stream)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        od = OracleDecode(seed=args.seed, fmt=FORMATS[args.format])
        od.run(1)
        dt = od.run(args.cpu_repeats)
        cpu = {"value": od.value(args.cpu_repeats, dt), "unit": UNIT, "cores": od.threads, "kind": "oracle",
               "sample": od.describe(args.cpu_repeats), "seconds": round(dt, 2),
               "lane_layer_ms": 1000.0 * dt / args.cpu_repeats}
        od.threads = 1
        r1 = max(1, args.cpu_repeats // 16)
        dt1 = od.run(r1)
        cpu["one_core"] = {"value": od.value(r1, dt1), "unit": UNIT, "cores": 1, "sample": od.describe(r1),
                           "seconds": round(dt1, 2), "lane_layer_ms": 1000.0 * dt1 / r1}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f16 mma / f32 accumulate (2-bit codes)", "data": "synthetic",
                "config": _config({"ms_per_attention_call": call_ms, "peak_source": peak_src,
                                   "step_calls": args.step_calls, "format": args.format}, args.format),
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak,
                             "traffic": _decode_traffic() if args.format == "hq2b" else None,
                             "kernel": ("paged_decode_attn (decode_hq2b_main + decode_hq2b_combine), one layer"
                                        if args.format == "hq2b" else
                                        ("paged_decode_attn (rotate_q_kernel + decode_hq2b_main<centred> + "
                                         "decode_hq2b_combine), one layer") if args.format == "hq2b_had" else
                                        ("paged_decode_attn (decode_hq2b_main<per-token K> + decode_hq2b_combine), "
                                         "one layer") if args.format == "hq2b_tok" else
                                        "paged_decode_attn (decode_fp8_split + attn_combine), one layer"
                                        if args.format == "fp8" else
                                        "paged_decode_attn (attn_split_generic + attn_combine, CUDA cores), one layer"),
                             "algorithmic_bytes_per_launch": attn_bytes},
                "cpu_baseline": cpu,
                "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
                "gpu_launches": (4 if args.format == "hq2b_had" else 3) * L * args.steps,
                "clocks": clk,
                "prefill": prefill,
                "prefill_format_variants": prefill_fmts,
                "mixed_shared_prefix": mixed,
                "needle_hq2b_and_bf16": needle,
                "page_moves": moves}
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_page_moves(dw, stream, reps=5):
    """Bit-exact page moves of one lane's whole context (640 pages of the 27B geometry, every layer
    and head, 377 MB): gather to a pinned host arena, scatter back, and gather to a device arena;
    next to one contiguous cudaMemcpyAsync of the same bytes each way (the copy engines)."""
    import torch

    from compressed_paged_kv_quant_gb300 import kvq
    ids = torch.from_numpy(dw.wl.page_table[0][dw.wl.page_table[0] >= 0].copy()).to(dw.device)
    pb = kvq.page_bytes(dw.g)
    nbytes = ids.numel() * pb
    host = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    devbuf = torch.empty(nbytes, dtype=torch.uint8, device=dw.device)

    def timed(fn):
        ts = []
        with torch.cuda.stream(stream):
            fn()
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                fn()
                e1.record(stream)
                stream.synchronize()
                ts.append(e0.elapsed_time(e1))
        return statistics.median(ts)

    st = stream.cuda_stream
    g_h = timed(lambda: kvq.pages_gather(dw.g, dw.cache.pool, ids, host, dw.cache.status, st))
    s_h = timed(lambda: kvq.pages_scatter(dw.g, dw.cache.pool, ids, host, dw.cache.status, st))
    g_d = timed(lambda: kvq.pages_gather(dw.g, dw.cache.pool, ids, devbuf, dw.cache.status, st))
    c_dh = timed(lambda: host.copy_(devbuf, non_blocking=True))
    c_hd = timed(lambda: devbuf.copy_(host, non_blocking=True))
    assert dw.cache.read_status() == 0, "device status flagged during page moves"
    gbs = lambda ms, factor=1: factor * nbytes / (ms / 1e3) / 1e9
    return {"workload": f"{ids.numel()} pages x {pb} B (one lane, all layers and heads)", "bytes": nbytes,
            "gather_to_pinned_host_gbs": gbs(g_h), "scatter_from_pinned_host_gbs": gbs(s_h),
            "gather_device_to_device_gbs": gbs(g_d, 2),
            "memcpy_device_to_host_gbs": gbs(c_dh), "memcpy_host_to_device_gbs": gbs(c_hd),
            "note": "device-to-device counts read + write bytes; host legs count the bytes moved"}


def _graph_ms(stream, fn, reps, warm=3):
    """ms per replay of one CUDA graph of fn() (run once eagerly first), CUDA events on the stream."""
    import torch
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / reps


def run_mixed(args, dev, stream):
    """The mixed pool with shared prefixes (1 x 131,072 + 8 x 4,096 tokens, the short lanes'
    first 2,048 tokens on 32 shared pages, window 64): one decode step per layer through
    kvq_decode_step in one CUDA graph, and the attention call alone.  GB/s on the unique
    compressed bytes (pages in the pool) and on the logical ones (every lane's tokens)."""
    import torch

    from compressed_paged_kv_quant_gb300 import kvq, synth
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    wl = synth.mixed_shared_27b(layers=args.layers)
    L, H = wl.num_layers, wl.num_kv_heads
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl, kvq.FMT_HQ2B, dev, fill=None, stream=stream.cuda_stream)
        dw.fill_history([n - 1 for n in wl.seq_len], chunk=16384)
        qs = [dw.step_q(l) for l in range(L)]
        kvs = [dw.step_kv(l) for l in range(L)]
        ws, _ = dw.decode_buffers()
        outs = torch.empty((L, wl.lanes, wl.num_q_heads, 256), dtype=torch.float32, device=dev)
    stream.synchronize()

    def step():
        for l in range(L):
            dw.decode_step(l, qs[l], kvs[l][0], kvs[l][1], ws, outs[l])

    def attn():
        for l in range(L):
            dw.decode(l, qs[l], ws, outs[l])

    reps = max(10, args.steps // 4)
    step_ms = _graph_ms(stream, step, reps)
    call_ms = _graph_ms(stream, attn, reps) / L
    assert dw.cache.read_status() == 0, "device status flagged in the mixed-pool leg"
    unique = wl.pool_pages * 64 * H * KV_BYTES["hq2b"]
    logical = sum(wl.seq_len) * H * KV_BYTES["hq2b"]
    peak, _ = _peaks()
    gbs = lambda b: b / (call_ms / 1e3) / 1e9
    return {"workload": "mixed_27b: 1 x 131,072 + 8 x 4,096 tokens (first 2,048 of the short lanes on 32 shared "
                        f"pages), window 64, {L} layers, 4 KV heads, 24 q heads, 2-bit pages",
            "ms_per_step": step_ms, "ms_per_attention_call": call_ms,
            "unique_bytes_per_layer": unique, "logical_bytes_per_layer": logical,
            "gbs_unique": gbs(unique), "gbs_logical": gbs(logical), "frac_unique": gbs(unique) / peak,
            "context_tokens_per_s": sum(wl.seq_len) / (step_ms / 1e3),
            "l2_policy": f"inputs larger than L2 ({unique * L / 1e9:.2f} GB of pages per step)"}


def run_needle(args, dev, stream, reps=30):
    """The needle workload (1 layer, 4 KV heads, 24 q heads, 131,072 tokens): one attention call
    over the 2-bit pool (75.5 MB, smaller than L2) and over the BF16 pool (537 MB), L2 flushed by
    a 256 MB write before every timed call; CUDA events around each call."""
    import torch

    from compressed_paged_kv_quant_gb300 import kvq, synth
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    wl = synth.needle_131k()
    n, H = wl.seq_len[0], wl.num_kv_heads
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    peak, _ = _peaks()
    res = {"workload": "needle_131072: 1 layer, 4 KV heads, 24 q heads, 131,072 tokens, one needle",
           "l2_policy": "256 MB buffer written before every timed call"}
    for fmt in ("hq2b", "bf16"):
        with torch.cuda.stream(stream):
            dw = DeviceWorkload(wl, getattr(kvq, FORMATS[fmt]), dev, fill=None, stream=stream.cuda_stream)
            dw.fill_history([n], chunk=16384)
            q = dw.step_q(0)
            ws, out = dw.decode_buffers()
            for _ in range(3):
                dw.decode(0, q, ws, out)
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
            for e0, e1 in ev:
                flush.fill_(1)
                e0.record(stream)
                dw.decode(0, q, ws, out)
                e1.record(stream)
        stream.synchronize()
        assert dw.cache.read_status() == 0, "device status flagged in the needle leg"
        ms = statistics.median(e0.elapsed_time(e1) for e0, e1 in ev)
        nbytes = n * H * KV_BYTES[fmt]
        res[fmt] = {"ms_per_attention_call": ms, "bytes": nbytes, "gbs": nbytes / (ms / 1e3) / 1e9,
                    "frac": nbytes / (ms / 1e3) / 1e9 / peak}
        del dw
        torch.cuda.empty_cache()
    res["hq2b_over_bf16_time"] = res["hq2b"]["ms_per_attention_call"] / res["bf16"]["ms_per_attention_call"]
    return res


def prefill_flops(prefix, chunk, q_heads):
    """Causal attention FLOPs of one layer: 4 * 256 per (query, key) pair per query head."""
    pairs = chunk * prefix + chunk * (chunk + 1) // 2
    return 4.0 * 256 * pairs * q_heads


def run_prefill(args, dev, stream, fmt="hq2b", layers=None, steps=None):
    """Chunked prefill over a compressed prefix (65,536 + 1,024 tokens, 16 layers): each layer
    appends the chunk's K/V, then paged_prefill_attn with a garbage-filled workspace."""
    import torch

    from compressed_paged_kv_quant_gb300 import kvq, synth
    from compressed_paged_kv_quant_gb300.workload import DeviceWorkload
    prefix, chunk = args.prefill_prefix, 1024
    wl = synth.chunked_prefill_27b(prefix=prefix, chunk=chunk, layers=layers or args.layers)
    L = wl.num_layers
    with torch.cuda.stream(stream):
        dw = DeviceWorkload(wl, getattr(kvq, FORMATS[fmt]), dev, fill=None, stream=stream.cuda_stream)
        dw.fill_history([prefix], chunk=16384)
        ks = [wl.kv_torch(l, 0, prefix, chunk, 0, dev) for l in range(L)]
        vs = [wl.kv_torch(l, 0, prefix, chunk, 1, dev) for l in range(L)]
        qs = [wl.q_torch(l, 0, prefix, chunk, dev) for l in range(L)]
        ws, out = dw.prefill_buffers(chunk)
        ws.view(torch.int32).fill_(-1)                       # garbage: the kernels never read unwritten bytes
        i32 = lambda xs: torch.tensor(xs, dtype=torch.int32, device=dev)
        sp, nn, to = i32([prefix]), i32([chunk]), i32([0])
        qp, nq, qo = i32([prefix]), i32([chunk]), i32([0])

    def step(timed=None):
        for l in range(L):
            kvq.kv_quant_append(dw.g, l, dw.cache.pool, dw.cache.ring, dw.page_table, sp, nn, to, chunk, ks[l], vs[l],
                                dw.cache.status, stream.cuda_stream)
            if timed is not None:
                timed[l][0].record(stream)
            kvq.paged_prefill_attn(dw.g, l, dw.cache.pool, dw.cache.ring, 0, dw.page_table, qp, nq, qo, chunk,
                                   dw.seq_len, dw.max_seq_len, qs[l], dw.sm_scale, ws, out, dw.cache.status,
                                   stream.cuda_stream)
            if timed is not None:
                timed[l][1].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(2):
            step()
    stream.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    call_ms = []
    steps = max(2, steps or args.prefill_steps)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            step(ev)
            stream.synchronize()
            call_ms += [x.elapsed_time(y) for x, y in ev]
        e1.record(stream)
    stream.synchronize()
    assert dw.cache.read_status() == 0, "device status flagged during prefill"
    step_ms = e0.elapsed_time(e1) / steps
    ms = statistics.median(call_ms)
    flops = prefill_flops(prefix, chunk, wl.num_q_heads)
    peak = 1925.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peak = float(json.load(f)["bf16_tflops"])
    except Exception:
        pass
    tflops = flops / (ms / 1000.0) / 1e12
    return {"workload": f"prefill_27b: {chunk}-token chunk over a {prefix}-token prefix, {L} layers, 24 q heads, "
                        f"{fmt} pages",
            "ms_per_layer_attention": ms, "ms_per_step": step_ms, "flop_per_layer": flops, "tflops": tflops,
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak, "peak_source": "measured bf16 dense (fp16 MMA runs at the same rate)"},
            "workspace": "filled with 0xFF before the timed steps, never zeroed"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-repeats", type=int, default=64,
                    help="oracle decodes of one lane-layer timed for the CPU baseline")
    # smaller cases of the same workload, for profiling only (the defaults are the benchmark)
    ap.add_argument("--lanes", type=int, default=WORKLOAD["lanes"])
    ap.add_argument("--ctx", type=int, default=WORKLOAD["ctx"])
    ap.add_argument("--layers", type=int, default=WORKLOAD["layers"])
    ap.add_argument("--format", default="hq2b", choices=sorted(FORMATS),
                    help="page format: hq2b (the benchmark's), hq2b_had (Walsh-Hadamard-rotated 2-bit), "
                         "hq2b_tok (K per token), fp8 (E4M3) or bf16 (the exact reference path); the "
                         "variants time decode only")
    ap.add_argument("--no-prefill", action="store_true")
    ap.add_argument("--no-legs", action="store_true", help="skip the mixed-pool and needle legs")
    ap.add_argument("--leg", default=None, choices=["mixed", "needle", "prefill"],
                    help="run one leg alone and print its JSON (for profiling)")
    ap.add_argument("--no-page-moves", action="store_true")
    ap.add_argument("--step-calls", default="fused", choices=["fused", "separate"],
                    help="one kvq_decode_step per layer, or kv_quant_append + paged_decode_attn")
    ap.add_argument("--prefill-prefix", type=int, default=65536)
    ap.add_argument("--prefill-steps", type=int, default=3)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.leg:
        return run_leg(args)
    return run_gpu(args)


def run_leg(args):
    """One leg alone on cuda:0 (a smaller command to profile under ncu)."""
    import torch

    from compressed_paged_kv_quant_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.Stream(device=dev)
    if args.leg == "prefill":
        res = run_prefill(args, dev, stream, fmt=args.format if args.format != "bf16" else "hq2b")
    else:
        res = {"mixed": run_mixed, "needle": run_needle}[args.leg](args, dev, stream)
    print(json.dumps({"leg": args.leg, "result": res}))
    return 0


if __name__ == "__main__":
    sys.exit(main())
