"""Benchmark: one decode-maximal hybrid batch through the LLaMA-13B layer.

Workload (one step): a prefill chunk of 256 tokens at offset 768 of a
1024-token prompt plus 18 decodes at context 1024, T = 274 rows, through one
LLaMA-13B decoder layer (hidden 5120, 40 heads x 128, SwiGLU FFN 13824),
bf16 weights ~N(0, 0.02), KV cache ~N(0, 1) in shuffled 16-token blocks.
Every step writes the batch's K/V and reads 399 MB of KV plus 634 MB of
weights, far more than the 126 MB L2, so no L2 flush is needed between steps.

Reported (one JSON line on rank 0):
  value      hybrid-batch tokens/s (T x steps / device time), inputs resident
  e2e        the same through hb_forward_host: pinned host x in, host y out
  decode     decode tok/s piggybacked (marginal over the chunk alone, the
             pages' definition) vs in a decode-only batch of the same 18
  roofline   the dominant kernel against MEASURED_PEAKS.json
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same batch

``--impl reference`` times the CPU oracle instead (the only reference arm:
the pages ship no code).  For N > 1 GPUs each rank runs an independent
replica (no collective on the data path); value sums the ranks' tokens over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "hybrid-batch tokens/s; decode tok/s piggybacked vs decode-only; % of TC/HBM roofline"
WORKLOAD = "llama13b-hybrid-c256@768-d18@1024"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


# --------------------------------------------------------------- clocks

class Clocks:
    """SM clock and clock-event reasons sampled during the timed region.

    Polls NVML (the driver's libnvidia-ml, through ctypes) about every
    millisecond from a thread, so even a timed region of a few milliseconds
    gets samples; falls back to nvidia-smi at 200 ms when NVML is missing."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.max_mhz = None
        self.nvml = None
        self.handle = None
        self.thread = None
        self.stop = False
        self.smi = None

    def _open_nvml(self):
        import ctypes
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
        except OSError:
            return False
        if lib.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = False
        try:
            import torch
            pr = torch.cuda.get_device_properties(self.gpu)
            bus = "%08x:%02x:%02x.0" % (getattr(pr, "pci_domain_id", 0), pr.pci_bus_id, pr.pci_device_id)
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
        except Exception:
            ok = False
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(self.gpu, ctypes.byref(h)) != 0:
            return False
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:  # NVML_CLOCK_SM
            self.max_mhz = float(mx.value)
        self.nvml, self.handle = lib, h
        return True

    def _poll(self):
        import ctypes
        mhz, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        get_r = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self.stop:
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0 and \
                    get_r(self.handle, ctypes.byref(rs)) == 0:
                self.samples.append((float(mhz.value), int(rs.value)))
            time.sleep(0.001)

    def __enter__(self):
        import threading
        if self._open_nvml():
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return self
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.smi = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={q}",
                                         "--format=csv,noheader,nounits", "-lms", "200"],
                                        stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.smi = None
        return self

    def __exit__(self, *a):
        self.stop = True
        if self.thread is not None:
            self.thread.join(timeout=5)
        if self.smi is not None:
            self.smi.terminate()
            try:
                self.smi.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.smi.kill()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            bits = [0x8, 0x40, 0x20, 0x4]
            try:
                with open(self.path) as f:
                    for line in f:
                        t = [x.strip() for x in line.split(",")]
                        if len(t) >= 6 and t[0].replace(".", "").isdigit():
                            r = sum(b for b, v in zip(bits, t[2:6]) if v.lower().startswith("active"))
                            self.samples.append((float(t[0]), r))
                            if t[1].replace(".", "").isdigit():
                                self.max_mhz = float(t[1])
                os.unlink(self.path)
            except OSError:
                pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"], "samples": 0}
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(m for m, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples),
                "source": "nvml" if self.nvml is not None else "nvidia-smi"}


# ----------------------------------------------------------- distributed

def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group("gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU oracle

def oracle_sample(w, target_s: float):
    """Time the oracle on the first rows of the chunk plus the first decodes.

    Rows are chosen so the sample respects causality (chunk rows 0..s-1) and
    grows until about target_s seconds of wall time.  Returns
    (rows_per_s, rows, seconds, threads).
    """
    from oracle import oracle as orc
    from chunked_prefill_hybrid_gb300 import synth
    threads = orc.max_threads()
    pools = orc.Pool(w.num_blocks, w.dims.n_kv_heads, w.dims.head_dim)
    for layer, s, k, v in w.prefix:
        if layer == 0:
            pools.write(s.block_table, 0, synth.bf16_to_f32(k).astype(np.float64),
                        synth.bf16_to_f32(v).astype(np.float64))
    x = synth.bf16_to_f32(w.x).astype(np.float64)
    T, C = w.T, w.batch.chunk_len

    def run(n_chunk, n_dec):
        rows = np.zeros(T, bool)
        rows[:n_chunk] = True
        rows[C:C + n_dec] = True
        t0 = time.perf_counter()
        orc.layer_forward(w.dims, w.weights[0], w.batch, x, pools, mirror=True, rows=rows)
        return time.perf_counter() - t0, int(rows.sum())

    dt, n = run(max(1, threads // 2), max(1, threads // 2))
    per_row = dt / n
    want = int(min(T, max(n, target_s / max(per_row, 1e-9))))
    n_dec = min(w.batch.n_decodes, want // 2)
    n_chunk = min(C, want - n_dec)
    dt, n = run(n_chunk, n_dec)
    return n / dt, n, dt, threads


def oracle_one_core(w, target_s: float):
    """The oracle on one thread over a bounded sample (first chunk rows and
    first decodes, about target_s seconds); returns (rows_per_s, rows, s)."""
    from oracle import oracle as orc
    threads = orc.max_threads()
    orc.set_threads(1)
    try:
        rps, n, dt, _ = oracle_sample(w, target_s)
    finally:
        orc.set_threads(threads)
    return rps, n, dt


def run_reference(args):
    """The reference arm: the CPU oracle on the host cores, same workload."""
    world, rank, local = dist_init(args.gpus)
    if rank != 0:
        return 0
    from chunked_prefill_hybrid_gb300 import workloads
    from oracle import oracle as orc
    orc.build()
    w = workloads.llama13b_hybrid(seed=2)
    per_step = []
    sample = None
    for i in range(args.warmup + args.steps):
        rps, n, dt, threads = oracle_sample(w, target_s=args.ref_seconds)
        if i >= args.warmup:
            per_step.append((rps, n, dt))
        sample = f"first {n // 2} chunk rows + decode rows ({n} rows of {w.T}), one layer, fp64, mirror mode"
    value = statistics.median([r for r, _, _ in per_step])
    ms = statistics.median([dt * 1e3 for _, _, dt in per_step])
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": 1, "T": w.T},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": sample, "one_core": dict(zip(("value", "rows", "seconds"),
                                                                    oracle_one_core(w, args.ref_seconds / 3)))},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------- GPU arm

def time_steps(torch, ctx, fn, steps, world):
    s = torch.cuda.current_stream()
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(s)
    for _ in range(steps):
        fn()
    e1.record(s)
    torch.cuda.synchronize()
    barrier(world)
    return e0.elapsed_time(e1)


def profiled(torch, ctx, fn, steps, world):
    """Per-kind (total ms, launches) over `steps` calls of fn, from the
    library's CUDA events around every launch."""
    ctx.profile(True)
    time_steps(torch, ctx, fn, steps, world)
    ctx.sync()
    prof = ctx.profile_read()
    ctx.profile(False)
    return prof


GEMM_KINDS = ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down")


def gemm_decode_cost(prof_hybrid, prof_chunk, prof_decode, steps, D):
    """Per-decode-token cost on the linear ops alone: the GEMM launches of
    each batch (each with its reduce pass), marginal over the chunk alone,
    (hybrid - chunk alone) / D, against decode-only / D.  The profiled times
    come from events around every launch, so each batch's sum leaves out the
    overlap of neighbouring launches in the same way."""
    def gemm_ms(prof):
        return sum(prof.get(k, (0.0, 0))[0] for k in GEMM_KINDS) / steps
    gh, gc, gd = gemm_ms(prof_hybrid), gemm_ms(prof_chunk), gemm_ms(prof_decode)
    marginal = (gh - gc) / D
    return {"ms_gemm_hybrid": gh, "ms_gemm_chunk_alone": gc, "ms_gemm_decode_only": gd,
            "per_decode_cost_ratio": (gd / D) / marginal if marginal > 0 else None}


# ncu summaries under profiles/ that carry a measured DRAM traffic figure for
# a kernel: "traffic_bytes_per_launch: N" and "sources: a b c" (files under
# the package's csrc/) with "sources_sha256: H" of their concatenated bytes.
# The figure is reported only while those sources are unchanged.
TRAFFIC_PROFILES = {
    "attention": "attention_llama13b_hybrid_c256_d18.md",
    "gemm_gate_up": "gemm_pair_gate_up_llama13b_hybrid_c256_d18.md",
}


TILE_CURVE_CHUNKS = list(range(200, 321)) + [64, 128, 384, 494, 512, 1024]


def tile_curve(args, torch, native, workloads, synth, world, rank):
    """Layer time against the chunk size C (LLaMA-13B layer, chunk at offset
    768, 18 decodes at ctx 1024): the GB300 form of the pages' tile-quantization
    curve (SARATHI summary, "The tile quantization effect", Figure 7: 256 vs 257).  The
    step in time every `quantum` rows of T = C + 18 is the tile a chunk size
    should be aligned to."""
    cmax = max(TILE_CURVE_CHUNKS)
    w = workloads.make("llama13b-tile-curve", synth.LLAMA_13B, 2 + rank, 768, cmax, [1024] * 18)
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx, poison=None)
    steps = max(10, min(args.steps, 50))
    points = []
    for C in sorted(TILE_CURVE_CHUNKS):
        b = synth.HybridBatch(w.batch.chunk, C, w.batch.decodes)
        spec = native.Spec(b)
        xc = torch.cat([x[:C], x[cmax:]]).contiguous()
        yc = torch.empty_like(xc)
        fn = lambda: ctx.forward(spec, xc, yc)
        for _ in range(args.warmup):
            fn()
        ctx.sync()
        ms = max_over_ranks(world, time_steps(torch, ctx, fn, steps, world)) / steps
        points.append({"chunk": C, "T": C + 18, "ms": round(ms, 5), "tok_s": round((C + 18) / ms * 1e3)})
    ctx.free()
    # rows at which the time steps up by more than 1.5 % over the previous chunk size
    steps_at = [p["T"] for a, p in zip(points, points[1:])
                if p["chunk"] == a["chunk"] + 1 and p["ms"] > a["ms"] * 1.015]
    if rank == 0:
        print(json.dumps({"tile_curve": WORKLOAD.replace("c256", "cX"), "steps_timed": steps,
                          "step_up_at_T": steps_at, "points": points}), flush=True)
    return 0


def prefill_sweep(args, torch, native, workloads, synth, world, rank):
    """The single-layer comparisons the pages make beside the hybrid batch
    (LLaMA-13B layer): prefill-only batches of T in {64, ..., 1024} tokens (one
    request at offset 0; SARATHI summary, section 2, Figure 4a, the prefill
    plateau at B x L >= 512), decode-only batches of B in {1, 2, 18} at context
    1024 with their per-token cost against the 1024-token prefill's (Figure 3:
    200x / 100x / 16.7x on an A6000), and Table 2's three batches of 1024 rows
    (prefill-only, decode-only of 4, hybrid of 1021 prompt tokens + 3 decodes)
    with the hybrid's marginal decode cost.  One JSON line."""
    w = workloads.make("llama13b-prefill-sweep", synth.LLAMA_13B, 2 + rank, 0, 1024, [1024] * 18)
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx, poison=None)
    steps = max(10, min(args.steps, 50))
    chunk, decs = w.batch.chunk, w.batch.decodes

    def timed(b, rows):
        spec = native.Spec(b)
        xi = rows.contiguous()
        yi = torch.empty_like(xi)
        fn = lambda: ctx.forward(spec, xi, yi)
        for _ in range(args.warmup):
            fn()
        ctx.sync()
        return max_over_ranks(world, time_steps(torch, ctx, fn, steps, world)) / steps

    prefill = {}
    for T in (64, 128, 256, 512, 1021, 1024):
        prefill[T] = timed(synth.HybridBatch(chunk, T, []), x[:T])
    decode = {}
    for B in (1, 2, 3, 4, 18):
        decode[B] = timed(synth.HybridBatch(None, 0, decs[:B]), x[1024:1024 + B])
    hybrid = timed(synth.HybridBatch(chunk, 1021, decs[:3]), torch.cat([x[:1021], x[1024:1027]]))
    ctx.free()
    per_tok_prefill = prefill[1024] / 1024
    line = {
        "prefill_sweep": "llama13b-layer", "steps_timed": steps,
        "prefill_only": [{"T": T, "ms": round(ms, 5), "tok_per_ms": round(T / ms, 1),
                          "us_per_token": round(ms / T * 1e3, 4)} for T, ms in sorted(prefill.items())],
        "decode_vs_prefill_per_token": [{"B": B, "ctx": 1024, "ms": round(decode[B], 5),
                                         "us_per_token": round(decode[B] / B * 1e3, 3),
                                         "ratio_to_prefill_1024": round(decode[B] / B / per_tok_prefill, 1)}
                                        for B in (1, 2, 18)],
        "table2_1024_rows": {"prefill_only_ms": round(prefill[1024], 5), "decode_only_4_ms": round(decode[4], 5),
                             "hybrid_1021_plus_3_ms": round(hybrid, 5),
                             "decode_only_us_per_token": round(decode[4] / 4 * 1e3, 3),
                             "hybrid_marginal_decode_us_per_token": round((hybrid - prefill[1021]) / 3 * 1e3, 3),
                             "marginal_decode_cost_ratio": round((decode[4] / 4) / ((hybrid - prefill[1021]) / 3), 2)
                             if hybrid > prefill[1021] else None},
        "pages_context": {"fig3_ratio_B1_B2_B18": [200, 100, 16.7], "fig4a_plateau_tok_per_ms": 180,
                          "table2_ms_per_token": {"prefill": 0.229, "decode": 12.49, "hybrid_marginal": 1.2},
                          "hardware": "A6000, FP16"}}
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def serve_bench(args, torch, native, workloads, synth, world, rank):
    """LLaMA-33B, 60 layers, serving a closed set of requests present at t = 0:
    prompts uniform in [512, 2048], max_new = max(1, round(P / r)) for each P:D
    ratio r; decode-maximal batching with chunks of 256 under a 512-token budget
    (Sarathi-Serve) against the request-level baseline (prefill-only and
    decode-only batches) on the same kernels.  KV pool = the HBM left after the
    weights.  Layer l's matrices are one seeded draw with rows rotated by l;
    the KV cache starts as bf16 1.0 everywhere (every read position is written
    by the loop before it is read)."""
    from chunked_prefill_hybrid_gb300 import sched, serve
    L = 60
    dims = synth.LLAMA_33B.with_layers(L)
    base = synth.layer_weights(dims, 4 + rank, 0)
    free, _ = torch.cuda.mem_get_info()
    w_bytes = L * 2 * sum(v.size for v in base.values())
    kv_tok = L * 2 * dims.n_kv_heads * dims.head_dim * 2
    num_blocks = int((free - w_bytes - 14 * 2**30) // (16 * kv_tok))
    max_pos, max_tokens, max_decodes = 4096, 4096, 512
    ctx = native.Context(native.model_config(dims, num_blocks, max_tokens, max_decodes, max_pos, n_layers=L))
    dev = {k: workloads.to_device(v) for k, v in base.items()}
    for l in range(L):
        ctx.load_layer(l, {k: (torch.roll(v, l, 0) if v.dim() == 2 else v) for k, v in dev.items()})
        ctx.sync()
    del dev, base
    ctx.fill_kv(0x3F80)
    x = workloads.to_device(synth.token_rows(4 + rank, (1,), max_tokens, dims.hidden))
    y = torch.empty_like(x)
    out = {}
    for r in [float(v) for v in args.serve_ratios.split(",")]:
        P = synth.uniform_ints(4 + rank, (2, int(r * 10)), args.serve_requests, 512, 2048)
        reqs = [(i, int(p), max(1, int(round(p / r)))) for i, p in enumerate(P)]
        row = {}
        for name, kw in (("decode_maximal", dict(chunk_size=256, token_budget=512)),
                         ("request_level", dict(chunk_size=1 << 20, token_budget=max_tokens,
                                                max_chunks_per_batch=16, max_decodes=max_decodes,
                                                request_level=1))):
            s = sched.Scheduler(num_blocks=num_blocks, max_blocks_per_seq=max_pos // 16, **kw)
            res = serve.run(ctx, s, reqs, x, y)
            row[name] = res.summary()
        dm, rl = row["decode_maximal"], row["request_level"]
        row["throughput_gain"] = dm["tokens_per_s"] / rl["tokens_per_s"]
        row["decode_throughput_gain"] = dm["decode_tokens_per_s"] / rl["decode_tokens_per_s"]
        out[f"pd_{r:g}"] = row
    ctx.free()
    if rank == 0:
        print(json.dumps({"serve": "llama33b-60L-c256-budget512", "requests": args.serve_requests,
                          "kv_blocks": num_blocks, "kv_tokens": num_blocks * 16, "results": out}), flush=True)
    return 0


def stack_bench(args, torch, native, workloads, synth, world, rank):
    """LLaMA-13B, all 40 layers: one hybrid iteration (chunk C at offset 768 +
    D decodes with contexts uniform in [128, 2048]) against a decode-only
    iteration of the same D decodes, for C in {128, 256, 512} and D from 1 to
    128; per-layer and whole-stack device time.  Layer l's matrices are one
    seeded draw with rows rotated by l; the KV cache holds bf16 1.0 (its values
    do not change the work)."""
    L = 40
    dims = synth.LLAMA_13B.with_layers(L)
    chunks, decodes = [128, 256, 512], [1, 8, 18, 32, 64, 128]
    dmax, cmax, off = max(decodes), max(chunks), 768
    ctxs = [int(c) for c in synth.uniform_ints(11 + rank, (9,), dmax, 128, 2048)]
    lengths = [off + cmax] + [c + 1 for c in ctxs]
    nb = sum(synth.blocks_needed(n) for n in lengths) + 8
    batch = synth.hybrid_batch(11 + rank, (7,), off, cmax, ctxs, nb)
    ctx = native.Context(native.model_config(dims, nb, cmax + dmax, dmax, max(lengths), n_layers=L))
    base = synth.layer_weights(synth.LLAMA_13B, 11 + rank, 0)
    dev = {k: workloads.to_device(v) for k, v in base.items()}
    for l in range(L):
        ctx.load_layer(l, {k: (torch.roll(v, l, 0) if v.dim() == 2 else v) for k, v in dev.items()})
        ctx.sync()
    del dev, base
    ctx.fill_kv(0x3F80)
    x = workloads.to_device(synth.token_rows(11 + rank, (8,), cmax + dmax, dims.hidden))
    y = torch.empty_like(x)
    steps = max(5, min(args.steps, 20))

    def timed(b):
        spec = native.Spec(b)
        for _ in range(3):
            ctx.forward(spec, x, y)
        ctx.sync()
        return max_over_ranks(world, time_steps(torch, ctx, lambda: ctx.forward(spec, x, y), steps, world)) / steps

    out = {"decode_only": {}, "hybrid": {}}
    for D in decodes:
        ms = timed(synth.HybridBatch(None, 0, batch.decodes[:D]))
        out["decode_only"][str(D)] = {"stack_ms": ms, "layer_us": ms / L * 1e3, "decode_tok_s": D / ms * 1e3}
    for C in chunks:
        ms_c = timed(synth.HybridBatch(batch.chunk, C, []))
        row = {"chunk_alone_stack_ms": ms_c}
        for D in decodes:
            ms = timed(synth.HybridBatch(batch.chunk, C, batch.decodes[:D]))
            marg = ms - ms_c
            dec = out["decode_only"][str(D)]["stack_ms"]
            row[str(D)] = {"stack_ms": ms, "layer_us": ms / L * 1e3, "tokens_s": (C + D) / ms * 1e3,
                           "piggybacked_decode_tok_s": D / marg * 1e3 if marg > 0 else None,
                           "per_decode_cost_ratio": dec / marg if marg > 0 else None}
        out["hybrid"][str(C)] = row
    ctx.free()
    if rank == 0:
        print(json.dumps({"stack": "llama13b-40L-hybrid", "chunk_offset": off, "decode_ctx": "U[128,2048]",
                          "steps_timed": steps, "kv_blocks": nb, "results": out}), flush=True)
    return 0


def sources_sha256(names):
    import hashlib
    h = hashlib.sha256()
    for n in names:
        with open(os.path.join(ROOT, "chunked_prefill_hybrid_gb300", "csrc", n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(kind):
    fn = TRAFFIC_PROFILES.get(kind)
    path = os.path.join(ROOT, "profiles", fn) if fn else None
    if not path or not os.path.exists(path):
        return None
    kv = {}
    with open(path) as f:
        for line in f:
            if ":" in line and line.split(":", 1)[0].strip() in ("traffic_bytes_per_launch", "sources",
                                                                   "sources_sha256"):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
    try:
        if sources_sha256(kv["sources"].split()) != kv["sources_sha256"]:
            return None  # the kernel changed since the counters were taken
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, OSError, ValueError):
        return None


def roofline_for(kind, prof, dims, T, D, ctx_len, pk):
    """Algorithmic bytes / flops of one launch of `kind` and its bound."""
    H, F, d = dims.hidden, dims.ffn, dims.head_dim
    nh, nkv = dims.n_heads, dims.n_kv_heads
    qkv = (nh + 2 * nkv) * d
    gemms = {  # (N_out, K, extra bytes written/read besides weights and X)
        "gemm_qkv": (qkv, H, T * qkv * 2),
        "gemm_o": (H, nh * d, T * H * 2 * 2),
        "gemm_gate_up": (2 * F, H, T * F * 2),
        "gemm_down": (H, F, T * H * 2 * 2),
    }
    ms, n = prof[kind]
    per_launch_s = ms / n / 1e3
    if kind in gemms:
        N, K, extra = gemms[kind]
        flops = 2.0 * T * N * K
        byts = N * K * 2 + T * K * 2 + extra
    elif kind == "attention":
        # KV reads of every key attended once per (sequence, kv head), plus q and o
        kv_keys = sum(ctx_len)
        byts = kv_keys * 2 * nkv * d * 2 + 2 * T * nh * d * 2
        flops = 0.0
    else:
        byts, flops = 0.0, 0.0
    t_mem = byts / (pk["hbm_gbs"] * 1e9)
    t_tc = flops / (pk["bf16_tflops"] * 1e12)
    if t_tc > t_mem:
        ach = flops / per_launch_s / 1e12
        return {"kernel": kind, "bound": "tensor", "achieved": ach, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": ach / pk["bf16_tflops"], "traffic": measured_traffic(kind), "algorithmic": flops,
                "per_launch_us": per_launch_s * 1e6, "peak_source": pk["source"] + " (burst)"}
    ach = byts / per_launch_s / 1e9
    return {"kernel": kind, "bound": "hbm", "achieved": ach, "peak": pk["hbm_gbs"], "unit": "GB/s",
            "frac": ach / pk["hbm_gbs"], "traffic": measured_traffic(kind), "algorithmic": byts,
            "per_launch_us": per_launch_s * 1e6, "peak_source": pk["source"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tile-curve", action="store_true",
                    help="time the LLaMA-13B hybrid layer against the chunk size (18 decodes at ctx 1024) and print "
                         "one JSON line with the curve instead of the benchmark line")
    ap.add_argument("--stack", action="store_true",
                    help="time the full LLaMA-13B stack (40 layers): hybrid batches of chunk C in {128, 256, 512} "
                         "+ D decodes against decode-only batches of the same D; one JSON line")
    ap.add_argument("--serve", action="store_true",
                    help="run the LLaMA-33B (60 layers) serving loop, decode-maximal vs the request-level baseline, "
                         "and print one JSON line with throughput, TTFT/ITL/TPOT and iteration uniformity")
    ap.add_argument("--serve-requests", type=int, default=128)
    ap.add_argument("--serve-ratios", default="1,5,10,50", help="P:D ratios r: max_new = max(1, round(P / r))")
    ap.add_argument("--prefill-sweep", action="store_true",
                    help="time prefill-only batches (T = 64..1024), decode-only batches (B = 1, 2, 18 at ctx 1024) "
                         "and the pages' Table 2 batches on one LLaMA-13B layer; one JSON line")
    ap.add_argument("--ncu-case", action="store_true",
                    help="run only the warm-up and --steps hybrid steps, untimed (the case ncu captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    world, rank, local = dist_init(args.gpus)
    import torch
    torch.cuda.set_device(local)
    import __graft_entry__
    __graft_entry__.build_library()
    from chunked_prefill_hybrid_gb300 import native, workloads, synth

    if args.tile_curve:
        return tile_curve(args, torch, native, workloads, synth, world, rank)
    if args.serve:
        return serve_bench(args, torch, native, workloads, synth, world, rank)
    if args.stack:
        return stack_bench(args, torch, native, workloads, synth, world, rank)
    if args.prefill_sweep:
        return prefill_sweep(args, torch, native, workloads, synth, world, rank)

    w = workloads.llama13b_hybrid(seed=2 + rank)
    dims = w.dims
    ctx = native.Context(workloads.config(w))
    x = workloads.upload(w, ctx, poison=None)
    y = torch.empty_like(x)
    spec = native.Spec(w.batch)
    T, D, C = w.T, w.batch.n_decodes, w.batch.chunk_len

    # comparison batches over the same pool and weights
    dec_only = native.Spec(synth.HybridBatch(None, 0, w.batch.decodes))
    x_dec = x[C:].contiguous()
    y_dec = torch.empty_like(x_dec)
    chunk_alone = native.Spec(synth.HybridBatch(w.batch.chunk, C, []))
    x_chk = x[:C].contiguous()
    y_chk = torch.empty_like(x_chk)

    def step():
        ctx.forward(spec, x, y)

    for _ in range(args.warmup):
        step()
    ctx.sync()
    if args.ncu_case:
        for _ in range(args.steps):
            step()
        ctx.sync()
        ctx.free()
        print(f"ncu case: {args.warmup} + {args.steps} steps of {WORKLOAD}", flush=True)
        return 0

    # 1) the headline: hybrid batch, inputs resident
    n0 = ctx.launch_count
    with Clocks(local) as clk:
        ms = time_steps(torch, ctx, step, args.steps, world)
    launches = (ctx.launch_count - n0) // args.steps
    ctx.sync()
    clocks = clk.summary()
    ms = max_over_ranks(world, ms)
    ms_step = ms / args.steps
    value = world * T * args.steps / (ms / 1e3)

    # 2) per-kernel timing of the same step (CUDA events around every launch)
    ctx.profile(True)
    time_steps(torch, ctx, step, args.steps, world)
    ctx.sync()
    prof = ctx.profile_read()
    ctx.profile(False)
    total = sum(v[0] for v in prof.values())
    kernels = {k: {"ms_per_launch": v[0] / v[1], "launches_per_step": v[1] / args.steps,
                   "share": v[0] / total if total else None} for k, v in prof.items()}
    pk = peaks()
    dominant = max(prof, key=lambda k: prof[k][0])
    ctx_lens = [w.batch.chunk.cached + C] + [s.cached + 1 for s in w.batch.decodes]
    roof = roofline_for(dominant, prof, dims, T, D, ctx_lens, pk)
    roof_all = {k: roofline_for(k, prof, dims, T, D, ctx_lens, pk) for k in prof if k.startswith(("gemm", "attention"))}

    # 3) decode tokens/s: piggybacked (marginal over the chunk alone) vs decode-only
    for _ in range(3):
        ctx.forward(chunk_alone, x_chk, y_chk)
        ctx.forward(dec_only, x_dec, y_dec)
    ctx.sync()
    ms_chunk = time_steps(torch, ctx, lambda: ctx.forward(chunk_alone, x_chk, y_chk), args.steps, world) / args.steps
    ms_dec = time_steps(torch, ctx, lambda: ctx.forward(dec_only, x_dec, y_dec), args.steps, world) / args.steps
    marginal_ms = ms_step - ms_chunk
    decode = {"piggybacked_tok_s": D / (marginal_ms / 1e3) if marginal_ms > 0 else None,
              "decode_only_tok_s": D / (ms_dec / 1e3),
              "per_decode_cost_ratio": (ms_dec / D) / (marginal_ms / D) if marginal_ms > 0 else None,
              "ms_hybrid": ms_step, "ms_chunk_alone": ms_chunk, "ms_decode_only": ms_dec}

    # 4) end to end through the public host-buffer calls: every step copies its
    # input rows from pinned host memory and writes its output rows to pinned
    # host memory.  The headline uses the asynchronous call (the host plans
    # step i+1 while the GPU runs step i; one hb_sync after the last step);
    # the waiting call is reported beside it.
    xh = torch.empty((T, dims.hidden), dtype=torch.int16, pin_memory=True)
    xh.copy_(x.cpu())
    yh = torch.empty_like(xh).pin_memory()

    def host_steps(call):
        for _ in range(3):
            call(spec, xh.data_ptr(), yh.data_ptr())
        ctx.sync()
        barrier(world)
        t0 = time.perf_counter()
        for _ in range(args.steps):
            call(spec, xh.data_ptr(), yh.data_ptr())
        ctx.sync()
        return max_over_ranks(world, time.perf_counter() - t0)

    e2e_s = host_steps(ctx.forward_host_async_ptr)
    sync_s = host_steps(ctx.forward_host_ptr)
    e2e = {"value": world * T * args.steps / e2e_s, "unit": "tokens/s",
           "h2d_bytes_per_step": T * dims.hidden * 2, "d2h_bytes_per_step": T * dims.hidden * 2,
           "call": "hb_forward_host_async per step, one hb_sync after the timed steps",
           "waiting_call_value": world * T * args.steps / sync_s}

    # 5) the per-decode cost on GEMM time alone (an extra figure: the line stays valid without it)
    try:
        prof_chunk = profiled(torch, ctx, lambda: ctx.forward(chunk_alone, x_chk, y_chk), args.steps, world)
        prof_dec = profiled(torch, ctx, lambda: ctx.forward(dec_only, x_dec, y_dec), args.steps, world)
        decode["gemm_time"] = gemm_decode_cost(prof, prof_chunk, prof_dec, args.steps, D)
    except Exception as e:  # noqa: BLE001
        decode["gemm_time"] = {"error": str(e)[:200]}

    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "layers": 1, "T": T, "chunk": C, "chunk_offset": w.batch.chunk.cached,
                       "decodes": D, "decode_ctx": 1024, "parallelism": f"replicas{world}",
                       "l2": "inputs larger than L2 (634 MB weights + 399 MB KV read per step)"},
            "e2e": e2e, "gpu_launches": int(launches * args.steps), "launches_per_step": int(launches),
            "clocks": clocks, "decode": decode, "roofline": roof, "kernels": kernels, "rooflines": roof_all}

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rps, n, dt, threads = oracle_sample(w, target_s=10.0)
        line["cpu_baseline"] = {"value": rps, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"{n} of {w.T} rows (first chunk rows + first decodes), one layer, "
                                          f"fp64 mirror mode, {dt:.1f} s"}
        r1, n1, dt1 = oracle_one_core(w, target_s=3.0)
        line["cpu_baseline"]["one_core"] = {"value": r1, "unit": "tokens/s", "cores": 1,
                                            "sample": f"{n1} rows, {dt1:.1f} s"}
    ctx.free()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
